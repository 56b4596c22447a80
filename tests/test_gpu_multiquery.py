"""GPU parity: pkv_multiquery_attn (speculative verification, prefill chunks)
against the float64 causal oracle. Tolerance as for decode:
|gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise for fp16 / bf16 caches,
|gpu - oracle| <= 2e-2 for INT8 caches (the oracle on the dequantised cache)."""

import numpy as np
import pytest

import oracle
from _pkv_helpers import GpuCase, OracleCase, assert_attention_close, out_to_f64, to_dev
from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload, variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


def _sync():
    import torch
    torch.cuda.synchronize()


def run_mq(g, q, cu_q, max_q, num_parts=0):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    cfg = g.cfg
    qd = q if isinstance(q, torch.Tensor) else to_dev(q)
    cu = cu_q if isinstance(cu_q, torch.Tensor) else to_dev(np.asarray(cu_q, np.int32))
    out = torch.full(qd.shape, float("nan"), dtype=qd.dtype, device="cuda")
    ws = torch.empty(B.pkv_multiquery_workspace_size(cfg.batch, cfg.num_q_heads, max_q, g.k_cache,
                                                     num_parts), dtype=torch.uint8, device="cuda")
    B.pkv_multiquery_attn(qd, cu, max_q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                          cfg.softmax_scale, out, ws, num_parts, g.status, k_scales=g.k_scales,
                          v_scales=g.v_scales)
    return out


def want_mq(w, o, seqs=None):
    return oracle.paged_multiquery_attention(w.q, w.cu_q, o.k, o.v, w.block_tables,
                                             w.context_lens, w.cfg.softmax_scale, o.ks, o.vs,
                                             seqs=seqs)


SMALL = {
    "spec_verify": variant(CONFIGS["spec_verify"], batch=12, len_groups=((12, 5, 900),)),
    "prefill_chunk": variant(CONFIGS["prefill_chunk"], batch=3, q_len=40, max_len=700,
                             len_groups=((3, 40, 700),)),
    "mha_q3_d64": variant(CONFIGS["mha7b"], batch=5, num_q_heads=4, num_kv_heads=4, head_dim=64,
                          q_len=3, max_len=400, len_groups=((5, 3, 400),)),
    "g2_q9_f16": variant(CONFIGS["gqa8b"], batch=6, num_q_heads=8, num_kv_heads=4,
                         kv_dtype="f16", q_dtype="f16", src_dtype="f16", q_len=9,
                         len_groups=((6, 9, 500),)),
    "g4_q1": variant(CONFIGS["gqa8b"], batch=9, len_groups=((9, 1, 700),)),
    # 7 x 4 = 28, 9 x 4 = 36 and 4 x 8 = 32 rows: the 16-rows-per-warp kernel
    # (24 rows or fewer take the short-run kernel, rows on the MMA's N side)
    "g4_q7": variant(CONFIGS["spec_verify"], batch=7, q_len=7, len_groups=((7, 7, 600),)),
    "g4_q9": variant(CONFIGS["spec_verify"], batch=7, q_len=9, len_groups=((7, 9, 600),)),
    "g8_q4_f16": variant(CONFIGS["gqa70b"], batch=5, q_len=4, kv_dtype="f16", q_dtype="f16",
                         src_dtype="f16", len_groups=((5, 4, 700),)),
    "g2_q8_d64": variant(CONFIGS["gqa8b"], batch=6, num_q_heads=4, num_kv_heads=2, head_dim=64,
                         q_len=8, len_groups=((6, 8, 500),)),
    "g8_q3_f16": variant(CONFIGS["gqa70b"], batch=5, q_len=3, kv_dtype="f16", q_dtype="f16",
                         src_dtype="f16", len_groups=((5, 3, 700),)),
    # group 8 (64 q / 8 kv heads)
    "g8_q5": variant(CONFIGS["gqa70b"], batch=8, q_len=5, len_groups=((8, 5, 800),)),
    # INT8 caches (the mma.sync kernel with codes entering as fp16 carriers)
    "int8_q5": variant(CONFIGS["spec_verify_int8"], batch=12, len_groups=((12, 5, 900),)),
    "int8_q9_d64_f16": variant(CONFIGS["spec_verify_int8"], batch=6, num_q_heads=8,
                               num_kv_heads=4, head_dim=64, q_dtype="f16", src_dtype="f16",
                               q_len=9, len_groups=((6, 9, 500),)),
    "int8_g8_q3": variant(CONFIGS["spec_verify_int8"], batch=6, num_q_heads=64, q_len=3,
                          len_groups=((6, 3, 600),)),
    "int8_g1_q2": variant(CONFIGS["spec_verify_int8"], batch=5, num_q_heads=4, num_kv_heads=4,
                          q_len=2, len_groups=((5, 2, 400),)),
    # 7 queries x group 4 = 28 rows over an INT8 cache at head_dim 128: the
    # 32-row kernel (24 rows or fewer take the short-run INT8 kernel)
    "int8_q7": variant(CONFIGS["spec_verify_int8"], batch=7, q_len=7, len_groups=((7, 7, 600),)),
    "int8_q3_f16": variant(CONFIGS["spec_verify_int8"], batch=6, q_dtype="f16", src_dtype="f16",
                           q_len=3, len_groups=((6, 3, 500),)),
}
_cache = {}


def case(name):
    if name not in _cache:
        w = make_workload(SMALL[name])
        g, o = GpuCase(w), OracleCase(w)
        _cache[name] = (w, g, o, want_mq(w, o))
    return _cache[name]


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("parts", [0, 1, 3, 17])
def test_multiquery_small(name, parts):
    w, g, o, want = case(name)
    out = run_mq(g, w.q, w.cu_q, w.cfg.q_len, parts)
    _sync()
    assert_attention_close(out_to_f64(out), want, w.cfg.kv_dtype == "i8", f"{name} parts={parts}")
    assert int(g.status.item()) == 0


def test_one_query_per_sequence_matches_decode_kernel():
    import torch
    w, g, o, want = case("g4_q1")
    out = run_mq(g, w.q, w.cu_q, 1)
    ref, _ = g.decode()
    _sync()
    a, b = out_to_f64(out), out_to_f64(ref)
    assert_attention_close(a, want, False, "q_len 1")
    assert np.abs(a - b).max() < 2e-2


def test_variable_query_counts_including_empty():
    w, g, o, _ = case("prefill_chunk")
    rng = np.random.default_rng(5)
    qmax = w.cfg.q_len
    ns = np.array([0, 17, qmax], np.int32)[: w.cfg.batch]
    rng.shuffle(ns)
    rows = [w.q[b * qmax: b * qmax + int(ns[b])] for b in range(w.cfg.batch)]
    qv = np.concatenate(rows)
    cu = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    want = oracle.paged_multiquery_attention(qv, cu, o.k, o.v, w.block_tables, w.context_lens,
                                             w.cfg.softmax_scale)
    for parts in (0, 2, 9):
        out = run_mq(g, qv, cu, qmax, parts)
        _sync()
        assert_attention_close(out_to_f64(out), want, False, f"varlen parts={parts}")


@pytest.mark.parametrize("name", ["spec_verify", "int8_q5"])
@pytest.mark.parametrize("parts", [0, 3, 40])
def test_short_runs_with_variable_query_counts(name, parts):
    """Speculative verification with 0..5 queries per sequence (the short-run
    kernels, bf16 and INT8): every row against the causal oracle."""
    w, g, o, _ = case(name)
    rng = np.random.default_rng(11)
    qmax = w.cfg.q_len
    ns = rng.integers(0, qmax + 1, size=w.cfg.batch).astype(np.int32)
    ns[:3] = (0, 1, qmax)
    rows = [w.q[b * qmax: b * qmax + int(ns[b])] for b in range(w.cfg.batch)]
    qv = np.concatenate(rows)
    cu = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    want = oracle.paged_multiquery_attention(qv, cu, o.k, o.v, w.block_tables, w.context_lens,
                                             w.cfg.softmax_scale, o.ks, o.vs)
    out = run_mq(g, qv, cu, qmax, parts)
    _sync()
    assert int(g.status.item()) == 0
    assert_attention_close(out_to_f64(out), want, w.cfg.kv_dtype == "i8",
                           f"short varlen {name} parts={parts}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "i8"])
@pytest.mark.parametrize("n", [48, 33])
def test_first_prefill_chunk_from_position_zero(dtype, n):
    """The whole context is new (L == n): query i sees only tokens 0..i, so
    the first rows average two or three values and expose any rounding of
    the probabilities (INT8: a bf16 q over an INT8 cache)."""
    qd = "bf16" if dtype == "i8" else dtype
    cfg = variant(CONFIGS["prefill_chunk"], batch=4, q_len=n, max_len=64,
                  len_groups=((4, n, n),), kv_dtype=dtype, q_dtype=qd, src_dtype=qd)
    w = make_workload(cfg)
    assert (w.context_lens == n).all()
    g, o = GpuCase(w), OracleCase(w)
    want = want_mq(w, o)
    for parts in (0, 5):
        out = run_mq(g, w.q, w.cu_q, n, parts)
        _sync()
        assert_attention_close(out_to_f64(out), want, dtype == "i8",
                               f"{dtype} from 0 parts={parts}")


# Query runs that fill 128-row tiles (q_len * g >= 128) take the tcgen05 kernel.
TC = {
    "g4_d128_bf16": variant(CONFIGS["prefill_chunk"], batch=3, q_len=64, max_len=2000,
                            len_groups=((3, 64, 2000),)),
    "g2_d64_f16": variant(CONFIGS["prefill_chunk"], batch=3, num_q_heads=8, num_kv_heads=4,
                          head_dim=64, kv_dtype="f16", q_dtype="f16", src_dtype="f16", q_len=100,
                          max_len=1200, len_groups=((3, 100, 1200),)),
    "g1_d128_two_tiles": variant(CONFIGS["prefill_chunk"], batch=2, num_q_heads=4, num_kv_heads=4,
                                 q_len=150, max_len=700, len_groups=((2, 150, 700),)),
    # scores spread over a wide range: running maxima jump by more than 2^8
    "g4_wide_scores": variant(CONFIGS["prefill_chunk"], batch=2, q_len=40, max_len=1500,
                              len_groups=((2, 40, 1500),), q_std=6.0),
    "g8_d128_bf16": variant(CONFIGS["prefill_chunk"], batch=2, num_q_heads=64, q_len=40,
                            max_len=900, len_groups=((2, 40, 900),)),
}


@pytest.mark.parametrize("name", list(TC))
def test_tensor_core_row_tiles(name):
    cfg = TC[name]
    assert cfg.q_len * (cfg.num_q_heads // cfg.num_kv_heads) >= 128
    w = make_workload(cfg)
    g, o = GpuCase(w), OracleCase(w)
    want = oracle.paged_multiquery_attention(w.q, w.cu_q, o.k, o.v, w.block_tables,
                                             w.context_lens, w.cfg.softmax_scale)
    out = run_mq(g, w.q, w.cu_q, w.cfg.q_len)
    _sync()
    got = out_to_f64(out)
    assert np.isfinite(got).all()
    assert_attention_close(got, want, False, name)
    assert int(g.status.item()) == 0


def test_long_query_runs_over_an_int8_cache():
    """Query runs that would fill 128-row tiles: over an INT8 cache the
    mma.sync kernel serves them (the tcgen05 kernel takes 16-bit operands)."""
    cfg = variant(CONFIGS["spec_verify_int8"], batch=3, q_len=64, max_len=1500,
                  len_groups=((3, 64, 1500),))
    w = make_workload(cfg)
    g, o = GpuCase(w), OracleCase(w)
    want = want_mq(w, o)
    for parts in (0, 7):
        out = run_mq(g, w.q, w.cu_q, cfg.q_len, parts)
        _sync()
        assert_attention_close(out_to_f64(out), want, True, f"int8 q_len 64 parts={parts}")
    assert int(g.status.item()) == 0


@pytest.mark.parametrize("name", ["spec_verify", "prefill_chunk"])   # mma.sync / tcgen05 kernel
def test_bad_block_entry_and_length_are_flagged(name):
    """An out-of-pool table entry and a length beyond the table are flagged on
    the status word; the over-long sequence's rows are not written and the
    other sequences stay exact."""
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w, g, o, want = case(name)
    bt = g.block_tables.clone()
    bt[0, 1] = w.num_blocks + 7                       # outside the pool
    lens = g.context_lens.clone()
    lens[1] = bt.shape[1] * 16 + 64                   # longer than the table
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd = to_dev(w.q)
    out = torch.full(qd.shape, float("nan"), dtype=qd.dtype, device="cuda")
    cu = to_dev(np.asarray(w.cu_q, np.int32))
    nbytes = B.pkv_multiquery_workspace_size(w.cfg.batch, w.cfg.num_q_heads, w.cfg.q_len,
                                             g.k_cache, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    B.pkv_multiquery_attn(qd, cu, w.cfg.q_len, g.k_cache, g.v_cache, bt, lens,
                          w.cfg.softmax_scale, out, ws, 0, status)
    _sync()
    st = int(status.item())
    assert st & B.DEV_BAD_BLOCK and st & B.DEV_BAD_LENGTH
    got = out_to_f64(out)
    rows = lambda b: np.arange(w.cu_q[b], w.cu_q[b + 1])   # noqa: E731
    assert np.isnan(got[rows(1)]).all()               # not written
    keep = np.concatenate([rows(b) for b in range(2, w.cfg.batch)])
    assert_attention_close(got[keep], want[keep], False, f"{name} other sequences")


def test_too_many_queries_are_flagged_not_written():
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w, g, o, _ = case("spec_verify")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g_status, g.status = g.status, status
    try:
        out = run_mq(g, w.q, w.cu_q, w.cfg.q_len - 1)   # max_q_len below the real n_b
        _sync()
    finally:
        g.status = g_status
    assert int(status.item()) & B.DEV_BAD_LENGTH
    assert torch.isnan(out.float()).all()            # nothing written


@pytest.mark.slow
@pytest.mark.parametrize("name", ["spec_verify", "prefill_chunk", "spec_verify_int8"])
def test_multiquery_full_size_sampled(name):
    w = make_workload(CONFIGS[name])
    g, o = GpuCase(w), OracleCase(w)
    lens = w.context_lens
    order = np.argsort(lens)
    seqs = sorted(set(order[:2].tolist() + order[-2:].tolist() +
                      np.linspace(0, w.cfg.batch - 1, min(8, w.cfg.batch)).astype(int).tolist()))
    want = want_mq(w, o, seqs=seqs)
    out = run_mq(g, w.q, w.cu_q, w.cfg.q_len)
    _sync()
    got = out_to_f64(out)
    rows = np.concatenate([np.arange(w.cu_q[b], w.cu_q[b + 1]) for b in seqs])
    assert_attention_close(got[rows], want, w.cfg.kv_dtype == "i8", name)
    assert np.isfinite(got).all()
    assert int(g.status.item()) == 0

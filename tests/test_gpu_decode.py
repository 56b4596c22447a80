"""GPU parity: pkv_decode_attn / split / combine against the float64 oracle.

Tolerance (bf16/fp16 KV): |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise;
INT8 KV: |gpu - oracle(dequantised cache)| <= 2e-2.
"""

import numpy as np
import pytest

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


SMALL = {
    "tiny": CONFIGS["tiny"],
    "mha7b": variant(CONFIGS["mha7b"], batch=6, len_groups=((6, 1, 700),)),
    "gqa8b": variant(CONFIGS["gqa8b"], batch=24, len_groups=((24, 1, 1500),)),
    "gqa8b_int8": variant(CONFIGS["gqa8b_int8"], batch=16, len_groups=((16, 1, 900),)),
    "skewed": variant(CONFIGS["skewed"], batch=12, max_len=9000,
                      len_groups=((3, 3000, 9000), (9, 16, 256))),
    # remaining built variants: head_dim 64 with bf16 and INT8, group 2
    "bf16_d64_g2": variant(CONFIGS["gqa8b"], batch=10, num_q_heads=8, num_kv_heads=4,
                           head_dim=64, len_groups=((10, 1, 600),)),
    "i8_d64_g1_f16": variant(CONFIGS["gqa8b_int8"], batch=7, num_q_heads=4, num_kv_heads=4,
                             head_dim=64, q_dtype="f16", src_dtype="f16",
                             len_groups=((7, 1, 400),)),
    "i8_d128_g2": variant(CONFIGS["gqa8b_int8"], batch=7, num_q_heads=8, num_kv_heads=4,
                          len_groups=((7, 1, 400),)),
    "f16_d128_g4": variant(CONFIGS["gqa8b"], batch=9, kv_dtype="f16", q_dtype="f16",
                           src_dtype="f16", len_groups=((9, 1, 500),)),
    # group 8: eight query heads per KV head (64 q / 8 kv heads, the 70B-class shape)
    "bf16_d128_g8": variant(CONFIGS["gqa8b"], batch=8, num_q_heads=64, num_kv_heads=8,
                            len_groups=((8, 1, 900),)),
    "i8_d128_g8": variant(CONFIGS["gqa8b_int8"], batch=6, num_q_heads=64, num_kv_heads=8,
                          len_groups=((6, 1, 600),)),
    "f16_d64_g8": variant(CONFIGS["gqa8b"], batch=7, num_q_heads=16, num_kv_heads=2,
                          head_dim=64, kv_dtype="f16", q_dtype="f16", src_dtype="f16",
                          len_groups=((7, 1, 500),)),
}

_cache = {}


def case(name):
    if name not in _cache:
        w = make_workload(SMALL[name])
        _cache[name] = (w, GpuCase(w), OracleCase(w).attention())
    return _cache[name]


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("parts", [0, 1, 3, 37])
def test_decode_small(name, parts):
    w, g, want = case(name)
    out, _ = g.decode(num_parts=parts)
    _sync()
    assert_attention_close(out_to_f64(out), want, w.cfg.kv_dtype == "i8", f"{name} parts={parts}")
    assert int(g.status.item()) == 0


@pytest.mark.parametrize("name", ["gqa8b", "skewed", "gqa8b_int8"])
def test_partition_invariance(name):
    """Any number of workers gives the same result within rounding."""
    w, g, want = case(name)
    outs = []
    for parts in (2, 5, 64, 400, 5000):
        out, _ = g.decode(num_parts=parts)
        _sync()
        got = out_to_f64(out)
        assert_attention_close(got, want, w.cfg.kv_dtype == "i8", f"{name} parts={parts}")
        outs.append(got)
    spread = max(float(np.abs(a - outs[0]).max()) for a in outs)
    assert spread < 2e-2


def test_split_then_combine_equals_attn():
    import torch
    w, g, want = case("skewed")
    a, _ = g.decode(num_parts=29)
    out = torch.full_like(a, float("nan"))
    _, ws = g.decode(num_parts=29, split_only=True, out=out)
    from paged_kv_decode_05_gb300 import binding as B
    B.pkv_decode_combine(out, g.k_cache, ws, num_parts=29)
    _sync()
    assert torch.equal(out.view(torch.int16), a.view(torch.int16))


def test_empty_and_single_token_sequences():
    cfg = variant(CONFIGS["gqa8b"], batch=9, len_groups=((9, 0, 3),))
    w = make_workload(cfg)
    assert (w.context_lens == 0).any() and (w.context_lens == 1).any()
    g = GpuCase(w)
    want = OracleCase(w).attention()
    for parts in (0, 1, 4):
        out, _ = g.decode(num_parts=parts)
        _sync()
        got = out_to_f64(out)
        assert np.all(got[w.context_lens == 0] == 0)
        assert_attention_close(got, want, False, f"tiny lengths parts={parts}")


@pytest.mark.parametrize("parts", [0, 37])
def test_large_batch_short_sequences(parts):
    """Batch 8192 (the largest supported) of 0..40-token sequences.

    At this batch each combine CTA looks after a run of segments, some empty
    and some split over two workers; every 7th sequence is checked.
    """
    cfg = variant(CONFIGS["gqa8b"], batch=8192, len_groups=((1024, 0, 0), (7168, 1, 40)),
                  max_len=64)
    w = make_workload(cfg)
    assert (w.context_lens == 0).sum() >= 1024
    g = GpuCase(w)
    seqs = list(range(0, 8192, 7)) + [8191]
    want = OracleCase(w).attention(seqs=seqs)
    out, _ = g.decode(num_parts=parts)
    _sync()
    got = out_to_f64(out)
    assert np.all(got[w.context_lens == 0] == 0)
    assert_attention_close(got[seqs], want, False, f"batch 8192 parts={parts}")


@pytest.mark.parametrize("base,parts", [("gqa8b", 0), ("gqa8b", 501), ("gqa8b_int8", 0),
                                        ("gqa8b_int8", 77)])
def test_batch_above_the_exact_prefix(base, parts):
    """1001 sequences: the split kernel keeps every 4th block-prefix entry in
    shared memory (251 chunks, the last holding one sequence) and walks the
    rest; runs of empty sequences cover whole chunks. Every sequence is
    checked."""
    cfg = variant(CONFIGS[base], batch=1001, max_len=320,
                  len_groups=((300, 1, 200), (20, 0, 0), (400, 1, 300), (281, 0, 50)))
    w = make_workload(cfg)
    g = GpuCase(w)
    want = OracleCase(w).attention()
    out, _ = g.decode(num_parts=parts)
    _sync()
    got = out_to_f64(out)
    assert int(g.status.item()) == 0
    assert np.all(got[w.context_lens == 0] == 0)
    assert_attention_close(got, want, cfg.kv_dtype == "i8", f"batch 1001 {base} parts={parts}")


def test_stale_nan_rows_are_never_read():
    """Rows past each context hold NaN; the output must stay finite and right."""
    w, g, want = case("gqa8b")
    out, _ = g.decode()
    _sync()
    assert np.isfinite(out_to_f64(out)).all()


def test_bad_block_entry_and_length_are_flagged_not_read():
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w, g, _ = case("gqa8b")
    bt = g.block_tables.clone()
    bt[3, 0] = w.num_blocks + 5          # outside the pool
    lens = g.context_lens.clone()
    lens[5] = bt.shape[1] * 16 + 100     # longer than the table
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(g.q)
    ws = torch.empty(B.pkv_decode_workspace_size(w.cfg.batch, w.cfg.num_q_heads, g.k_cache, 0),
                     dtype=torch.uint8, device="cuda")
    B.pkv_decode_attn(g.q, g.k_cache, g.v_cache, bt, lens, w.cfg.softmax_scale, out, ws,
                      num_parts=0, dev_status=status)
    _sync()
    st = int(status.item())
    assert st & B.DEV_BAD_BLOCK and st & B.DEV_BAD_LENGTH


# ------------------------------------------------------------- full sizes ---
FULL_SAMPLES = 24


def _full(name):
    key = "full:" + name
    if key not in _cache:
        w = make_workload(CONFIGS[name])
        g = GpuCase(w)
        lens = w.context_lens
        order = np.argsort(lens)
        seqs = sorted(set(order[:4].tolist() + order[-6:].tolist() +
                          np.linspace(0, w.cfg.batch - 1, FULL_SAMPLES - 10).astype(int).tolist()))
        want = OracleCase(w).attention(seqs=seqs)
        _cache[key] = (w, g, seqs, want)
    return _cache[key]


@pytest.mark.parametrize("spread", [False, True])
def test_int8_large_value_scales(spread):
    """INT8 V scales far above the fp16 range of the probabilities' carrier:
    2^24 everywhere (the output scales exactly), or 2^20 .. 2^24 varying by
    block, so that a piece meets ever larger scales midway."""
    import torch
    cfg = variant(CONFIGS["gqa8b_int8"], batch=6, len_groups=((6, 100, 700),))
    w = make_workload(cfg)
    g, o = GpuCase(w), OracleCase(w)
    blk = np.arange(w.num_blocks)
    f = 2.0 ** (20 + (blk * 7) % 5) if spread else np.full(w.num_blocks, 2.0 ** 24)
    o.vs = (o.vs.astype(np.float64) * f[:, None]).astype(np.float32)
    g.v_scales.copy_(torch.from_numpy(o.vs).cuda())
    want = o.attention()
    for parts in (0, 7):
        out, _ = g.decode(num_parts=parts)
        _sync()
        got = out_to_f64(out)
        assert np.isfinite(got).all()
        err = np.abs(got - want)
        assert (err <= 2e-2 * 2.0 ** 20 + 1e-2 * np.abs(want)).all(), (spread, parts, err.max())
    assert int(g.status.item()) == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["tiny", "mha7b", "gqa8b", "gqa8b_int8", "skewed"])
def test_decode_full_size_sampled(name):
    """The benchmark's launch configuration (default workers) at full size."""
    w, g, seqs, want = _full(name)
    out, _ = g.decode(num_parts=0)
    _sync()
    got = out_to_f64(out)
    assert_attention_close(got[seqs], want, w.cfg.kv_dtype == "i8", name)
    assert int(g.status.item()) == 0
    assert np.isfinite(got).all()
    # every row is a convex combination of V rows: bounded by the V range
    if w.cfg.kv_dtype != "i8":
        assert np.abs(got).max() <= 8.0 * max(w.cfg.kv_std, 1.0)
    _cache.pop("full:" + name)

"""The bounded-wait timeout path, exercised without any GPU fault.

Every wait of the paged kernels on an in-kernel copy is bounded: when it runs
out, the kernel sets PKV_DEV_TIMEOUT, stops the waiting work, waits (again
bounded) for the copies it did issue and returns, so the CUDA context stays
usable. The test hooks of include/pkv_testing.h arm the first stage of one
worker (or CTA) for 16 bytes more than its copies deliver, with a short
limit: the wait runs out for certain, no memory is touched out of bounds and
nothing hangs. Each test
then checks that the call returned within the limit's order of magnitude,
that the status says so, and that a normal call on the same context still
matches the oracle.
"""

import time

import numpy as np
import pytest

import oracle
from _pkv_helpers import GpuCase, OracleCase, assert_attention_close, out_to_f64, to_dev
from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload, variant

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000      # 20 ms per bounded wait


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


def _decode_case(kv):
    base = CONFIGS["gqa8b_int8"] if kv == "i8" else CONFIGS["gqa8b"]
    cfg = variant(base, batch=6, len_groups=((6, 100, 700),))
    w = make_workload(cfg)
    return w, GpuCase(w), OracleCase(w)


@pytest.mark.parametrize("kv", ["bf16", "i8"])
def test_decode_wait_that_runs_out(kv):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w, g, o = _decode_case(kv)
    cfg = w.cfg
    parts = 7
    ws = torch.empty(B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, g.k_cache, parts),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(g.q)
    # no stall, short limit: the same result as the public entry point, bitwise
    B.pkv_testing_decode_attn_stall(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                    cfg.softmax_scale, out, ws, LIMIT_NS, -1, g.k_scales,
                                    g.v_scales, parts, status)
    ref, _ = g.decode(num_parts=parts)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # worker 3's first unit stalls: its wait runs out, the call comes back, the
    # status says so
    t0 = time.time()
    B.pkv_testing_decode_attn_stall(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                    cfg.softmax_scale, out, ws, LIMIT_NS, 3, g.k_scales,
                                    g.v_scales, parts, status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) & B.DEV_TIMEOUT
    assert elapsed < 3.0, elapsed       # 20 ms limit + a bounded drain, far below the 4 s default
    # the context is still usable: a normal call matches the oracle
    got, _ = g.decode(num_parts=parts)
    torch.cuda.synchronize()
    assert int(g.status.item()) == 0
    assert_attention_close(out_to_f64(got), o.attention(), kv == "i8", f"after a stall ({kv})")


def test_decode_stall_hook_rejects_bad_arguments():
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w, g, _ = _decode_case("bf16")
    cfg = w.cfg
    ws = torch.empty(B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, g.k_cache, 4),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(g.q)
    for limit, unit in ((5_000_000_000, -1), (LIMIT_NS, -2)):
        with pytest.raises(B.PkvError) as e:
            B.pkv_testing_decode_attn_stall(g.q, g.k_cache, g.v_cache, g.block_tables,
                                            g.context_lens, cfg.softmax_scale, out, ws, limit,
                                            unit, num_parts=4)
        assert e.value.code == 1


MQ = {
    # 5 queries x group 4 = 20 rows: the short-run split kernels (bf16, INT8)
    "spec_verify": variant(CONFIGS["spec_verify"], batch=6, len_groups=((6, 5, 600),)),
    "spec_verify_int8": variant(CONFIGS["spec_verify_int8"], batch=6, len_groups=((6, 5, 600),)),
    # 7 x 4 = 28 and 10 x 4 = 40 rows: the 16-rows-per-warp split kernel (two
    # and four consumer warps)
    "rows28": variant(CONFIGS["spec_verify"], batch=6, q_len=7, len_groups=((6, 7, 600),)),
    "rows40": variant(CONFIGS["spec_verify"], batch=6, q_len=10, len_groups=((6, 10, 600),)),
    # 64 queries x group 4 = 256 rows: the tcgen05 kernel
    "prefill_chunk": variant(CONFIGS["prefill_chunk"], batch=2, q_len=64, max_len=500,
                             len_groups=((2, 64, 500),)),
}


@pytest.mark.parametrize("name", list(MQ))
def test_multiquery_wait_that_runs_out(name):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w = make_workload(MQ[name])
    g, o = GpuCase(w), OracleCase(w)
    cfg = w.cfg
    nq = cfg.q_len
    q, cu = to_dev(w.q), to_dev(w.cu_q)
    ws = torch.empty(B.pkv_multiquery_workspace_size(cfg.batch, cfg.num_q_heads, nq, g.k_cache, 5),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    B.pkv_testing_multiquery_attn_stall(q, cu, nq, g.k_cache, g.v_cache, g.block_tables,
                                        g.context_lens, cfg.softmax_scale, out, ws, LIMIT_NS, 0,
                                        5, status, k_scales=g.k_scales, v_scales=g.v_scales)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    st = int(status.item())
    assert st & B.DEV_TIMEOUT and st & 0x1f00, hex(st)
    assert elapsed < 3.0, elapsed
    # a normal call on the same context matches the oracle
    B.pkv_multiquery_attn(q, cu, nq, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                          cfg.softmax_scale, out, ws, 5, g.status, k_scales=g.k_scales,
                          v_scales=g.v_scales)
    torch.cuda.synchronize()
    assert int(g.status.item()) == 0
    want = oracle.paged_multiquery_attention(w.q, w.cu_q, o.k, o.v, w.block_tables,
                                             w.context_lens, cfg.softmax_scale, o.ks, o.vs)
    assert_attention_close(out_to_f64(out), want, cfg.kv_dtype == "i8", f"{name} after a stall")

"""GPU parity: pkv_copy_blocks (copy-on-write fork / rollback) against the oracle."""

import numpy as np
import pytest

import oracle
from _pkv_helpers import (GpuCase, OracleCase, assert_attention_close, out_to_f64, to_dev,
                          to_host_bits)
from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload, variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


def _pairs(w, n, rng):
    used = np.unique(w.block_tables[w.block_tables >= 0])
    free = np.setdiff1d(np.arange(w.num_blocks), used)
    n = min(n, free.size)
    return (rng.choice(used, n, replace=False).astype(np.int32),
            rng.choice(free, n, replace=False).astype(np.int32))


@pytest.mark.parametrize("name", ["gqa8b", "gqa8b_int8", "tiny"])
def test_copy_blocks_bit_exact(name):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    cfg = CONFIGS[name] if name == "tiny" else variant(CONFIGS[name], batch=12,
                                                           len_groups=((12, 1, 700),))
    w = make_workload(cfg)
    g, o = GpuCase(w, stale="zero"), OracleCase(w)   # both pools start at zero
    rng = np.random.default_rng(3)
    src, dst = _pairs(w, 20, rng)
    src = np.concatenate([src, [w.num_blocks + 3, 0]]).astype(np.int32)    # one out of pool
    dst = np.concatenate([dst, [1, -2]]).astype(np.int32)                  # one negative
    B.pkv_copy_blocks(g.k_cache, g.v_cache, to_dev(src), to_dev(dst), g.k_scales, g.v_scales,
                      g.status)
    oracle.copy_blocks(o.k, o.v, src, dst, o.ks, o.vs)
    torch.cuda.synchronize()
    assert int(g.status.item()) & B.DEV_BAD_BLOCK
    gk, gv = to_host_bits(g.k_cache), to_host_bits(g.v_cache)
    live = np.unique(np.concatenate([w.block_tables[w.block_tables >= 0], dst[(dst >= 0) &
                                                                            (dst < w.num_blocks)]]))
    assert np.array_equal(gk[live], o.k[live]) and np.array_equal(gv[live], o.v[live])
    if o.ks is not None:
        assert np.array_equal(g.k_scales.cpu().numpy()[live], o.ks[live])
        assert np.array_equal(g.v_scales.cpu().numpy()[live], o.vs[live])


def test_fork_then_append_then_attend():
    """Copy-on-write in use: a sequence whose last block is shared gets a copy,
    its table is pointed at the copy, the new token lands there, and attention
    over both the forked and the original sequence matches the oracle."""
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    cfg = variant(CONFIGS["gqa8b"], batch=6, len_groups=((6, 40, 300),))
    w = make_workload(cfg)
    # before the step: seq 1 becomes a fork of seq 0 sharing seq 0's blocks
    w.block_tables[1] = w.block_tables[0]
    w.context_lens[1] = w.context_lens[0]
    L = int(w.context_lens[0])
    free = np.setdiff1d(np.arange(w.num_blocks), w.block_tables[w.block_tables >= 0])
    last = (L - 1) // 16
    src, dst = np.array([w.block_tables[0, last]], np.int32), np.array([free[0]], np.int32)
    w.block_tables[1, last] = free[0]          # private copy for the writer
    w.step_slots[1] = int(free[0]) * 16 + (L - 1) % 16
    keep_step = (w.k_step.copy(), w.v_step.copy(), w.step_slots.copy())
    g = GpuCase(w, append_step=False)
    o = OracleCase(w, append_step=False)
    # fork on both sides, then the decode step's append, then attention
    B.pkv_copy_blocks(g.k_cache, g.v_cache, to_dev(src), to_dev(dst), dev_status=g.status)
    oracle.copy_blocks(o.k, o.v, src, dst)
    k_step, v_step, slots = keep_step
    g.append(k_step, v_step, slots)
    oracle.append_copy(o.k, o.v, k_step, v_step, slots)
    out, _ = g.decode()
    torch.cuda.synchronize()
    assert_attention_close(out_to_f64(out), o.attention(), False, "fork + append + attend")
    assert int(g.status.item()) == 0

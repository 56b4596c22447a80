"""pkv_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc: runtimes that plan all
device memory ahead of time and own the allocator, and latency-critical
serving loops that must not allocate (or pay the synchronisation a cudaFree
brings). For them the library offers a variant whose scratch is a fixed array
compiled into the library, so neither the caller nor the library allocates.

These tests call it through the C ABI and compare it with the workspace entry
point, pkv_decode_attn, on two calls in a row with different shapes (the
second call finds the first call's contents in the shared array), on an INT8
cache, and at the size limit: the largest worker count whose scratch fits the
array is accepted, one more worker is rejected. The file is named to be
collected last.
"""

import numpy as np
import pytest

from _pkv_helpers import GpuCase, assert_attention_close, out_to_f64
from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload, variant

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20   # PKV_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


def _free_bytes():
    import torch
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def _noalloc_vs_workspace(cfg, num_parts=0, g=None):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    if g is None:
        g = GpuCase(make_workload(cfg))
    ref, _ = g.decode(num_parts=num_parts)          # existing entry point, caller workspace
    out = torch.full_like(ref, float("nan"))
    free_before = _free_bytes()
    B.pkv_decode_attn_noalloc(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                              cfg.softmax_scale, out, g.k_scales, g.v_scales, num_parts,
                              g.status)
    # nothing was allocated (device-wide free memory; nothing else runs on the GPU)
    assert _free_bytes() == free_before
    assert int(g.status.item()) == 0
    got, want = out_to_f64(out), out_to_f64(ref)
    assert np.isfinite(got).all()
    assert_attention_close(got, want, cfg.kv_dtype == "i8", cfg.name)
    return g


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    first = variant(CONFIGS["gqa8b"], batch=24, len_groups=((24, 1, 1500),))
    second = variant(CONFIGS["skewed"], batch=12, max_len=9000,
                     len_groups=((3, 3000, 9000), (9, 16, 256)))
    _noalloc_vs_workspace(first)
    _noalloc_vs_workspace(second)


def test_noalloc_int8_cache():
    cfg = variant(CONFIGS["gqa8b_int8"], batch=20, len_groups=((20, 1, 1200),))
    g = _noalloc_vs_workspace(cfg)
    _noalloc_vs_workspace(cfg, num_parts=37, g=g)


def _largest_fitting_parts(B, cfg, k_cache):
    """The largest num_parts whose decode scratch fits the built-in array."""
    lo, hi = 1, 1 << 16
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, k_cache, mid) <= LIMIT:
            lo = mid
        else:
            hi = mid - 1
    return lo


@pytest.mark.parametrize("base", ["gqa8b", "gqa8b_int8"])
def test_noalloc_at_its_size_limit(base):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    cfg = variant(CONFIGS[base], batch=24, len_groups=((24, 1, 2000),))
    g = GpuCase(make_workload(cfg))
    parts = _largest_fitting_parts(B, cfg, g.k_cache)
    need = B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, g.k_cache, parts)
    assert LIMIT - 4096 < need <= LIMIT
    assert B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, g.k_cache, parts + 1) > LIMIT
    _noalloc_vs_workspace(cfg, num_parts=parts, g=g)          # just fits: accepted
    out = torch.empty_like(g.q)
    with pytest.raises(B.PkvError) as e:                     # one worker more: rejected
        B.pkv_decode_attn_noalloc(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                  cfg.softmax_scale, out, g.k_scales, g.v_scales, parts + 1)
    assert e.value.code == 3


def test_noalloc_rejects_work_beyond_its_scratch():
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    cfg = variant(CONFIGS["gqa8b"], batch=8192, len_groups=((8192, 1, 8),), max_len=16)
    w = make_workload(cfg)
    g = GpuCase(w)
    need = B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, g.k_cache, 0)
    assert need > LIMIT
    out = torch.empty_like(g.q)
    with pytest.raises(B.PkvError) as e:
        B.pkv_decode_attn_noalloc(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                  cfg.softmax_scale, out)
    assert e.value.code == 3

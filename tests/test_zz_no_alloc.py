"""pkv_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc: runtimes that plan all
device memory ahead of time and own the allocator, and latency-critical
serving loops that must not allocate (or pay the synchronisation a cudaFree
brings). For them the library offers a variant whose scratch is a fixed array
compiled into the library, so neither the caller nor the library allocates.

These tests call it through the C ABI and compare it with the workspace entry
point, pkv_decode_attn, on two calls in a row with different shapes (the
second call finds the first call's contents in the shared array). The file is
named to be collected last.
"""

import numpy as np
import pytest

from _pkv_helpers import GpuCase, assert_attention_close, out_to_f64
from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload, variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


def _noalloc_vs_workspace(cfg):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w = make_workload(cfg)
    g = GpuCase(w)
    ref, _ = g.decode(num_parts=0)           # existing entry point, caller workspace
    out = torch.full_like(ref, float("nan"))
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    B.pkv_decode_attn_noalloc(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                              cfg.softmax_scale, out, g.k_scales, g.v_scales, 0, g.status)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before   # nothing was allocated
    assert int(g.status.item()) == 0
    got, want = out_to_f64(out), out_to_f64(ref)
    assert np.isfinite(got).all()
    assert_attention_close(got, want, cfg.kv_dtype == "i8", cfg.name)


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    first = variant(CONFIGS["gqa8b"], batch=24, len_groups=((24, 1, 1500),))
    second = variant(CONFIGS["skewed"], batch=12, max_len=9000,
                     len_groups=((3, 3000, 9000), (9, 16, 256)))
    _noalloc_vs_workspace(first)
    _noalloc_vs_workspace(second)


def test_noalloc_rejects_work_beyond_its_scratch():
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    cfg = variant(CONFIGS["gqa8b"], batch=8192, len_groups=((8192, 1, 8),), max_len=16)
    w = make_workload(cfg)
    g = GpuCase(w)
    need = B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, g.k_cache, 0)
    assert need > (16 << 20)
    out = torch.empty_like(g.q)
    with pytest.raises(B.PkvError) as e:
        B.pkv_decode_attn_noalloc(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                  cfg.softmax_scale, out)
    assert e.value.code == 3

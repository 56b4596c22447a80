"""The decode step (append + split + combine) captured in a CUDA graph.

Replaying a captured step must give exactly what the eager calls give, and
stay within tolerance of the oracle; the library's launches (with their
programmatic-dependent-launch attributes) must be capturable.
"""

import numpy as np
import pytest

from _pkv_helpers import GpuCase, OracleCase, assert_attention_close, out_to_f64
from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload, variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


@pytest.mark.parametrize("mode", ["append_attn", "step"])
@pytest.mark.parametrize("name", ["gqa8b", "gqa8b_int8", "tiny"])
def test_graph_replay_equals_eager(name, mode):
    """``append_attn``: pkv_append + pkv_decode_attn; ``step``: pkv_decode_step
    (16-bit: the split kernel writes the rows; INT8: its one-row append kernel).
    Replaying appends the same rows again, which leaves the cache unchanged."""
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    cfg = CONFIGS[name] if name == "tiny" else variant(CONFIGS[name], batch=20,
                                                           len_groups=((20, 1, 1200),))
    w = make_workload(cfg)
    g = GpuCase(w, append_step=False)
    def dev(a):
        b = a.view(np.int16) if a.dtype == np.uint16 else a
        return torch.from_numpy(np.ascontiguousarray(b)).cuda()
    k_step, v_step, slots = dev(w.k_step), dev(w.v_step), dev(w.step_slots)
    if w.k_step.dtype == np.uint16:
        k_step, v_step = k_step.view(torch.bfloat16), v_step.view(torch.bfloat16)
    ws = torch.empty(B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, g.k_cache),
                     dtype=torch.uint8, device="cuda")
    out_graph = torch.empty_like(g.q)

    def step(out):
        if mode == "step":
            B.pkv_decode_step(g.q, k_step, v_step, g.k_cache, g.v_cache, g.block_tables,
                              g.context_lens, cfg.softmax_scale, out, ws, 0, g.status,
                              k_scales=g.k_scales, v_scales=g.v_scales)
            return
        B.pkv_append(k_step, v_step, slots, g.k_cache, g.v_cache, g.k_scales, g.v_scales,
                     g.append_ws, g.status)
        B.pkv_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                          cfg.softmax_scale, out, ws, g.k_scales, g.v_scales, 0, g.status)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):           # warm up outside capture
        step(out_graph)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(out_graph)
    out_graph.zero_()
    for _ in range(3):
        graph.replay()
    out_eager = torch.empty_like(g.q)
    step(out_eager)
    torch.cuda.synchronize()
    assert torch.equal(out_graph.view(torch.int16), out_eager.view(torch.int16))
    assert int(g.status.item()) == 0
    want = OracleCase(w).attention()
    assert_attention_close(out_to_f64(out_graph), want, cfg.kv_dtype == "i8", name)


@pytest.mark.parametrize("name", ["spec_verify", "spec_verify_int8", "prefill_chunk"])
def test_multiquery_graph_replay_equals_eager(name):
    """pkv_multiquery_attn (short-run kernels, the tcgen05 kernel) captured in a
    CUDA graph: replays give the eager output bit for bit."""
    import torch
    from _pkv_helpers import to_dev
    from paged_kv_decode_05_gb300 import binding as B
    base = CONFIGS[name]
    cfg = (variant(base, batch=2, q_len=64, max_len=500, len_groups=((2, 64, 500),))
           if name == "prefill_chunk" else variant(base, batch=12, len_groups=((12, 5, 900),)))
    w = make_workload(cfg)
    g = GpuCase(w)
    q, cu = to_dev(w.q), to_dev(w.cu_q)
    nq = cfg.q_len
    ws = torch.empty(B.pkv_multiquery_workspace_size(cfg.batch, cfg.num_q_heads, nq, g.k_cache, 0),
                     dtype=torch.uint8, device="cuda")

    def run(out):
        B.pkv_multiquery_attn(q, cu, nq, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                              cfg.softmax_scale, out, ws, 0, g.status, k_scales=g.k_scales,
                              v_scales=g.v_scales)

    out_graph = torch.empty_like(q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(out_graph)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(out_graph)
    out_graph.zero_()
    for _ in range(3):
        graph.replay()
    out_eager = torch.empty_like(q)
    run(out_eager)
    torch.cuda.synchronize()
    assert int(g.status.item()) == 0
    assert torch.equal(out_graph.view(torch.int16), out_eager.view(torch.int16))

"""GPU parity: pkv_decode_step (fused append + attention) equals pkv_append +
pkv_decode_attn bit for bit (cache and output) and matches the oracle."""

import numpy as np
import pytest

from _pkv_helpers import (GpuCase, OracleCase, assert_attention_close, out_to_f64, to_dev,
                          to_host_bits)
from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload, variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


@pytest.mark.parametrize("name,cfg", [
    ("gqa8b", variant(CONFIGS["gqa8b"], batch=24, len_groups=((24, 0, 1500),))),
    ("skewed", variant(CONFIGS["skewed"], batch=12, max_len=9000,
                       len_groups=((3, 3000, 9000), (9, 16, 256)))),
    ("tiny", CONFIGS["tiny"]),
    ("mha_d128", variant(CONFIGS["mha7b"], batch=5, len_groups=((5, 1, 600),))),
    ("g8_d128", variant(CONFIGS["gqa8b"], batch=6, num_q_heads=64, num_kv_heads=8,
                        len_groups=((6, 0, 700),))),
    # the new token in row 0 (no cache rows copied), row 15, and L = 0
    ("edges", variant(CONFIGS["gqa8b"], batch=14, len_groups=(
        (2, 0, 0), (2, 1, 1), (2, 16, 16), (2, 17, 17), (2, 31, 31), (2, 32, 32), (2, 33, 33)))),
])
@pytest.mark.parametrize("parts", [0, 7])
def test_fused_step_equals_append_then_attend(name, cfg, parts):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w = make_workload(cfg)
    fused = GpuCase(w, append_step=False)      # cache holds the fill only
    ref = GpuCase(w, append_step=True)
    ref_out, _ = ref.decode(num_parts=parts)
    out = torch.full_like(fused.q, float("nan"))
    ws = torch.empty(B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, fused.k_cache, parts),
                     dtype=torch.uint8, device="cuda")
    B.pkv_decode_step(fused.q, to_dev(w.k_step), to_dev(w.v_step), fused.k_cache, fused.v_cache,
                      fused.block_tables, fused.context_lens, cfg.softmax_scale, out, ws, parts,
                      fused.status)
    torch.cuda.synchronize()
    assert int(fused.status.item()) == 0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    bits = lambda t: to_host_bits(t).view(np.uint16)   # noqa: E731  (stale rows hold NaN)
    assert np.array_equal(bits(fused.k_cache), bits(ref.k_cache))
    assert np.array_equal(bits(fused.v_cache), bits(ref.v_cache))
    want = OracleCase(w).attention()
    assert_attention_close(out_to_f64(out), want, False, name)


@pytest.mark.parametrize("name,cfg", [
    ("gqa8b_int8", variant(CONFIGS["gqa8b_int8"], batch=24, len_groups=((24, 0, 1500),))),
    # the new token in row 0 (a fresh block), rows 15 and 16 (across a block
    # boundary), and L = 0
    ("int8_edges", variant(CONFIGS["gqa8b_int8"], batch=14, len_groups=(
        (2, 0, 0), (2, 1, 1), (2, 16, 16), (2, 17, 17), (2, 31, 31), (2, 32, 32), (2, 33, 33)))),
    ("int8_d64_f16", variant(CONFIGS["gqa8b_int8"], batch=6, num_q_heads=8, num_kv_heads=4,
                             head_dim=64, q_dtype="f16", src_dtype="f16",
                             len_groups=((6, 1, 500),))),
])
@pytest.mark.parametrize("grow", [1.0, 4.0])
@pytest.mark.parametrize("parts", [0, 7])
def test_int8_step_equals_append_then_attend(name, cfg, grow, parts):
    """INT8 caches: pkv_decode_step (the step's one-row append kernel, then
    the split and combine) writes the same codes and scales as pkv_append
    with the same slots and returns the same output bit for bit. With the
    new rows scaled by 4 nearly every touched tile's scale grows, so those
    tiles are requantised."""
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w = make_workload(cfg)
    k_rows = to_dev(w.k_step) * grow          # exact: a power of two, far from overflow
    v_rows = to_dev(w.v_step) * grow
    fused = GpuCase(w, append_step=False)
    ref = GpuCase(w, append_step=False)
    B.pkv_append(k_rows, v_rows, to_dev(w.step_slots), ref.k_cache, ref.v_cache, ref.k_scales,
                 ref.v_scales, ref.append_ws, ref.status)
    ref_out, _ = ref.decode(num_parts=parts)
    out = torch.full_like(fused.q, float("nan"))
    ws = torch.empty(B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, fused.k_cache, parts),
                     dtype=torch.uint8, device="cuda")
    B.pkv_decode_step(fused.q, k_rows, v_rows, fused.k_cache, fused.v_cache, fused.block_tables,
                      fused.context_lens, cfg.softmax_scale, out, ws, parts, fused.status,
                      k_scales=fused.k_scales, v_scales=fused.v_scales)
    torch.cuda.synchronize()
    assert int(fused.status.item()) == 0
    assert torch.equal(fused.k_cache, ref.k_cache) and torch.equal(fused.v_cache, ref.v_cache)
    assert torch.equal(fused.k_scales.view(torch.int32), ref.k_scales.view(torch.int32))
    assert torch.equal(fused.v_scales.view(torch.int32), ref.v_scales.view(torch.int32))
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    if grow == 1.0:
        want = OracleCase(w).attention()
        assert_attention_close(out_to_f64(out), want, True, name)

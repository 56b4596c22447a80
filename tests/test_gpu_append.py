"""GPU parity: pkv_append against the oracle, bit for bit (fp16, bf16, INT8)."""

import numpy as np
import pytest

from _pkv_helpers import GpuCase, OracleCase, to_dev, to_host_bits
from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload, variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


SMALL = {
    "tiny": CONFIGS["tiny"],
    "mha7b": variant(CONFIGS["mha7b"], batch=6, len_groups=((6, 1, 700),)),
    "gqa8b": variant(CONFIGS["gqa8b"], batch=20, len_groups=((20, 1, 900),)),
    "gqa8b_int8": variant(CONFIGS["gqa8b_int8"], batch=20, len_groups=((20, 1, 900),)),
    "int8_d64_f16src": variant(CONFIGS["gqa8b_int8"], batch=9, head_dim=64, src_dtype="f16",
                               q_dtype="f16", len_groups=((9, 1, 300),)),
    "skewed": variant(CONFIGS["skewed"], batch=10, max_len=6000,
                      len_groups=((2, 2500, 6000), (8, 16, 256))),
}


def _compare_caches(g, o, what):
    gk, gv = to_host_bits(g.k_cache), to_host_bits(g.v_cache)
    assert gk.dtype == o.k.dtype
    # every row the workload wrote must match bit for bit
    w = g.w
    slots = np.concatenate([w.fill_slots, w.step_slots[w.step_slots >= 0]])
    blk, row = slots // 16, slots % 16
    assert np.array_equal(gk[blk, :, row, :], o.k[blk, :, row, :]), what
    assert np.array_equal(gv[blk, :, row, :], o.v[blk, :, row, :]), what
    if o.ks is not None:
        assert np.array_equal(gk, o.k), what      # whole pool, incl. requantised rows
        assert np.array_equal(gv, o.v), what
        assert np.array_equal(g.k_scales.cpu().numpy(), o.ks), what
        assert np.array_equal(g.v_scales.cpu().numpy(), o.vs), what


@pytest.mark.parametrize("name", list(SMALL))
def test_append_bit_exact_small(name):
    w = make_workload(SMALL[name])
    g = GpuCase(w)
    o = OracleCase(w)
    import torch
    torch.cuda.synchronize()
    _compare_caches(g, o, name)
    assert int(g.status.item()) == 0


def test_append_leaves_other_rows_untouched():
    import torch
    w = make_workload(SMALL["gqa8b"])
    g = GpuCase(w, stale="nan")
    torch.cuda.synchronize()
    gk = to_host_bits(g.k_cache).transpose(0, 2, 1, 3).reshape(-1, w.cfg.num_kv_heads, 128)
    written = np.zeros(gk.shape[0], bool)
    written[w.fill_slots] = True
    written[w.step_slots[w.step_slots >= 0]] = True
    assert np.all(gk[~written] == 0x7FC0)


def test_append_negative_and_out_of_pool_slots():
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    w = make_workload(SMALL["gqa8b_int8"])
    g = GpuCase(w)
    o = OracleCase(w)
    # a call whose slots are all skipped (-1) or out of the pool changes nothing
    bad = np.array([-1, w.num_blocks * 16, -5, w.num_blocks * 16 + 7], np.int64)
    k = w.k_step[:4].copy()
    g.append(k, k, bad)
    torch.cuda.synchronize()
    assert int(g.status.item()) & B.DEV_BAD_SLOT
    _compare_caches(g, o, "after skipped slots")


def test_int8_requantise_path_and_repeat_step():
    """The decode-step token grows some tile scales; repeating it is a no-op."""
    import torch
    w = make_workload(SMALL["gqa8b_int8"])
    g = GpuCase(w)
    o = OracleCase(w)
    o_before = OracleCase(w, append_step=False)
    grew = (o.ks != o_before.ks) & (o_before.ks != 0)
    assert grew.any(), "workload should exercise the grow-and-requantise branch"
    g.append(w.k_step, w.v_step, w.step_slots)
    torch.cuda.synchronize()
    _compare_caches(g, o, "repeated step")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["gqa8b", "gqa8b_int8"])
def test_append_bit_exact_full_size(name):
    import torch
    w = make_workload(CONFIGS[name])
    g = GpuCase(w)
    o = OracleCase(w)
    torch.cuda.synchronize()
    _compare_caches(g, o, name)
    assert int(g.status.item()) == 0

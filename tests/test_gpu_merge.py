"""pkv_merge_states (the split-K reduce on its own) against the oracle's merge.

Each case draws attention problems (scores, values) per (row, head), cuts
each problem's tokens into random pieces, takes every piece's state with
``oracle.partial_state`` and rounds the states to fp32 (what the GPU reads).
The expected output is ``oracle.merge_states`` of those same fp32 states, in
float64; the GPU's output is compared element by element within the
fp16 / bf16 output bound used throughout (|g - o| <= 2e-3 + 1e-2 |o|).
"""

import numpy as np
import pytest

import oracle
from _pkv_helpers import TOL_ABS, TOL_REL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_05_gb300.build import build
    build()


def make_states(rows, heads, D, seed, max_pieces=6, empty_rows=(), score_std=3.0):
    """Random pieces per (row, head); every head of a row has the same number
    of pieces (states are stored [S, H, ...]). Returns fp32 arrays, row_ptr
    and the float64 expected outputs."""
    rng = np.random.default_rng(seed)
    m_l, l_l, o_l, ptr = [], [], [], [0]
    want = np.zeros((rows, heads, D))
    want_m = np.full((rows, heads), -np.inf)
    want_l = np.zeros((rows, heads))
    for r in range(rows):
        k = 0 if r in empty_rows else int(rng.integers(1, max_pieces + 1))
        pieces = np.zeros((k, heads)), np.zeros((k, heads)), np.zeros((k, heads, D))
        for h in range(heads if k else 0):
            n = int(rng.integers(k, k + 300))
            s = rng.normal(0, score_std, n)
            v = rng.normal(0, 1, (n, D))
            cuts = np.sort(rng.choice(np.arange(1, n), k - 1, replace=False)) if k > 1 else []
            for i, (a, b) in enumerate(zip([0, *cuts], [*cuts, n])):
                m, l, o = oracle.partial_state(s[a:b], v[a:b])
                pieces[0][i, h], pieces[1][i, h], pieces[2][i, h] = m, l, o
        pm, pl, po = (x.astype(np.float32) for x in pieces)
        for h in range(heads):
            if k:
                st = [(float(pm[i, h]), float(pl[i, h]), po[i, h].astype(np.float64))
                      for i in range(k)]
                want[r, h] = oracle.merge_states(st)
                want_m[r, h] = pm[:, h].max()
                want_l[r, h] = sum(np.exp(np.float64(pm[i, h]) - want_m[r, h]) *
                                   np.float64(pl[i, h])
                                   for i in range(k))
        m_l.append(pm); l_l.append(pl); o_l.append(po)
        ptr.append(ptr[-1] + k)
    cat = lambda xs, shape: np.concatenate(xs) if xs else np.zeros(shape, np.float32)  # noqa: E731
    return (cat(m_l, (0, heads)), cat(l_l, (0, heads)), cat(o_l, (0, heads, D)),
            np.array(ptr, np.int32), want, want_m, want_l)


def run_merge(pm, pl, po, ptr, dtype, status=None, with_ml=True):
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    R, H, D = len(ptr) - 1, po.shape[1], po.shape[2]
    out = torch.full((R, H, D), float("nan"), dtype=dtype, device="cuda")
    om = torch.full((R, H), float("nan"), dtype=torch.float32, device="cuda") if with_ml else None
    ol = torch.full((R, H), float("nan"), dtype=torch.float32, device="cuda") if with_ml else None
    B.pkv_merge_states(dev(pm), dev(pl), dev(po), dev(ptr), out, om, ol, status)
    torch.cuda.synchronize()
    res = out.float().cpu().numpy().astype(np.float64)
    if with_ml:
        return res, om.cpu().numpy(), ol.cpu().numpy()
    return res


def assert_close(got, want, what):
    err = np.abs(got - want)
    bad = err > TOL_ABS + TOL_REL * np.abs(want)
    assert not bad.any(), f"{what}: {int(bad.sum())} bad, max abs err {err.max():.3e}"


@pytest.mark.parametrize("D", [64, 128, 256, 36])
@pytest.mark.parametrize("dtype_name", ["bf16", "f16"])
def test_merge_matches_oracle(D, dtype_name):
    import torch
    dtype = torch.bfloat16 if dtype_name == "bf16" else torch.float16
    pm, pl, po, ptr, want, want_m, want_l = make_states(37, 4, D, seed=D, empty_rows=(3, 20))
    got, om, ol = run_merge(pm, pl, po, ptr, dtype)
    assert_close(got, want, f"D={D} {dtype_name}")
    assert np.array_equal(om, want_m.astype(np.float32))      # the max of fp32 inputs
    ok = want_l > 0
    assert np.allclose(ol[ok], want_l[ok], rtol=1e-5, atol=0)
    assert np.all(ol[~ok] == 0) and np.all(np.isneginf(om[~ok]))
    assert np.all(got[3] == 0) and np.all(got[20] == 0)        # rows without states


def test_merge_of_merges_is_the_merge():
    """Merging the merged states of two halves of every row's pieces gives the
    merge of all pieces (the split identity, one level up)."""
    import torch
    pm, pl, po, ptr, want, _, _ = make_states(16, 2, 128, seed=7, max_pieces=8)
    # level 1: each row's pieces cut into two groups -> 2 rows per original row
    ptr2 = []
    for r in range(16):
        a, b = int(ptr[r]), int(ptr[r + 1])
        mid = (a + b) // 2
        ptr2 += [a, mid]
    ptr2 = np.array(ptr2 + [int(ptr[-1])], np.int32)
    g1, m1, l1 = run_merge(pm, pl, po, ptr2, torch.bfloat16)
    # the level-1 outputs are bf16-rounded: rebuild states from them in fp32
    o1 = (g1 * l1[:, :, None].astype(np.float64)).astype(np.float32)
    got = run_merge(m1, l1, o1, np.arange(0, 33, 2, dtype=np.int32), torch.bfloat16,
                    with_ml=False)
    assert_close(got, want, "two-level merge")


def test_states_without_tokens_contribute_nothing():
    import torch
    pm, pl, po, ptr, want, _, _ = make_states(8, 2, 64, seed=11)
    # one extra empty state (m = -inf, l = 0, o = NaN) appended to every row
    R, H, D = 8, 2, 64
    m2, l2, o2, p2 = [], [], [], [0]
    for r in range(R):
        a, b = int(ptr[r]), int(ptr[r + 1])
        m2.append(np.concatenate([pm[a:b], np.full((1, H), -np.inf, np.float32)]))
        l2.append(np.concatenate([pl[a:b], np.zeros((1, H), np.float32)]))
        o2.append(np.concatenate([po[a:b], np.full((1, H, D), np.nan, np.float32)]))
        p2.append(p2[-1] + (b - a) + 1)
    got = run_merge(np.concatenate(m2), np.concatenate(l2), np.concatenate(o2),
                    np.array(p2, np.int32), torch.bfloat16, with_ml=False)
    assert_close(got, want, "with empty states")


def test_wide_score_range():
    """Pieces whose maxima differ by far more than the fp32 exponent range of
    exp(m_i - M) behave as the oracle says: the low pieces vanish."""
    import torch
    pm, pl, po, ptr, want, _, _ = make_states(12, 4, 128, seed=5, score_std=200.0)
    got = run_merge(pm, pl, po, ptr, torch.bfloat16, with_ml=False)
    assert_close(got, want, "wide score range")


def test_bad_row_range_is_flagged_and_zeroed():
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    pm, pl, po, ptr, want, _, _ = make_states(6, 2, 64, seed=3)
    bad = ptr.copy()
    bad[3] = bad[-1] + 5           # row 2 ends past the states, row 3 starts past them
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_merge(pm, pl, po, bad, torch.bfloat16, status=status, with_ml=False)
    assert int(status.item()) & B.DEV_BAD_INDEX
    assert np.all(got[2] == 0) and np.all(got[3] == 0)
    for r in (0, 1, 4, 5):
        assert_close(got[r], want[r], f"row {r}")

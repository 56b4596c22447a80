"""Invariants of the seeded workload generator (CPU only)."""

import numpy as np
import pytest

from paged_kv_decode_05_gb300.workloads import (CONFIGS, algorithmic_bytes, make_workload,
                                                variant)

SMALL = {
    "tiny": CONFIGS["tiny"],
    "mha7b": variant(CONFIGS["mha7b"], batch=6, len_groups=((6, 512, 2048),)),
    "gqa8b": variant(CONFIGS["gqa8b"], batch=9, len_groups=((9, 128, 4096),)),
    "gqa8b_int8": variant(CONFIGS["gqa8b_int8"], batch=5, len_groups=((5, 1, 300),)),
    "skewed": variant(CONFIGS["skewed"], batch=10, max_len=9000,
                      len_groups=((3, 3000, 9000), (7, 16, 256))),
    "gqa70b": variant(CONFIGS["gqa70b"], batch=5, len_groups=((5, 128, 900),)),
    "spec_verify": variant(CONFIGS["spec_verify"], batch=7, len_groups=((7, 5, 600),)),
    "prefill_chunk": variant(CONFIGS["prefill_chunk"], batch=3, q_len=40, max_len=700,
                             len_groups=((3, 40, 700),)),
    "skewed_q3": variant(CONFIGS["skewed"], batch=9, max_len=5000, q_len=3,
                         len_groups=((2, 3000, 5000), (7, 16, 100))),
}


def _check(w):
    cfg = w.cfg
    bs = cfg.block_size
    lens = w.context_lens.astype(np.int64)
    nblk = -(-lens // bs)
    t = w.block_tables
    assert t.shape == (cfg.batch, cfg.max_blocks_per_seq)
    for b in range(cfg.batch):
        assert np.all(t[b, :nblk[b]] >= 0) and np.all(t[b, :nblk[b]] < w.num_blocks)
        assert np.all(t[b, nblk[b]:] == -1)
    nq = cfg.q_len
    written = set()
    for s in w.fill_slots.tolist():
        assert s not in written
        written.add(s)
    assert w.cu_q.tolist() == [nq * b for b in range(cfg.batch + 1)]
    assert w.q.shape[0] == cfg.batch * nq == w.step_slots.size
    for b in range(cfg.batch):
        if lens[b] == 0:
            assert np.all(w.step_slots[b * nq:(b + 1) * nq] == -1)
            continue
        for p in range(int(lens[b]) - nq):
            assert int(t[b, p // bs]) * bs + p % bs in written
        for k in range(nq):
            p = int(lens[b]) - nq + k
            s = int(t[b, p // bs]) * bs + p % bs
            assert w.step_slots[b * nq + k] == s and s not in written
    assert len(set(w.step_slots[w.step_slots >= 0].tolist())) == int(nq * (lens > 0).sum())
    return nblk


@pytest.mark.parametrize("name", list(SMALL))
def test_generator_invariants(name):
    w = make_workload(SMALL[name])
    nblk = _check(w)
    cfg = w.cfg
    used = np.concatenate([w.block_tables[b, :nblk[b]] for b in range(cfg.batch)])
    if cfg.prefix_share == 0:
        assert len(set(used.tolist())) == used.size
    else:
        owner = {}
        for b in range(cfg.batch):
            for j in range(nblk[b]):
                owner.setdefault(int(w.block_tables[b, j]), set()).add(b)
        for blk, seqs in owner.items():
            if len(seqs) > 1:
                assert len({s // cfg.share_group for s in seqs}) == 1
        for b in range(cfg.batch):   # blocks receiving new tokens are private
            for p in range(int(w.context_lens[b]) - cfg.q_len, int(w.context_lens[b])):
                assert owner[int(w.block_tables[b, p // 16])] == {b}
        assert w.shared_blocks > 0
    if cfg.num_blocks is None:
        assert w.num_blocks == -(-w.notes["demand_blocks"] * 11 // 10)
    lo = min(g[1] for g in cfg.len_groups) if cfg.len_groups else 0
    hi = max(g[2] for g in cfg.len_groups) if cfg.len_groups else cfg.max_len
    assert w.context_lens.min() >= lo and w.context_lens.max() <= hi


def test_tiny_config_matches_its_statement():
    w = make_workload(CONFIGS["tiny"])
    assert w.context_lens.tolist() == [17, 64, 100, 129]
    assert w.num_blocks == 64
    assert int((-(-w.context_lens // 16)).sum()) == 22
    assert w.q.dtype == np.float16 and w.k_fill.dtype == np.float16
    assert w.block_tables.shape == (4, 9)


def test_seeded_determinism_and_seed_sensitivity():
    cfg = SMALL["gqa8b"]
    a, b = make_workload(cfg), make_workload(cfg)
    for f in ("context_lens", "block_tables", "q", "k_fill", "v_fill", "k_step", "fill_slots"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    c = make_workload(cfg, seed=1)
    assert not np.array_equal(a.context_lens, c.context_lens)


def test_value_distribution_and_chunking():
    from paged_kv_decode_05_gb300.workloads import _normals
    a = _normals(np.random.default_rng(5), (10000, 3, 7), 1.0, "bf16", chunk_rows=4096)
    b = _normals(np.random.default_rng(5), (10000, 3, 7), 1.0, "bf16", chunk_rows=777)
    assert np.array_equal(a, b)
    cfg = variant(CONFIGS["mha7b"], batch=4, len_groups=((4, 512, 600),))
    w = make_workload(cfg)
    x = (w.k_fill.astype(np.uint32) << 16).view(np.float32)
    assert abs(float(x.std()) - 0.5) < 0.01 and abs(float(x.mean())) < 0.01


def test_algorithmic_bytes_formula():
    cfg = CONFIGS["gqa8b"]
    lens = np.array([16, 17] + [1] * 254, dtype=np.int32)
    T = int(lens.sum())
    nblk = 1 + 2 + 254
    assert algorithmic_bytes(cfg, lens) == T * 2 * 8 * 128 * 2 + 256 * 32 * 128 * 2 + nblk * 4
    assert algorithmic_bytes(CONFIGS["gqa8b_int8"], lens) == \
        T * 2 * 8 * 128 + 256 * 32 * 128 * 2 + nblk * 4 + nblk * 8 * 2 * 4

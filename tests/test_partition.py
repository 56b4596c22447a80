"""The split kernel's work partition, checked by brute force on the CPU.

The decode split cuts the unit stream (sequence b, kv head, unit j) into W
equal contiguous ranges (a unit is one 16-token block for fp16 / bf16 caches
and two consecutive blocks of the sequence for INT8 caches, so a sequence of
L tokens has ceil(L / 16) or ceil(L / 32) units per kv head; the partition is
the same either way); a (b, kv head) segment crossing ranges leaves one
partial state per range at slot ``segment + worker``, and the combine finds a
segment's ranges as ``worker_of(first unit) .. worker_of(last unit)`` minus
empty ranges. This restates that index arithmetic in Python and checks, for
random batches, that every unit is decoded back to itself, that the combine
visits exactly the workers that wrote pieces, and that slots never collide;
and that the lookup over the strided block prefix used above 256 sequences
finds the same sequence as the exact prefix.
The multi-query split's partition (row tiles over the blocks their queries
can see) is checked the same way.
"""

import bisect
import random


def worker_of(u, U, W):
    return ((u + 1) * W - 1) // U


def nonempty(w, U, W):
    return w * U // W < (w + 1) * U // W


def test_partition_slots_and_combine_ranges():
    rng = random.Random(0)
    for _ in range(2000):
        B, hkv, W = rng.randint(1, 12), rng.randint(1, 4), rng.randint(1, 60)
        nblk = [rng.choice([0, 0, 1, 2, 3, 7, 20]) for _ in range(B)]
        prefix = [0]
        for n in nblk:
            prefix.append(prefix[-1] + n)
        U = prefix[-1] * hkv
        pieces = {}
        for w in range(W):
            for u in range(w * U // W, (w + 1) * U // W):
                x = u // hkv
                b = max(i for i in range(B) if prefix[i] <= x)
                nb = prefix[b + 1] - prefix[b]
                assert nb > 0
                kvh, j = divmod(u - hkv * prefix[b], nb)
                assert u == hkv * prefix[b] + kvh * nb + j
                pieces.setdefault(b * hkv + kvh, set()).add(w)
        slots = set()
        for seg, ws in pieces.items():
            b, kvh = divmod(seg, hkv)
            uf = hkv * prefix[b] + kvh * nblk[b]
            wf, wl = worker_of(uf, U, W), worker_of(uf + nblk[b] - 1, U, W)
            assert ws == {w for w in range(wf, wl + 1) if nonempty(w, U, W)}
            if len(ws) > 1:
                for w in ws:
                    assert seg + w not in slots and seg + w < B * hkv + W
                    slots.add(seg + w)



PREFIX_ENTRIES = 256   # shared-memory block prefix entries of the decode split


def strided_lookup(x, coarse, stride, nblk):
    """The split kernel's unit lookup over a strided prefix: the last chunk
    whose first sequence starts at or before x, then a walk over its
    sequences. Returns (b, first unit of b, units of b)."""
    lo = 0
    step = 128
    while step:
        if lo + step < len(coarse) - 1 and coarse[lo + step] <= x:
            lo += step
        step >>= 1
    first = coarse[lo]
    b = lo * stride
    last = min(b + stride, len(nblk)) - 1
    nb = nblk[b]
    while b < last and x >= first + nb:
        first += nb
        b += 1
        nb = nblk[b]
    return b, first, nb


def test_strided_prefix_lookup_matches_exact_prefix():
    """Above 256 sequences the kernel keeps every stride-th prefix entry in
    shared memory and walks the rest; it must find the same sequence as the
    exact prefix, through runs of empty sequences and a ragged last chunk."""
    rng = random.Random(1)
    for _ in range(60):
        B = rng.choice([257, 300, 511, 1000, 1001, 4097, 8192])
        stride = 1 if B <= PREFIX_ENTRIES else -(-B // PREFIX_ENTRIES)
        chunks = -(-B // stride)
        assert chunks <= PREFIX_ENTRIES
        nblk = [rng.choice([0, 0, 1, 2, 5]) for _ in range(B)]
        for _ in range(rng.randint(0, 4)):          # long empty runs
            a = rng.randrange(B)
            for i in range(a, min(B, a + rng.randint(1, 3 * stride))):
                nblk[i] = 0
        prefix = [0]
        for n in nblk:
            prefix.append(prefix[-1] + n)
        coarse = [prefix[c * stride] for c in range(chunks)] + [prefix[B]]
        for x in range(prefix[B]):
            b = bisect.bisect_right(prefix, x) - 1   # the exact rule: last b with prefix[b] <= x
            assert strided_lookup(x, coarse, stride, nblk) == (b, prefix[b], nblk[b])

# ----------------------------------------------------- multi-query kernel ---
# The multi-query split orders units (sequence b, kv head, row tile t, block j)
# over the blocks each 16 NW-row tile can see; row r of a tile is query r // g
# of the sequence, which sits at position L - n + r // g. A piece of a tile
# that crosses ranges leaves its rows at slot (b * hkv + kvh) * tmax + t + w.

def tile_blocks(n, L, t, RT, G):
    q_last = min(n - 1, ((t + 1) * RT - 1) // G)
    return (L - n + q_last) // 16 + 1


def units_per_head(n, L, RT, G):
    if n == 0:
        return 0
    return sum(tile_blocks(n, L, t, RT, G) for t in range(-(-n * G // RT)))


def test_multiquery_partition_slots_tiles_and_combine_ranges():
    rng = random.Random(1)
    for _ in range(1500):
        B, hkv = rng.randint(1, 6), rng.randint(1, 3)
        # tile heights of the 16-rows-per-warp kernel (16, 32, 64) and of the
        # short-run kernels (8, 16 or 24 rows on the MMA's N side, one tile)
        G, RT = rng.choice([1, 2, 4, 8]), rng.choice([8, 16, 24, 32, 64])
        max_q = rng.randint(1, 20) if RT in (32, 64) or rng.random() < 0.5 else max(1, RT // G)
        ns = [rng.choice([0, 1, rng.randint(0, max_q)]) for _ in range(B)]
        Ls = [n + rng.randint(0, 90) for n in ns]
        tmax = -(-max_q * G // RT)
        prefix = [0]
        for n, L in zip(ns, Ls):
            prefix.append(prefix[-1] + hkv * units_per_head(n, L, RT, G))
        U = prefix[-1]
        W0 = rng.randint(1, 60)
        W = max(1, min(W0, U // 4))
        # brute force: the blocks a tile's rows can see are those up to its
        # last row's position
        for n, L in zip(ns, Ls):
            for t in range(-(-n * G // RT) if n else 0):
                rows = range(t * RT, min((t + 1) * RT, n * G))
                last_pos = max(L - n + r // G for r in rows)
                assert tile_blocks(n, L, t, RT, G) == last_pos // 16 + 1
        # every unit, in order, and the pieces the split kernel writes
        order = [(b, k, t, j) for b in range(B) for k in range(hkv)
                 for t in range(-(-ns[b] * G // RT) if ns[b] else 0)
                 for j in range(tile_blocks(ns[b], Ls[b], t, RT, G))]
        assert len(order) == U
        pieces = {}
        for w in range(W):
            for u in range(w * U // W, (w + 1) * U // W):
                b, k, t, j = order[u]
                pieces.setdefault((b, k, t), {}).setdefault(w, []).append(j)
        slots = set()
        for (b, k, t), by_worker in pieces.items():
            nb = tile_blocks(ns[b], Ls[b], t, RT, G)
            per_head = units_per_head(ns[b], Ls[b], RT, G)
            cum = sum(tile_blocks(ns[b], Ls[b], tt, RT, G) for tt in range(t))
            uf = prefix[b] + k * per_head + cum
            ul = uf + nb - 1
            assert order[uf] == (b, k, t, 0) and order[ul] == (b, k, t, nb - 1)
            wf, wl = ((uf + 1) * W - 1) // U, ((ul + 1) * W - 1) // U
            assert set(by_worker) == set(range(wf, wl + 1))
            if wf == wl:   # finished inside one worker: written directly
                assert by_worker[wf] == list(range(nb))
                continue
            for w in by_worker:
                s = (b * hkv + k) * tmax + t + w
                assert s not in slots and s < B * hkv * tmax + W
                slots.add(s)

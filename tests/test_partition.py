"""The split kernel's work partition, checked by brute force on the CPU.

The decode split cuts the unit stream (sequence b, kv head, block j) into W
equal contiguous ranges; a (b, kv head) segment crossing ranges leaves one
partial state per range at slot ``segment + worker``, and the combine finds a
segment's ranges as ``worker_of(first unit) .. worker_of(last unit)`` minus
empty ranges. This restates that index arithmetic in Python and checks, for
random batches, that every unit is decoded back to itself, that the combine
visits exactly the workers that wrote pieces, and that slots never collide.
"""

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

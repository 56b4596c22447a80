"""Float64 paged decode attention, written from its plain definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Definition (one query token per sequence, "decode step"): for sequence ``b``
with context length ``L`` and query head ``h``, let ``hkv = h // g`` with
``g = Hq / Hkv``. Token ``p`` (``0 <= p < L``) lives in physical block
``block_tables[b, p // bs]`` at row ``p % bs``. With ``k_p``/``v_p`` that
token's key/value rows,

    s_p   = scale * <q[b, h], k_p>
    out   = sum_p softmax(s)_p * v_p          (max-subtracted softmax)

and ``out = 0`` when ``L == 0``.

Sources: block pool + per-sequence logical->physical page table, KV gathered
from non-contiguous blocks inside the kernel (Continuous-Batching-LLM-
Inference-Engine README, feature list "Paged KV-cache", "PagedAttention
kernel"); the decoder "reads block table" and dispatches the attention kernel
(paged-inference-engine, Connections); paged decode attention kernel
(mini-inference-engine, component "Paged decode attention"); INT8 paged KV
(paged-inference-engine overview). Readings where the pages are silent:

* GQA grouping is contiguous: query head ``h`` reads KV head ``h // g``.
* An INT8 cache value dequantises as ``code * scale[block, kv_head]``; the
  product of an 8-bit integer and an fp32 scale is exact in float64.
* The split-K merge state of a chunk is ``(m, l, o)`` with ``m`` the chunk's
  max score, ``l = sum exp(s - m)`` and ``o = sum exp(s - m) v`` (unnormalised).
"""

from __future__ import annotations

import numpy as np


def decode_kv(x: np.ndarray) -> np.ndarray:
    """Decode stored cache / query values to float64, exactly.

    ``np.uint16`` holds bfloat16 bit patterns (the upper half of an IEEE
    binary32), ``np.float16`` holds IEEE binary16, ``np.int8`` holds raw codes
    (scales are applied by the caller). float32/float64 pass through.
    """
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if x.dtype in (np.float16, np.float32, np.float64, np.int8):
        return x.astype(np.float64)
    raise TypeError(f"unsupported stored dtype {x.dtype}")


def _gather_sequence(cache, scales, block_tables, b, L, block_size):
    """Walk sequence ``b``'s block table token by token.

    Returns float64 rows ``[L, Hkv, D]``. Position ``p`` maps to
    ``(block_tables[b, p // block_size], p % block_size)``.
    """
    pos = np.arange(L)
    blk = block_tables[b, pos // block_size].astype(np.int64)
    row = pos % block_size
    rows = decode_kv(cache[blk, :, row, :])  # [L, Hkv, D]
    if scales is not None:
        rows = rows * scales[blk, :].astype(np.float64)[:, :, None]
    return rows


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens,
                           softmax_scale, k_scales=None, v_scales=None,
                           block_size=16, seqs=None):
    """Single-query attention over a paged KV cache, in float64.

    q            [B, Hq, D]        query (uint16 bf16 bits / float16 / float)
    k_cache      [NB, Hkv, bs, D]  keys   (uint16 / float16 / int8 / float)
    v_cache      [NB, Hkv, bs, D]  values
    block_tables [B, MB] int32     physical block of each logical block
    context_lens [B] int32         tokens per sequence (incl. the new one)
    k_scales, v_scales [NB, Hkv] float32, required for int8 caches
    seqs         optional list of sequence indices to evaluate

    Returns float64 ``[len(seqs), Hq, D]``.
    """
    B, Hq, D = q.shape
    NB, Hkv, bs, Dk = k_cache.shape
    assert bs == block_size and Dk == D and Hq % Hkv == 0
    if k_cache.dtype == np.int8:
        assert k_scales is not None and v_scales is not None
    g = Hq // Hkv
    if seqs is None:
        seqs = range(B)
    seqs = list(seqs)
    out = np.zeros((len(seqs), Hq, D), dtype=np.float64)
    for i, b in enumerate(seqs):
        L = int(context_lens[b])
        if L == 0:
            continue
        K = _gather_sequence(k_cache, k_scales, block_tables, b, L, bs)
        V = _gather_sequence(v_cache, v_scales, block_tables, b, L, bs)
        qb = decode_kv(q[b])
        for h in range(Hq):
            kvh = h // g
            s = float(softmax_scale) * (K[:, kvh, :] @ qb[h])
            w = np.exp(s - s.max())
            out[i, h] = (w @ V[:, kvh, :]) / w.sum()
    return out


def partial_state(scores, values):
    """Merge state ``(m, l, o)`` of one chunk of tokens (float64).

    scores [n] already scaled; values [n, D]. ``o`` is unnormalised.
    """
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    m = scores.max()
    w = np.exp(scores - m)
    return m, w.sum(), w @ values


def merge_states(states):
    """Combine chunk states into the attention output.

    With ``M = max_i m_i``:
    ``out = sum_i exp(m_i - M) o_i / sum_i exp(m_i - M) l_i``.
    This is the split-K (flash-decoding) reduce; it equals the unsplit
    softmax-weighted sum for any partition of the tokens into chunks.
    """
    ms = np.array([s[0] for s in states], dtype=np.float64)
    M = ms.max()
    num = 0.0
    den = 0.0
    for (m, l, o) in states:
        a = np.exp(m - M)
        num = num + a * np.asarray(o, dtype=np.float64)
        den = den + a * l
    return num / den


def paged_multiquery_attention(q, cu_q, k_cache, v_cache, block_tables, context_lens,
                               softmax_scale, k_scales=None, v_scales=None, block_size=16,
                               seqs=None):
    """Several new query tokens per sequence, causal among themselves (float64).

    The target model of speculative decoding scores the draft's K tokens plus
    one in a single batched pass (Continuous-Batching-LLM-Inference-Engine
    README, feature list "Speculative decoding"), and a continuous-batching
    scheduler mixes decode tokens with prefill chunks (mini-inference-engine
    overview). Both are attention of ``n_b`` new query tokens per sequence
    over the paged cache, which already holds them. Reading: sequence ``b``
    owns query rows ``cu_q[b] .. cu_q[b+1]-1`` (``n_b`` of them, in position
    order), its cache holds ``L_b = context_lens[b]`` tokens including those
    ``n_b``, and query ``i`` sits at position ``p_i = L_b - n_b + i`` and attends
    to positions ``0 .. p_i``.

    q [total_q, Hq, D]; cu_q int [B+1]. Returns float64 rows for the selected
    sequences' queries, concatenated in sequence order.
    """
    total_q, Hq, D = q.shape
    NB, Hkv, bs, Dk = k_cache.shape
    assert bs == block_size and Dk == D and Hq % Hkv == 0
    g = Hq // Hkv
    B = len(cu_q) - 1
    seqs = list(range(B)) if seqs is None else list(seqs)
    rows = []
    for b in seqs:
        n = int(cu_q[b + 1] - cu_q[b])
        L = int(context_lens[b])
        assert 0 <= n <= L or n == 0
        out = np.zeros((n, Hq, D), dtype=np.float64)
        if n:
            K = _gather_sequence(k_cache, k_scales, block_tables, b, L, bs)
            V = _gather_sequence(v_cache, v_scales, block_tables, b, L, bs)
            for i in range(n):
                p = L - n + i
                qi = decode_kv(q[int(cu_q[b]) + i])
                for h in range(Hq):
                    kvh = h // g
                    s = float(softmax_scale) * (K[:p + 1, kvh, :] @ qi[h])
                    w = np.exp(s - s.max())
                    out[i, h] = (w @ V[:p + 1, kvh, :]) / w.sum()
        rows.append(out)
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, Hq, D))

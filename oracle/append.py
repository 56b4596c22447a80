"""KV-cache append (cache write) oracle: bit copy and INT8 quantise-on-append.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources: the Llama forward "writes and reads" the paged KV cache
(mini-inference-engine, Connections); the engine "writes KV cache" and paged
attention "maps cache slots" (low-latency-distributed-llm-serving-
infrastructure, Connections); paged INT8 KV storage (paged-inference-engine
overview). The pages give no slot formula and no quantisation rule. Readings:

* A slot is ``block * block_size + row``; a negative slot means "skip".
* fp16 / bf16 caches store the new rows bit for bit.
* INT8 caches: symmetric codes in [-127, 127] with one fp32 scale per
  (block, kv_head), separately for K and V, ``scale = absmax / 127`` and
  round-to-nearest-even. Tokens arrive incrementally, so each call applies,
  per (block, kv_head) tile touched by the call (K and V separately):

    a   = max |x| over the call's new values in the tile   (fp32, exact)
    s_c = a / 127                                          (fp32 RN divide)
    s_o = the tile's stored scale (pool scales start at 0)
    s   = s_c            if s_o == 0
          s_o            if s_c <= s_o                     (no requantise)
          s_c            otherwise, and every stored code of the tile is
                         requantised  q' = rne((float(q) * s_o) / s),
                         evaluated left to right in fp32
    new codes: q = clamp(rne(x / s), -127, 127), and q = 0 when s == 0.

  A tile filled by one call therefore has exactly ``scale = absmax / 127``.
"""

from __future__ import annotations

import numpy as np

_F32_127 = np.float32(127.0)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (``np.uint16``) -> float32, exactly."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def quantize_int8(x: np.ndarray, s) -> np.ndarray:
    """``clamp(rne(x / s), -127, 127)`` in fp32; 0 where ``s == 0``.

    ``x`` float32, ``s`` float32 scalar or array broadcastable to ``x``.
    """
    x = np.asarray(x, dtype=np.float32)
    s = np.asarray(s, dtype=np.float32)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    with np.errstate(over="ignore"):
        y = np.rint(x / safe)  # fp32 RN division, then ties-to-even
    y = np.clip(y, -127.0, 127.0)
    y = np.where(s == 0, np.float32(0.0), y)
    return y.astype(np.int8)


def requantize_int8(codes: np.ndarray, s_old, s_new) -> np.ndarray:
    """``rne((float(q) * s_old) / s_new)`` in fp32, left to right."""
    t = codes.astype(np.float32) * np.asarray(s_old, dtype=np.float32)
    t = t.astype(np.float32) / np.asarray(s_new, dtype=np.float32)
    return np.rint(t.astype(np.float32)).astype(np.int8)


def append_copy(k_cache, v_cache, k_new, v_new, slot_mapping, block_size=16):
    """Write ``k_new[n], v_new[n]`` ([N, Hkv, D]) to slot ``slot_mapping[n]``.

    In place, bit for bit (fp16 / bf16 caches). Negative slots are skipped.
    """
    slots = np.asarray(slot_mapping, dtype=np.int64)
    keep = slots >= 0
    blk = slots[keep] // block_size
    row = slots[keep] % block_size
    k_cache[blk, :, row, :] = k_new[keep]
    v_cache[blk, :, row, :] = v_new[keep]


def _append_int8_one(cache, scales, new_f32, slots, block_size):
    """Apply the INT8 append rule to one of K or V (in place)."""
    NB, Hkv, bs, D = cache.shape
    valid = slots >= 0
    n_idx = np.nonzero(valid)[0]
    if n_idx.size == 0:
        return
    blk = slots[n_idx] // block_size
    row = slots[n_idx] % block_size
    rows = new_f32[n_idx]                                   # [n, Hkv, D] f32
    row_amax = np.abs(rows).max(axis=2)                      # [n, Hkv]   exact
    tile = (blk[:, None] * Hkv + np.arange(Hkv)[None, :])    # [n, Hkv]
    flat_scales = scales.reshape(-1)
    flat_cache = cache.reshape(NB * Hkv, bs, D)

    touched, inv = np.unique(tile.reshape(-1), return_inverse=True)
    a = np.zeros(touched.size, dtype=np.float32)
    np.maximum.at(a, inv, row_amax.reshape(-1).astype(np.float32))

    s_c = (a / _F32_127).astype(np.float32)
    s_o = flat_scales[touched].astype(np.float32)
    grow = (s_o != 0) & (s_c > s_o)
    s = np.where(s_o == 0, s_c, np.where(s_c <= s_o, s_o, s_c)).astype(np.float32)

    if grow.any():
        t = touched[grow]
        flat_cache[t] = requantize_int8(flat_cache[t], s_o[grow][:, None, None],
                                        s[grow][:, None, None])
    flat_scales[touched] = s

    s_rows = flat_scales[tile]                                # [n, Hkv]
    codes = quantize_int8(rows, s_rows[:, :, None])
    cache[blk[:, None], np.arange(Hkv)[None, :], row[:, None], :] = codes


def append_int8(k_cache, v_cache, k_scales, v_scales, k_new, v_new,
                slot_mapping, block_size=16):
    """INT8 quantise-on-append for one call (in place).

    k_cache, v_cache  [NB, Hkv, bs, D] int8
    k_scales, v_scales [NB, Hkv] float32 (0 = never written)
    k_new, v_new      [N, Hkv, D] float32 (exact bf16 / fp16 source values,
                      or np.uint16 bf16 bit patterns)
    Duplicate non-negative slots within one call are a caller error.
    """
    slots = np.asarray(slot_mapping, dtype=np.int64)
    if k_new.dtype == np.uint16:
        k_new = bf16_bits_to_f32(k_new)
        v_new = bf16_bits_to_f32(v_new)
    k_new = np.asarray(k_new, dtype=np.float32)
    v_new = np.asarray(v_new, dtype=np.float32)
    _append_int8_one(k_cache, k_scales, k_new, slots, block_size)
    _append_int8_one(v_cache, v_scales, v_new, slots, block_size)


def copy_blocks(k_cache, v_cache, src_blocks, dst_blocks, k_scales=None, v_scales=None):
    """Copy whole physical blocks ``src -> dst`` (all kv heads, K and V, and
    the INT8 scales when given), pair by pair in order (in place).

    The copy-on-write step of a paged KV cache: a block shared by several
    sequences (reference count > 1) gets a private copy before one of them
    writes to it, and speculative decoding rolls a rejected draft back to such
    copies (Continuous-Batching-LLM-Inference-Engine README, feature list
    "Paged KV-cache": copy-on-write reference counting; "Speculative
    decoding": KV-cache rollback uses the copy-on-write). Reading: a pair
    with an id outside the pool is skipped; a destination that is also a
    source in the same call is a caller error.
    """
    NB = k_cache.shape[0]
    for s, d in zip(np.asarray(src_blocks).tolist(), np.asarray(dst_blocks).tolist()):
        if not (0 <= s < NB and 0 <= d < NB):
            continue
        k_cache[d] = k_cache[s]
        v_cache[d] = v_cache[s]
        if k_scales is not None:
            k_scales[d] = k_scales[s]
            v_scales[d] = v_scales[s]

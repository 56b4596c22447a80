"""Seeded synthetic decode-step workloads (block pools, tables, lengths, values).

This module only draws inputs. It holds none of the attention or quantisation
arithmetic, so both the CUDA path (tests, bench) and the CPU oracle can be fed
from it without sharing any of the method.

Recipe (every config):

* RNG: ``numpy.random.default_rng(seed)`` (PCG64), draws in this order:
  context lengths -> pool shuffle -> q -> fill K -> fill V -> new-token K/V.
* Values: standard normals drawn in float32, times the config's std, rounded
  to the stored 16-bit type with round-to-nearest-even (bf16 as bit patterns
  in ``np.uint16``, fp16 as ``np.float16``).
* Pool: ``num_blocks`` physical blocks of ``block_size = 16`` tokens. Unless a
  config fixes the pool size, it is the blocks in use plus 10 %, rounded up.
  A seeded permutation of the pool hands out blocks in sequence order, so every
  table is scattered over the pool.
* Each sequence's last ``q_len`` tokens (positions ``L - q_len .. L - 1``;
  one token for a decode step) are the step's new tokens; positions
  ``0 .. L - q_len - 1`` form the bulk "fill" appended beforehand.
* Prefix sharing (skewed mix): sequences are taken 4 at a time in batch order;
  member ``i`` of a group reads the group's shared physical blocks for its
  first ``min(prefix, 16 * floor((L_i - q_len) / 16))`` tokens, so the blocks
  that receive its new tokens are always private (copy-on-write safe). The
  shared prefix is written once.

The five decode configurations are the shapes of a paged-KV serving loop's
decode step: a tiny fp16 case, an MHA 7B-shape batch, a Llama-3-8B-shape GQA
batch (bf16 and INT8 KV) and a skewed long-context mix with shared prefixes.
Three more cover adjacent work: a 70B-class decode batch with 8 query heads
per KV head, speculative verification and chunked prefill.
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str          # "f16" | "bf16" | "i8"  (cache storage)
    q_dtype: str           # "f16" | "bf16"         (query / output)
    src_dtype: str         # "f16" | "bf16"         (rows handed to append)
    len_groups: tuple      # ((count, lo, hi), ...) uniform integer ranges
    max_len: int           # sizes the block-table width
    kv_std: float = 1.0
    q_std: float = 1.0
    fixed_lens: tuple | None = None
    num_blocks: int | None = None
    prefix_share: int = 0
    share_group: int = 4
    seed: int = 0
    block_size: int = BLOCK_SIZE
    q_len: int = 1         # new query tokens per sequence (1 = decode)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_blocks_per_seq(self) -> int:
        return -(-self.max_len // self.block_size)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


CONFIGS = {
    "tiny": DecodeConfig(
        name="tiny", batch=4, num_q_heads=4, num_kv_heads=4, head_dim=64,
        kv_dtype="f16", q_dtype="f16", src_dtype="f16",
        len_groups=(), fixed_lens=(17, 64, 100, 129), max_len=129,
        num_blocks=64, seed=0),
    "mha7b": DecodeConfig(
        name="mha7b", batch=64, num_q_heads=32, num_kv_heads=32, head_dim=128,
        kv_dtype="bf16", q_dtype="bf16", src_dtype="bf16",
        len_groups=((64, 512, 2048),), max_len=2048, kv_std=0.5),
    "gqa8b": DecodeConfig(
        name="gqa8b", batch=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
        kv_dtype="bf16", q_dtype="bf16", src_dtype="bf16",
        len_groups=((256, 128, 4096),), max_len=4096),
    "gqa8b_int8": DecodeConfig(
        name="gqa8b_int8", batch=256, num_q_heads=32, num_kv_heads=8,
        head_dim=128, kv_dtype="i8", q_dtype="bf16", src_dtype="bf16",
        len_groups=((256, 128, 4096),), max_len=4096),
    "skewed": DecodeConfig(
        name="skewed", batch=128, num_q_heads=32, num_kv_heads=8, head_dim=128,
        kv_dtype="bf16", q_dtype="bf16", src_dtype="bf16",
        len_groups=((8, 32768, 131072), (120, 16, 256)), max_len=131072,
        prefix_share=2048),
    "gqa70b": DecodeConfig(
        name="gqa70b", batch=256, num_q_heads=64, num_kv_heads=8, head_dim=128,
        kv_dtype="bf16", q_dtype="bf16", src_dtype="bf16",
        len_groups=((256, 128, 4096),), max_len=4096),
    "spec_verify": DecodeConfig(
        name="spec_verify", batch=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
        kv_dtype="bf16", q_dtype="bf16", src_dtype="bf16",
        len_groups=((256, 128, 4096),), max_len=4096, q_len=5),
    "prefill_chunk": DecodeConfig(
        name="prefill_chunk", batch=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
        kv_dtype="bf16", q_dtype="bf16", src_dtype="bf16",
        len_groups=((8, 512, 8192),), max_len=8192, q_len=512),
    "spec_verify_int8": DecodeConfig(
        name="spec_verify_int8", batch=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
        kv_dtype="i8", q_dtype="bf16", src_dtype="bf16",
        len_groups=((256, 128, 4096),), max_len=4096, q_len=5),
}

# One-line workload descriptions, for bench output and docs.
DESCRIPTIONS = {
    "tiny": "tiny fp16: B=4, L={17,64,100,129}, 4/4 heads, D=64, pool 64 blocks",
    "mha7b": "MHA 7B-shape bf16: B=64, 32/32 heads, D=128, L~U[512,2048]",
    "gqa8b": "GQA Llama-3-8B-shape bf16: B=256, 32 q / 8 kv heads, D=128, L~U[128,4096]",
    "gqa8b_int8": "GQA Llama-3-8B-shape INT8 KV: B=256, 32/8 heads, D=128, L~U[128,4096]",
    "skewed": "skewed long-context bf16: 8 x L~U[32768,131072] + 120 x L~U[16,256], "
              "32/8 heads, D=128, 2048-token CoW prefix per 4 sequences",
    "gqa70b": "GQA 70B-class-shape bf16: B=256, 64 q / 8 kv heads (group 8), D=128, "
              "L~U[128,4096]",
    "spec_verify": "speculative verification bf16: B=256, 4 draft tokens + 1 per sequence, "
                   "32/8 heads, D=128, L~U[128,4096]",
    "prefill_chunk": "chunked prefill bf16: B=8, 512-token chunk per sequence after a cached "
                     "prefix, 32/8 heads, D=128, L~U[512,8192]",
    "spec_verify_int8": "speculative verification over an INT8 cache: B=256, 4 draft tokens + 1 "
                        "per sequence, 32/8 heads, D=128, L~U[128,4096]",
}


def variant(cfg: DecodeConfig, **changes) -> DecodeConfig:
    """Same config family with some fields replaced (smaller test cases)."""
    return dataclasses.replace(cfg, **changes)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _to_stored(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x_f32)
    if dtype == "f16":
        return x_f32.astype(np.float16)
    raise ValueError(dtype)


def _normals(rng, shape, std, dtype, chunk_rows=4096):
    """Draw ``shape`` normals in float32, in row chunks along axis 0, then round.

    The chunks are consecutive draws from one stream, so the values do not
    depend on the chunk size.
    """
    n = shape[0]
    out = np.empty(shape, dtype=np.uint16 if dtype == "bf16" else np.float16)
    if n == 0:
        return out
    buf = np.empty((min(n, chunk_rows),) + tuple(shape[1:]), dtype=np.float32)
    for s in range(0, n, chunk_rows):
        e = min(n, s + chunk_rows)
        x = buf[:e - s]
        rng.standard_normal(out=x, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = _to_stored(x, dtype)
    return out


@dataclass
class Workload:
    cfg: DecodeConfig
    context_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray          # int32 [B, MB], -1 past the end
    num_blocks: int
    q: np.ndarray                     # [B, Hq, D] uint16 (bf16) / float16
    fill_slots: np.ndarray            # int64 [Nf]
    k_fill: np.ndarray                # [Nf, Hkv, D] source dtype
    v_fill: np.ndarray
    step_slots: np.ndarray            # int64 [B*q_len], -1 if L == 0
    k_step: np.ndarray                # [B*q_len, Hkv, D] source dtype
    v_step: np.ndarray
    cu_q: np.ndarray = None           # int32 [B+1] query rows of each sequence
    shared_blocks: int = 0            # physical blocks referenced by >1 seq
    notes: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())


def _draw_lengths(cfg, rng):
    if cfg.fixed_lens is not None:
        lens = np.array(cfg.fixed_lens, dtype=np.int64)
    else:
        parts = [rng.integers(lo, hi, size=cnt, endpoint=True)
                 for (cnt, lo, hi) in cfg.len_groups]
        lens = np.concatenate(parts).astype(np.int64)
    assert lens.size == cfg.batch, (lens.size, cfg.batch)
    assert lens.max(initial=0) <= cfg.max_len
    return lens


def make_workload(cfg: DecodeConfig, seed: int | None = None) -> Workload:
    """Build the seeded workload for ``cfg`` (see module docstring)."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    bs = cfg.block_size
    B, Hkv, Hq, D = cfg.batch, cfg.num_kv_heads, cfg.num_q_heads, cfg.head_dim
    MB = cfg.max_blocks_per_seq

    lens = _draw_lengths(cfg, rng)
    nq = cfg.q_len
    assert nq >= 1 and (nq == 1 or lens.min(initial=nq) >= nq), "each sequence holds its queries"
    nblk = -(-lens // bs)

    # Which leading tokens of each sequence are read from shared blocks.
    shared_len = np.zeros(B, dtype=np.int64)
    if cfg.prefix_share > 0:
        G = cfg.share_group
        groups = [list(range(g0, min(B, g0 + G))) for g0 in range(0, B, G)]
        for members in groups:
            for i in members:
                if lens[i] > 0:
                    shared_len[i] = min(cfg.prefix_share, bs * ((lens[i] - cfg.q_len) // bs))
    else:
        groups = [[i] for i in range(B)]

    # Physical blocks in use, in allocation order.
    demand = 0
    for members in groups:
        demand += int(shared_len[members].max(initial=0)) // bs
        demand += int(sum(nblk[i] - shared_len[i] // bs for i in members))
    NB = cfg.num_blocks if cfg.num_blocks is not None else -(-demand * 11 // 10)
    assert demand <= NB, (demand, NB)
    perm = rng.permutation(NB).astype(np.int64)

    tables = np.full((B, MB), -1, dtype=np.int32)
    cursor = 0
    fill_slot_parts = []
    shared_total = 0
    for members in groups:
        n_shared = int(shared_len[members].max(initial=0)) // bs
        shared = perm[cursor:cursor + n_shared]
        cursor += n_shared
        if n_shared and len(members) > 1:
            shared_total += n_shared
        if n_shared:  # the shared prefix rows are written once
            pos = np.arange(n_shared * bs)
            fill_slot_parts.append(shared[pos // bs] * bs + pos % bs)
        for i in members:
            own_shared = int(shared_len[i]) // bs
            n_priv = int(nblk[i]) - own_shared
            priv = perm[cursor:cursor + n_priv]
            cursor += n_priv
            tables[i, :own_shared] = shared[:own_shared]
            tables[i, own_shared:own_shared + n_priv] = priv
            # private fill rows: positions shared_len .. L-q_len-1
            pos = np.arange(int(shared_len[i]), max(int(lens[i]) - nq, int(shared_len[i])))
            if pos.size:
                fill_slot_parts.append(tables[i, pos // bs].astype(np.int64) * bs + pos % bs)
    assert cursor == demand

    fill_slots = (np.concatenate(fill_slot_parts) if fill_slot_parts
                  else np.zeros(0, dtype=np.int64)).astype(np.int64)
    step_slots = np.full(B * nq, -1, dtype=np.int64)
    for i in range(B):
        for k in range(nq):
            p = int(lens[i]) - nq + k
            if p >= 0:
                step_slots[i * nq + k] = int(tables[i, p // bs]) * bs + p % bs

    q = _normals(rng, (B * nq, Hq, D), cfg.q_std, cfg.q_dtype)
    Nf = fill_slots.size
    k_fill = _normals(rng, (Nf, Hkv, D), cfg.kv_std, cfg.src_dtype)
    v_fill = _normals(rng, (Nf, Hkv, D), cfg.kv_std, cfg.src_dtype)
    k_step = _normals(rng, (B * nq, Hkv, D), cfg.kv_std, cfg.src_dtype)
    v_step = _normals(rng, (B * nq, Hkv, D), cfg.kv_std, cfg.src_dtype)

    return Workload(cfg=cfg, context_lens=lens.astype(np.int32), block_tables=tables,
                    num_blocks=int(NB), q=q, fill_slots=fill_slots, k_fill=k_fill,
                    v_fill=v_fill, step_slots=step_slots, k_step=k_step, v_step=v_step,
                    shared_blocks=shared_total, notes={"demand_blocks": demand},
                    cu_q=(np.arange(B + 1) * nq).astype(np.int32))


def algorithmic_bytes(cfg: DecodeConfig, context_lens: np.ndarray) -> int:
    """Bytes one decode-attention call must read at minimum.

    Logical KV tokens read (a shared block counts once per sequence reading
    it) for K and V, the queries, the used block-table entries and, for INT8,
    the per-(block, kv_head) K and V scales.
    """
    lens = np.asarray(context_lens, dtype=np.int64)
    esz = {"f16": 2, "bf16": 2, "i8": 1}
    T = int(lens.sum())
    nblk = int((-(-lens // cfg.block_size)).sum())
    kv = T * 2 * cfg.num_kv_heads * cfg.head_dim * esz[cfg.kv_dtype]
    q = cfg.batch * cfg.q_len * cfg.num_q_heads * cfg.head_dim * esz[cfg.q_dtype]
    tables = nblk * 4
    scales = nblk * cfg.num_kv_heads * 2 * 4 if cfg.kv_dtype == "i8" else 0
    return kv + q + tables + scales

"""Shared helpers for the GPU parity tests.

The same seeded workload feeds both sides. The GPU side fills its cache with
the library's own ``pkv_append`` (bulk fill, then the decode step's token);
the oracle side builds its cache with ``oracle.append_*`` from the same rows.
Nothing computed on the GPU is ever handed to the oracle.
"""

from __future__ import annotations

import numpy as np

import oracle
from paged_kv_decode_05_gb300.workloads import make_workload

NAN16 = {"bf16": 0x7FC0, "f16": 0x7E00}
TOL_ABS, TOL_REL = 2e-3, 1e-2      # bf16 / fp16 KV: |g - o| <= 2e-3 + 1e-2 |o|
TOL_I8 = 2e-2                       # INT8 KV: |g - o_dequant| <= 2e-2


def torch_dtype(name):
    import torch
    return {"bf16": torch.bfloat16, "f16": torch.float16, "i8": torch.int8}[name]


def to_dev(a: np.ndarray, dtype_name: str | None = None):
    """Host array -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host_bits(t) -> np.ndarray:
    """CUDA tensor -> numpy with bf16 as uint16 bit patterns."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def out_to_f64(t) -> np.ndarray:
    return oracle.decode_kv(to_host_bits(t))


class GpuCase:
    """GPU-side state for one workload: cache filled through pkv_append."""

    def __init__(self, w, stale="nan", append_step=True):
        import torch
        from paged_kv_decode_05_gb300 import binding as B
        self.w, self.cfg = w, w.cfg
        cfg = w.cfg
        shape = (w.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
        if cfg.kv_dtype == "i8":
            self.k_cache = torch.zeros(shape, dtype=torch.int8, device="cuda")
            self.v_cache = torch.zeros(shape, dtype=torch.int8, device="cuda")
            self.k_scales = torch.zeros(shape[:2], dtype=torch.float32, device="cuda")
            self.v_scales = torch.zeros(shape[:2], dtype=torch.float32, device="cuda")
            nbytes = B.pkv_append_workspace_size(self.k_cache)
            self.append_ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        else:
            dt = torch_dtype(cfg.kv_dtype)
            fill = NAN16[cfg.kv_dtype] if stale == "nan" else 0
            raw = torch.full(shape, fill if fill < 0x8000 else fill - 0x10000,
                             dtype=torch.int16, device="cuda")
            self.k_cache = raw.view(dt)
            self.v_cache = raw.clone().view(dt)
            self.k_scales = self.v_scales = None
            self.append_ws = None
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.q = to_dev(w.q)
        self.block_tables = to_dev(w.block_tables)
        self.context_lens = to_dev(w.context_lens)
        self.append(w.k_fill, w.v_fill, w.fill_slots)
        if append_step:
            self.append(w.k_step, w.v_step, w.step_slots)

    def append(self, k, v, slots):
        from paged_kv_decode_05_gb300 import binding as B
        if slots.size == 0:
            return
        B.pkv_append(to_dev(k), to_dev(v), to_dev(slots), self.k_cache, self.v_cache,
                     self.k_scales, self.v_scales, self.append_ws, self.status)

    def decode(self, num_parts=0, split_only=False, out=None):
        import torch
        from paged_kv_decode_05_gb300 import binding as B
        cfg = self.cfg
        if out is None:
            out = torch.empty(self.q.shape, dtype=self.q.dtype, device="cuda")
        ws = torch.empty(B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, self.k_cache,
                                                     num_parts), dtype=torch.uint8, device="cuda")
        fn = B.pkv_decode_split if split_only else B.pkv_decode_attn
        fn(self.q, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
           cfg.softmax_scale, out, ws, self.k_scales, self.v_scales, num_parts, self.status)
        return out, ws


class OracleCase:
    """Oracle-side cache for the same workload, built by the oracle's append."""

    def __init__(self, w, append_step=True):
        cfg = w.cfg
        shape = (w.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
        self.w = w
        if cfg.kv_dtype == "i8":
            self.k = np.zeros(shape, np.int8)
            self.v = np.zeros(shape, np.int8)
            self.ks = np.zeros(shape[:2], np.float32)
            self.vs = np.zeros(shape[:2], np.float32)
            oracle.append_int8(self.k, self.v, self.ks, self.vs, w.k_fill, w.v_fill, w.fill_slots)
            if append_step:
                oracle.append_int8(self.k, self.v, self.ks, self.vs, w.k_step, w.v_step,
                                   w.step_slots)
        else:
            dt = np.uint16 if cfg.kv_dtype == "bf16" else np.float16
            self.k = np.zeros(shape, dt)
            self.v = np.zeros(shape, dt)
            self.ks = self.vs = None
            oracle.append_copy(self.k, self.v, w.k_fill, w.v_fill, w.fill_slots)
            if append_step:
                oracle.append_copy(self.k, self.v, w.k_step, w.v_step, w.step_slots)

    def attention(self, seqs=None):
        w = self.w
        return oracle.paged_decode_attention(w.q, self.k, self.v, w.block_tables,
                                             w.context_lens, w.cfg.softmax_scale,
                                             self.ks, self.vs, seqs=seqs)


def error_figures(got, want):
    """max |g - o| and max |g - o| / |o| over the elements with |o| >= 0.2."""
    err = np.abs(got - want)
    big = np.abs(want) >= 0.2
    rel = float((err[big] / np.abs(want[big])).max()) if big.any() else 0.0
    return float(err.max()) if err.size else 0.0, rel


def assert_attention_close(got, want, int8: bool, what=""):
    """Element-wise bound (bf16 / fp16 KV: 2e-3 + 1e-2 |o|; INT8: 2e-2);
    returns (max abs error, max relative error where |o| >= 0.2)."""
    err = np.abs(got - want)
    if int8:
        bad = err > TOL_I8
    else:
        bad = err > TOL_ABS + TOL_REL * np.abs(want)
    max_abs, max_rel = error_figures(got, want)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, first at "
                             f"{tuple(i)}: got {got[tuple(i)]!r} want {want[tuple(i)]!r}; "
                             f"max abs err {max_abs:.3e}, max rel err (|o| >= 0.2) {max_rel:.3e}")
    return max_abs, max_rel


def workload(cfg):
    return make_workload(cfg)

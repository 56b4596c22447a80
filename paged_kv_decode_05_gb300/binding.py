"""Thin ctypes binding over ``libpkv.so`` (argument marshalling only).

Each function has the name of the C entry point it calls (``include/pkv.h``),
takes torch CUDA tensors, passes their device pointers, sizes and the current
CUDA stream, and raises :class:`PkvError` on a non-OK status. All arithmetic
runs in the library's kernels; there is no other code path. If the library
has not been built, loading it raises.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB, up_to_date

PKV_F16, PKV_BF16, PKV_I8 = 0, 1, 2
STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
          3: "PKV_ERR_WORKSPACE", 4: "PKV_ERR_CUDA"}
DEV_BAD_BLOCK, DEV_BAD_LENGTH, DEV_BAD_SLOT, DEV_TIMEOUT, DEV_BAD_INDEX = 1, 2, 4, 8, 16
BLOCK_SIZE = 16


class PkvError(RuntimeError):
    def __init__(self, func, code, msg):
        super().__init__(f"{func}: {msg}")
        self.code = code


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int)]


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_DESC = ctypes.POINTER(CacheDesc)

_SIGS = {
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_append_workspace_size": (_SZ, [_DESC]),
    "pkv_append": (ctypes.c_int, [_P, _P, ctypes.c_int, _I32, _P, _P, _P, _P, _P, _DESC, _P, _SZ,
                                  _P, _P]),
    "pkv_decode_default_parts": (_I32, [_I32, _I32, _I32, _DESC]),
    "pkv_decode_workspace_size": (_SZ, [_I32, _I32, _DESC, _I32]),
    "pkv_decode_attn": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, _P, _DESC, _P, _I32, _P,
                                       _I32, _I32, ctypes.c_float, _P, _P, _SZ, _I32, _P, _P]),
    "pkv_decode_split": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, _P, _DESC, _P, _I32, _P,
                                        _I32, _I32, ctypes.c_float, _P, _P, _SZ, _I32, _P, _P]),
    "pkv_decode_combine": (ctypes.c_int, [_DESC, _I32, _I32, ctypes.c_int, _P, _P, _SZ, _I32, _P]),
    "pkv_decode_step": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, _P, _P, _P, _DESC, _P, _I32,
                                       _P, _I32, _I32, ctypes.c_float, _P, _P, _SZ, _I32, _I32,
                                       _P, _P]),
    "pkv_copy_blocks": (ctypes.c_int, [_P, _P, _P, _P, _DESC, _P, _P, _I32, _P, _P]),
    "pkv_multiquery_workspace_size": (_SZ, [_I32, _I32, _I32, _DESC, _I32]),
    "pkv_multiquery_attn": (ctypes.c_int, [_P, ctypes.c_int, _P, _I32, _P, _P, _P, _P, _DESC, _P,
                                           _I32, _P, _I32, _I32, ctypes.c_float, _P, _P, _SZ,
                                           _I32, _P, _P]),
    "pkv_decode_attn_noalloc": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, _P, _DESC, _P, _I32,
                                               _P, _I32, _I32, ctypes.c_float, _P, _I32, _P, _P]),
    "pkv_merge_states": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64, _P, _I32, _I32, _I32,
                                        ctypes.c_int, _P, _P, _P, _P, _P]),
    # test hooks (include/pkv_testing.h)
    "pkv_testing_decode_attn_stall": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, _P, _DESC, _P,
                                                     _I32, _P, _I32, _I32, ctypes.c_float, _P, _P,
                                                     _SZ, _I32, ctypes.c_uint64, _I32,
                                                     _P, _P]),
    "pkv_testing_multiquery_kernel": (ctypes.c_int, [_I32, _I32, _I32, _DESC, ctypes.c_int, _I32,
                                                     _P, _P]),
    "pkv_testing_multiquery_attn_stall": (ctypes.c_int, [_P, ctypes.c_int, _P, _I32, _P, _P, _P,
                                                         _P, _DESC, _P, _I32, _P, _I32, _I32,
                                                         ctypes.c_float, _P, _P, _SZ, _I32,
                                                         ctypes.c_uint64, _I32, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """Load ``libpkv.so`` once; raise if it is missing or older than its sources."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built: run paged_kv_decode_05_gb300.build.build()")
        if not up_to_date():
            raise RuntimeError(f"{LIB} is older than its sources: rebuild it")
        L = ctypes.CDLL(LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _check(func, code):
    if code != 0:
        raise PkvError(func, code, lib().pkv_status_string(code).decode())


def _dtype_code(t):
    import torch
    m = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.int8: PKV_I8}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def cache_desc(k_cache) -> CacheDesc:
    """Describe a ``[num_blocks, num_kv_heads, 16, head_dim]`` cache tensor."""
    NB, H, bs, D = k_cache.shape
    return CacheDesc(NB, bs, H, D, _dtype_code(k_cache))


def pkv_status_string(code: int) -> str:
    return lib().pkv_status_string(code).decode()


def pkv_append_workspace_size(k_cache) -> int:
    return int(lib().pkv_append_workspace_size(ctypes.byref(cache_desc(k_cache))))


def pkv_append(k_new, v_new, slot_mapping, k_cache, v_cache, k_scales=None, v_scales=None,
               workspace=None, dev_status=None, stream=None):
    """Write ``k_new/v_new [N, Hkv, D]`` to the cache at ``slot_mapping [N] int64``."""
    desc = cache_desc(k_cache)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib().pkv_append(_ptr(k_new), _ptr(v_new), _dtype_code(k_new), int(k_new.shape[0]),
                            _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales),
                            _ptr(v_scales), ctypes.byref(desc), _ptr(workspace), ws_bytes,
                            _ptr(dev_status), _stream(stream))
    _check("pkv_append", code)


def pkv_decode_default_parts(batch, num_q_heads, k_cache, device=None) -> int:
    import torch
    dev = torch.cuda.current_device() if device is None else device
    return int(lib().pkv_decode_default_parts(dev, batch, num_q_heads,
                                              ctypes.byref(cache_desc(k_cache))))


def pkv_decode_workspace_size(batch, num_q_heads, k_cache, num_parts=0) -> int:
    return int(lib().pkv_decode_workspace_size(batch, num_q_heads,
                                               ctypes.byref(cache_desc(k_cache)), num_parts))


def _decode(name, q, k_cache, v_cache, block_tables, context_lens, softmax_scale, out,
            workspace, k_scales, v_scales, num_parts, dev_status, stream):
    desc = cache_desc(k_cache)
    B, Hq, D = q.shape
    code = getattr(lib(), name)(
        _ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
        ctypes.byref(desc), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
        B, Hq, float(softmax_scale), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), int(num_parts), _ptr(dev_status),
        _stream(stream))
    _check(name, code)


def pkv_decode_attn(q, k_cache, v_cache, block_tables, context_lens, softmax_scale, out,
                    workspace, k_scales=None, v_scales=None, num_parts=0, dev_status=None,
                    stream=None):
    """``out [B, Hq, D] = softmax(scale q K^T) V`` over each sequence's paged KV."""
    _decode("pkv_decode_attn", q, k_cache, v_cache, block_tables, context_lens, softmax_scale,
            out, workspace, k_scales, v_scales, num_parts, dev_status, stream)


def pkv_decode_split(q, k_cache, v_cache, block_tables, context_lens, softmax_scale, out,
                     workspace, k_scales=None, v_scales=None, num_parts=0, dev_status=None,
                     stream=None):
    _decode("pkv_decode_split", q, k_cache, v_cache, block_tables, context_lens, softmax_scale,
            out, workspace, k_scales, v_scales, num_parts, dev_status, stream)


def pkv_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, softmax_scale,
                    out, workspace, num_parts=0, dev_status=None, stream=None, run_combine=True,
                    k_scales=None, v_scales=None):
    """Write ``k_new/v_new [B, Hkv, D]`` at each sequence's last position, then attend
    (``run_combine=False``: split phase only; :func:`pkv_decode_combine` must follow).
    INT8 caches take their ``k_scales/v_scales``."""
    desc = cache_desc(k_cache)
    B, Hq, D = q.shape
    code = lib().pkv_decode_step(
        _ptr(q), _dtype_code(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scales), _ptr(v_scales),
        ctypes.byref(desc), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
        B, Hq, float(softmax_scale), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), int(num_parts), int(bool(run_combine)),
        _ptr(dev_status), _stream(stream))
    _check("pkv_decode_step", code)


def pkv_decode_combine(out, k_cache, workspace, num_parts=0, stream=None):
    """Merge the partial states a preceding :func:`pkv_decode_split` left in ``workspace``."""
    desc = cache_desc(k_cache)
    B, Hq, D = out.shape
    code = lib().pkv_decode_combine(ctypes.byref(desc), B, Hq, _dtype_code(out), _ptr(out),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    int(num_parts), _stream(stream))
    _check("pkv_decode_combine", code)


def pkv_copy_blocks(k_cache, v_cache, src_blocks, dst_blocks, k_scales=None, v_scales=None,
                    dev_status=None, stream=None):
    """Copy whole blocks ``src_blocks[i] -> dst_blocks[i]`` (int32 device tensors)."""
    desc = cache_desc(k_cache)
    code = lib().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
                                 ctypes.byref(desc), _ptr(src_blocks), _ptr(dst_blocks),
                                 int(src_blocks.numel()), _ptr(dev_status), _stream(stream))
    _check("pkv_copy_blocks", code)


def pkv_multiquery_workspace_size(batch, num_q_heads, max_q_len, k_cache, num_parts=0) -> int:
    return int(lib().pkv_multiquery_workspace_size(batch, num_q_heads, max_q_len,
                                                   ctypes.byref(cache_desc(k_cache)), num_parts))


def pkv_multiquery_attn(q, cu_q, max_q_len, k_cache, v_cache, block_tables, context_lens,
                        softmax_scale, out, workspace, num_parts=0, dev_status=None, stream=None,
                        k_scales=None, v_scales=None):
    """Causal attention of ``cu_q``-delimited new queries ``q [total_q, Hq, D]``
    (``k_scales``, ``v_scales``: INT8 caches only)."""
    desc = cache_desc(k_cache)
    code = lib().pkv_multiquery_attn(
        _ptr(q), _dtype_code(q), _ptr(cu_q), int(max_q_len), _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scales), _ptr(v_scales), ctypes.byref(desc), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(context_lens),
        int(cu_q.numel() - 1), int(q.shape[1]), float(softmax_scale), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), int(num_parts), _ptr(dev_status),
        _stream(stream))
    _check("pkv_multiquery_attn", code)


def pkv_decode_attn_noalloc(q, k_cache, v_cache, block_tables, context_lens, softmax_scale, out,
                            k_scales=None, v_scales=None, num_parts=0, dev_status=None,
                            stream=None):
    """:func:`pkv_decode_attn` using the library's built-in scratch array.

    For callers that cannot allocate device memory: no workspace is passed and
    nothing is allocated. Raises PkvError(PKV_ERR_WORKSPACE) when the sizes
    need more scratch than the built-in array holds.
    """
    desc = cache_desc(k_cache)
    B, Hq, D = q.shape
    code = lib().pkv_decode_attn_noalloc(
        _ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
        ctypes.byref(desc), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
        B, Hq, float(softmax_scale), _ptr(out), int(num_parts), _ptr(dev_status),
        _stream(stream))
    _check("pkv_decode_attn_noalloc", code)


def pkv_merge_states(part_m, part_l, part_o, row_ptr, out, out_m=None, out_l=None,
                     dev_status=None, stream=None):
    """Merge partial states ``(m, l, o)`` (``[S, H]``, ``[S, H]``, ``[S, H, D]`` fp32):
    row ``r`` of ``out [R, H, D]`` merges states ``row_ptr[r] .. row_ptr[r+1]-1``."""
    S, H, D = part_o.shape
    R = int(row_ptr.numel()) - 1
    code = lib().pkv_merge_states(_ptr(part_m), _ptr(part_l), _ptr(part_o), int(S),
                                  _ptr(row_ptr), R, int(H), int(D), _dtype_code(out), _ptr(out),
                                  _ptr(out_m), _ptr(out_l), _ptr(dev_status), _stream(stream))
    _check("pkv_merge_states", code)


def pkv_testing_decode_attn_stall(q, k_cache, v_cache, block_tables, context_lens, softmax_scale,
                                  out, workspace, wait_limit_ns, stall_worker, k_scales=None,
                                  v_scales=None, num_parts=0, dev_status=None, stream=None):
    """Test hook: :func:`pkv_decode_attn` whose worker ``stall_worker`` never completes
    the wait for its first unit (bounded by ``wait_limit_ns``); see ``include/pkv_testing.h``."""
    desc = cache_desc(k_cache)
    B, Hq, D = q.shape
    code = lib().pkv_testing_decode_attn_stall(
        _ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
        ctypes.byref(desc), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
        B, Hq, float(softmax_scale), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), int(num_parts), int(wait_limit_ns),
        int(stall_worker), _ptr(dev_status), _stream(stream))
    _check("pkv_testing_decode_attn_stall", code)


def pkv_testing_multiquery_attn_stall(q, cu_q, max_q_len, k_cache, v_cache, block_tables,
                                      context_lens, softmax_scale, out, workspace, wait_limit_ns,
                                      stall_cta, num_parts=0, dev_status=None, stream=None,
                                      k_scales=None, v_scales=None):
    """Test hook: :func:`pkv_multiquery_attn` whose CTA ``stall_cta`` stalls."""
    desc = cache_desc(k_cache)
    code = lib().pkv_testing_multiquery_attn_stall(
        _ptr(q), _dtype_code(q), _ptr(cu_q), int(max_q_len), _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scales), _ptr(v_scales), ctypes.byref(desc), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(context_lens),
        int(cu_q.numel() - 1), int(q.shape[1]), float(softmax_scale), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), int(num_parts), int(wait_limit_ns),
        int(stall_cta), _ptr(dev_status), _stream(stream))
    _check("pkv_testing_multiquery_attn_stall", code)


MQ_KERNELS = {0: "mq_tc_kernel", 1: "mqt_split_kernel", 2: "mqt_i8_split_kernel",
              3: "mq_split_kernel"}


def pkv_testing_multiquery_kernel(batch, num_q_heads, max_q_len, desc, q_dtype, num_parts=16):
    """Test hook: (kernel name, rows per tile) that pkv_multiquery_attn runs for
    these sizes, from the library's own planner (no GPU needed)."""
    kernel, rt = ctypes.c_int32(-1), ctypes.c_int32(0)
    code = lib().pkv_testing_multiquery_kernel(int(batch), int(num_q_heads), int(max_q_len),
                                               ctypes.byref(desc), int(q_dtype), int(num_parts),
                                               ctypes.byref(kernel), ctypes.byref(rt))
    _check("pkv_testing_multiquery_kernel", code)
    return MQ_KERNELS[kernel.value], rt.value

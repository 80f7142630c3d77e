"""GB300 tree-verify attention: Python binding of the C ABI in include/tree_attn.h.

Every function here only marshals arguments (torch tensors -> pointer, byte
count, dtype code; the current CUDA stream) into the C library; all work runs
in the library's CUDA kernels.  Importing this module loads the in-tree
``_build/libtree_attn.so`` (compiling it first when it is missing or older than
its sources) and raises if that fails: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build_mod

__all__ = [
    "TA_OK", "TreeParams", "QuantParams", "TreeAttentionError", "lib", "library_path",
    "tree_attn_tmp_bytes", "tree_attn_num_splits", "tree_attn_workspace_bytes", "tree_attn_fwd",
    "tree_attn_fwd_causal", "tree_attn_fwd_parents", "tree_attn_fwd_ex", "tree_attn_status_offset",
    "tree_attn_reduce", "tree_attn_fwd_noalloc", "quant_sdpa_num_splits", "quant_sdpa_tmp_bytes",
    "quant_sdpa_fwd", "ta_last_error", "ta_launch_count", "quant_sdpa_uses_tensor_cores",
    "quant_sdpa_kernel_family", "KERNEL_WARP_MMA",
    "ta_test_quant_sdpa_fwd_wait_limit", "quant_sdpa_fwd_tree", "tree_attention", "quant_sdpa", "tree_params", "quant_params",
    "tree_mask_build", "TreeOptions", "KERNEL_AUTO", "KERNEL_CUDA_CORES", "KERNEL_TENSOR_CORES",
]

TA_OK = 0
TA_F32, TA_F16, TA_BF16, TA_U32, TA_I32 = 0, 1, 2, 3, 4
KERNEL_AUTO, KERNEL_CUDA_CORES, KERNEL_TENSOR_CORES, KERNEL_WARP_MMA = 0, 1, 2, 3
MASK_DENSE, MASK_CAUSAL, MASK_PARENTS = 0, 1, 2
STATUS_NAMES = {0: "TA_OK", 1: "TA_ERR_INVALID_ARGUMENT", 2: "TA_ERR_BUFFER_TOO_SMALL",
                3: "TA_ERR_OVERFLOW", 4: "TA_ERR_UNSUPPORTED", 5: "TA_ERR_CUDA"}


class TreeAttentionError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class Buf(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("bytes", ctypes.c_uint64), ("dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class TreeParams(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_uint32), ("n_kv_heads", ctypes.c_uint32),
                ("head_dim", ctypes.c_uint32), ("kv_seq_len", ctypes.c_uint32),
                ("kv_capacity", ctypes.c_uint32), ("scale", ctypes.c_float), ("nwg", ctypes.c_uint32),
                ("q_l", ctypes.c_uint32), ("mask_stride", ctypes.c_uint32)]


class QuantParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_uint32), ("n_q_heads", ctypes.c_uint32),
                ("n_kv_heads", ctypes.c_uint32), ("dim", ctypes.c_uint32), ("tokens", ctypes.c_uint32),
                ("bits", ctypes.c_uint32), ("group_size", ctypes.c_uint32),
                ("has_sinks", ctypes.c_uint32), ("window_size", ctypes.c_uint32),
                ("scale", ctypes.c_float), ("nwg", ctypes.c_uint32), ("kernel", ctypes.c_uint32)]


class TreeOptions(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("mask_kind", ctypes.c_int32), ("window_start", ctypes.c_uint32),
                ("reserved", ctypes.c_int32)]


def library_path() -> str:
    return _build_mod.LIB


def _load() -> ctypes.CDLL:
    # (Re)build the in-tree library when it is missing or older than its
    # sources; a failed build raises, so the package never imports without it.
    path = _build_mod.build()
    if not os.path.exists(path):
        raise ImportError("tree_masked_speculative_gb300: %s is missing" % path)
    L = ctypes.CDLL(path)
    P, B = ctypes.c_void_p, ctypes.POINTER(Buf)
    PT, PQ = ctypes.POINTER(TreeParams), ctypes.POINTER(QuantParams)
    u32 = ctypes.c_uint32
    L.tree_attn_tmp_bytes.argtypes = [u32, u32, u32, u32]
    L.tree_attn_tmp_bytes.restype = ctypes.c_size_t
    L.tree_attn_num_splits.argtypes = [PT]
    L.tree_attn_num_splits.restype = u32
    L.tree_attn_workspace_bytes.argtypes = [PT]
    L.tree_attn_workspace_bytes.restype = ctypes.c_size_t
    L.tree_attn_fwd.argtypes = [PT, B, B, B, B, B, B, P]
    L.tree_attn_fwd.restype = ctypes.c_int
    L.tree_attn_fwd_causal.argtypes = [PT, u32, B, B, B, B, B, P]
    L.tree_attn_fwd_causal.restype = ctypes.c_int
    L.tree_attn_fwd_parents.argtypes = [PT, B, B, B, B, B, B, P]
    L.tree_attn_fwd_parents.restype = ctypes.c_int
    L.tree_attn_fwd_ex.argtypes = [PT, ctypes.POINTER(TreeOptions), B, B, B, B, B, B, P]
    L.tree_attn_fwd_ex.restype = ctypes.c_int
    L.tree_attn_status_offset.argtypes = [PT]
    L.tree_attn_status_offset.restype = ctypes.c_size_t
    L.tree_attn_reduce.argtypes = [PT, B, B, P]
    L.tree_attn_reduce.restype = ctypes.c_int
    L.tree_attn_fwd_noalloc.argtypes = [PT, B, B, B, B, B, P]
    L.tree_attn_fwd_noalloc.restype = ctypes.c_int
    L.quant_sdpa_num_splits.argtypes = [PQ]
    L.quant_sdpa_num_splits.restype = u32
    L.quant_sdpa_tmp_bytes.argtypes = [PQ]
    L.quant_sdpa_tmp_bytes.restype = ctypes.c_size_t
    L.quant_sdpa_fwd.argtypes = [PQ] + [B] * 12 + [P]
    L.quant_sdpa_fwd.restype = ctypes.c_int
    L.ta_last_error.argtypes = []
    L.ta_last_error.restype = ctypes.c_char_p
    L.ta_launch_count.argtypes = []
    L.ta_launch_count.restype = ctypes.c_uint64
    L.quant_sdpa_fwd_tree.argtypes = [PQ, u32] + [B] * 12 + [P]
    L.quant_sdpa_fwd_tree.restype = ctypes.c_int
    L.ta_test_quant_sdpa_fwd_wait_limit.argtypes = [u32, PQ] + [B] * 12 + [P]
    L.ta_test_quant_sdpa_fwd_wait_limit.restype = ctypes.c_int
    L.quant_sdpa_uses_tensor_cores.argtypes = [PQ]
    L.quant_sdpa_uses_tensor_cores.restype = ctypes.c_int
    L.quant_sdpa_kernel_family.argtypes = [PQ]
    L.quant_sdpa_kernel_family.restype = ctypes.c_int
    L.tree_mask_build.argtypes = [PT, B, B, P]
    L.tree_mask_build.restype = ctypes.c_int
    return L


lib = _load()

_DTYPE_CODE = {torch.float32: TA_F32, torch.float16: TA_F16, torch.bfloat16: TA_BF16,
               torch.int32: TA_U32}
_U32 = getattr(torch, "uint32", None)
if _U32 is not None:
    _DTYPE_CODE[_U32] = TA_U32


def buf(t: Optional[torch.Tensor], dtype_code: Optional[int] = None):
    """Describe a tensor as a ta_buf passed by reference; None = absent buffer
    (a NULL descriptor).  int32 tensors are passed as U32 (packed words, bool
    masks)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    code = _DTYPE_CODE.get(t.dtype) if dtype_code is None else dtype_code
    if code is None:
        raise ValueError("unsupported dtype %s" % t.dtype)
    return ctypes.byref(Buf(t.data_ptr(), t.numel() * t.element_size(), code, 0))


def raw_buf(ptr: int, nbytes: int, dtype_code: int) -> Buf:
    return Buf(ptr, nbytes, dtype_code, 0)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int):
    if status != TA_OK:
        raise TreeAttentionError(status, lib.ta_last_error().decode())


def ta_last_error() -> str:
    return lib.ta_last_error().decode()


def ta_launch_count() -> int:
    return int(lib.ta_launch_count())


def quant_sdpa_uses_tensor_cores(p: QuantParams) -> int:
    return int(lib.quant_sdpa_uses_tensor_cores(ctypes.byref(p)))


def quant_sdpa_kernel_family(p: QuantParams) -> int:
    return int(lib.quant_sdpa_kernel_family(ctypes.byref(p)))


def tree_params(n_heads, n_kv_heads, head_dim, kv_seq_len, kv_capacity, scale, q_l, mask_stride,
                nwg=0) -> TreeParams:
    return TreeParams(n_heads, n_kv_heads, head_dim, kv_seq_len, kv_capacity, scale, nwg, q_l,
                      mask_stride)


def quant_params(batch, n_q_heads, n_kv_heads, dim, tokens, bits, group_size, has_sinks,
                 window_size, scale, nwg=0, kernel=KERNEL_AUTO) -> QuantParams:
    return QuantParams(batch, n_q_heads, n_kv_heads, dim, tokens, bits, group_size, has_sinks,
                       window_size, scale, nwg, kernel)


def tree_attn_tmp_bytes(n_heads: int, head_dim: int, q_l: int, nwg: int) -> int:
    return int(lib.tree_attn_tmp_bytes(n_heads, head_dim, q_l, nwg))


def tree_attn_num_splits(p: TreeParams) -> int:
    return int(lib.tree_attn_num_splits(ctypes.byref(p)))


def tree_attn_workspace_bytes(p: TreeParams) -> int:
    return int(lib.tree_attn_workspace_bytes(ctypes.byref(p)))


def tree_attn_fwd(p: TreeParams, q, k, v, mask, tmp, out, stream=None):
    _check(lib.tree_attn_fwd(ctypes.byref(p), buf(q), buf(k), buf(v), buf(mask), buf(tmp),
                             buf(out), _stream(stream)))


def tree_attn_fwd_parents(p: TreeParams, parents, q, k, v, tmp, out, stream=None):
    _check(lib.tree_attn_fwd_parents(ctypes.byref(p), buf(parents, TA_I32), buf(q), buf(k), buf(v), buf(tmp),
                                     buf(out), _stream(stream)))


def tree_attn_fwd_causal(p: TreeParams, window_start: int, q, k, v, tmp, out, stream=None):
    _check(lib.tree_attn_fwd_causal(ctypes.byref(p), window_start, buf(q), buf(k), buf(v),
                                    buf(tmp), buf(out), _stream(stream)))


def tree_attn_fwd_ex(p: TreeParams, kernel: int, mask_kind: int, window_start: int, q, k, v, mask, tmp, out,
                     stream=None):
    """Main pass with an explicit kernel family (KERNEL_*) and mask form (MASK_*:
    `mask` is the dense mask, unused, or the int32 parent array)."""
    o = TreeOptions(kernel, mask_kind, window_start, 0)
    m = buf(mask, TA_I32) if mask_kind == MASK_PARENTS else (buf(mask) if mask_kind == MASK_DENSE else None)
    _check(lib.tree_attn_fwd_ex(ctypes.byref(p), ctypes.byref(o), buf(q), buf(k), buf(v), m, buf(tmp), buf(out),
                                _stream(stream)))


def tree_attn_status_offset(p: TreeParams) -> int:
    return int(lib.tree_attn_status_offset(ctypes.byref(p)))


def tree_attn_reduce(p: TreeParams, tmp, out, stream=None):
    _check(lib.tree_attn_reduce(ctypes.byref(p), buf(tmp), buf(out), _stream(stream)))


def tree_attn_fwd_noalloc(p: TreeParams, q, k, v, mask, out, stream=None):
    """Main pass + merge with the library's static scratch (no tmp buffer); for
    callers that cannot allocate device memory.  mask=None: implicit causal."""
    _check(lib.tree_attn_fwd_noalloc(ctypes.byref(p), buf(q), buf(k), buf(v), buf(mask), buf(out),
                                     _stream(stream)))


def quant_sdpa_num_splits(p: QuantParams) -> int:
    return int(lib.quant_sdpa_num_splits(ctypes.byref(p)))


def quant_sdpa_tmp_bytes(p: QuantParams) -> int:
    return int(lib.quant_sdpa_tmp_bytes(ctypes.byref(p)))


def _quant_bufs(queries, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, sinks, mask_bool,
                mask_float, tmp, out):
    return (buf(queries), buf(k_packed, TA_U32), buf(k_scales), buf(k_biases), buf(v_packed, TA_U32),
            buf(v_scales), buf(v_biases), buf(sinks), buf(mask_bool, TA_U32) if mask_bool is not None else None,
            buf(mask_float), buf(tmp), buf(out))


def quant_sdpa_fwd(p: QuantParams, queries, k_packed, k_scales, k_biases, v_packed, v_scales,
                   v_biases, sinks, mask_bool, mask_float, tmp, out, stream=None):
    _check(lib.quant_sdpa_fwd(ctypes.byref(p), *_quant_bufs(queries, k_packed, k_scales, k_biases, v_packed,
                                                            v_scales, v_biases, sinks, mask_bool, mask_float,
                                                            tmp, out), _stream(stream)))


def quant_sdpa_fwd_tree(p: QuantParams, q_l: int, parents, queries, k_packed, k_scales, k_biases, v_packed,
                        v_scales, v_biases, sinks, mask_bool, tmp, out, stream=None):
    """Quantized-KV attention of draft-tree rows (row q = node q % q_l) with the
    tree mask as the int32 parent array of the last q_l tokens."""
    b = _quant_bufs(queries, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, sinks, mask_bool, None,
                    tmp, out)
    _check(lib.quant_sdpa_fwd_tree(ctypes.byref(p), q_l, buf(parents, TA_I32), *b[:9], b[10], b[11],
                                   _stream(stream)))


def ta_test_quant_sdpa_fwd_wait_limit(first_wait_polls: int, p: QuantParams, queries, k_packed, k_scales,
                                      k_biases, v_packed, v_scales, v_biases, sinks, mask_bool, mask_float, tmp,
                                      out, stream=None):
    """Test hook: quant_sdpa_fwd (CUDA-core kernel) whose first copy wait per CTA
    gives up after `first_wait_polls` polls (0: at once)."""
    _check(lib.ta_test_quant_sdpa_fwd_wait_limit(first_wait_polls, ctypes.byref(p),
                                                 *_quant_bufs(queries, k_packed, k_scales, k_biases, v_packed,
                                                              v_scales, v_biases, sinks, mask_bool, mask_float,
                                                              tmp, out), _stream(stream)))


# ------------------------------------------------------------- conveniences
def tree_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: Optional[torch.Tensor],
                   *, n_heads: int, n_kv_heads: int, kv_seq_len: int, scale: float,
                   mask_stride: Optional[int] = None, nwg: int = 0, window_start: int = 0,
                   tmp: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   parents: Optional[torch.Tensor] = None, kernel: int = KERNEL_AUTO,
                   stream=None) -> torch.Tensor:
    """One verify step (main pass + reduce) on device tensors.  mask=None uses the
    implicit causal mask starting at window_start, or, with `parents` (int32
    [q_l] on the device), the tree mask of that parent array.  `kernel` picks
    the main pass's kernel family (KERNEL_*).  Returns out [q_l, n_heads, D]."""
    H, L, D = q.shape
    C = k.shape[1]
    stride = mask_stride if mask_stride is not None else (mask.shape[1] if mask is not None else kv_seq_len)
    p = tree_params(n_heads, n_kv_heads, D, kv_seq_len, C, scale, L, stride, nwg)
    if tmp is None:
        ws = tree_attn_workspace_bytes(p)
        if ws >= 2 ** 63:
            raise TreeAttentionError(1, "invalid tree-attention parameters")
        tmp = torch.empty((ws + 3) // 4, dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty((L, n_heads, D), dtype=torch.float32, device=q.device)
    if parents is not None:
        if mask is not None:
            raise ValueError("give either a dense mask or a parent array, not both")
        tree_attn_fwd_ex(p, kernel, MASK_PARENTS, 0, q, k, v, parents, tmp, out, stream)
    elif mask is None:
        tree_attn_fwd_ex(p, kernel, MASK_CAUSAL, window_start, q, k, v, None, tmp, out, stream)
    else:
        tree_attn_fwd_ex(p, kernel, MASK_DENSE, 0, q, k, v, mask, tmp, out, stream)
    tree_attn_reduce(p, tmp, out, stream)
    return out


def quant_sdpa(inputs: dict, *, batch: int, n_q_heads: int, n_kv_heads: int, dim: int, tokens: int,
               bits: int, group_size: int, has_sinks: int, window_size: int, scale: float,
               nwg: int = 0, out_dtype: Optional[torch.dtype] = None, tmp=None, out=None,
               kernel: int = KERNEL_AUTO, tree_parents: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """Quantized-KV attention on device tensors (dict as made by workloads.make_quant_inputs).
    With `tree_parents` (int32 [q_l] on the device) the rows are draft-tree nodes
    (row q = node q % q_l) masked by that tree over the last q_l tokens, and the
    dict's float mask is not used."""
    p = quant_params(batch, n_q_heads, n_kv_heads, dim, tokens, bits, group_size, has_sinks,
                     window_size, scale, nwg, kernel)
    dev = inputs["queries"].device
    if tmp is None:
        nb = quant_sdpa_tmp_bytes(p)
        if nb >= 2 ** 63:
            raise TreeAttentionError(1, "invalid quantized-SDPA parameters")
        tmp = torch.zeros(max(1, (nb + 3) // 4), dtype=torch.float32, device=dev)   # error word = 0
    if out is None:
        out = torch.empty((batch * n_q_heads, dim), dtype=out_dtype or inputs["queries"].dtype,
                          device=dev)
    if tree_parents is not None:
        quant_sdpa_fwd_tree(p, int(tree_parents.numel()), tree_parents, inputs["queries"], inputs["k_packed"],
                            inputs["k_scales"], inputs["k_biases"], inputs["v_packed"], inputs["v_scales"],
                            inputs["v_biases"], inputs["sinks"] if has_sinks else None, inputs.get("mask_bool"),
                            tmp, out, stream)
        return out
    quant_sdpa_fwd(p, inputs["queries"], inputs["k_packed"], inputs["k_scales"], inputs["k_biases"],
                   inputs["v_packed"], inputs["v_scales"], inputs["v_biases"],
                   inputs["sinks"] if has_sinks else None, inputs.get("mask_bool"),
                   inputs.get("mask_float"), tmp, out, stream)
    return out


def tree_mask_build(p: TreeParams, parents: torch.Tensor, mask: torch.Tensor, stream=None):
    """Dense tree mask [q_l, mask_stride] f32 from parents [q_l] int32, on the device."""
    _check(lib.tree_mask_build(ctypes.byref(p), buf(parents, TA_I32), buf(mask), _stream(stream)))

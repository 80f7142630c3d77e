"""Float64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product library never does,
and this package never imports the product library.

The arithmetic lives in ``oracle.c`` (plain C, binary64, no blocking or
fusion); this module compiles it with gcc on first use and marshals numpy /
torch-CPU arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library next to it (plain gcc, no -march)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_tree_attention.argtypes = [I, I, I, I, I, ctypes.c_double, I, I, P, P, P, I,
                                                  P, I, I, P, P, I]
            lib.oracle_tree_attention.restype = I
            lib.oracle_quant_sdpa.argtypes = [I, I, I, I, I, I, I, I, I, ctypes.c_double, I, P,
                                              P, P, P, P, P, P, P, P, P, I, P, P, I]
            lib.oracle_quant_sdpa.restype = I
            lib.oracle_decode.argtypes = [I, ctypes.c_int64, P, P]
            lib.oracle_decode.restype = None
            lib.oracle_dequant_token.argtypes = [I, I, I, I, I, P, P, P, I, I, P]
            lib.oracle_dequant_token.restype = I
            lib.oracle_tree_mask.argtypes = [P, I, I, I, P]
            lib.oracle_tree_mask.restype = I
            _lib = lib
    return _lib


def _np(x) -> Optional[np.ndarray]:
    """torch CPU tensor / numpy array -> contiguous numpy array (raw bits kept)."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype in (torch.float16, torch.bfloat16):
                return x.view(torch.int16).numpy().view(np.uint16)
            if x.dtype == torch.int32:
                return x.numpy().view(np.uint32)
            return x.numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(x)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def decode(dtype: str, raw) -> np.ndarray:
    """Widen raw f32 / f16 / bf16 storage to float64 with the oracle's own decoder."""
    a = _np(raw)
    out = np.empty(a.size, dtype=np.float64)
    _load().oracle_decode(DTYPE_CODES[dtype], a.size, _ptr(a), _ptr(out))
    return out.reshape(a.shape)


def tree_attention(q, k, v, mask, *, n_heads: int, n_kv_heads: int, head_dim: int,
                   kv_seq_len: int, kv_capacity: int, scale: float, q_l: int,
                   mask_stride: int, kv_dtype: str, window_start: int = 0,
                   rows: Optional[Sequence[tuple]] = None,
                   threads: Optional[int] = None) -> np.ndarray:
    """Masked softmax attention in float64.

    q [n_heads, q_l, D] f32; k, v [n_kv_heads, kv_capacity, D]; mask
    [q_l, mask_stride] f32 or None for the implicit causal mask (row i attends
    [window_start, kv_seq_len - q_l + i]).  Returns [q_l, n_heads, D] float64,
    or [len(rows), D] for rows given as (h, i) pairs.
    """
    qa = _np(q).astype(np.float32, copy=False)
    ka, va = _np(k), _np(v)
    ma = None if mask is None else _np(mask).astype(np.float32, copy=False)
    sel = None
    if rows is not None:
        sel = np.asarray([h * q_l + i for (h, i) in rows], dtype=np.int32)
        out = np.empty((len(sel), head_dim), dtype=np.float64)
    else:
        out = np.empty((q_l, n_heads, head_dim), dtype=np.float64)
    rc = _load().oracle_tree_attention(
        n_heads, n_kv_heads, head_dim, kv_seq_len, kv_capacity, float(scale), q_l, mask_stride,
        _ptr(qa), _ptr(ka), _ptr(va), DTYPE_CODES[kv_dtype], _ptr(ma), window_start,
        0 if sel is None else len(sel), _ptr(sel), _ptr(out), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_tree_attention: bad shapes")
    return out


def quant_sdpa(inputs: dict, *, batch: int, n_q_heads: int, n_kv_heads: int, dim: int,
               tokens: int, bits: int, group_size: int, has_sinks: int, window_size: int,
               scale: float, dtype: str, rows: Optional[Sequence[int]] = None,
               threads: Optional[int] = None) -> np.ndarray:
    """Attention over the affine-quantized cache in float64: [B*nQ, dim] or [len(rows), dim]."""
    a = {k: _np(v) for k, v in inputs.items()}
    sel = None if rows is None else np.asarray(list(rows), dtype=np.int32)
    n = batch * n_q_heads if sel is None else len(sel)
    out = np.empty((n, dim), dtype=np.float64)
    sinks = a.get("sinks")
    if sinks is None:
        sinks = np.zeros(n_q_heads, dtype=np.float32)
    sinks = sinks.astype(np.float32, copy=False)
    rc = _load().oracle_quant_sdpa(
        batch, n_q_heads, n_kv_heads, dim, tokens, bits, group_size, has_sinks, window_size,
        float(scale), DTYPE_CODES[dtype], _ptr(a["queries"]), _ptr(a["k_packed"]),
        _ptr(a["k_scales"]), _ptr(a["k_biases"]), _ptr(a["v_packed"]), _ptr(a["v_scales"]),
        _ptr(a["v_biases"]), _ptr(sinks), _ptr(a.get("mask_bool")), _ptr(a.get("mask_float")),
        0 if sel is None else len(sel), _ptr(sel), _ptr(out), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_quant_sdpa: bad shapes")
    return out


def dequant_token(packed, scales, biases, *, dim: int, tokens: int, bits: int,
                  group_size: int, dtype: str, kv: int, t: int) -> np.ndarray:
    """The oracle's dequantized values of token t of KV row kv."""
    p, s, b = _np(packed), _np(scales), _np(biases)
    out = np.empty(dim, dtype=np.float64)
    _load().oracle_dequant_token(dim, tokens, bits, group_size, DTYPE_CODES[dtype], _ptr(p),
                                 _ptr(s), _ptr(b), kv, t, _ptr(out))
    return out


def tree_oracle_for(wl, inp: dict, rows=None, mask="explicit", window_start: int = 0,
                    threads=None) -> np.ndarray:
    """Convenience: oracle for a workloads.TreeWorkload and its generated inputs."""
    return tree_attention(inp["q"], inp["k"], inp["v"], None if mask is None else inp["mask"],
                          n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim,
                          kv_seq_len=wl.kv_seq_len, kv_capacity=wl.kv_capacity, scale=wl.scale,
                          q_l=wl.q_l, mask_stride=wl.mask_stride, kv_dtype=wl.kv_dtype,
                          window_start=window_start, rows=rows, threads=threads)


def quant_oracle_for(wl, inp: dict, rows=None, threads=None) -> np.ndarray:
    """Convenience: oracle for a workloads.QuantWorkload and its generated inputs."""
    return quant_sdpa(inp, batch=wl.batch, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads,
                      dim=wl.dim, tokens=wl.tokens, bits=wl.bits, group_size=wl.group_size,
                      has_sinks=wl.has_sinks, window_size=wl.window_size, scale=wl.scale,
                      dtype=wl.dtype, rows=rows, threads=threads)


def tree_mask(parents, *, kv_seq_len: int, mask_stride: int) -> np.ndarray:
    """Dense tree mask [q_l, mask_stride] f32 (0 / -65504) from a parent array
    (oracle_tree_mask in oracle.c)."""
    par = np.ascontiguousarray(np.asarray(parents, dtype=np.int32))
    q_l = int(par.shape[0])
    out = np.empty((q_l, mask_stride), dtype=np.float32)
    st = _load().oracle_tree_mask(_ptr(par), q_l, kv_seq_len, mask_stride, _ptr(out))
    if st != 0:
        raise ValueError("oracle_tree_mask: invalid sizes (status %d)" % st)
    return out

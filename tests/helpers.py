"""Shared helpers of the GPU tests: run the library on workload inputs and
compare with the float64 oracle under the stated tolerance."""
import math

import numpy as np
import torch

import oracle
import workloads as W

# Tolerance for f32 outputs: |gpu - ref| <= ATOL + RTOL * |ref| per element.
ATOL = 2e-3
RTOL = 1e-3


def assert_close(got, ref, atol=ATOL, rtol=RTOL, extra_ulp_dtype=None, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    tol = atol + rtol * np.abs(ref)
    if extra_ulp_dtype is not None:
        tol = tol + ulp(ref, extra_ulp_dtype)
    err = np.abs(got - ref)
    bad = err > tol
    if np.any(bad):
        idx = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError("%s: %d of %d elements out of tolerance; worst at %s: got %r ref %r "
                             "(max abs err %.3g)" % (what, int(bad.sum()), bad.size, idx, got[idx],
                                                     ref[idx], float(err.max())))
    return float(err.max())


def ulp(x, dtype: str):
    """One unit in the last place of |x| in f16 / bf16 (for outputs stored in T)."""
    mant = {"f16": 10, "bf16": 7}[dtype]
    ax = np.maximum(np.abs(x), 1e-30)
    e = np.floor(np.log2(ax))
    e = np.maximum(e, -14 if dtype == "f16" else -126)
    return np.power(2.0, e - mant)


def to_dev(inp: dict, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_tree(ta, wl: W.TreeWorkload, inp: dict, *, causal=False, window_start=0, nwg=None, kernel=0):
    d = to_dev(inp)
    out = ta.tree_attention(d["q"], d["k"], d["v"], None if causal else d["mask"],
                            n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads, kv_seq_len=wl.kv_seq_len,
                            scale=wl.scale, mask_stride=wl.mask_stride,
                            nwg=wl.nwg if nwg is None else nwg, window_start=window_start, kernel=kernel)
    torch.cuda.synchronize()
    return out


def run_quant(ta, wl: W.QuantWorkload, inp: dict, *, nwg=None, out_dtype=None, kernel=0):
    d = to_dev(inp)
    out = ta.quant_sdpa(d, batch=wl.batch, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads,
                        dim=wl.dim, tokens=wl.tokens, bits=wl.bits, group_size=wl.group_size,
                        has_sinks=wl.has_sinks, window_size=wl.window_size, scale=wl.scale,
                        nwg=wl.nwg if nwg is None else nwg, out_dtype=out_dtype, kernel=kernel)
    torch.cuda.synchronize()
    return out


def small_tree(name="small", H=4, Hk=2, D=128, N=200, C=256, L=5, stride=None, kv_dtype="f16",
               topology="dynamic", seed=7, nwg=0, kv_std=1.0, scale=None) -> W.TreeWorkload:
    return W.TreeWorkload(name=name, n_heads=H, n_kv_heads=Hk, head_dim=D, kv_seq_len=N,
                          kv_capacity=C, q_l=L, mask_stride=stride or N,
                          scale=scale if scale is not None else 1.0 / math.sqrt(D),
                          kv_dtype=kv_dtype, topology=topology, branching=(3, 2, 2, 1, 1),
                          kv_std=kv_std, nwg=nwg, seed=seed)

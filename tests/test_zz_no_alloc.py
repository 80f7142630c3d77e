"""The allocation-free verify step (tree_attn_fwd_noalloc), called through the
C ABI, against the regular entry points (tree_attn_fwd + tree_attn_reduce with
a caller tmp buffer).

tree_attn_fwd_noalloc exists for callers that cannot allocate device memory
when they run the verify step (engines that plan every device byte up front,
plugins inside a framework that owns the allocator, decode loops that cannot
take an allocation's synchronization).  It keeps its scratch in a static
16 MiB device array, so it is checked here on two calls in a row (the second
call sees the first call's leftovers) and on a request that does not fit.
This file runs last so that a failure here leaves every other test already run.
"""
import ctypes

import pytest
import torch

import workloads as W
from helpers import ATOL, RTOL, assert_close, small_tree, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tree_masked_speculative_gb300 as m
    return m


def _regular(ta, p, d, causal):
    ws = ta.tree_attn_workspace_bytes(p)
    tmp = torch.empty((ws + 3) // 4, dtype=torch.float32, device="cuda")
    out = torch.empty((p.q_l, p.n_heads, p.head_dim), dtype=torch.float32, device="cuda")
    if causal:
        ta.tree_attn_fwd_causal(p, 0, d["q"], d["k"], d["v"], tmp, out)
    else:
        ta.tree_attn_fwd(p, d["q"], d["k"], d["v"], d["mask"], tmp, out)
    ta.tree_attn_reduce(p, tmp, out)
    torch.cuda.synchronize()
    return out


def _noalloc(ta, p, d, causal):
    out = torch.full((p.q_l, p.n_heads, p.head_dim), float("nan"), device="cuda")
    st = ta.lib.tree_attn_fwd_noalloc(
        ctypes.byref(p), ta.buf(d["q"]), ta.buf(d["k"]), ta.buf(d["v"]),
        None if causal else ta.buf(d["mask"]), ta.buf(out),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ta.TA_OK, ta.ta_last_error()
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("wl,causal", [
    (W.PR1_CHAIN, False),
    (W.PR1_CHAIN, True),
    (small_tree(H=24, Hk=4, D=256, N=1500, C=2048, L=32, kv_dtype="f16", nwg=8), False),
    (small_tree(H=8, Hk=2, D=512, N=700, C=700, L=6, kv_dtype="bf16", nwg=5, seed=11), False),
], ids=["pr1", "pr1_causal", "tree_d256_f16", "tree_d512_bf16"])
def test_noalloc_matches_regular_entry_points_twice(ta, wl, causal):
    inp = W.make_tree_inputs(wl)
    d = to_dev(inp)
    p = ta.tree_params(wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.kv_seq_len, wl.kv_capacity,
                       wl.scale, wl.q_l, wl.mask_stride, wl.nwg)
    assert ta.tree_attn_workspace_bytes(p) <= 16 << 20
    ref = _regular(ta, p, d, causal).cpu().numpy()
    for _ in range(2):
        got = _noalloc(ta, p, d, causal).cpu().numpy()
        assert_close(got, ref, atol=ATOL, rtol=RTOL, what="noalloc vs regular")


def test_noalloc_after_a_different_shape_reuses_scratch(ta):
    big = small_tree(H=16, Hk=2, D=256, N=900, C=900, L=12, kv_dtype="bf16", nwg=6, seed=3)
    small = small_tree(H=4, Hk=2, D=128, N=100, C=128, L=3, kv_dtype="f16", nwg=2, seed=4)
    for wl in (big, small, big):
        d = to_dev(W.make_tree_inputs(wl))
        p = ta.tree_params(wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.kv_seq_len,
                           wl.kv_capacity, wl.scale, wl.q_l, wl.mask_stride, wl.nwg)
        assert_close(_noalloc(ta, p, d, False).cpu().numpy(),
                     _regular(ta, p, d, False).cpu().numpy())


def test_noalloc_rejects_requests_beyond_its_scratch(ta):
    wl = W.FIXED_TREE.with_(nwg=64)           # 768 rows x 64 splits x 258 x 4 B > 16 MiB
    p = ta.tree_params(wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.kv_seq_len, wl.kv_capacity,
                       wl.scale, wl.q_l, wl.mask_stride, wl.nwg)
    assert ta.tree_attn_workspace_bytes(p) > 16 << 20
    x = torch.zeros(16, device="cuda")
    b = ta.buf(x)
    before = ta.ta_launch_count()
    st = ta.lib.tree_attn_fwd_noalloc(ctypes.byref(p), b, b, b, b, b, None)
    assert st == 4 and "static scratch" in ta.ta_last_error()
    assert ta.ta_launch_count() == before


def test_noalloc_call_allocates_no_device_memory(ta):
    """The defining claim: after a first call (which may load the module), a
    call leaves the device's free memory unchanged.  Every tensor the calls use
    exists before the first reading."""
    wl = small_tree(H=24, Hk=4, D=256, N=1500, C=2048, L=32, kv_dtype="f16", nwg=8)
    d = to_dev(W.make_tree_inputs(wl))
    p = ta.tree_params(wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.kv_seq_len, wl.kv_capacity,
                       wl.scale, wl.q_l, wl.mask_stride, wl.nwg)
    out = torch.empty((p.q_l, p.n_heads, p.head_dim), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (ctypes.byref(p), ta.buf(d["q"]), ta.buf(d["k"]), ta.buf(d["v"]), ta.buf(d["mask"]), ta.buf(out),
            stream)
    assert ta.lib.tree_attn_fwd_noalloc(*args) == ta.TA_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert ta.lib.tree_attn_fwd_noalloc(*args) == ta.TA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0

"""GPU parity of the quantized-KV attention path against the float64 oracle,
called through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_close, run_quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tree_masked_speculative_gb300 as m
    return m


@pytest.fixture(params=[2, 1, 3], ids=["tensor_cores", "cuda_cores", "warp_mma"])
def kern(request):
    """Every test runs on the three kernel families: the tcgen05 kernel and the
    warp-MMA kernel (each where its shape rules allow it; other shapes fall
    back to CUDA cores) and the CUDA-core one."""
    return request.param


def qwl(B=2, nQ=8, nKV=2, dim=128, N=300, bits=4, G=64, sinks=1, window=0, dtype="f16",
        fmask="none", bfrac=0.0, nwg=0, seed=3):
    return W.QuantWorkload(name="small", batch=B, n_q_heads=nQ, n_kv_heads=nKV, dim=dim, tokens=N,
                           bits=bits, group_size=G, has_sinks=sinks, window_size=window,
                           scale=1.0 / math.sqrt(dim), dtype=dtype, float_mask=fmask,
                           bool_mask_frac=bfrac, nwg=nwg, seed=seed)


QCASES = [
    dict(),
    dict(bits=8, dtype="bf16", sinks=0),
    dict(dim=64, G=32, N=77, nwg=1),
    dict(dim=96, G=32, bits=4, N=130, nwg=3),
    dict(dim=96, G=32, bits=8, N=130, nwg=2, dtype="bf16"),
    dict(dim=256, bits=8, window=100, N=500, fmask="alibi", bfrac=0.1, dtype="bf16", sinks=0),
    dict(dim=512, bits=4, G=128, N=200, nwg=2),
    dict(dim=512, bits=8, G=64, N=150, bfrac=0.3, dtype="bf16"),
    dict(nQ=16, nKV=2, N=257, window=33),          # 8 query rows per KV row
    dict(nQ=32, nKV=2, N=129, bits=8, dtype="bf16", fmask="alibi", bfrac=0.2),   # 16 rows, 4 row groups
    dict(nQ=4, nKV=4, N=100, dim=128, nwg=2),      # 1 row per KV row
    dict(dim=128, G=32, bits=8, N=333, window=200, fmask="alibi", bfrac=0.1, sinks=1, dtype="bf16"),
    dict(nQ=6, nKV=2, N=64, nwg=1),                # 3 rows per KV row
    dict(N=31, window=500),
    # both masks with 16-byte aligned rows (tokens a multiple of 8): the bulk-copy staging of masked chunks
    dict(dim=256, bits=8, N=512, fmask="alibi", bfrac=0.1, dtype="bf16", sinks=0),
    dict(dim=128, bits=4, N=256, window=100, fmask="alibi", bfrac=0.2, nwg=2),
    dict(dim=64, G=32, bits=8, N=192, bfrac=0.3, nwg=1),
    # eight scale groups per token (two accumulator sets of the warp-MMA scores)
    dict(dim=256, G=32, bits=4, N=300, nwg=3),
    dict(dim=256, G=32, bits=8, N=256, fmask="alibi", bfrac=0.1, dtype="bf16"),
    dict(dim=128, G=32, bits=8, nQ=12, nKV=2, N=320, window=150),   # 6 rows per KV row: a partial row group
    # 16 or more query rows per KV row: the warp-MMA kernel's wide form (16 rows per warp)
    dict(nQ=40, nKV=2, N=300, window=120),                                  # 20 rows: a partial 16-row group
    dict(nQ=32, nKV=2, N=256, dim=64, G=64, fmask="alibi"),                 # 16 float-mask rows by bulk copies
    dict(nQ=32, nKV=1, N=512, bits=8, G=32, dtype="bf16", bfrac=0.2),       # 32 rows, bool-mask rows by bulk copies
    dict(nQ=32, nKV=2, N=512, bits=8, fmask="alibi", bfrac=0.1, nwg=1),     # both masks (32 rows): lanes' cp.async
    dict(nQ=64, nKV=2, N=190, dim=64, G=32, bits=8, sinks=1, nwg=2),        # 32 rows, ragged last chunk
]


@pytest.mark.parametrize("kw", QCASES, ids=[str(i) for i in range(len(QCASES))])
def test_quant_matches_oracle(ta, kern, kw):
    wl = qwl(**kw)
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    got32 = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got32, ref, what="quant f32 out %r" % (kw,))
    gotT = run_quant(ta, wl, inp, kernel=kern).cpu().double().numpy()
    assert_close(gotT, ref, extra_ulp_dtype=wl.dtype, what="quant T out %r" % (kw,))


def test_quant_no_visible_token_gives_zero_and_sink_only(ta, kern):
    wl = qwl(N=70, sinks=1, bfrac=0.0, nwg=2)
    inp = W.make_quant_inputs(wl)
    inp["mask_bool"] = torch.ones((wl.rows, wl.tokens), dtype=torch.int32)
    inp["mask_bool"][3] = 0
    got = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern).cpu()
    assert torch.all(got[3] == 0.0)
    wl0 = wl.with_(has_sinks=0)
    got0 = run_quant(ta, wl0, inp, out_dtype=torch.float32, kernel=kern).cpu()
    assert torch.all(got0[3] == 0.0)
    assert_close(got.double().numpy(), oracle.quant_oracle_for(wl, inp))


def test_quant_error_word_stays_clear(ta, kern):
    wl = qwl(N=700, bits=8, dtype="bf16", fmask="alibi", bfrac=0.1, window=300)
    inp = W.make_quant_inputs(wl)
    p = ta.quant_params(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.dim, wl.tokens, wl.bits,
                        wl.group_size, wl.has_sinks, wl.window_size, wl.scale, 0, kern)
    nb = ta.quant_sdpa_tmp_bytes(p)
    assert nb >= 256
    tmp = torch.zeros((nb + 3) // 4, dtype=torch.float32, device="cuda")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = ta.quant_sdpa(d, batch=wl.batch, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads,
                        dim=wl.dim, tokens=wl.tokens, bits=wl.bits, group_size=wl.group_size,
                        has_sinks=wl.has_sinks, window_size=wl.window_size, scale=wl.scale,
                        out_dtype=torch.float32, tmp=tmp, kernel=kern)
    torch.cuda.synchronize()
    assert int(tmp[:1].view(torch.int32).item()) == 0
    assert_close(out.cpu().double().numpy(), oracle.quant_oracle_for(wl, inp))


def test_quant_split_invariance(ta, kern):
    wl = qwl(N=2000, bits=8, dtype="bf16")
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    outs = [run_quant(ta, wl, inp, nwg=n, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
            for n in (1, 3, 15)]
    for o in outs:
        assert_close(o, ref)


def test_quant_b4_workload_full(ta, kern):
    wl = W.QUANT_B4
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, kernel=kern).cpu().double().numpy()
    assert_close(got, ref, extra_ulp_dtype=wl.dtype, what="quant b4 workload")
    got32 = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got32, ref, what="quant b4 workload f32")


def test_quant_b8_masks_workload_full(ta, kern):
    wl = W.QUANT_B8_MASKS
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, kernel=kern).cpu().double().numpy()
    assert_close(got, ref, extra_ulp_dtype=wl.dtype, what="quant b8 workload")
    got32 = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got32, ref, what="quant b8 workload f32")


@pytest.mark.parametrize("bits,dtype", [(4, "f16"), (8, "bf16")])
def test_quant_cache_verified_with_a_tree_mask(ta, kern, bits, dtype):
    """q_l draft-tree nodes per head verified against a quantized cache through
    the same call: the nodes are extra query rows (n_q_heads * q_l of them,
    ordered (batch, head, node), so each KV row serves heads_per_kv * q_l rows)
    and each row's tree mask is its additive float mask (0 / -65504)."""
    B, nQ, nKV, q_l, N = 2, 4, 2, 6, 300
    wl = qwl(B=B, nQ=nQ * q_l, nKV=nKV, dim=128, N=N, bits=bits, G=64, sinks=0, dtype=dtype)
    inp = W.make_quant_inputs(wl)
    par = W.fixed_tree_parents((2, 2, 1), q_l)
    tm = oracle.tree_mask(par, kv_seq_len=N, mask_stride=N)             # [q_l, N]
    T = torch.float16 if dtype == "f16" else torch.bfloat16
    inp["mask_float"] = torch.from_numpy(np.tile(tm, (B * nQ, 1))).to(T)
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got, ref, what="quant cache x tree mask")
    # the same token sets given as a bool mask instead of an additive one
    inp_b = dict(inp)
    del inp_b["mask_float"]
    inp_b["mask_bool"] = torch.from_numpy(np.tile((tm == 0.0).astype(np.int32), (B * nQ, 1)))
    got_b = run_quant(ta, wl, inp_b, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got_b, ref, what="quant cache x tree mask as a bool mask")


def test_quant_many_rows_per_kv_row(ta, kern):
    """48 query rows per KV row: two row blocks of the tensor-core kernel, a
    ragged last tile, a window that starts inside a tile, both masks."""
    wl = qwl(B=1, nQ=48, nKV=1, dim=128, N=777, bits=4, G=32, sinks=1, window=600, fmask="alibi",
             bfrac=0.2, dtype="bf16")
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got, ref, what="48 rows per KV row")
    gotT = run_quant(ta, wl, inp, kernel=kern).cpu().double().numpy()
    assert_close(gotT, ref, extra_ulp_dtype=wl.dtype, what="48 rows per KV row, T out")


def test_quant_tree_workload_full(ta, kern):
    """The draft-tree workload on a quantized cache at full size (256 rows over
    8 KV rows, 16384 tokens, per-row tree masks)."""
    wl = W.QUANT_TREE
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got, ref, what="quant tree workload f32")


def test_quant_more_splits_than_tiles(ta, kern):
    """A forced split count above the number of 128-token tiles: the splits
    without a token leave an empty partial (S = 0) that the merge skips."""
    wl = qwl(N=200, nwg=5, sinks=1, dtype="bf16")
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, nwg=5, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got, ref, what="more splits than tiles")


@pytest.mark.parametrize("bits,dtype", [(8, "bf16"), (4, "f16")])
def test_quant_peaked_softmax_plain_tolerance(ta, kern, bits, dtype):
    """A peaked softmax with a running max that moves many times: 16 rows per KV
    row (the tensor-core kernel's shape), queries scaled by 4 (exact in f16 /
    bf16) and a large attention scale.  A single f16 P would move the output by
    up to 2^-11 of the attended V spread (8-bit codes: V up to about 13); the
    kernels are held to the plain tolerance."""
    wl = qwl(B=1, nQ=32, nKV=2, dim=128, N=1200, bits=bits, G=64, sinks=1, dtype=dtype)
    wl = wl.with_(scale=1.5)
    inp = W.make_quant_inputs(wl)
    inp["queries"] = inp["queries"] * 4.0
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern).cpu().double().numpy()
    assert_close(got, ref, what="quant peaked softmax")


def test_bounded_wait_timeout_sets_status_and_returns(ta):
    """The failure path of the bounded waits, exercised without any fault: the
    test hook gives every CTA's first K/V copy wait a bound of zero polls, so
    it gives up at once.  Each CTA then ORs 1 into the status word, lets its
    issued copies land (normal bound) and returns; the call completes, the
    status is set, and the context stays usable for a normal call."""
    wl = qwl(B=2, nQ=8, nKV=2, dim=128, N=2000, bits=4, G=64, sinks=1, dtype="f16")
    inp = W.make_quant_inputs(wl)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    for nwg, kernel in ((1, 1), (0, 1), (1, 3), (0, 3)):
        p = ta.quant_params(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.dim, wl.tokens, wl.bits, wl.group_size,
                            wl.has_sinks, wl.window_size, wl.scale, nwg, kernel)
        nb = ta.quant_sdpa_tmp_bytes(p)
        tmp = torch.zeros((nb + 3) // 4, dtype=torch.float32, device="cuda")
        out = torch.zeros((wl.rows, wl.dim), dtype=torch.float32, device="cuda")
        args = (d["queries"], d["k_packed"], d["k_scales"], d["k_biases"], d["v_packed"], d["v_scales"],
                d["v_biases"], d["sinks"], None, None, tmp, out)
        ta.ta_test_quant_sdpa_fwd_wait_limit(0, p, *args)
        torch.cuda.synchronize()
        assert int(tmp[:1].view(torch.int32).item()) & 1 == 1
        tmp.zero_()
        ta.quant_sdpa_fwd(p, *args)
        torch.cuda.synchronize()
        assert int(tmp[:1].view(torch.int32).item()) == 0
        assert_close(out.cpu().double().numpy(), oracle.quant_oracle_for(wl, inp), what="after a timeout")
    # the hook refuses the tensor-core kernel
    p2 = ta.quant_params(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.dim, wl.tokens, wl.bits, wl.group_size,
                         wl.has_sinks, wl.window_size, wl.scale, 0, 2)
    tmp2 = torch.zeros((ta.quant_sdpa_tmp_bytes(p2) + 3) // 4, dtype=torch.float32, device="cuda")
    before = ta.ta_launch_count()
    with pytest.raises(ta.TreeAttentionError, match="CUDA-core or warp-MMA kernel only"):
        ta.ta_test_quant_sdpa_fwd_wait_limit(0, p2, *args[:-2], tmp2, out)
    assert ta.ta_launch_count() == before


def test_bounded_wait_timeout_two_warp_form(ta):
    """The same failure path on the warp-MMA kernel's two-warp form (64 packed
    words per token; with and without masks): both warps give up at their
    first wait, the value warp lets every copy it issued land, and the CTA
    leaves through its final barrier with the status set."""
    assert ta.quant_sdpa_kernel_family(ta.quant_params(1, 8, 2, 256, 640, 8, 64, 0, 0, 0.1, 0, 3)) == \
        ta.KERNEL_WARP_MMA
    for fmask, bfrac in (("none", 0.0), ("alibi", 0.1)):
        wl = qwl(B=2, nQ=8, nKV=2, dim=256, N=640, bits=8, G=64, sinks=0, dtype="bf16", fmask=fmask, bfrac=bfrac)
        inp = W.make_quant_inputs(wl)
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        for nwg in (1, 0):
            p = ta.quant_params(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.dim, wl.tokens, wl.bits, wl.group_size,
                                wl.has_sinks, wl.window_size, wl.scale, nwg, 3)
            tmp = torch.zeros((ta.quant_sdpa_tmp_bytes(p) + 3) // 4, dtype=torch.float32, device="cuda")
            out = torch.zeros((wl.rows, wl.dim), dtype=torch.float32, device="cuda")
            args = (d["queries"], d["k_packed"], d["k_scales"], d["k_biases"], d["v_packed"], d["v_scales"],
                    d["v_biases"], None, d.get("mask_bool"), d.get("mask_float"), tmp, out)
            ta.ta_test_quant_sdpa_fwd_wait_limit(0, p, *args)
            torch.cuda.synchronize()
            assert int(tmp[:1].view(torch.int32).item()) & 1 == 1
            tmp.zero_()
            ta.quant_sdpa_fwd(p, *args)
            torch.cuda.synchronize()
            assert int(tmp[:1].view(torch.int32).item()) == 0
            assert_close(out.cpu().double().numpy(), oracle.quant_oracle_for(wl, inp), what="two-warp, after a timeout")


def test_bounded_wait_timeout_wide_form(ta):
    """The same failure path on the warp-MMA kernel's wide form (16 query rows
    per warp), with its copies by bulk copies (float mask) and by the lanes'
    cp.async (both masks on 16 rows)."""
    for fmask, bfrac in (("none", 0.0), ("alibi", 0.0), ("alibi", 0.2)):
        wl = qwl(B=2, nQ=32, nKV=2, dim=128, N=1024, bits=4, G=64, sinks=1, dtype="f16", fmask=fmask, bfrac=bfrac)
        inp = W.make_quant_inputs(wl)
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        for nwg in (1, 0):
            p = ta.quant_params(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.dim, wl.tokens, wl.bits, wl.group_size,
                                wl.has_sinks, wl.window_size, wl.scale, nwg, 3)
            tmp = torch.zeros((ta.quant_sdpa_tmp_bytes(p) + 3) // 4, dtype=torch.float32, device="cuda")
            out = torch.zeros((wl.rows, wl.dim), dtype=torch.float32, device="cuda")
            args = (d["queries"], d["k_packed"], d["k_scales"], d["k_biases"], d["v_packed"], d["v_scales"],
                    d["v_biases"], d["sinks"], d.get("mask_bool"), d.get("mask_float"), tmp, out)
            ta.ta_test_quant_sdpa_fwd_wait_limit(0, p, *args)
            torch.cuda.synchronize()
            assert int(tmp[:1].view(torch.int32).item()) & 1 == 1
            tmp.zero_()
            ta.quant_sdpa_fwd(p, *args)
            torch.cuda.synchronize()
            assert int(tmp[:1].view(torch.int32).item()) == 0
            assert_close(out.cpu().double().numpy(), oracle.quant_oracle_for(wl, inp), what="wide form, after a timeout")


TREE_CASES = [
    # q_l, bits, dtype, dim, G, N, window, bool fraction, sinks, heads per KV row
    (8, 4, "f16", 128, 64, 700, 0, 0.0, 0, 4),      # 32 rows per KV row
    (4, 8, "bf16", 128, 32, 333, 200, 0.1, 1, 2),   # window and bool mask
    (16, 4, "bf16", 64, 32, 129, 0, 0.0, 1, 1),     # 16 rows
    (32, 4, "f16", 128, 64, 500, 0, 0.0, 0, 1),     # the largest tree
    (1, 8, "f16", 256, 64, 90, 0, 0.2, 1, 3),       # a single node
    (8, 4, "f16", 128, 64, 1000, 0, 0.0, 0, 4),
]


@pytest.mark.parametrize("q_l,bits,dtype,dim,G,N,window,bfrac,sinks,hpk", TREE_CASES,
                         ids=[str(i) for i in range(len(TREE_CASES))])
def test_quant_tree_as_parent_array(ta, kern, q_l, bits, dtype, dim, G, N, window, bfrac, sinks, hpk):
    """A draft tree verified on a quantized cache with the tree mask given as the
    parent array of the last q_l tokens (no mask read): the same output, bit for
    bit, as the dense additive mask that tree_mask_build's rule gives, and the
    oracle on that dense mask."""
    wl = qwl(B=2, nQ=2 * hpk * q_l, nKV=2, dim=dim, G=G, N=N, bits=bits, sinks=sinks, window=window,
             dtype=dtype, fmask="tree%d" % q_l, bfrac=bfrac, seed=q_l * 7 + N)
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    dense = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=kern)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    par = torch.tensor(inp["tree_parents"], dtype=torch.int32, device="cuda")
    tree = ta.quant_sdpa(d, batch=wl.batch, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads, dim=wl.dim,
                         tokens=wl.tokens, bits=wl.bits, group_size=wl.group_size, has_sinks=wl.has_sinks,
                         window_size=wl.window_size, scale=wl.scale, out_dtype=torch.float32, kernel=kern,
                         tree_parents=par)
    torch.cuda.synchronize()
    assert_close(tree.cpu().double().numpy(), ref, what="quant tree as parents")
    assert torch.equal(tree, dense)


def test_quant_tree_workload_as_parent_array(ta, kern):
    wl = W.QUANT_TREE
    inp = W.make_quant_inputs(wl)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    par = torch.tensor(inp["tree_parents"], dtype=torch.int32, device="cuda")
    got = ta.quant_sdpa(d, batch=wl.batch, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads, dim=wl.dim,
                        tokens=wl.tokens, bits=wl.bits, group_size=wl.group_size, has_sinks=wl.has_sinks,
                        window_size=wl.window_size, scale=wl.scale, out_dtype=torch.float32, kernel=kern,
                        tree_parents=par)
    torch.cuda.synchronize()
    assert_close(got.cpu().double().numpy(), oracle.quant_oracle_for(wl, inp), what="quant tree workload, parents")

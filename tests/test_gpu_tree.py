"""GPU parity of the tree-verify attention path against the float64 oracle,
called through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_close, run_tree, small_tree, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tree_masked_speculative_gb300 as m
    return m


@pytest.fixture(params=[0, 1], ids=["auto", "fma"])
def path(request):
    """The main pass's kernel family: 0 = automatic (tensor cores for 16-bit K/V
    and >= 16 rows per KV head), 1 = CUDA cores."""
    return request.param


CASES = [
    # H, Hk, D, N, C, L, kv_dtype, nwg
    (4, 2, 128, 256, 256, 8, "f32", 32),      # pages' PR1 reference shape
    (4, 2, 128, 200, 256, 5, "f16", 0),       # ragged last chunk
    (6, 3, 256, 333, 400, 7, "bf16", 3),
    (8, 1, 512, 97, 128, 3, "f16", 2),
    (2, 2, 128, 31, 31, 1, "f32", 1),         # one split, single partial chunk
    (12, 4, 128, 1000, 1024, 16, "bf16", 0),  # 48 rows per KV head
    (16, 2, 256, 517, 600, 20, "f16", 5),     # 160 rows per KV head
    (8, 4, 512, 260, 300, 9, "bf16", 0),
    (4, 2, 256, 150, 160, 4, "f32", 2),       # f32 K/V at each head dimension (CUDA-core kernel)
    (4, 2, 512, 100, 128, 3, "f32", 0),
    (16, 2, 512, 700, 700, 20, "bf16", 3),    # 160 rows: two row tiles per O half
    (20, 1, 512, 400, 416, 15, "f16", 2),     # 300 rows: three row tiles
    (16, 2, 256, 3000, 3008, 8, "f16", 12),   # 12 splits merged in a 12-CTA cluster (two rounds of 8)
]


@pytest.mark.parametrize("H,Hk,D,N,C,L,kvd,nwg", CASES)
def test_tree_matches_oracle(ta, path, H, Hk, D, N, C, L, kvd, nwg):
    wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=C, L=L, kv_dtype=kvd, nwg=nwg, seed=H * 100 + N)
    inp = W.make_tree_inputs(wl)
    got = run_tree(ta, wl, inp, kernel=path).cpu().numpy()
    ref = oracle.tree_oracle_for(wl, inp)
    assert_close(got, ref, what="tree %s" % (wl,))


def test_tree_mask_stride_padding_and_tail_cells_ignored(ta, path):
    wl = small_tree(H=4, Hk=2, D=256, N=150, C=160, L=6, stride=192, kv_dtype="f16", nwg=2)
    inp = W.make_tree_inputs(wl)
    inp["mask"][:, 150:] = 0.0            # cells past kv_seq_len would attend if read
    got = run_tree(ta, wl, inp, kernel=path).cpu().numpy()
    ref = oracle.tree_oracle_for(wl, inp)
    assert_close(got, ref)


def test_explicit_causal_mask_bit_identical_to_implicit(ta, path):
    """The pages' byte-identity contract, on our own two kernels."""
    for (H, Hk, D, N, L, kvd, nwg, ws) in [(4, 2, 128, 256, 8, "f32", 32, 0),
                                           (24, 4, 256, 700, 32, "f16", 0, 0),
                                           (8, 2, 512, 300, 12, "bf16", 3, 0),
                                           (4, 1, 128, 500, 4, "f16", 4, 130)]:
        wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=N, L=L, kv_dtype=kvd, nwg=nwg, topology="chain")
        inp = W.make_tree_inputs(wl)
        inp["mask"] = W.causal_mask(L, N, N, window_start=ws)
        explicit = run_tree(ta, wl, inp, kernel=path)
        implicit = run_tree(ta, wl, inp, kernel=path, causal=True, window_start=ws)
        assert torch.equal(explicit, implicit), (H, D, kvd)
        assert_close(explicit.cpu().numpy(),
                     oracle.tree_oracle_for(wl, inp, mask=None, window_start=ws))


# (H, Hk): 4/2 gives 2*L rows per KV head (CUDA-core kernel for small L),
# 16/2 gives 8*L rows per KV head (tensor-core kernel for 16-bit K/V).
@pytest.mark.parametrize("H,Hk,D", [(4, 2, 128), (16, 2, 128), (16, 2, 256), (8, 1, 512)])
def test_single_attended_key_returns_value_row_exactly(ta, path, H, Hk, D):
    wl = small_tree(H=H, Hk=Hk, D=D, N=300, C=300, L=3, kv_dtype="bf16", nwg=4)
    inp = W.make_tree_inputs(wl)
    inp["mask"][:] = W.MASKED
    keys = [5, 177, 299]
    for i, j in enumerate(keys):
        inp["mask"][i, j] = 0.0
    got = run_tree(ta, wl, inp, kernel=path).cpu()
    g = H // Hk
    for i, j in enumerate(keys):
        for h in range(H):
            assert torch.equal(got[i, h], inp["v"][h // g, j].float()), (i, h)


@pytest.mark.parametrize("H,Hk,D,kvd", [(4, 2, 256, "f16"), (24, 4, 256, "f16"), (16, 2, 512, "bf16"),
                                        (12, 1, 128, "bf16")])
def test_fully_masked_rows_and_dead_chunks(ta, path, H, Hk, D, kvd):
    wl = small_tree(H=H, Hk=Hk, D=D, N=640, C=640, L=6, kv_dtype=kvd, nwg=3)
    inp = W.make_tree_inputs(wl)
    m = inp["mask"]
    m[2] = W.MASKED                        # row with no attended key -> zeros
    m[:, 64:320] = W.MASKED                # chunks no row attends: never loaded
    m[4, 330:640] = W.MASKED               # a row whose last chunks are dead for it alone
    got = run_tree(ta, wl, inp, kernel=path).cpu().numpy()
    assert np.all(got[2] == 0.0)
    assert_close(got, oracle.tree_oracle_for(wl, inp))


def test_all_keys_dead_for_every_row(ta, path):
    wl = small_tree(H=16, Hk=2, D=128, N=200, C=200, L=4, kv_dtype="f16", nwg=2)
    inp = W.make_tree_inputs(wl)
    inp["mask"][:] = W.MASKED
    got = run_tree(ta, wl, inp, kernel=path).cpu().numpy()
    assert np.all(got == 0.0)


@pytest.mark.parametrize("D,kvd", [(128, "bf16"), (128, "f16"), (512, "bf16"), (256, "f16")])
def test_large_logits_exercise_rescaling(ta, path, D, kvd):
    """Logit ranges far above the lazy-rescale slack, growing along the keys so the
    running max moves many times, and a peaked softmax (a few keys carry the
    weight): the case where a 16-bit P would move the output by up to 2^-8
    (bf16) of the attended V spread.  Held to the plain tolerance."""
    wl = small_tree(H=16, Hk=2, D=D, N=1500, C=1500, L=4, kv_dtype=kvd, nwg=2, scale=1.0)
    inp = W.make_tree_inputs(wl)
    ramp = torch.linspace(0.1, 3.0, wl.kv_seq_len).view(1, -1, 1) * (128.0 / D) ** 0.5
    inp["k"] = (inp["k"].float() * ramp).to(W.DTYPES[kvd])
    # quarters are exact in f16 and bf16, so the logits carry no Q-rounding error and the
    # comparison isolates the rescaling of O and S and the rounding of P
    inp["q"] = torch.round(inp["q"] * 4.0) / 4.0
    got = run_tree(ta, wl, inp, kernel=path).cpu().numpy()
    ref = oracle.tree_oracle_for(wl, inp)
    assert_close(got, ref, what="peaked softmax D %d %s" % (D, kvd))


@pytest.mark.parametrize("H,Hk,D,N,L,kvd,nwg", [
    (16, 2, 128, 700, 8, "bf16", 3),    # 64 rows per KV head: tensor cores
    (24, 4, 256, 900, 32, "f16", 0),    # the fixed tree's shape, two row tiles
    (8, 1, 512, 500, 20, "bf16", 2),    # two O halves, two row tiles
    (4, 2, 256, 300, 5, "f16", 2),      # 10 rows: CUDA cores
    (4, 2, 128, 256, 8, "f32", 4),      # f32 K/V: CUDA cores
    (16, 2, 512, 333, 9, "f32", 0),
])
def test_additive_float_mask_values(ta, path, H, Hk, D, N, L, kvd, nwg):
    """Finite, non-binary mask cells are added to the scaled logit
    (tree_attention_impl: logit = fma(qk, scale, mask)); cells <= -65504 drop
    the key.  Mixed chunks carry biases, some chunks stay all-zero
    (all-attended), some are dead for every row."""
    wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=N, L=L, kv_dtype=kvd, nwg=nwg, seed=N + D)
    inp = W.make_tree_inputs(wl)
    g = torch.Generator().manual_seed(N * 7 + L)
    bias = torch.rand((L, wl.mask_stride), generator=g) * 7.0 - 4.0        # U(-4, 3)
    m = inp["mask"]
    att = m == 0.0
    m = torch.where(att, bias, m)
    m[:, :64] = 0.0                                       # two all-attended chunks
    m[:, 64:128] = W.MASKED                               # two dead chunks
    m[0, 200] = -3.0e4                                    # large but finite bias
    m[1, 130:140] = 1.0e-3
    inp["mask"] = m.contiguous()
    got = run_tree(ta, wl, inp, kernel=path).cpu().numpy()
    ref = oracle.tree_oracle_for(wl, inp)
    assert_close(got, ref, what="additive mask %s" % (wl,))


def test_device_status_word_is_cleared_and_stays_zero(ta):
    """The status word at tree_attn_status_offset: set to 0 by every main pass
    (the buffer starts as garbage here) and left 0 when every wait completed."""
    wl = small_tree(H=24, Hk=4, D=256, N=900, C=1024, L=32, kv_dtype="f16", nwg=6)
    inp = to_dev(W.make_tree_inputs(wl))
    p = ta.tree_params(wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.kv_seq_len, wl.kv_capacity,
                       wl.scale, wl.q_l, wl.mask_stride, wl.nwg)
    ws = ta.tree_attn_workspace_bytes(p)
    off = ta.tree_attn_status_offset(p)
    tmp = torch.full(((ws + 3) // 4,), 123.0, device="cuda")
    out = torch.empty((wl.q_l, wl.n_heads, wl.head_dim), device="cuda")
    for kernel in (0, 1):
        tmp.view(torch.int32)[off // 4] = 0x5A5A
        ta.tree_attn_fwd_ex(p, kernel, ta.MASK_DENSE, 0, inp["q"], inp["k"], inp["v"], inp["mask"], tmp, out)
        ta.tree_attn_reduce(p, tmp, out)
        torch.cuda.synchronize()
        assert tmp.view(torch.int32)[off // 4].item() == 0


def test_split_count_invariance(ta, path):
    wl = small_tree(H=8, Hk=2, D=128, N=1000, C=1000, L=8, kv_dtype="f16")
    inp = W.make_tree_inputs(wl)
    ref = oracle.tree_oracle_for(wl, inp)
    outs = [run_tree(ta, wl, inp, kernel=path, nwg=n).cpu().numpy() for n in (1, 2, 7, 32)]
    for o in outs:
        assert_close(o, ref)
    assert_close(outs[0], outs[-1], atol=1e-4, rtol=1e-4)


@pytest.mark.parametrize("H,Hk,D,L", [(4, 2, 128, 5), (16, 2, 256, 5)])
def test_output_guard_bytes_untouched(ta, path, H, Hk, D, L):
    wl = small_tree(H=H, Hk=Hk, D=D, N=200, C=256, L=L, kv_dtype="f16", nwg=3)
    inp = to_dev(W.make_tree_inputs(wl))
    p = ta.tree_params(H, Hk, D, 200, 256, wl.scale, L, 200, 3)
    ws = ta.tree_attn_workspace_bytes(p)
    tmp_full = torch.full(((ws + 3) // 4 + 1024,), 7.0, device="cuda")
    out_full = torch.full((L * H * D + 1024,), 7.0, device="cuda")
    tmp, out = tmp_full[:(ws + 3) // 4], out_full[:L * H * D]
    ta.tree_attn_fwd_ex(p, path, ta.MASK_DENSE, 0, inp["q"], inp["k"], inp["v"], inp["mask"], tmp, out)
    ta.tree_attn_reduce(p, tmp, out)
    torch.cuda.synchronize()
    assert torch.all(tmp_full[(ws + 3) // 4:] == 7.0)
    assert torch.all(out_full[L * H * D:] == 7.0)


def test_pr1_reference_workload_full(ta, path):
    wl = W.PR1_CHAIN
    inp = W.make_tree_inputs(wl)
    got = run_tree(ta, wl, inp, kernel=path)
    assert_close(got.cpu().numpy(), oracle.tree_oracle_for(wl, inp))
    implicit = run_tree(ta, wl, inp, kernel=path, causal=True)
    assert torch.equal(got, implicit)


def test_fixed_tree_workload_full(ta):
    wl = W.FIXED_TREE
    inp = W.make_tree_inputs(wl)
    got = run_tree(ta, wl, inp).cpu().numpy()
    assert_close(got, oracle.tree_oracle_for(wl, inp), what="fixed tree")


def test_dynamic_tree_workload_full(ta):
    """The dynamic asymmetric tree at full size (32 heads x 64 nodes over 32768
    bf16 keys of head dim 512), every one of its 2048 output rows against the
    oracle, in the launch configuration the benchmark times."""
    wl = W.DYNAMIC_TREE
    inp = W.make_tree_inputs(wl)
    got = run_tree(ta, wl, inp).cpu().numpy()
    assert_close(got, oracle.tree_oracle_for(wl, inp), what="dynamic tree, all rows")


# ------------------------------------------------------------ tree mask builder
MASK_CASES = [
    ("fixed", 32, 4096, 8192),        # the fixed-tree workload's shape (stride 8192 > N)
    ("dynamic", 64, 32768, 32768),    # the dynamic-tree workload's shape
    ("chain", 8, 256, 256),
    ("dynamic", 1, 5, 7),             # a single node; stride not a multiple of 4
    ("dynamic", 100, 1000, 1003),
    ("fixed", 17, 17, 17),            # no prefix
    ("dynamic", 300, 5000, 5004),     # more than 256 nodes
]


def _parents(topology, L, seed=5):
    if topology == "chain":
        return W.chain_parents(L)
    if topology == "fixed":
        return W.fixed_tree_parents((4, 2, 2, 2, 2, 1, 1), L)
    return W.dynamic_tree_parents(L, torch.Generator().manual_seed(seed))


@pytest.mark.parametrize("topology,L,N,S", MASK_CASES, ids=[str(i) for i in range(len(MASK_CASES))])
def test_tree_mask_build_matches_oracle(ta, topology, L, N, S):
    par = _parents(topology, L)
    p = ta.tree_params(8, 2, 128, N, N, 0.1, L, S, 0)
    d_par = torch.tensor(par, dtype=torch.int32, device="cuda")
    full = torch.full((L * S + 64,), 7.0, device="cuda")           # guard cells after the mask
    mask = full[:L * S].view(L, S)
    ta.tree_mask_build(p, d_par, mask)
    torch.cuda.synchronize()
    ref = oracle.tree_mask(par, kv_seq_len=N, mask_stride=S)
    got = mask.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))   # bit-exact
    assert torch.all(full[L * S:] == 7.0)


def test_tree_mask_build_feeds_the_verify_pass(ta):
    # the device-built mask gives the same attention output, bit for bit, as the host-built one
    wl = small_tree(H=8, Hk=2, D=128, N=600, C=640, L=12, kv_dtype="f16", topology="fixed")
    inp = W.make_tree_inputs(wl)
    par = W.fixed_tree_parents(wl.branching, wl.q_l)
    out_host = run_tree(ta, wl, inp)
    p = ta.tree_params(wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.kv_seq_len, wl.kv_capacity, wl.scale,
                       wl.q_l, wl.mask_stride, wl.nwg)
    d_mask = torch.empty((wl.q_l, wl.mask_stride), device="cuda")
    ta.tree_mask_build(p, torch.tensor(par, dtype=torch.int32, device="cuda"), d_mask)
    inp2 = dict(inp)
    inp2["mask"] = d_mask.cpu()
    out_dev = run_tree(ta, wl, inp2)
    assert torch.equal(out_host, out_dev)


# ------------------------------------------------- tree mask as a parent array
def _run_parents(ta, wl, inp, parents, nwg=None, kernel=0):
    d = to_dev(inp)
    par = torch.tensor(parents, dtype=torch.int32, device="cuda")
    out = ta.tree_attention(d["q"], d["k"], d["v"], None, n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads,
                            kv_seq_len=wl.kv_seq_len, scale=wl.scale, mask_stride=wl.mask_stride,
                            nwg=wl.nwg if nwg is None else nwg, parents=par, kernel=kernel)
    torch.cuda.synchronize()
    return out


PARENT_CASES = [
    # H, Hk, D, N, C, L, kv_dtype, topology, nwg
    (24, 4, 256, 1000, 1024, 32, "f16", "fixed", 0),     # tensor cores, two row tiles
    (16, 2, 512, 700, 700, 20, "bf16", "dynamic", 3),    # D 512, two O halves
    (8, 2, 128, 300, 320, 13, "f16", "chain", 2),
    (4, 2, 128, 256, 256, 8, "f32", "chain", 32),        # CUDA cores (f32 K/V)
    (4, 4, 256, 90, 96, 3, "bf16", "dynamic", 0),        # CUDA cores (R = 3)
    (2, 1, 128, 40, 40, 1, "f16", "dynamic", 1),         # a single node, one split
    (8, 2, 128, 64, 64, 64, "f16", "dynamic", 0),        # no prefix: every key is a tree node
    (2, 1, 128, 600, 600, 256, "f16", "chain", 0),       # the largest tree, a 256-deep chain
    (4, 1, 256, 900, 900, 200, "bf16", "dynamic", 4),    # 800 rows, bitsets of 7 words
]


@pytest.mark.parametrize("H,Hk,D,N,C,L,kvd,topo,nwg", PARENT_CASES, ids=[str(i) for i in range(len(PARENT_CASES))])
def test_parent_array_mask_bit_identical_to_dense(ta, path, H, Hk, D, N, C, L, kvd, topo, nwg):
    """The parent-array entry gives, bit for bit, what the dense-mask entry gives
    for the mask the device builder writes from the same parents; both match
    the oracle on the host-built mask."""
    wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=C, L=L, kv_dtype=kvd, topology="chain", nwg=nwg, seed=N + L)
    inp = W.make_tree_inputs(wl)
    par = _parents(topo, L, seed=N)
    inp["mask"] = W.tree_mask(par, N, N)
    got = _run_parents(ta, wl, inp, par, kernel=path)
    p = ta.tree_params(H, Hk, D, N, C, wl.scale, L, N, nwg)
    d_mask = torch.empty((L, N), device="cuda")
    ta.tree_mask_build(p, torch.tensor(par, dtype=torch.int32, device="cuda"), d_mask)
    inp_dev = dict(inp)
    inp_dev["mask"] = d_mask.cpu()
    dense = run_tree(ta, wl, inp_dev, kernel=path)
    assert torch.equal(got, dense)
    assert_close(got.cpu().numpy(), oracle.tree_oracle_for(wl, inp), what="parents %s" % topo)


def test_parent_array_out_of_range_values_end_chains(ta):
    """Values outside [-1, i) end a node's chain there, as in the mask builder."""
    wl = small_tree(H=16, Hk=2, D=128, N=400, C=400, L=12, kv_dtype="f16", nwg=2)
    inp = W.make_tree_inputs(wl)
    par = [-1, 0, 0, 7, 1, -5, 3, 2, 100, 4, 9, 8]    # 3 -> 7 (not smaller), 5 -> -5, 8 -> 100
    ref_par = [-1, 0, 0, -1, 1, -1, 3, 2, -1, 4, 9, 8]
    inp["mask"] = W.tree_mask(ref_par, wl.kv_seq_len, wl.mask_stride)
    got = _run_parents(ta, wl, inp, par).cpu().numpy()
    assert_close(got, oracle.tree_oracle_for(wl, inp))


def test_parent_array_dynamic_tree_workload(ta):
    """The dynamic-tree workload at full size: the parent-array entry equals the
    dense-mask entry bit for bit on every output."""
    wl = W.DYNAMIC_TREE
    inp = W.make_tree_inputs(wl)
    dense = run_tree(ta, wl, inp)
    got = _run_parents(ta, wl, inp, inp["parents"])
    assert torch.equal(got, dense)

"""Pins for the float64 oracle: checks against library routines, closed forms,
hand-worked values from the pages and invariants, never against itself."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ decoders
def test_decode_f16_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode("f16", bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_bf16_all_bit_patterns_match_torch():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ours = oracle.decode("bf16", bits.view(torch.bfloat16))
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ------------------------------------------------------------ tree oracle
def _rand_tree_case(seed, H, Hk, D, N, C, L, stride, kv_dtype, p_attend=0.6, full_rows=True):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((H, L, D), generator=g)
    k = torch.randn((Hk, C, D), generator=g).to(W.DTYPES[kv_dtype])
    v = torch.randn((Hk, C, D), generator=g).to(W.DTYPES[kv_dtype])
    att = torch.rand((L, stride), generator=g) < p_attend
    if full_rows:
        att[:, 0] = True           # every row attends at least one key
    mask = torch.where(att, torch.tensor(0.0), torch.tensor(W.MASKED)).float()
    return q, k, v, mask


def _sdpa_reference(q, k, v, mask, N, scale):
    """torch's scaled_dot_product_attention in float64 with GQA (enable_gqa)."""
    qq = q.double().unsqueeze(0)                                   # [1, H, L, D]
    kk = k[:, :N].double().unsqueeze(0)                            # [1, Hk, N, D]
    vv = v[:, :N].double().unsqueeze(0)
    am = (mask[:, :N] == 0.0).unsqueeze(0).unsqueeze(0)            # True = attend
    o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=am, scale=scale, enable_gqa=True)
    return o[0]                                                    # [H, L, D]


@pytest.mark.parametrize("kv_dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("H,Hk,L", [(4, 2, 3), (6, 3, 5), (2, 2, 1), (8, 1, 4)])
def test_tree_oracle_matches_torch_sdpa(kv_dtype, H, Hk, L):
    D, N, C, stride = 8, 37, 45, 40
    q, k, v, mask = _rand_tree_case(7 + H + L, H, Hk, D, N, C, L, stride, kv_dtype)
    scale = 0.37
    got = oracle.tree_attention(q, k, v, mask, n_heads=H, n_kv_heads=Hk, head_dim=D,
                                kv_seq_len=N, kv_capacity=C, scale=scale, q_l=L,
                                mask_stride=stride, kv_dtype=kv_dtype)
    ref = _sdpa_reference(q, k, v, mask, N, scale).permute(1, 0, 2).numpy()   # -> [L, H, D]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("kv_dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("H,Hk,L", [(4, 2, 3), (6, 3, 5), (8, 1, 4)])
def test_tree_oracle_additive_mask_matches_torch_sdpa_float_mask(kv_dtype, H, Hk, L):
    """The mask is added to the scaled logit (mlx-native tree_attention.metal,
    tree_attention_impl: logit = fma(qk, scale, mask)): finite, non-binary
    cells shift the logits, cells <= -65504 drop the key.  torch SDPA with a
    float attn_mask (the cell where attended, -inf where masked) computes the
    same softmax; a 0 / -65504 mask could not tell adding from gating."""
    D, N, C, stride = 8, 37, 45, 40
    q, k, v, mask = _rand_tree_case(31 + H + L, H, Hk, D, N, C, L, stride, kv_dtype)
    g = torch.Generator().manual_seed(77 + H)
    bias = torch.rand((L, stride), generator=g) * 7.0 - 4.0          # U(-4, 3)
    att = mask == 0.0
    mask = torch.where(att, bias, mask)
    mask[0, 1] = -1.0e30                                              # below -65504: masked too
    mask[0, 0] = 2.5                                                  # row 0 keeps an attended key
    scale = 0.37
    got = oracle.tree_attention(q, k, v, mask, n_heads=H, n_kv_heads=Hk, head_dim=D, kv_seq_len=N,
                                kv_capacity=C, scale=scale, q_l=L, mask_stride=stride, kv_dtype=kv_dtype)
    fm = mask[:, :N].double()
    fm = torch.where(fm <= W.MASKED, torch.tensor(-math.inf, dtype=torch.float64), fm)
    qq = q.double().unsqueeze(0)
    kk = k[:, :N].double().unsqueeze(0)
    vv = v[:, :N].double().unsqueeze(0)
    ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=fm.unsqueeze(0).unsqueeze(0), scale=scale,
                                         enable_gqa=True)[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # and the bias matters: without it the result moves
    plain = oracle.tree_attention(q, k, v, torch.where(mask > W.MASKED, torch.tensor(0.0), mask), n_heads=H,
                                  n_kv_heads=Hk, head_dim=D, kv_seq_len=N, kv_capacity=C, scale=scale, q_l=L,
                                  mask_stride=stride, kv_dtype=kv_dtype)
    assert np.max(np.abs(plain - got)) > 1e-3


def test_tree_oracle_row_subset_matches_full():
    H, Hk, D, N, C, L = 6, 2, 16, 50, 64, 4
    q, k, v, mask = _rand_tree_case(3, H, Hk, D, N, C, L, N, "f16")
    kw = dict(n_heads=H, n_kv_heads=Hk, head_dim=D, kv_seq_len=N, kv_capacity=C, scale=0.25,
              q_l=L, mask_stride=N, kv_dtype="f16")
    full = oracle.tree_attention(q, k, v, mask, **kw)
    rows = [(5, 3), (0, 0), (2, 1)]
    sub = oracle.tree_attention(q, k, v, mask, rows=rows, **kw)
    for s, (h, i) in enumerate(rows):
        assert np.array_equal(sub[s], full[i, h])


def test_tree_oracle_closed_form_golden():
    gdat = _golden("tree_closed_form.json")
    L = len(gdat["mask_rows"])
    N = len(gdat["c"])
    q = torch.full((1, L, 1), gdat["q"][0])
    k = torch.tensor([math.log(c) for c in gdat["c"]], dtype=torch.float32).view(1, N, 1)
    v = torch.tensor(gdat["v"], dtype=torch.float32).view(1, N, 1)
    mask = torch.tensor(gdat["mask_rows"], dtype=torch.float32)
    got = oracle.tree_attention(q, k, v, mask, n_heads=1, n_kv_heads=1, head_dim=1, kv_seq_len=N,
                                kv_capacity=N, scale=1.0, q_l=L, mask_stride=N, kv_dtype="f32")
    np.testing.assert_allclose(got[:, 0, 0], gdat["expected"], rtol=2e-7, atol=0)


def test_tree_oracle_zero_query_gives_mean_of_attended_values():
    H, Hk, D, N, L = 4, 2, 8, 33, 3
    q, k, v, mask = _rand_tree_case(11, H, Hk, D, N, N, L, N, "f32")
    q.zero_()
    got = oracle.tree_attention(q, k, v, mask, n_heads=H, n_kv_heads=Hk, head_dim=D,
                                kv_seq_len=N, kv_capacity=N, scale=1.0, q_l=L, mask_stride=N,
                                kv_dtype="f32")
    g = H // Hk
    for h in range(H):
        for i in range(L):
            att = (mask[i, :N] == 0).numpy()
            expect = v[h // g, :N].double().numpy()[att].mean(axis=0)
            np.testing.assert_allclose(got[i, h], expect, rtol=1e-13, atol=1e-13)


def test_tree_oracle_single_attended_key_returns_its_value_row_exactly():
    H, Hk, D, N, L = 4, 4, 16, 40, 2
    q, k, v, _ = _rand_tree_case(5, H, Hk, D, N, N, L, N, "bf16")
    mask = torch.full((L, N), W.MASKED)
    mask[0, 17] = 0.0
    mask[1, 39] = 0.0
    got = oracle.tree_attention(q, k, v, mask, n_heads=H, n_kv_heads=Hk, head_dim=D, kv_seq_len=N,
                                kv_capacity=N, scale=3.0, q_l=L, mask_stride=N, kv_dtype="bf16")
    for h in range(H):
        assert np.array_equal(got[0, h], v[h, 17].double().numpy())
        assert np.array_equal(got[1, h], v[h, 39].double().numpy())


def test_tree_oracle_output_is_convex_combination():
    H, Hk, D, N, L = 4, 2, 8, 64, 4
    q, k, v, mask = _rand_tree_case(9, H, Hk, D, N, N, L, N, "f16")
    q *= 4.0
    got = oracle.tree_attention(q, k, v, mask, n_heads=H, n_kv_heads=Hk, head_dim=D, kv_seq_len=N,
                                kv_capacity=N, scale=1.0, q_l=L, mask_stride=N, kv_dtype="f16")
    for h in range(H):
        for i in range(L):
            vv = v[h // 2, :N].double().numpy()[(mask[i] == 0).numpy()]
            assert np.all(got[i, h] >= vv.min(axis=0) - 1e-12)
            assert np.all(got[i, h] <= vv.max(axis=0) + 1e-12)


def test_tree_oracle_fully_masked_row_outputs_zero():
    H, Hk, D, N, L = 2, 1, 8, 20, 3
    q, k, v, mask = _rand_tree_case(1, H, Hk, D, N, N, L, N, "f32")
    mask[1] = W.MASKED
    got = oracle.tree_attention(q, k, v, mask, n_heads=H, n_kv_heads=Hk, head_dim=D, kv_seq_len=N,
                                kv_capacity=N, scale=0.5, q_l=L, mask_stride=N, kv_dtype="f32")
    assert np.all(got[1] == 0.0)
    assert np.all(np.abs(got[0]) > 0)


def test_tree_oracle_chain_mask_equals_implicit_causal():
    """The pages' tree=1 parity contract: an explicit causal mask gives the same
    result as the implicit causal mask."""
    wl = W.PR1_CHAIN
    inp = W.make_tree_inputs(wl)
    explicit = oracle.tree_oracle_for(wl, inp)
    implicit = oracle.tree_oracle_for(wl, inp, mask=None)
    assert np.array_equal(explicit, implicit)
    # with a sliding-window start the implicit mask equals causal_mask(window_start)
    m = W.causal_mask(wl.q_l, wl.kv_seq_len, wl.mask_stride, window_start=100)
    inp2 = dict(inp, mask=m)
    a = oracle.tree_oracle_for(wl, inp2)
    b = oracle.tree_oracle_for(wl, inp, mask=None, window_start=100)
    assert np.array_equal(a, b)


def test_tree_oracle_gqa_equals_duplicated_kv_heads():
    H, Hk, D, N, L = 6, 2, 8, 30, 3
    q, k, v, mask = _rand_tree_case(21, H, Hk, D, N, N, L, N, "f32")
    kw = dict(head_dim=D, kv_seq_len=N, kv_capacity=N, scale=0.4, q_l=L, mask_stride=N,
              kv_dtype="f32")
    gqa = oracle.tree_attention(q, k, v, mask, n_heads=H, n_kv_heads=Hk, **kw)
    kd = k.repeat_interleave(H // Hk, dim=0).contiguous()
    vd = v.repeat_interleave(H // Hk, dim=0).contiguous()
    mha = oracle.tree_attention(q, kd, vd, mask, n_heads=H, n_kv_heads=H, **kw)
    assert np.array_equal(gqa, mha)


def test_tree_oracle_key_permutation_invariance():
    H, Hk, D, N, L = 4, 2, 8, 48, 4
    q, k, v, mask = _rand_tree_case(31, H, Hk, D, N, N, L, N, "f32")
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(0))
    kw = dict(n_heads=H, n_kv_heads=Hk, head_dim=D, kv_seq_len=N, kv_capacity=N, scale=0.6,
              q_l=L, mask_stride=N, kv_dtype="f32")
    a = oracle.tree_attention(q, k, v, mask, **kw)
    b = oracle.tree_attention(q, k[:, perm].contiguous(), v[:, perm].contiguous(),
                              mask[:, perm].contiguous(), **kw)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_tree_oracle_ignores_cells_and_rows_beyond_kv_seq_len():
    H, Hk, D, N, C, L, stride = 4, 2, 8, 30, 40, 3, 36
    q, k, v, mask = _rand_tree_case(41, H, Hk, D, N, C, L, stride, "f16")
    kw = dict(n_heads=H, n_kv_heads=Hk, head_dim=D, kv_seq_len=N, kv_capacity=C, scale=0.5,
              q_l=L, mask_stride=stride, kv_dtype="f16")
    a = oracle.tree_attention(q, k, v, mask, **kw)
    m2 = mask.clone()
    m2[:, N:] = 0.0                           # cells >= kv_seq_len flipped to "attend"
    k2, v2 = k.clone(), v.clone()
    k2[:, N:] = float("nan")                  # capacity tail is never read
    v2[:, N:] = float("nan")
    b = oracle.tree_attention(q, k2, v2, m2, **kw)
    assert np.array_equal(a, b)


def test_fixed_tree_topology_golden():
    gdat = _golden("fixed_tree_parents.json")
    assert W.fixed_tree_parents((4, 2, 2, 1, 1), 32) == gdat["parents"]


def test_tree_mask_rows_attend_prefix_ancestors_and_self():
    parents = [-1, 0, 0, 1, 3]
    m = W.tree_mask(parents, kv_seq_len=12, mask_stride=16)
    prefix = 12 - 5
    expect_sets = [{0}, {0, 1}, {0, 2}, {0, 1, 3}, {0, 1, 3, 4}]
    for i, s in enumerate(expect_sets):
        row = m[i]
        assert torch.all(row[:prefix] == 0.0)
        for j in range(5):
            assert (row[prefix + j] == 0.0) == (j in s)
        assert torch.all(row[12:] == W.MASKED)


# ----------------------------------------------------------- quant oracle
def _pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """Test-side packer: element d goes to bits (d % pf) * bits of word d // pf."""
    pf = 32 // bits
    c = codes.reshape(*codes.shape[:-1], -1, pf).astype(np.uint64)
    w = np.zeros(c.shape[:-1], dtype=np.uint64)
    for e in range(pf):
        w |= c[..., e] << np.uint64(e * bits)
    return w.astype(np.uint32)


def test_quant_pack_golden_words_and_unit_affine_dequant():
    gdat = _golden("quant_pack_words.json")
    for case in gdat["cases"]:
        bits = case["bits"]
        codes = np.array(case["codes"], dtype=np.uint32)
        words = np.array([int(w, 16) for w in case["words"]], dtype=np.uint32)
        assert np.array_equal(_pack(codes, bits), words)
        dim = len(codes)
        packed = words.reshape(1, 1, -1)
        one = torch.ones((1, 1, 1), dtype=torch.float16)
        zero = torch.zeros((1, 1, 1), dtype=torch.float16)
        got = oracle.dequant_token(packed, one, zero, dim=dim, tokens=1, bits=bits,
                                   group_size=dim, dtype="f16", kv=0, t=0)
        assert np.array_equal(got, codes.astype(np.float64))


def test_quant_dequant_affine_per_group():
    bits, dim, G, N = 4, 32, 16, 3
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 16, size=(2, N, dim)).astype(np.uint32)
    packed = _pack(codes, bits)
    sc = torch.tensor(rng.uniform(0.5, 2.0, size=(2, N, dim // G)), dtype=torch.bfloat16)
    bi = torch.tensor(rng.normal(size=(2, N, dim // G)), dtype=torch.bfloat16)
    got = oracle.dequant_token(packed, sc, bi, dim=dim, tokens=N, bits=bits, group_size=G,
                               dtype="bf16", kv=1, t=2)
    s = sc[1, 2].double().numpy().repeat(G)
    b = bi[1, 2].double().numpy().repeat(G)
    assert np.array_equal(got, s * codes[1, 2] + b)


def _quant_case(seed, B, nQ, nKV, dim, N, bits, G, dtype, has_sinks, window, bool_frac, fmask):
    g = torch.Generator().manual_seed(seed)
    T = W.DTYPES[dtype]
    rows, kvr = B * nQ, B * nKV
    rng = np.random.default_rng(seed)
    codes_k = rng.integers(0, 1 << bits, size=(kvr, N, dim)).astype(np.uint32)
    codes_v = rng.integers(0, 1 << bits, size=(kvr, N, dim)).astype(np.uint32)
    inp = {
        "queries": torch.randn((rows, dim), generator=g).to(T),
        "k_packed": _pack(codes_k, bits), "v_packed": _pack(codes_v, bits),
        "k_scales": (torch.rand((kvr, N, dim // G), generator=g) * 0.04 + 0.01).to(T),
        "k_biases": (torch.randn((kvr, N, dim // G), generator=g) * 0.1).to(T),
        "v_scales": (torch.rand((kvr, N, dim // G), generator=g) * 0.04 + 0.01).to(T),
        "v_biases": (torch.randn((kvr, N, dim // G), generator=g) * 0.1).to(T),
        "sinks": torch.randn((nQ,), generator=g),
        "mask_bool": None, "mask_float": None,
    }
    if bool_frac > 0:
        inp["mask_bool"] = (torch.rand((rows, N), generator=g) >= bool_frac).to(torch.int32)
    if fmask:
        inp["mask_float"] = (torch.randn((rows, N), generator=g) * 2.0).to(T)
    kw = dict(batch=B, n_q_heads=nQ, n_kv_heads=nKV, dim=dim, tokens=N, bits=bits, group_size=G,
              has_sinks=has_sinks, window_size=window, scale=1.0 / math.sqrt(dim), dtype=dtype)
    return inp, kw


def _dequant_all(inp, kw, which):
    kvr = kw["batch"] * kw["n_kv_heads"]
    N, dim = kw["tokens"], kw["dim"]
    out = np.empty((kvr, N, dim))
    for kv in range(kvr):
        for t in range(N):
            out[kv, t] = oracle.dequant_token(inp[which + "_packed"], inp[which + "_scales"],
                                              inp[which + "_biases"], dim=dim, tokens=N,
                                              bits=kw["bits"], group_size=kw["group_size"],
                                              dtype=kw["dtype"], kv=kv, t=t)
    return out


def _quant_sdpa_reference(inp, kw):
    """torch SDPA (float64, GQA over the B*nQ rows) on the dequantized cache, with
    the sink as an extra zero key/value whose additive bias is the sink logit."""
    B, nQ, nKV, N, dim = kw["batch"], kw["n_q_heads"], kw["n_kv_heads"], kw["tokens"], kw["dim"]
    rows = B * nQ
    kd = torch.tensor(_dequant_all(inp, kw, "k"))
    vd = torch.tensor(_dequant_all(inp, kw, "v"))
    zeros = torch.zeros((B * nKV, 1, dim), dtype=torch.float64)
    kd = torch.cat([kd, zeros], 1)
    vd = torch.cat([vd, zeros], 1)
    bias = torch.zeros((rows, N + 1), dtype=torch.float64)
    if inp["mask_float"] is not None:
        bias[:, :N] += inp["mask_float"].double()
    if inp["mask_bool"] is not None:
        bias[:, :N] = torch.where(inp["mask_bool"] != 0, bias[:, :N], torch.tensor(-math.inf))
    if kw["window_size"]:
        t = torch.arange(N)
        bias[:, :N] = torch.where(t + kw["window_size"] > N - 1, bias[:, :N], torch.tensor(-math.inf))
    if kw["has_sinks"]:
        bias[:, N] = inp["sinks"].double()[torch.arange(rows) % nQ]
    else:
        bias[:, N] = -math.inf
    q = inp["queries"].double().view(1, rows, 1, dim)
    o = F.scaled_dot_product_attention(q, kd.unsqueeze(0), vd.unsqueeze(0),
                                       attn_mask=bias.view(1, rows, 1, N + 1),
                                       scale=kw["scale"], enable_gqa=True)
    return o.view(rows, dim).numpy()


@pytest.mark.parametrize("bits,dim,G,dtype,has_sinks,window,bool_frac,fmask", [
    (4, 32, 16, "f16", 1, 0, 0.0, False),
    (8, 32, 32, "bf16", 0, 0, 0.0, False),
    (4, 64, 32, "bf16", 1, 7, 0.0, False),
    (8, 16, 16, "f16", 0, 0, 0.3, False),
    (4, 32, 32, "f16", 1, 0, 0.0, True),
    (8, 32, 16, "bf16", 1, 9, 0.25, True),
])
def test_quant_oracle_matches_torch_sdpa(bits, dim, G, dtype, has_sinks, window, bool_frac, fmask):
    inp, kw = _quant_case(bits + dim + window, 2, 4, 2, dim, 23, bits, G, dtype, has_sinks,
                          window, bool_frac, fmask)
    got = oracle.quant_sdpa(inp, **kw)
    ref = _quant_sdpa_reference(inp, kw)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_quant_single_token_with_sink_closed_form():
    inp, kw = _quant_case(3, 1, 2, 1, 32, 1, 8, 32, "f16", 1, 0, 0.0, False)
    got = oracle.quant_sdpa(inp, **kw)
    kd = _dequant_all(inp, kw, "k")[0, 0]
    vd = _dequant_all(inp, kw, "v")[0, 0]
    for r in range(2):
        q = inp["queries"][r].double().numpy()
        ell = float(np.dot(q * kw["scale"], kd))
        s = float(inp["sinks"][r])
        expect = vd * math.exp(ell) / (math.exp(ell) + math.exp(s))
        np.testing.assert_allclose(got[r], expect, rtol=1e-12, atol=1e-15)


def test_quant_special_cases_reduce_to_base():
    inp, kw = _quant_case(5, 2, 4, 2, 32, 19, 4, 16, "bf16", 0, 0, 0.0, False)
    base = oracle.quant_sdpa(inp, **kw)
    # window >= tokens is the same as no window
    assert np.array_equal(oracle.quant_sdpa(inp, **dict(kw, window_size=19)), base)
    assert np.array_equal(oracle.quant_sdpa(inp, **dict(kw, window_size=500)), base)
    # an all-ones bool mask is the same as none
    ones = dict(inp, mask_bool=torch.ones((8, 19), dtype=torch.int32))
    assert np.array_equal(oracle.quant_sdpa(ones, **kw), base)
    # a very negative sink is the same as no sink
    neg = dict(inp, sinks=torch.full((4,), -1.0e4))
    np.testing.assert_allclose(oracle.quant_sdpa(neg, **dict(kw, has_sinks=1)), base,
                               rtol=1e-15, atol=0)
    # a constant float bias without a sink changes nothing (shift invariance) ...
    cb = dict(inp, mask_float=torch.full((8, 19), 3.0).to(torch.bfloat16))
    np.testing.assert_allclose(oracle.quant_sdpa(cb, **kw), base, rtol=1e-12, atol=1e-14)
    # ... but with a sink it does
    with_sink = oracle.quant_sdpa(inp, **dict(kw, has_sinks=1))
    with_sink_cb = oracle.quant_sdpa(cb, **dict(kw, has_sinks=1))
    assert np.max(np.abs(with_sink - with_sink_cb)) > 1e-3


def test_quant_no_visible_token_and_no_sink_gives_zero():
    inp, kw = _quant_case(8, 1, 2, 1, 16, 10, 8, 16, "f16", 0, 0, 0.0, False)
    inp["mask_bool"] = torch.zeros((2, 10), dtype=torch.int32)
    inp["mask_bool"][1, 4] = 1
    got = oracle.quant_sdpa(inp, **kw)
    assert np.all(got[0] == 0.0)
    vd = _dequant_all(inp, kw, "v")[0, 4]
    assert np.array_equal(got[1], vd)           # single visible token -> its value row


def test_quant_oracle_row_subset_and_gqa_mapping():
    inp, kw = _quant_case(12, 2, 4, 2, 32, 15, 8, 32, "f16", 1, 0, 0.0, False)
    full = oracle.quant_sdpa(inp, **kw)
    sub = oracle.quant_sdpa(inp, rows=[7, 2], **kw)
    assert np.array_equal(sub[0], full[7]) and np.array_equal(sub[1], full[2])


# ------------------------------------------------------------- tree mask builder
def test_tree_mask_oracle_hand_golden():
    g = json.load(open(os.path.join(GOLDEN, "tree_mask_small.json")))
    m = oracle.tree_mask(g["parents"], kv_seq_len=g["kv_seq_len"], mask_stride=g["mask_stride"])
    assert m.shape == (len(g["parents"]), g["mask_stride"])
    for i, cols in enumerate(g["attended_positions"]):
        want = np.full(g["mask_stride"], -65504.0, dtype=np.float32)
        want[cols] = 0.0
        assert np.array_equal(m[i], want), i


def test_tree_mask_oracle_chain_is_causal():
    # a chain (node i's parent is i - 1) attends exactly keys [0, N - L + i]
    L, N, S = 9, 40, 45
    m = oracle.tree_mask([-1] + list(range(L - 1)), kv_seq_len=N, mask_stride=S)
    j = np.arange(S)[None, :]
    i = np.arange(L)[:, None]
    assert np.array_equal(m == 0.0, (j <= N - L + i))


def test_tree_mask_oracle_matches_transitive_closure():
    rng = np.random.default_rng(11)
    for L in (1, 2, 7, 33):
        par = [-1] + [int(rng.integers(0, i)) for i in range(1, L)]
        N, S = L + 17, L + 20
        m = oracle.tree_mask(par, kv_seq_len=N, mask_stride=S)
        # reachability by repeated squaring of (I + child->parent edges)
        A = np.eye(L, dtype=bool)
        for i, p in enumerate(par):
            if p >= 0:
                A[i, p] = True
        R = A.copy()
        for _ in range(max(1, int(np.ceil(np.log2(L))) + 1)):
            R = R | ((R.astype(np.int64) @ R.astype(np.int64)) > 0)
        P = N - L
        assert np.all(m[:, :P] == 0.0)
        assert np.array_equal(m[:, P:N] == 0.0, R)
        assert np.all(m[:, N:] == -65504.0)


def test_tree_mask_oracle_invalid_links_end_the_chain():
    # node 1 names a later node as its parent and node 3 itself: both chains stop there
    m = oracle.tree_mask([-1, 2, 1, 3], kv_seq_len=6, mask_stride=6)
    att = (m == 0.0)
    P = 2
    assert list(np.flatnonzero(att[1][P:])) == [1]
    assert list(np.flatnonzero(att[2][P:])) == [1, 2]
    assert list(np.flatnonzero(att[3][P:])) == [3]

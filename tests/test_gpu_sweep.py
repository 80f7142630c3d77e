"""Seeded sweeps of random shapes through both paths, against the float64
oracle: head counts, head dimensions, KV types, lengths (ragged chunks and
tiles), tree sizes and topologies, split counts, and for the quantized path
bits, group sizes, rows per KV row, windows, sinks and masks - on both kernel
families.  Catches shape-dependent faults that the hand-picked cases miss."""
import math
import random

import pytest
import torch

import oracle
import workloads as W
from helpers import assert_close, run_quant, run_tree, small_tree

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tree_masked_speculative_gb300 as m
    return m


def _tree_case(rng):
    D = rng.choice([128, 256, 512])
    Hk = rng.choice([1, 2, 4])
    g = rng.choice([1, 2, 3, 4, 8])
    L = rng.choice([1, 2, 5, 8, 13, 24, 32])
    N = rng.randint(max(L, 20), 1400 if D < 512 else 700)
    C = N + rng.choice([0, 7, 64])
    kvd = rng.choice(["f32", "f16", "bf16"])
    topo = rng.choice(["dynamic", "fixed", "chain"])
    nwg = rng.choice([0, 0, 1, 3, 7])
    return dict(H=Hk * g, Hk=Hk, D=D, N=N, C=C, L=L, kv_dtype=kvd, topology=topo, nwg=nwg,
                seed=rng.randint(1, 10 ** 6))


TREE_SWEEP = [_tree_case(random.Random(1000 + i)) for i in range(18)]


@pytest.mark.parametrize("kw", TREE_SWEEP, ids=[str(i) for i in range(len(TREE_SWEEP))])
def test_tree_sweep(ta, kw):
    wl = small_tree(**kw)
    inp = W.make_tree_inputs(wl)
    ref = oracle.tree_oracle_for(wl, inp)
    got = run_tree(ta, wl, inp).cpu().double().numpy()
    assert_close(got, ref, what="tree sweep %r" % (kw,))


def _quant_case(rng):
    bits = rng.choice([4, 8])
    dim = rng.choice([64, 128, 256] if bits == 4 else [64, 128])
    G = rng.choice([g for g in (32, 64, 128) if dim % g == 0 and g <= dim])
    nKV = rng.choice([1, 2])
    rep = rng.choice([1, 3, 4, 8, 16, 20, 32, 40])
    N = rng.randint(40, 900)
    window = rng.choice([0, 0, rng.randint(1, N)])
    fmask = rng.choice(["none", "alibi"])
    bfrac = rng.choice([0.0, 0.0, 0.15])
    return dict(batch=rng.choice([1, 2]), n_q_heads=nKV * rep, n_kv_heads=nKV, dim=dim, tokens=N, bits=bits,
                group_size=G, has_sinks=rng.choice([0, 1]), window_size=window, dtype=rng.choice(["f16", "bf16"]),
                float_mask=fmask, bool_mask_frac=bfrac, nwg=rng.choice([0, 0, 1, 5]), seed=rng.randint(1, 10 ** 6))


QUANT_SWEEP = [_quant_case(random.Random(2000 + i)) for i in range(18)]


@pytest.mark.parametrize("path", [2, 1], ids=["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("kw", QUANT_SWEEP, ids=[str(i) for i in range(len(QUANT_SWEEP))])
def test_quant_sweep(ta, kw, path):
    wl = W.QuantWorkload(name="sweep", scale=1.0 / math.sqrt(kw["dim"]), **kw)
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=path).cpu().double().numpy()
    assert_close(got, ref, what="quant sweep %r" % (kw,))


def _layout_case(rng):
    """Mask rows padded past N (mask_stride > N), or the implicit causal mask
    with a random window start."""
    kw = _tree_case(rng)
    N = kw["N"]
    kw["stride"] = N + rng.choice([0, 5, 64, 333])
    causal = rng.random() < 0.5
    ws = rng.randint(0, N - kw["L"]) if causal and rng.random() < 0.6 else 0
    return kw, causal, ws


LAYOUT_SWEEP = [_layout_case(random.Random(3000 + i)) for i in range(12)]


@pytest.mark.parametrize("case", LAYOUT_SWEEP, ids=[str(i) for i in range(len(LAYOUT_SWEEP))])
def test_tree_layout_sweep(ta, case):
    kw, causal, ws = case
    wl = small_tree(**kw)
    inp = W.make_tree_inputs(wl)
    ref = oracle.tree_oracle_for(wl, inp, mask=None if causal else "explicit", window_start=ws)
    got = run_tree(ta, wl, inp, causal=causal, window_start=ws).cpu().double().numpy()
    assert_close(got, ref, what="tree layout sweep %r causal=%d ws=%d" % (kw, causal, ws))


def _draft_tree_case(rng):
    """Draft-tree nodes on a quantized cache: n_q_heads = heads x q_l rows, each
    block of q_l rows carrying the fixed tree's float mask."""
    kw = _quant_case(rng)
    q_l = rng.choice([4, 8, 16])
    heads = rng.choice([1, 2, 4])
    kw["n_q_heads"] = kw["n_kv_heads"] * heads * q_l
    kw["float_mask"] = "tree%d" % q_l
    kw["window_size"] = 0
    return kw


DRAFT_SWEEP = [_draft_tree_case(random.Random(4000 + i)) for i in range(10)]


@pytest.mark.parametrize("path", [2, 1], ids=["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("kw", DRAFT_SWEEP, ids=[str(i) for i in range(len(DRAFT_SWEEP))])
def test_quant_draft_tree_sweep(ta, kw, path):
    wl = W.QuantWorkload(name="sweep", scale=1.0 / math.sqrt(kw["dim"]), **kw)
    inp = W.make_quant_inputs(wl)
    ref = oracle.quant_oracle_for(wl, inp)
    got = run_quant(ta, wl, inp, out_dtype=torch.float32, kernel=path).cpu().double().numpy()
    assert_close(got, ref, what="quant draft-tree sweep %r" % (kw,))

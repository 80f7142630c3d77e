"""GPU parity of the tree tensor-core kernel's flattened CTA-pair schedule.

With head dim 512 and more than 128 rows per KV head the main pass runs as CTA
pairs.  When the library picks the split count and the uniform split would leave
SMs idle (the number of units, KV heads x pairs of row tiles, does not divide
the pair-groups the GPU holds), each pair-group takes a contiguous range of the
(unit, key tile) positions that may cross from one unit into the next; each part
leaves its own partial slot and the slots no group fills are marked empty.
These cases pick shapes that take that path on a GPU with 152 SMs (38
pair-groups) and compare with the float64 oracle, bit-identity contracts
included."""
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


def _flat_slots(H, Hk, L, N):
    """Partial slots the flattened schedule leaves per row, or None when the
    shape keeps the uniform split on this GPU: the most pair-groups that one
    unit's key tiles meet when U x tpu positions are cut into G ranges
    [g W / G, (g + 1) W / G)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    G = sms // 4
    R = H // Hk * L
    n_rt = (R + 127) // 128
    U = Hk * ((n_rt + 1) // 2)
    tpu = ((N + 31) // 32 + 3) // 4
    Wp = U * tpu
    if R <= 128 or U > G or G % U == 0 or Wp < G:
        return None
    owner = [max(g for g in range(G) if g * Wp // G <= P) for P in range(Wp)]
    return max(owner[(u + 1) * tpu - 1] - owner[u * tpu] + 1 for u in range(U))


FLAT_CASES = [
    # H, Hk, D, N, C, L, kv_dtype: R = H / Hk * L > 128 rows per KV head
    (32, 4, 512, 700, 704, 40, "bf16"),    # 320 rows: 2 pairs of row tiles per KV head, 8 units of 6 tiles
    (24, 3, 512, 2000, 2000, 24, "f16"),   # 192 rows: 3 units of 16 tiles
    (40, 5, 512, 1200, 1216, 20, "bf16"),  # 160 rows: 5 units of 10 tiles, a ragged last chunk
]


@pytest.mark.parametrize("H,Hk,D,N,C,L,kvd", FLAT_CASES)
def test_flat_schedule_matches_oracle(ta, H, Hk, D, N, C, L, kvd):
    slots = _flat_slots(H, Hk, L, N)
    if slots is None:
        pytest.skip("this GPU keeps the uniform split for the shape")
    wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=C, L=L, kv_dtype=kvd, nwg=0, seed=N + L)
    p = ta.tree_params(H, Hk, D, N, C, wl.scale, L, N, 0)
    assert ta.tree_attn_num_splits(p) == slots
    inp = W.make_tree_inputs(wl)
    got = run_tree(ta, wl, inp).cpu().numpy()
    assert_close(got, oracle.tree_oracle_for(wl, inp), what="flat %s" % (wl,))


def test_flat_schedule_dead_chunks_and_masked_rows(ta):
    """Chunks no row attends are skipped inside a group's range (a segment may
    hold no live tile at all) and a row with no attended key gives zeros."""
    H, Hk, D, N, L = 32, 4, 512, 1500, 40
    assert _flat_slots(H, Hk, L, N) is not None
    wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=N, L=L, kv_dtype="bf16", nwg=0, seed=3)
    inp = W.make_tree_inputs(wl)
    m = inp["mask"]
    m[5] = W.MASKED
    m[:, 96:900] = W.MASKED
    m[11, 1000:1460] = W.MASKED
    got = run_tree(ta, wl, inp).cpu().numpy()
    assert np.all(got[5] == 0.0)
    assert_close(got, oracle.tree_oracle_for(wl, inp))


def test_flat_schedule_explicit_causal_bit_identical_to_implicit(ta):
    H, Hk, D, N, L = 24, 3, 512, 2000, 24
    assert _flat_slots(H, Hk, L, N) is not None
    wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=N, L=L, kv_dtype="bf16", nwg=0, topology="chain")
    inp = W.make_tree_inputs(wl)
    inp["mask"] = W.causal_mask(L, N, N, window_start=200)
    explicit = run_tree(ta, wl, inp)
    implicit = run_tree(ta, wl, inp, causal=True, window_start=200)
    assert torch.equal(explicit, implicit)
    assert_close(explicit.cpu().numpy(), oracle.tree_oracle_for(wl, inp, mask=None, window_start=200))


def test_flat_schedule_parent_array_bit_identical_to_dense(ta):
    H, Hk, D, N, L = 32, 4, 512, 700, 40
    assert _flat_slots(H, Hk, L, N) is not None
    wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=N, L=L, kv_dtype="bf16", nwg=0, topology="chain", seed=9)
    inp = W.make_tree_inputs(wl)
    par = W.dynamic_tree_parents(L, torch.Generator().manual_seed(9))
    inp["mask"] = W.tree_mask(par, N, N)
    d = to_dev(inp)
    out = ta.tree_attention(d["q"], d["k"], d["v"], None, n_heads=H, n_kv_heads=Hk, kv_seq_len=N,
                            scale=wl.scale, mask_stride=N, nwg=0,
                            parents=torch.tensor(par, dtype=torch.int32, device="cuda"))
    dense = run_tree(ta, wl, inp)
    torch.cuda.synchronize()
    assert torch.equal(out, dense)
    assert_close(out.cpu().numpy(), oracle.tree_oracle_for(wl, inp))


def test_uniform_split_kept_when_the_units_divide_the_groups(ta):
    """Two KV heads of one row-tile pair divide 38 groups: the uniform split
    count (38 / 2 = 19 per unit, capped by the key tiles) stays."""
    H, Hk, D, N, L = 16, 2, 512, 4000, 20
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if (sms // 4) % 2 != 0:
        pytest.skip("needs an even number of pair-groups")
    assert _flat_slots(H, Hk, L, N) is None
    wl = small_tree(H=H, Hk=Hk, D=D, N=N, C=N, L=L, kv_dtype="bf16", nwg=0, seed=4)
    inp = W.make_tree_inputs(wl)
    assert_close(run_tree(ta, wl, inp).cpu().numpy(), oracle.tree_oracle_for(wl, inp))

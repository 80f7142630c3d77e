"""Seeded synthetic inputs for the tree-verify and quantized-KV attention workloads.

This module only draws random numbers and lays them out.  It holds none of the
attention arithmetic: both the CPU oracle (``oracle/``) and the CUDA library
(``tree_masked_speculative_gb300``) consume what it returns, and neither imports
the other.

Tree topologies (chains, fixed trees, dynamic asymmetric trees) are turned into
the explicit ``[q_l, mask_stride]`` float mask the tree-attention kernel reads
(0.0 = attend, -65504.0 = masked), as described in the header comment of the
tree-attention Metal shader (mlx-native ``tree_attention.metal``) and in the
``tree_attention`` buffer docs of ``tree_attention.rs``.  How the mask is built
from a topology is not shown on those pages; here a tree node attends the
committed prefix, its ancestors and itself.

Draw order (all from one ``torch.Generator`` seeded with ``seed``):
  tree workloads : [dynamic parents] -> Q -> K -> V  (K/V drawn over the full
                   kv_capacity so the unused tail holds finite data)
  quant workloads: queries -> k_packed -> k_scales -> k_biases -> v_packed ->
                   v_scales -> v_biases -> sinks -> bool-mask subsets
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

MASKED = -65504.0
ATTENDED = 0.0

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


# ----------------------------------------------------------------------------
# Tree-attention workloads
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class TreeWorkload:
    name: str
    n_heads: int
    n_kv_heads: int
    head_dim: int
    kv_seq_len: int
    kv_capacity: int
    q_l: int
    mask_stride: int
    scale: float
    kv_dtype: str            # "f32" | "f16" | "bf16"
    topology: str            # "chain" | "fixed" | "dynamic"
    branching: tuple = ()    # fixed trees: children per node at each depth
    kv_std: float = 1.0
    q_std: float = 1.0
    nwg: int = 0             # 0 = library's choice
    seed: int = 0

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    @property
    def kv_bytes(self) -> int:
        """K and V bytes of positions [0, kv_seq_len), once per KV head."""
        elt = torch.tensor([], dtype=DTYPES[self.kv_dtype]).element_size()
        return 2 * self.n_kv_heads * self.kv_seq_len * self.head_dim * elt

    def with_(self, **kw) -> "TreeWorkload":
        return dataclasses.replace(self, **kw)


def fixed_tree_parents(branching, n_nodes: int) -> List[int]:
    """Breadth-first node list of a tree whose depth-d nodes each have
    branching[d] children; node 0 is the root.  Truncated to n_nodes."""
    parents = [-1]
    level = [0]
    depth = 0
    while len(parents) < n_nodes and depth < len(branching) and level:
        nxt = []
        for p in level:
            for _ in range(branching[depth]):
                if len(parents) >= n_nodes:
                    break
                parents.append(p)
                nxt.append(len(parents) - 1)
        level = nxt
        depth += 1
    if len(parents) < n_nodes:
        raise ValueError("branching factors give fewer than n_nodes nodes")
    return parents


def dynamic_tree_parents(n_nodes: int, gen: torch.Generator) -> List[int]:
    """Node 0 is the root; node i >= 1 takes a parent drawn uniformly from 0..i-1."""
    parents = [-1]
    for i in range(1, n_nodes):
        parents.append(int(torch.randint(0, i, (1,), generator=gen).item()))
    return parents


def chain_parents(n_nodes: int) -> List[int]:
    return [-1] + list(range(n_nodes - 1))


def ancestor_sets(parents: List[int]) -> List[List[int]]:
    out = []
    for i in range(len(parents)):
        s = []
        j = i
        while j >= 0:
            s.append(j)
            j = parents[j]
        out.append(sorted(s))
    return out


def tree_mask(parents: List[int], kv_seq_len: int, mask_stride: int,
              fill_tail: float = MASKED) -> torch.Tensor:
    """Explicit mask [q_l, mask_stride] f32.  Tree node i sits at KV position
    kv_seq_len - q_l + i and attends the prefix [0, kv_seq_len - q_l) plus its
    ancestors and itself.  Cells j >= kv_seq_len hold ``fill_tail`` (the kernel
    ignores them)."""
    q_l = len(parents)
    prefix = kv_seq_len - q_l
    if prefix < 0:
        raise ValueError("q_l > kv_seq_len")
    m = torch.full((q_l, mask_stride), MASKED, dtype=torch.float32)
    m[:, :prefix] = ATTENDED
    for i, anc in enumerate(ancestor_sets(parents)):
        for a in anc:
            m[i, prefix + a] = ATTENDED
    if mask_stride > kv_seq_len:
        m[:, kv_seq_len:] = fill_tail
    return m


def causal_mask(q_l: int, kv_seq_len: int, mask_stride: int, window_start: int = 0,
                fill_tail: float = MASKED) -> torch.Tensor:
    """Row i attends keys [window_start, kv_seq_len - q_l + i]."""
    m = torch.full((q_l, mask_stride), MASKED, dtype=torch.float32)
    for i in range(q_l):
        hi = kv_seq_len - q_l + i
        if hi >= window_start:
            m[i, window_start:hi + 1] = ATTENDED
    if mask_stride > kv_seq_len:
        m[:, kv_seq_len:] = fill_tail
    return m


def tree_parents_for(wl: TreeWorkload, gen: torch.Generator) -> List[int]:
    if wl.topology == "chain":
        return chain_parents(wl.q_l)
    if wl.topology == "fixed":
        return fixed_tree_parents(wl.branching, wl.q_l)
    if wl.topology == "dynamic":
        return dynamic_tree_parents(wl.q_l, gen)
    raise ValueError(wl.topology)


def make_tree_inputs(wl: TreeWorkload) -> dict:
    """Host tensors: q [H, L, D] f32, k/v [Hk, C, D] kv_dtype, mask [L, stride] f32."""
    g = torch.Generator().manual_seed(wl.seed)
    parents = tree_parents_for(wl, g)
    H, Hk, D, C, L = wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.kv_capacity, wl.q_l
    q = (torch.randn((H, L, D), generator=g, dtype=torch.float32) * wl.q_std).contiguous()
    kvd = DTYPES[wl.kv_dtype]
    k = (torch.randn((Hk, C, D), generator=g, dtype=torch.float32) * wl.kv_std).to(kvd)
    v = (torch.randn((Hk, C, D), generator=g, dtype=torch.float32) * wl.kv_std).to(kvd)
    mask = tree_mask(parents, wl.kv_seq_len, wl.mask_stride)
    return {"q": q, "k": k, "v": v, "mask": mask, "parents": parents}


# The five named workloads.  Sizes follow the pages' problem statement; where a
# size is left open the plainest reading is taken (kv_capacity = kv_seq_len and
# scale = 1/sqrt(head_dim) for the dynamic tree; sigma = 0.5 for "N(0, 0.5)").
PR1_CHAIN = TreeWorkload(
    name="pr1_chain_h4_kv2_d128_n256_q8_f32", n_heads=4, n_kv_heads=2, head_dim=128,
    kv_seq_len=256, kv_capacity=256, q_l=8, mask_stride=256, scale=1.0 / math.sqrt(128),
    kv_dtype="f32", topology="chain", nwg=32, seed=1001)

FIXED_TREE = TreeWorkload(
    name="fixed_tree_h24_kv4_d256_n4096_q32_f16", n_heads=24, n_kv_heads=4, head_dim=256,
    kv_seq_len=4096, kv_capacity=8192, q_l=32, mask_stride=4096, scale=1.0 / 16.0,
    kv_dtype="f16", topology="fixed", branching=(4, 2, 2, 1, 1), seed=1002)

DYNAMIC_TREE = TreeWorkload(
    name="dynamic_tree_h32_kv8_d512_n32768_q64_bf16", n_heads=32, n_kv_heads=8, head_dim=512,
    kv_seq_len=32768, kv_capacity=32768, q_l=64, mask_stride=32768,
    scale=1.0 / math.sqrt(512), kv_dtype="bf16", topology="dynamic", kv_std=0.5, seed=1003)


# ----------------------------------------------------------------------------
# Affine-quantized KV workloads
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class QuantWorkload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    dim: int
    tokens: int
    bits: int
    group_size: int
    has_sinks: int
    window_size: int
    scale: float
    dtype: str                  # T: "f16" | "bf16"
    float_mask: str = "none"    # "none" | "alibi" | "tree<q_l>": n_q_heads = heads x q_l draft
                                # nodes (rows (batch, head, node)), each row's fixed-tree mask
    bool_mask_frac: float = 0.0  # 0 = no bool mask
    nwg: int = 0
    seed: int = 0

    @property
    def repeat_count(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def rows(self) -> int:
        return self.batch * self.n_q_heads

    @property
    def kv_rows(self) -> int:
        return self.batch * self.n_kv_heads

    @property
    def window_tokens(self) -> int:
        return self.tokens if self.window_size == 0 else min(self.window_size, self.tokens)

    @property
    def bytes_per_token(self) -> int:
        """Packed words + scales + biases of one token of K (same for V)."""
        words = self.dim * self.bits // 32
        groups = self.dim // self.group_size
        return 4 * words + 2 * 2 * groups

    @property
    def kv_bytes(self) -> int:
        """K and V bytes of the tokens inside the window, once per KV head."""
        return 2 * self.kv_rows * self.window_tokens * self.bytes_per_token

    def with_(self, **kw) -> "QuantWorkload":
        return dataclasses.replace(self, **kw)


def alibi_mask(rows: int, n_q_heads: int, tokens: int, dtype: torch.dtype) -> torch.Tensor:
    """ALiBi bias slope_h * (t - tokens + 1), slope_h = 2^(-8 h / n_q_heads) with a
    1-based head index h = (row mod n_q_heads) + 1."""
    h = (torch.arange(rows, dtype=torch.float64) % n_q_heads) + 1.0
    slope = torch.pow(2.0, -8.0 * h / n_q_heads)
    t = torch.arange(tokens, dtype=torch.float64) - (tokens - 1)
    return (slope[:, None] * t[None, :]).to(torch.float32).to(dtype).contiguous()


def make_quant_inputs(wl: QuantWorkload) -> dict:
    """Host tensors laid out as the quantized-SDPA page states:
    queries [B*nQ, dim] T; k/v_packed [B*nKV, N, dim*bits/32] u32 (int32 storage);
    k/v_scales and k/v_biases [B*nKV, N, dim/G] T; sinks [nQ] f32;
    mask_bool [B*nQ, N] u32 (or None); mask_float [B*nQ, N] T (or None);
    tree_parents: for a "tree<q_l>" float mask, the parent list of that draft
    tree (row r is node r % q_l over the last q_l tokens), else None."""
    g = torch.Generator().manual_seed(wl.seed)
    T = DTYPES[wl.dtype]
    rows, kvr, N = wl.rows, wl.kv_rows, wl.tokens
    words = wl.dim * wl.bits // 32
    groups = wl.dim // wl.group_size
    queries = torch.randn((rows, wl.dim), generator=g, dtype=torch.float32).to(T)

    def packed():
        # Uniformly random 32-bit words hold independent uniform codes in every
        # bits-wide field, which is what "codes uniform 0..2^bits-1" asks for.
        return torch.randint(-(2 ** 31), 2 ** 31, (kvr, N, words), generator=g,
                             dtype=torch.int64).to(torch.int32)

    def scales():
        return (torch.rand((kvr, N, groups), generator=g, dtype=torch.float32) * 0.04 + 0.01).to(T)

    def biases():
        return (torch.randn((kvr, N, groups), generator=g, dtype=torch.float32) * 0.1).to(T)

    k_packed, k_scales, k_biases = packed(), scales(), biases()
    v_packed, v_scales, v_biases = packed(), scales(), biases()
    sinks = torch.randn((wl.n_q_heads,), generator=g, dtype=torch.float32)
    mask_bool = None
    if wl.bool_mask_frac > 0:
        n_zero = int(round(wl.bool_mask_frac * N))
        mask_bool = torch.ones((rows, N), dtype=torch.int32)
        for r in range(rows):
            idx = torch.randperm(N, generator=g)[:n_zero]
            mask_bool[r, idx] = 0
    mask_float = None
    tree_parents = None
    if wl.float_mask == "alibi":
        mask_float = alibi_mask(rows, wl.n_q_heads, N, T)
    elif wl.float_mask.startswith("tree"):
        q_l = int(wl.float_mask[len("tree"):])
        tree_parents = fixed_tree_parents((4, 2, 2, 1, 1), q_l)
        tm = tree_mask(tree_parents, N, N)      # [q_l, N]
        mask_float = tm.repeat(rows // q_l, 1).to(T)
    return {"queries": queries, "k_packed": k_packed, "k_scales": k_scales,
            "k_biases": k_biases, "v_packed": v_packed, "v_scales": v_scales,
            "v_biases": v_biases, "sinks": sinks, "mask_bool": mask_bool,
            "mask_float": mask_float, "tree_parents": tree_parents}


QUANT_B4 = QuantWorkload(
    name="quant_b4_B4_q32_kv8_d128_n16384_sinks_f16", batch=4, n_q_heads=32, n_kv_heads=8,
    dim=128, tokens=16384, bits=4, group_size=64, has_sinks=1, window_size=0,
    scale=1.0 / math.sqrt(128), dtype="f16", seed=1004)

QUANT_B8_MASKS = QuantWorkload(
    name="quant_b8_B8_q32_kv8_d256_n65536_w4096_alibi_bool_bf16", batch=8, n_q_heads=32,
    n_kv_heads=8, dim=256, tokens=65536, bits=8, group_size=64, has_sinks=0,
    window_size=4096, scale=1.0 / math.sqrt(256), dtype="bf16", float_mask="alibi",
    bool_mask_frac=0.1, seed=1005)

# A draft tree verified on a quantized cache: 32 heads x 8 fixed-tree nodes as
# query rows over 8 KV heads (32 rows per KV row), 4-bit d128 cache.
QUANT_TREE = QuantWorkload(
    name="quant_tree_B1_h32xq8_kv8_d128_n16384_4bit_f16", batch=1, n_q_heads=256, n_kv_heads=8,
    dim=128, tokens=16384, bits=4, group_size=64, has_sinks=0, window_size=0,
    scale=1.0 / math.sqrt(128), dtype="f16", float_mask="tree8", seed=1006)

TREE_WORKLOADS = {w.name: w for w in (PR1_CHAIN, FIXED_TREE, DYNAMIC_TREE)}
QUANT_WORKLOADS = {w.name: w for w in (QUANT_B4, QUANT_B8_MASKS, QUANT_TREE)}

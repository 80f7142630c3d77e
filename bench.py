#!/usr/bin/env python3
"""Benchmark of the tree-verify attention step (and the quantized-KV variant).

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dynamic_tree|fixed_tree|pr1_chain|quant_b4|quant_b8_masks|quant_tree]

A step is one verify pass over one batch of synthetic inputs: mask compaction
+ main pass + split merge (tree), or main pass + merge (quantized).  The
headline is KV-cache bytes streamed per second (K and V of positions
[0, kv_seq_len), once per KV head) over the device-timed region.  Inputs are
resident in HBM; K/V rotate over enough copies that the bytes read per pass of
the rotation exceed 3x the L2 size, so every step reads cold K/V.  Prints one
JSON line.  The default workload is the largest single-GPU one, the dynamic
asymmetric tree (537 MB of K/V per step).

One GPU per process: the verify step of one sequence never needs more, and
the library has no multi-GPU path, so --gpus > 1 (or a multi-rank launch) is
refused with an error.  The reference arm (--impl reference, the float64 CPU
oracle) runs on rank 0 alone; other ranks exit at once.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "tree-verify attention KV GB/s and % of HBM roofline; μs per verify step"
WORKLOADS = {"pr1_chain": W.PR1_CHAIN, "fixed_tree": W.FIXED_TREE, "dynamic_tree": W.DYNAMIC_TREE,
             "quant_b4": W.QUANT_B4, "quant_b8_masks": W.QUANT_B8_MASKS, "quant_tree": W.QUANT_TREE}
L2_BYTES = 129 * 1024 * 1024
GRAPH_STEPS = 500


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dynamic_tree", choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile", action="store_true",
                    help="run --warmup eager steps and exit (a short, graph-free run for a profiler)")
    ap.add_argument("--mask-build", action="store_true",
                    help="tree workloads: also time the device-side tree-mask build from the parent array")
    ap.add_argument("--kernel", type=int, default=0, choices=[0, 1, 2, 3],
                    help="kernel family of the main pass: 0 automatic, 1 CUDA cores, 2 tcgen05 tensor cores "
                         "where the shape allows them, 3 (quantized only) warp MMA where the shape allows it")
    ap.add_argument("--tree-mask", default="dense", choices=["dense", "parents"],
                    help="tree and draft-tree workloads: the mask as the dense array (tree_attn_fwd, "
                         "quant_sdpa_fwd) or as the parent array (tree_attn_fwd_parents, quant_sdpa_fwd_tree)")
    ap.add_argument("--kv-sets", type=int, default=0,
                    help="K/V copies to rotate over (0 = enough to exceed 3x L2)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def refuse_multi_gpu(args, ws):
    """This bench (and the library) runs one GPU per process; a request for more
    is an error, not a silently smaller run."""
    if args.gpus != 1 or ws != 1:
        sys.stderr.write("bench.py: one GPU per process (got --gpus %d, WORLD_SIZE %d); the library has no "
                         "multi-GPU path\n" % (args.gpus, ws))
        sys.exit(2)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(device_index)
        self.ident = ident

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names[1:], parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------- tree arm
class TreeBench:
    def __init__(self, ta, wl: W.TreeWorkload, dev, kv_sets=0, tree_mask="dense", kernel=0):
        self.ta, self.wl, self.dev = ta, wl, dev
        self.kernel = kernel
        inp = W.make_tree_inputs(wl)
        self.host = inp
        self.q = inp["q"].to(dev)
        self.mask = inp["mask"].to(dev)
        per_set = wl.kv_bytes + self.q.numel() * 4 + self.mask.numel() * 4
        self.nsets = kv_sets or max(1, math.ceil(3 * L2_BYTES / per_set))
        k, v = inp["k"].to(dev), inp["v"].to(dev)
        self.ks = [k] + [k.clone() for _ in range(self.nsets - 1)]
        self.vs = [v] + [v.clone() for _ in range(self.nsets - 1)]
        self.p = ta.tree_params(wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.kv_seq_len,
                                wl.kv_capacity, wl.scale, wl.q_l, wl.mask_stride, wl.nwg)
        self.nwg = ta.tree_attn_num_splits(self.p)
        ws = ta.tree_attn_workspace_bytes(self.p)
        self.tmp = torch.empty((ws + 3) // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((wl.q_l, wl.n_heads, wl.head_dim), dtype=torch.float32, device=dev)
        self.bytes_per_step = wl.kv_bytes
        self.name = wl.name
        self.dtype = wl.kv_dtype
        self.parents = torch.tensor(inp["parents"], dtype=torch.int32, device=dev) if "parents" in inp else None
        self.use_parents = tree_mask == "parents"
        self.fwd_label = ("ancestor bitsets + mask compaction + main pass (tree_attn_fwd_parents)"
                          if self.use_parents else "mask compaction + main pass (tree_attn_fwd)")
        self.traffic_key = traffic_key(wl.name, self.use_parents, kernel)
        self.built_mask = None

    def mask_step(self, i):
        """The device-side tree-mask build from the parent array (into its own buffer)."""
        if self.built_mask is None:
            self.built_mask = torch.empty_like(self.mask)
        self.ta.tree_mask_build(self.p, self.parents, self.built_mask)

    def _fwd(self, q, m, k, v):
        ta = self.ta
        kind = ta.MASK_PARENTS if self.use_parents else ta.MASK_DENSE
        ta.tree_attn_fwd_ex(self.p, self.kernel, kind, 0, q, k, v, m, self.tmp, self.out)

    def step(self, i, fwd_only=False):
        s = i % self.nsets
        self._fwd(self.q, self.parents if self.use_parents else self.mask, self.ks[s], self.vs[s])
        if not fwd_only:
            self.ta.tree_attn_reduce(self.p, self.tmp, self.out)

    def status_word(self):
        """The device status word of the last main pass (0 = every bounded wait completed)."""
        off = self.ta.tree_attn_status_offset(self.p)
        return int(self.tmp.view(torch.int32)[off // 4].item())

    def config(self):
        wl = self.wl
        return {"workload": wl.name, "n_heads": wl.n_heads, "n_kv_heads": wl.n_kv_heads,
                "head_dim": wl.head_dim, "kv_seq_len": wl.kv_seq_len, "kv_capacity": wl.kv_capacity,
                "q_l": wl.q_l, "kv_dtype": wl.kv_dtype, "splits": self.nwg,
                "tree_mask": "parent array" if self.use_parents else "dense f32",
                "l2": "rotating %d K/V sets, %.0f MB read per rotation (> 3x L2)" % (
                    self.nsets, self.nsets * self.bytes_per_step / 1e6)}

    # end to end through host buffers: Q, mask, K/V[0:N) in, output out
    def e2e_setup(self):
        wl = self.wl
        N = wl.kv_seq_len
        self.h_q = self.host["q"].pin_memory()
        self.h_mask = (torch.tensor(self.host["parents"], dtype=torch.int32) if self.use_parents
                       else self.host["mask"]).pin_memory()
        self.h_k = self.host["k"][:, :N].contiguous().pin_memory()
        self.h_v = self.host["v"][:, :N].contiguous().pin_memory()
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.e2e_h2d = sum(t.numel() * t.element_size() for t in (self.h_q, self.h_mask, self.h_k, self.h_v))
        self.e2e_d2h = self.h_out.numel() * 4
        # two device input sets: step i + 1's inputs land in one while step i reads the other
        m = self.parents if self.use_parents else self.mask
        k1 = self.ks[1] if self.nsets > 1 else self.ks[0].clone()
        v1 = self.vs[1] if self.nsets > 1 else self.vs[0].clone()
        self.e2e_sets = [(self.q, m, self.ks[0], self.vs[0]), (self.q.clone(), m.clone(), k1, v1)]

    def e2e_copy_in(self, i):
        N = self.wl.kv_seq_len
        q, m, k, v = self.e2e_sets[i % 2]
        q.copy_(self.h_q, non_blocking=True)
        m.copy_(self.h_mask, non_blocking=True)
        for h in range(self.wl.n_kv_heads):   # contiguous [N, D] runs, one copy each
            k[h, :N].copy_(self.h_k[h], non_blocking=True)
            v[h, :N].copy_(self.h_v[h], non_blocking=True)

    def e2e_compute(self, i):
        q, m, k, v = self.e2e_sets[i % 2]
        self._fwd(q, m, k, v)
        self.ta.tree_attn_reduce(self.p, self.tmp, self.out)
        self.h_out.copy_(self.out, non_blocking=True)

    def cpu_reference(self, rows, threads):
        import oracle
        return oracle.tree_oracle_for(self.wl, self.host, rows=rows, threads=threads)

    def all_rows(self):
        return [(h, i) for h in range(self.wl.n_heads) for i in range(self.wl.q_l)]


# ------------------------------------------------------------ quant arm
class QuantBench:
    def __init__(self, ta, wl: W.QuantWorkload, dev, kv_sets=0, kernel=0, tree_mask="dense"):
        self.ta, self.wl, self.dev = ta, wl, dev
        inp = W.make_quant_inputs(wl)
        self.oracle_inputs = inp             # the same mask, dense, for the CPU baseline
        # a draft-tree workload may take its tree mask as the parent array (no mask read)
        self.tree = None
        if tree_mask == "parents" and inp.get("tree_parents") is not None:
            self.tree = torch.tensor(inp["tree_parents"], dtype=torch.int32, device=dev)
            inp = dict(inp, mask_float=None)
        self.host = inp
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        self.d = d
        per_set = wl.kv_bytes
        self.nsets = kv_sets or max(1, math.ceil(3 * L2_BYTES / per_set))
        kv_keys = ["k_packed", "k_scales", "k_biases", "v_packed", "v_scales", "v_biases"]
        self.sets = [{k: d[k] for k in kv_keys}]
        for _ in range(self.nsets - 1):
            self.sets.append({k: d[k].clone() for k in kv_keys})
        self.p = ta.quant_params(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.dim, wl.tokens, wl.bits,
                                 wl.group_size, wl.has_sinks, wl.window_size, wl.scale, wl.nwg, kernel)
        self.nwg = ta.quant_sdpa_num_splits(self.p)
        nb = ta.quant_sdpa_tmp_bytes(self.p)
        # the status word (tmp's first 32-bit word) is sticky: zeroed here, ORed by the kernel
        self.tmp = torch.zeros(max(1, (nb + 3) // 4), dtype=torch.float32, device=dev)
        self.out = torch.empty((wl.rows, wl.dim), dtype=d["queries"].dtype, device=dev)
        self.bytes_per_step = wl.kv_bytes
        self.name = wl.name
        self.dtype = "u%d" % wl.bits
        self.family = ta.quant_sdpa_kernel_family(self.p)
        self.tc = self.family != ta.KERNEL_CUDA_CORES
        fam = {ta.KERNEL_TENSOR_CORES: ("quant_tc_kernel (tcgen05 tensor cores)", "tcgen05 tensor cores"),
               ta.KERNEL_WARP_MMA: ("quant_mma_kernel (warp MMA tensor cores)", "warp MMA tensor cores"),
               ta.KERNEL_CUDA_CORES: ("quant_kernel (CUDA cores)", "CUDA cores")}
        kern, self.family_name = fam[self.family]
        rep = wl.n_q_heads // wl.n_kv_heads
        if self.family == ta.KERNEL_WARP_MMA and rep >= 16 and wl.dim in (64, 128) and wl.group_size in (32, 64):
            kern = "quant_mma16_kernel (warp MMA tensor cores, 16 rows per warp)"
        call = "quant_sdpa_fwd_tree" if self.tree is not None else "quant_sdpa_fwd"
        self.fwd_label = "main pass (%s) + split merge (%s, one call)" % (kern, call)
        self.traffic_key = traffic_key(wl.name, self.tree is not None, kernel)

    def _fwd(self, e, kv):
        if self.tree is not None:
            self.ta.quant_sdpa_fwd_tree(self.p, int(self.tree.numel()), self.tree, e["queries"], kv["k_packed"],
                                        kv["k_scales"], kv["k_biases"], kv["v_packed"], kv["v_scales"],
                                        kv["v_biases"], e["sinks"] if self.wl.has_sinks else None,
                                        e.get("mask_bool"), self.tmp, self.out)
        else:
            self.ta.quant_sdpa_fwd(self.p, e["queries"], kv["k_packed"], kv["k_scales"], kv["k_biases"],
                                   kv["v_packed"], kv["v_scales"], kv["v_biases"],
                                   e["sinks"] if self.wl.has_sinks else None, e.get("mask_bool"),
                                   e.get("mask_float"), self.tmp, self.out)

    def step(self, i, fwd_only=False):
        self._fwd(self.d, self.sets[i % self.nsets])

    def config(self):
        wl = self.wl
        return {"workload": wl.name, "batch": wl.batch, "n_q_heads": wl.n_q_heads,
                "n_kv_heads": wl.n_kv_heads, "dim": wl.dim, "tokens": wl.tokens, "bits": wl.bits,
                "group_size": wl.group_size, "window_size": wl.window_size, "splits": self.nwg,
                "kernel": self.family_name,
                "tree_mask": "parent array" if self.tree is not None else None,
                "l2": "rotating %d K/V sets, %.0f MB read per rotation (> 3x L2)" % (
                    self.nsets, self.nsets * self.bytes_per_step / 1e6)}

    def e2e_setup(self):
        wl = self.wl
        lo = wl.tokens - wl.window_tokens
        self.h = {}
        for k in ("queries", "k_packed", "k_scales", "k_biases", "v_packed", "v_scales", "v_biases"):
            t = self.host[k]
            if k != "queries":
                t = t[:, lo:]
            self.h[k] = t.contiguous().pin_memory()
        for k in ("mask_bool", "mask_float"):
            if self.host.get(k) is not None and not (k == "mask_float" and self.tree is not None):
                self.h[k] = self.host[k][:, lo:].contiguous().pin_memory()
        if self.tree is not None:
            self.h["tree_parents"] = self.tree.cpu().pin_memory()
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.e2e_h2d = sum(t.numel() * t.element_size() for t in self.h.values())
        self.e2e_d2h = self.h_out.numel() * self.h_out.element_size()
        # two device input sets: step i + 1's inputs land in one while step i reads the other
        first = dict(self.d)
        first.update(self.sets[0])
        kv = set(self.sets[0])
        second = {k: (v.clone() if isinstance(v, torch.Tensor) and k not in kv else v) for k, v in self.d.items()}
        second.update(self.sets[1] if self.nsets > 1 else {k: v.clone() for k, v in self.sets[0].items()})
        self.e2e_sets = [first, second]

    def e2e_copy_in(self, i):
        wl = self.wl
        lo = wl.tokens - wl.window_tokens
        e = self.e2e_sets[i % 2]
        e["queries"].copy_(self.h["queries"], non_blocking=True)
        for k in ("k_packed", "k_scales", "k_biases", "v_packed", "v_scales", "v_biases"):
            e[k][:, lo:].copy_(self.h[k], non_blocking=True)
        for k in ("mask_bool", "mask_float"):
            if k in self.h:
                e[k][:, lo:].copy_(self.h[k], non_blocking=True)
        if self.tree is not None:
            self.tree.copy_(self.h["tree_parents"], non_blocking=True)

    def e2e_compute(self, i):
        e = self.e2e_sets[i % 2]
        self._fwd(e, e)
        self.h_out.copy_(self.out, non_blocking=True)

    def status_word(self):
        """ORed device status of every call since tmp was zeroed (0 = every bounded wait completed)."""
        return int(self.tmp[:1].view(torch.int32).item())

    def cpu_reference(self, rows, threads):
        import oracle
        return oracle.quant_oracle_for(self.wl, self.oracle_inputs, rows=rows, threads=threads)

    def all_rows(self):
        return list(range(self.wl.rows))


def make_bench(ta, name, dev, kv_sets=0, tree_mask="dense", kernel=0):
    wl = WORKLOADS[name]
    if isinstance(wl, W.TreeWorkload):
        return TreeBench(ta, wl, dev, kv_sets, tree_mask, kernel)
    return QuantBench(ta, wl, dev, kv_sets, kernel, tree_mask)


# ------------------------------------------------------------ timing
def capture(fn, n, start):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(start + i)
    return g


def timed_graph_steps(fn, steps, start):
    """Time exactly `steps` calls of fn on the device; returns (ms_total, launches_per_step)."""
    import tree_masked_speculative_gb300 as ta
    full, rem = divmod(steps, GRAPH_STEPS)
    c0 = ta.ta_launch_count()
    g = capture(fn, GRAPH_STEPS, start) if full else None
    per_step = (ta.ta_launch_count() - c0) / GRAPH_STEPS if full else None
    c1 = ta.ta_launch_count()
    gr = capture(fn, rem, start) if rem else None
    if per_step is None:
        per_step = (ta.ta_launch_count() - c1) / max(rem, 1)
    # one untimed replay of each graph first: a graph's first launch also
    # uploads it to the device, which is not a cost of the steps
    for gg in (g, gr):
        if gg is not None:
            gg.replay()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(full):
        g.replay()
    if gr is not None:
        gr.replay()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), per_step


def cpu_baseline(bench, seconds):
    rows = bench.all_rows()
    threads = host_threads()
    t0 = time.perf_counter()
    bench.cpu_reference(rows[:1], threads)
    t_row = max(time.perf_counter() - t0, 1e-6)
    n = max(1, min(len(rows), int(seconds / t_row * min(threads, len(rows)) * 0.5)))
    step = max(1, len(rows) // n)
    sample = rows[::step][:n]
    t0 = time.perf_counter()
    bench.cpu_reference(sample, threads)
    dt = time.perf_counter() - t0
    full_s = dt * len(rows) / len(sample)
    return {"value": bench.bytes_per_step / full_s / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d of %d query rows of one step (float64 C oracle, %d threads), %.1f s, "
                      "scaled to a full step" % (len(sample), len(rows), threads, dt)}


def check_status(bench, where):
    """Every bounded wait of the timed kernels completed (a timed-out wait would
    have left the output invalid)."""
    st = bench.status_word()
    if st != 0:
        raise RuntimeError("device status word %#x after the %s: a bounded wait gave up" % (st, where))
    return st


def run_ours(args):
    ws, rank, local = dist_env()
    refuse_multi_gpu(args, ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from tree_masked_speculative_gb300 import build as b
    b.build()
    import tree_masked_speculative_gb300 as ta

    bench = make_bench(ta, args.workload, dev, args.kv_sets, args.tree_mask, args.kernel)
    if args.profile:
        for i in range(max(1, args.warmup)):
            bench.step(i)
        torch.cuda.synchronize()
        check_status(bench, "profile steps")
        print(json.dumps({"profile_run": bench.name, "eager_steps": max(1, args.warmup)}), flush=True)
        return
    # warm-up (untimed): eager steps, then enough graph replays to bring clocks up
    for i in range(max(3, args.warmup)):
        bench.step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    g = capture(bench.step, GRAPH_STEPS, 0)
    t_end = time.time() + 1.0
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize()
    del g
    ms, launches_per_step = timed_graph_steps(bench.step, args.steps, 0)
    check_status(bench, "timed steps")
    # the dominant pass alone (mask compaction + main kernel), same rotation, for the roofline
    ms_fwd, _ = timed_graph_steps(lambda i: bench.step(i, fwd_only=True), args.steps, 0)
    ms_mask = None
    if args.mask_build and isinstance(bench, TreeBench) and bench.parents is not None:
        ms_mask, _ = timed_graph_steps(bench.mask_step, args.steps, 0)
    clocks = sampler.stop()

    # end to end: every step's inputs from pinned host memory and its output back, through the
    # public API; step i + 1's copies (second stream, second device input set) overlap step i.
    # The steps are captured in a CUDA graph (as a serving loop would), so the host's per-call
    # work is not timed; every copy still runs in every step.
    bench.e2e_setup()
    s = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        cur = torch.cuda.current_stream()
        for b in range(2):
            free[b].record(cur)
        for i in range(n):
            b = i % 2
            copy_s.wait_event(free[b])         # step i - 2 is done reading input set b
            with torch.cuda.stream(copy_s):
                bench.e2e_copy_in(i)
                ready[b].record(copy_s)
            cur.wait_event(ready[b])
            bench.e2e_compute(i)
            free[b].record(cur)
        cur.wait_stream(copy_s)

    e2e_run(3)
    torch.cuda.synchronize()
    per_graph = max(2, min(50, args.e2e_steps))
    replays = max(1, -(-args.e2e_steps // per_graph))
    e2e_steps = per_graph * replays
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge):
        e2e_run(per_graph)
    ge.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(replays):
        ge.replay()
    e1.record(s)                               # after the last output copy
    torch.cuda.synchronize()
    del ge
    ms_e2e = e0.elapsed_time(e1)
    status = check_status(bench, "end-to-end steps")

    peak, peak_kind = load_peaks()
    us_step = ms * 1e3 / args.steps
    value = bench.bytes_per_step * args.steps / (ms * 1e-3) / 1e9
    achieved = bench.bytes_per_step * args.steps / (ms_fwd * 1e-3) / 1e9
    traffic = committed_traffic(bench.traffic_key)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "us_per_step": round(us_step, 3), "pct_of_hbm_peak": round(100 * value / peak, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": bench.dtype,
        "data": "synthetic (seeded, shapes of the named workload)", "config": bench.config(),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": bench.fwd_label + ", timed alone",
                     "peak_kind": peak_kind + " (MEASURED_PEAKS hbm_gbs)"},
        "e2e": {"value": round(bench.bytes_per_step * e2e_steps / (ms_e2e * 1e-3) / 1e9, 2),
                "unit": "GB/s", "h2d_bytes_per_step": bench.e2e_h2d,
                "d2h_bytes_per_step": bench.e2e_d2h, "steps": e2e_steps,
                "us_per_step": round(ms_e2e * 1e3 / e2e_steps, 3),
                "overlap": "step i+1's host-to-device copies on a second stream during step i",
                "launch": "CUDA graphs of %d steps" % per_graph},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "device_status": status,
        "clocks": clocks,
    }
    if ms_mask is not None:
        mb = bench.mask.numel() * 4                       # every mask cell written once
        gbs = mb * args.steps / (ms_mask * 1e-3) / 1e9
        line["mask_build"] = {"us_per_build": round(ms_mask * 1e3 / args.steps, 3), "bytes": mb,
                              "achieved": round(gbs, 2), "unit": "GB/s", "peak": peak,
                              "frac": round(gbs / peak, 4), "bound": "hbm (writes)"}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(bench, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def traffic_key(name, parents, kernel):
    """Entry of the committed DRAM-traffic table for a workload run: the mask
    form and a forced kernel family select different kernels."""
    return name + ("|parents" if parents else "") + ("|kernel%d" % kernel if kernel else "")


def committed_traffic(key):
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    or None when absent or taken on an older version of the kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(key)
        if not ent:
            return None
        import hashlib
        h = hashlib.sha256()
        for rel in ent["sources"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        return ent["bytes_per_launch"] if h.hexdigest() == ent["sha256"] else None
    except Exception:
        return None


def run_reference(args):
    """The float64 CPU oracle as it stands, on this machine's host cores: each step
    computes a bounded sample of the workload's query rows."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return                       # the other ranks exit 0 without work
    import oracle
    oracle.build()

    class _NoDev:
        pass

    wl = WORKLOADS[args.workload]
    threads = host_threads()
    if isinstance(wl, W.TreeWorkload):
        host = W.make_tree_inputs(wl)
        rows = [(h, i) for h in range(wl.n_heads) for i in range(wl.q_l)]
        run = lambda sample: oracle.tree_oracle_for(wl, host, rows=sample, threads=threads)
        bytes_per_step = wl.kv_bytes
        cfg = {"workload": wl.name, "n_heads": wl.n_heads, "n_kv_heads": wl.n_kv_heads,
               "head_dim": wl.head_dim, "kv_seq_len": wl.kv_seq_len, "q_l": wl.q_l,
               "kv_dtype": wl.kv_dtype}
        dtype = "f64"
    else:
        host = W.make_quant_inputs(wl)
        rows = list(range(wl.rows))
        run = lambda sample: oracle.quant_oracle_for(wl, host, rows=sample, threads=threads)
        bytes_per_step = wl.kv_bytes
        cfg = {"workload": wl.name, "dim": wl.dim, "tokens": wl.tokens, "bits": wl.bits}
        dtype = "f64"
    t0 = time.perf_counter()
    run(rows[:threads])
    t_blk = time.perf_counter() - t0                    # one row per thread
    budget = 120.0
    total_steps = args.steps + args.warmup
    per_step_budget = budget / total_steps
    n = max(1, min(len(rows), int(per_step_budget / max(t_blk, 1e-6) * threads)))
    stride = max(1, len(rows) // n)
    sample = rows[::stride][:n]
    steps_run = args.steps
    est = t_blk * max(1, math.ceil(n / threads)) * total_steps
    if est > 3 * budget:
        steps_run = max(1, int(3 * budget / (t_blk * max(1, math.ceil(n / threads)))) - args.warmup)
    for _ in range(args.warmup):
        run(sample)
    t0 = time.perf_counter()
    for _ in range(steps_run):
        run(sample)
    dt = time.perf_counter() - t0
    full_step_s = dt / steps_run * len(rows) / len(sample)
    value = bytes_per_step / full_step_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": ws, "steps": steps_run, "warmup": args.warmup,
            "ms_per_step": full_step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic (seeded)", "config": cfg,
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle",
                             "sample": "%d of %d query rows per step, scaled to a full step"
                                       % (len(sample), len(rows))},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

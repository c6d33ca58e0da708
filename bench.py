"""Benchmark of one tree-verification step on GB300.

A step is the whole hot path over one batch: tree-causal paged attention with
the ancestor bits derived from the parent array and split-KV merge (tv_attn),
vocab argmax and greedy acceptance (tv_accept), for one layer's attention.
The metric is verified tree nodes per second per layer (nb * B / step time).

Default workload (the largest single-GPU one): 4 sequences, Qwen3-8B attention
shape (32 q / 8 kv heads, head dim 128, bf16), 32768-token prefixes in shuffled
16-token pages, 256-node best-first draft trees, 151936-entry bf16 logits.
Inputs are seeded synthetic tensors of those shapes, resident in HBM; L2 is
flushed (a 512 MB write) before every timed step.  The same process then
measures the four smaller workloads (``per_config``) with the same flush.

  python bench.py [--gpus N --steps K --warmup W] [--config 1..5] [--impl reference]

Under torchrun (N > 1) every rank runs an independent replica (the step has no
cross-GPU exchange); value = all ranks' nodes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "tree-verify attn verified nodes/s per layer; % of roofline (HBM or TC)"
UNIT = "nodes/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 data-sheet figures: HBM3e bandwidth and dense bf16 tensor throughput
NOMINAL_PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}
DEFAULT_CONFIG = 5


# ----------------------------------------------------------------------------- bookkeeping

def tree_depth(parent: np.ndarray) -> np.ndarray:
    d = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return d


def attn_bytes(w: wl.Workload) -> int:
    """K+V read once per (sequence, kv head) + Q + O (bf16) + LSE (fp32)."""
    kv = 2 * int(np.sum(w.prefix_lens.astype(np.int64) + w.B)) * w.Hkv * w.D * 2
    return kv + 2 * w.nb * w.B * w.Hq * w.D * 2 + w.nb * w.B * w.Hq * 4


def attn_flops(w: wl.Workload) -> int:
    """QK^T and PV over the prefix (dense) and over ancestor pairs only inside the tree."""
    tot = 0
    for b in range(w.nb):
        tot += 4 * w.Hq * w.D * (w.B * int(w.prefix_lens[b]) + int(np.sum(tree_depth(w.parent[b]) + 1)))
    return tot


def accept_bytes(w: wl.Workload) -> int:
    return w.nb * w.B * w.V * 2


def source_hash(name: str) -> str:
    import hashlib
    with open(os.path.join(ROOT, "tree_speculative_decoding_tv_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel: str, src: str, config):
    """DRAM bytes per launch (read + write) from the committed ncu summary of this kernel and
    workload (a config number, or a workload tag), or None when there is none or the kernel
    source changed since it was taken."""
    tag = f"config{config}" if isinstance(config, int) else config
    path = os.path.join(ROOT, "profiles", f"{kernel}_{tag}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = dict(line.split(":", 1) for line in text.splitlines() if line.startswith(("source_sha256_16:", "traffic_bytes_per_launch:")))
    if fields.get("source_sha256_16", "").strip() != source_hash(src):
        return None
    try:
        return float(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured (MEASURED_PEAKS.json)"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback (no MEASURED_PEAKS.json)"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = time.time()
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, t_begin: float, t_end: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        n = 0
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            n += 1
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples come ~100 ms apart from t0; keep the ones inside the timed window when there are any
        dt = (time.time() - self.t0) / max(1, len(rows))
        times = [self.t0 + (k + 0.5) * dt for k in range(len(rows))]
        inside = [r for r, t in zip(rows, times) if t_begin <= t <= t_end]
        sel = inside if inside else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in sel for k in range(4) if r[2][k].lower().startswith("active")})
        return {"sm_mhz": float(np.median([r[0] for r in sel])), "sm_max_mhz": max(r[1] for r in sel),
                "reasons": reasons, "samples": len(sel),
                "window": "a load window of the same steps plus the timed steps" if inside else "whole run"}


# ----------------------------------------------------------------------------- GPU arm

class Step:
    """Device-resident inputs, preallocated outputs and one verify step through the C ABI."""

    def __init__(self, w: wl.Workload, dev: str):
        import torch
        import tree_speculative_decoding_tv_gb300 as tv
        self.torch, self.tv, self.w = torch, tv, w

        def bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

        self.q, self.k, self.v = bf(w.q), bf(w.k_cache), bf(w.v_cache)
        self.bt, self.pl, self.parent, self.draft = i32(w.block_table), i32(w.prefix_lens), i32(w.parent), i32(w.draft)
        self.logits = bf(w.logits)
        W = (w.B + 31) // 32
        self.mask = torch.empty((w.nb, w.B, W), dtype=torch.int32, device=dev)
        self.depth = torch.empty((w.nb, w.B), dtype=torch.int32, device=dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((w.nb * w.B, w.Hq), dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        args = tv.attn_args(self.q, self.k, self.v, self.bt, self.pl, self.mask, self.o, self.lse, self.status)
        self.ws = torch.zeros(tv.attn_workspace_size(args), dtype=torch.uint8, device=dev)
        self.acc_out = (torch.empty(w.nb * w.B, dtype=torch.int32, device=dev),
                        torch.empty(w.nb, dtype=torch.int32, device=dev),
                        torch.empty((w.nb, w.B), dtype=torch.int32, device=dev),
                        torch.empty(w.nb, dtype=torch.int32, device=dev))
        self.acc_ws = torch.zeros(tv.accept_workspace_size(w.V, w.B, w.nb), dtype=torch.uint8, device=dev)
        # the attention (1, or 2 with the split-KV merge kernel), argmax, acceptance (the masks are folded in)
        self.launches_per_step = tv.attn_launches(tv.attn_args(self.q, self.k, self.v, self.bt, self.pl, None, self.o,
                                                               self.lse, self.status, parent=self.parent)) + 2
        self.g_step = self.g_attn = self.g_acc = None

    # The step is the folded form: the attention and the acceptance walk derive the ancestor
    # bits from the parent array, so no mask kernel runs (the fastest form measured; the
    # breakdown times the others).
    def _attn_stage(self):
        self.tv.attn(self.q, self.k, self.v, self.bt, self.pl, None, status=self.status, o=self.o, lse=self.lse,
                     workspace=self.ws, parent=self.parent)

    def _accept_stage(self):
        self.tv.accept(self.logits, self.draft, self.parent, None, status=self.status, out=self.acc_out,
                       workspace=self.acc_ws)

    def time_step_form(self, flush, steps, form):
        """Mean ms of one form of the whole step (its own graph, same flush, own outputs):
        "mask": tv_build_mask + attention (+ merge) + argmax + walk;
        "folded": attention and walk build the ancestor bits from the parent array (no mask kernel);
        "fused": folded, with argmax and walk in one kernel, tv_accept_fused."""
        torch, tv = self.torch, self.tv
        dev = self.q.device
        ws = torch.zeros(tv.accept_fused_workspace_size(self.w.V, self.w.B, self.w.nb), dtype=torch.uint8, device=dev)
        o, lse = torch.empty_like(self.o), torch.empty_like(self.lse)
        out = tuple(torch.empty_like(t) for t in self.acc_out)
        mask = torch.empty_like(self.mask)

        def step():
            if form == "mask":
                tv.build_mask(self.parent, status=self.status, mask=mask)
                tv.attn(self.q, self.k, self.v, self.bt, self.pl, mask, status=self.status, o=o, lse=lse,
                        workspace=self.ws)
                tv.accept(self.logits, self.draft, self.parent, mask, status=self.status, out=out, workspace=ws)
            else:
                tv.attn(self.q, self.k, self.v, self.bt, self.pl, None, status=self.status, o=o, lse=lse,
                        workspace=self.ws, parent=self.parent)
                if form == "folded":
                    tv.accept(self.logits, self.draft, self.parent, None, status=self.status, out=out, workspace=ws)
                else:
                    tv.accept_fused(self.logits, self.draft, self.parent, None, status=self.status, out=out,
                                    workspace=ws)

        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        return self.time_stage(g, flush, steps)

    def time_accept_fused(self, flush, steps, with_mask=True):
        """Mean ms of tv_accept_fused (argmax and walk in one kernel) on the same inputs, with the
        step's mask or building it from the parent array, for comparison with the two-kernel
        tv_accept the step uses (its own graph, same flush)."""
        torch, tv = self.torch, self.tv
        ws = torch.zeros(tv.accept_fused_workspace_size(self.w.V, self.w.B, self.w.nb), dtype=torch.uint8,
                         device=self.q.device)
        out = tuple(torch.empty_like(t) for t in self.acc_out)
        mask = None
        if with_mask:  # the step itself builds no mask array
            tv.build_mask(self.parent, status=self.status, mask=self.mask)
            mask = self.mask
        tv.accept_fused(self.logits, self.draft, self.parent, mask, status=self.status, out=out, workspace=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tv.accept_fused(self.logits, self.draft, self.parent, mask, status=self.status, out=out, workspace=ws)
        return self.time_stage(g, flush, steps)

    def capture(self):
        """Record the step into one CUDA graph (and each stage into its own graph, for the
        per-stage timing); replays launch the same kernels with no host work."""
        torch = self.torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._attn_stage()
            self._accept_stage()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.g_step, self.g_attn, self.g_acc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_step):
            self._attn_stage()
            self._accept_stage()
        with torch.cuda.graph(self.g_attn):
            self._attn_stage()
        with torch.cuda.graph(self.g_acc):
            self._accept_stage()
        torch.cuda.synchronize()

    def run(self, ev=None):
        """One step (one graph replay); ev = 2 events around it."""
        if ev is not None:
            ev[0].record()
        self.g_step.replay()
        if ev is not None:
            ev[1].record()

    def time_commit(self, flush, steps):
        """Mean ms of tv_kv_commit (commit of the accepted branch found by the step) replayed from
        its own graph with the same flush, and the bytes it moves.  Run last: it rewrites the
        caches' tree positions."""
        torch, tv = self.torch, self.tv
        n_acc, path = self.acc_out[1], self.acc_out[2]
        self.new_pl = torch.empty_like(self.pl)
        kv = (self.k.view(torch.int16), self.v.view(torch.int16))
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            tv.kv_commit(*kv, self.bt, self.pl, n_acc, path, new_prefix_lens=self.new_pl, status=self.status)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tv.kv_commit(*kv, self.bt, self.pl, n_acc, path, new_prefix_lens=self.new_pl, status=self.status)
        ms = self.time_stage(g, flush, steps)
        # rows that move (path[k] != k), K and V, read and written
        nacc, pth = n_acc.cpu().numpy(), path.cpu().numpy()
        moved = sum(int(np.sum(pth[b, 1:nacc[b] + 1] != np.arange(1, nacc[b] + 1))) for b in range(self.w.nb))
        return ms, moved * self.w.Hkv * 2 * self.w.D * 2 * 2

    # Per-depth candidate tables for tv_build_tree on the best-first workloads: K candidates
    # per depth (the recipe's child cap) drawn as the top K of Dirichlet(0.3) over 8, depth cap.
    TREE_SHAPES = {2: (16, 4), 3: (12, 3), 5: (24, 4)}

    def time_tree(self, config, flush, steps, w=1):
        """Mean ms of tv_build_tree for this workload's budget (its own graph, same flush), or None."""
        if config not in self.TREE_SHAPES:
            return None
        torch, tv = self.torch, self.tv
        Dmax, K = self.TREE_SHAPES[config]
        rng = np.random.default_rng(99)
        p = rng.dirichlet([0.3] * 8, size=(self.w.nb, Dmax))
        lp = np.log(-np.sort(-p, axis=-1)[..., :K] + 1e-12).astype(np.float32)
        tok = rng.integers(0, self.w.V, size=(self.w.nb, Dmax, K)).astype(np.int32)
        d_lp, d_tok = torch.from_numpy(lp).to(self.q.device), torch.from_numpy(tok).to(self.q.device)
        out = tv.build_tree(d_lp, d_tok, self.w.B, w, status=self.status)  # warm (outside the graph)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tv.build_tree(d_lp, d_tok, self.w.B, w, out=out, status=self.status)
        return self.time_stage(g, flush, steps)

    def time_gdn(self, flush, steps):
        """Mean ms of tv_gdn_tree on the Gated DeltaNet tree workload (its own graph, same flush)
        and that call's algorithmic bytes (q, k, v, gates, S0 in; O out); then the same for
        tv_gdn_commit along the tree's deepest root path (S0 in, the path's k/v/gates, S out)."""
        torch, tv = self.torch, self.tv
        g_w = wl.gdn_config(seed=5)
        dev = self.q.device
        f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        bf = lambda a: f(a.view(np.int16)).view(torch.bfloat16)
        q, k, v = bf(g_w.q), bf(g_w.k), bf(g_w.v)
        a, b, S0, par = f(g_w.alpha), f(g_w.beta), f(g_w.S0), f(g_w.parent)
        out = tv.gdn_tree(q, k, v, a, b, S0, par, status=self.status)  # warm (outside the graph)
        ws = torch.empty(tv.lib().tv_gdn_tree_workspace_size(g_w.nb, g_w.B, g_w.H, g_w.D), dtype=torch.uint8,
                         device=dev)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tv.gdn_tree(q, k, v, a, b, S0, par, out=out, workspace=ws, status=self.status)
        rows = g_w.nb * g_w.B * g_w.H
        nbytes = rows * g_w.D * (3 * 2 + 4) + rows * 8 + g_w.S0.nbytes + g_w.parent.nbytes
        ms = self.time_stage(g, flush, steps)
        # the state commit along the deepest root path (the longest accepted branch)
        h_par = g_w.parent[0]
        dep = np.zeros(g_w.B, np.int64)
        for i in range(1, g_w.B):
            dep[i] = dep[h_par[i]] + 1
        node, path = int(np.argmax(dep)), []
        while node != -1:
            path.append(node)
            node = int(h_par[node])
        path = path[::-1]
        p_host = np.full((1, g_w.B), -1, np.int32)
        p_host[0, :len(path)] = path
        n_acc = torch.tensor([len(path) - 1], dtype=torch.int32, device=dev)
        d_path = f(p_host)
        S_new = torch.empty_like(S0)
        tv.gdn_commit(k, v, a, b, S0, n_acc, d_path, out=S_new, status=self.status)
        torch.cuda.synchronize()
        gc = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gc):
            tv.gdn_commit(k, v, a, b, S0, n_acc, d_path, out=S_new, status=self.status)
        commit_ms = self.time_stage(gc, flush, steps)
        commit_bytes = 2 * g_w.S0.nbytes + len(path) * g_w.H * (g_w.D * 4 + 8)
        return ms, nbytes, g_w.name, commit_ms, commit_bytes, len(path)

    def time_stage(self, graph, flush, steps):
        """Mean ms of one stage graph replay, L2 flushed before each (CUDA events, current stream)."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            flush.zero_()
            a.record()
            graph.replay()
            b.record()
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank calls it (an all-reduce MAX); one rank returns ms."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(nodes_per_rank: int, world: int, total_ms: float, steps: int) -> float:
    """Whole-job throughput: every rank's nodes over the slowest rank's mean step time."""
    return nodes_per_rank * world / (total_ms / steps * 1e-3)


def stage_rooflines(w: wl.Workload, t_attn: float, t_acc: float, peaks: dict, peak_src: str, config):
    """Rooflines of the attention stage (tensor- or HBM-bound, whichever floor is higher) and of
    the acceptance stage (HBM), for stage times in seconds.  frac is against the measured peak
    (peaks), frac_nominal against the GB300 data-sheet figure (NOMINAL_PEAKS)."""
    ab, af, lb = attn_bytes(w), attn_flops(w), accept_bytes(w)
    kname = ("attention stage: tree_attn_kernel (ancestor bits from the parent array; split-KV merge inside, or "
             "tree_attn_merge_kernel after it when split tiles have many parts)")
    if af / (peaks["bf16_tflops"] * 1e12) >= ab / (peaks["hbm_gbs"] * 1e9):
        attn = {"kernel": kname, "bound": "tensor", "achieved": af / t_attn / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "peak_nominal": NOMINAL_PEAKS["bf16_tflops"]}
    else:
        attn = {"kernel": kname, "bound": "hbm", "achieved": ab / t_attn / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "peak_nominal": NOMINAL_PEAKS["hbm_gbs"]}
    acc = {"kernel": "argmax_span_kernel + accept_kernel (tv_accept)", "bound": "hbm",
           "achieved": lb / t_acc / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "peak_nominal": NOMINAL_PEAKS["hbm_gbs"]}
    for r, src, name in ((attn, "tv_attn.cu", "tree_attn_kernel"), (acc, "tv_accept.cu", "argmax_span_kernel")):
        r["frac"] = r["achieved"] / r["peak"]
        r["frac_nominal"] = r["achieved"] / r["peak_nominal"]
        r["peak_source"] = peak_src + " burst; frac_nominal is of the GB300 data-sheet figure"
        r["traffic"] = profiled_traffic(name, src, config)
        r["algorithmic_bytes"] = ab if src == "tv_attn.cu" else lb
        if src == "tv_attn.cu":
            r["algorithmic_flops"] = af
    return attn, acc


def measure_config(n: int, dev: str, flush, steps: int, warmup: int, seed: int) -> dict:
    """Step, attention-stage and acceptance-stage times of workload n, each from its own
    graph replayed `steps` times with the L2 flush before every replay (the headline's timing
    rules), and the stages' roofline fractions."""
    import torch
    w = wl.config(n, seed=seed)
    st = Step(w, dev)
    st.capture()
    for _ in range(warmup):
        st.run()
    torch.cuda.synchronize()
    step_ms = st.time_stage(st.g_step, flush, steps)
    attn_ms = st.time_stage(st.g_attn, flush, steps)
    acc_ms = st.time_stage(st.g_acc, flush, steps)
    if st.status.item() != 0:
        raise RuntimeError(f"device status {st.status.item()} on workload {n}")
    peaks, peak_src = load_peaks()
    attn, acc = stage_rooflines(w, attn_ms * 1e-3, acc_ms * 1e-3, peaks, peak_src, n)
    nodes = w.nb * w.B
    out = {"workload": wl.CONFIG_NAMES[n], "nodes_per_s": nodes / (step_ms * 1e-3), "step_us": step_ms * 1e3,
           "attention_stage_us": attn_ms * 1e3, "attention_bound": attn["bound"],
           "attention_frac": attn["frac"], "attention_frac_nominal": attn["frac_nominal"],
           "attention_traffic": attn["traffic"], "accept_us": acc_ms * 1e3, "accept_frac": acc["frac"],
           "accept_frac_nominal": acc["frac_nominal"], "attention_bytes": attn_bytes(w),
           "attention_flops": attn_flops(w), "accept_bytes": accept_bytes(w)}
    del st
    torch.cuda.empty_cache()
    return out


def run_gpu(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    w = wl.config(args.config, seed=1234 + rank)
    st = Step(w, dev)
    st.capture()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(local_rank)

    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    if st.status.item() != 0:
        raise RuntimeError(f"device status {st.status.item()} during warm-up")

    # The timed steps last milliseconds, shorter than one nvidia-smi sample, so the clocks
    # are sampled over a load window of the same steps (--clock-window seconds) that ends
    # where they start.
    # no collector pause on the host may fall between a step's start event and its launch
    # (the device work is unchanged; a stall there would add idle time to the step)
    gc.collect()
    gc.disable()
    t_begin = time.time()
    while time.time() - t_begin < args.clock_window:
        for _ in range(20):
            flush.zero_()
            st.run()
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()
        st.run(evs[k])
    torch.cuda.synchronize()
    t_end = time.time()
    if world > 1:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = float(np.sum(step_ms))
    # per-stage times for the roofline: each stage's own graph, same flush, second timed loop
    attn_stage_ms = st.time_stage(st.g_attn, flush, args.steps)
    acc_stage_ms = st.time_stage(st.g_acc, flush, args.steps)
    total_ms = max_over_ranks(total_ms, world, dev)
    clocks = sampler.stop(t_begin, t_end)
    if st.status.item() != 0:
        raise RuntimeError(f"device status {st.status.item()} in the timed region")

    # End to end: every step copies its inputs in from pinned host memory and its results
    # out.  Two device input sets (each with its own captured graph) let step k+1's inputs
    # stream in on a copy stream while step k computes; each step still waits for its own
    # copy, and its results are read back before the next step's results.
    sets = [st, Step(w, dev)]
    sets[1].capture()
    names = ("q", "logits", "parent", "draft", "bt", "pl")
    h_in = {n: getattr(st, n).cpu().pin_memory() for n in names}
    h_out = {n: torch.empty(getattr(st, n).shape, dtype=getattr(st, n).dtype).pin_memory() for n in ("o", "lse")}
    h_acc = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in st.acc_out[1:]]
    bi = sum(t.numel() * t.element_size() for t in h_in.values())
    bo = sum(t.numel() * t.element_size() for t in h_out.values()) + sum(t.numel() * t.element_size() for t in h_acc)
    copy_stream = torch.cuda.Stream()
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_free = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(k):
        b = k % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_free[b])  # the step that last used set b has read its inputs
            for n, t in h_in.items():
                getattr(sets[b], n).copy_(t, non_blocking=True)
            ev_in[b].record(copy_stream)

    def compute(k):
        b = k % 2
        cur = torch.cuda.current_stream()
        cur.wait_event(ev_in[b])
        sets[b].run()
        ev_free[b].record(cur)
        for n, t in h_out.items():
            t.copy_(getattr(sets[b], n), non_blocking=True)
        for t, s in zip(h_acc, sets[b].acc_out[1:]):
            t.copy_(s, non_blocking=True)

    # Small inputs (config 1: ~0.3 MB) are copied on the compute stream in step order: for
    # them a cross-stream event costs more than the overlap saves.
    pipelined = bi > (4 << 20)

    def e2e_run(steps):
        if not pipelined:
            for k in range(steps):
                for n, t in h_in.items():
                    getattr(st, n).copy_(t, non_blocking=True)
                st.run()
                for n, t in h_out.items():
                    t.copy_(getattr(st, n), non_blocking=True)
                for t, s in zip(h_acc, st.acc_out[1:]):
                    t.copy_(s, non_blocking=True)
            return
        copy_in(0)
        for k in range(steps):
            if k + 1 < steps:
                copy_in(k + 1)
            compute(k)

    e2e_run(max(2, min(args.warmup, 4)))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_run(args.steps)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if any(x.status.item() != 0 for x in sets):
        raise RuntimeError("device status set in the end-to-end run")
    commit_ms, commit_bytes = st.time_commit(flush, args.steps)
    tree_ms = st.time_tree(args.config, flush, args.steps)
    tree_w32_ms = st.time_tree(args.config, flush, args.steps, w=32)
    gdn_ms, gdn_bytes, gdn_name, gdn_commit_ms, gdn_commit_bytes, gdn_path_len = st.time_gdn(flush, args.steps)
    acc_fused_ms = st.time_accept_fused(flush, args.steps)
    acc_fused_nomask_ms = st.time_accept_fused(flush, args.steps, with_mask=False)
    forms_ms = {f: st.time_step_form(flush, args.steps, f) for f in ("mask", "folded", "fused")}
    if st.status.item() != 0:
        raise RuntimeError(f"device status {st.status.item()} in the commit stage")
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    per_config = {}
    if not args.no_per_config:
        del sets
        for n in sorted(wl.CONFIG_NAMES):
            if n != args.config:
                per_config[str(n)] = measure_config(n, dev, flush, args.steps, args.warmup, 1234 + rank)

    if rank != 0:
        return
    nodes = w.nb * w.B
    ms_per_step = total_ms / args.steps
    peaks, peak_src = load_peaks()
    t_attn = attn_stage_ms * 1e-3
    t_acc = acc_stage_ms * 1e-3
    ab, af, lb = attn_bytes(w), attn_flops(w), accept_bytes(w)
    attn_roof, acc_roof = stage_rooflines(w, t_attn, t_acc, peaks, peak_src, args.config)
    roof = attn_roof if t_attn >= t_acc else acc_roof
    out = {
        "metric": METRIC, "value": job_value(nodes, world, total_ms, args.steps), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the pages' Qwen3 workloads, random values)",
        "config": {"workload": wl.CONFIG_NAMES[args.config], "nb": w.nb, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "D": w.D, "prefix_lens": [int(x) for x in w.prefix_lens][:8], "V": w.V,
                   "l2": "flushed before every timed step (512 MB write)", "parallelism": f"replicas x{world}",
                   "launch": "one CUDA graph per step (attention with the ancestor bits from the parent array and "
                             "the split-KV merge, argmax, acceptance walk; %d launches), captured once"
                             % st.launches_per_step},
        "roofline": roof,
        "breakdown": {
            "attention_stage_ms": attn_stage_ms, "accept_ms": acc_stage_ms, "accept_fused_ms": acc_fused_ms,
            "accept_fused_nomask_ms": acc_fused_nomask_ms, "step_forms_ms": forms_ms,
            "step_forms_note": "each form of the whole step from its own graph with the same flush: mask = "
                               "tv_build_mask + attention + argmax + walk; folded = the attention and the walk "
                               "derive the ancestor bits from the parent array (no mask kernel); fused = folded "
                               "with tv_accept_fused (argmax and walk in one kernel)",
            "accept_note": "the step's acceptance is the two-kernel tv_accept (argmax, then the walk as a programmatic "
                           "dependent); accept_fused_ms is tv_accept_fused (one kernel) on the same inputs with the "
                           "step's mask, accept_fused_nomask_ms the same building the mask from the parent array",
            "stage_timing": "each stage's own graph replayed K times with the same L2 flush, after the timed steps",
            "attention_nodes_per_s": nodes / t_attn, "attention_roofline": attn_roof, "accept_roofline": acc_roof,
            "per_config": per_config,
            "per_config_note": "the other four workloads in the same process after the headline: each one's step, "
                               "attention stage and acceptance stage from their own graphs, K replays each with "
                               "the same 512 MB L2 flush before every replay; fractions of the measured peaks "
                               "(frac) and of the GB300 data-sheet peaks (frac_nominal)",
            "attention_bytes": ab, "attention_flops": af, "accept_bytes": lb,
            "kv_commit_ms": commit_ms, "kv_commit_bytes": commit_bytes,
            "build_tree_ms": tree_ms, "build_tree_w32_ms": tree_w32_ms,
            "build_tree_note": "tv_build_tree of this workload's budget from per-depth candidate tables, best-first "
                               "(w = 1) and in top-32 rounds (w = 32), each its own graph; not part of the step (it "
                               "precedes verification)",
            "gdn_tree_ms": gdn_ms, "gdn_tree_bytes": gdn_bytes, "gdn_tree_workload": gdn_name,
            "gdn_tree_roofline": {
                "kernel": "gdn_tree_kernel (tv_gdn_tree)", "bound": "hbm",
                "achieved": gdn_bytes / (gdn_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gdn_bytes / (gdn_ms * 1e-3) / (peaks["hbm_gbs"] * 1e9),
                "peak_source": peak_src + " burst", "algorithmic_bytes": gdn_bytes,
                "traffic": profiled_traffic("gdn_tree_kernel", "tv_gdn.cu", "gdn128")},
            "gdn_commit_ms": gdn_commit_ms, "gdn_commit_bytes": gdn_commit_bytes,
            "gdn_commit_note": f"tv_gdn_commit of the GDN workload's state along its deepest root path "
                               f"({gdn_path_len} nodes), its own graph",
            "gdn_tree_note": "tv_gdn_tree (Gated DeltaNet layer verified over the tree without rollback), its own "
                             "graph; a layer of the hybrid model's verification pass, not part of this attention "
                             "step; the dependent chain along each root path bounds it, not HBM",
            "kv_commit_note": "tv_kv_commit of the accepted branch, its own graph after the timed steps; not part "
                              "of the step (it rewrites the caches); latency-bound (a few KB moved)",
        },
        "clocks": clocks,
        "gpu_launches": st.launches_per_step * args.steps,
        "e2e": {"value": job_value(nodes, world, e2e_ms, args.steps), "unit": UNIT, "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo,
                "pipelined": pipelined,
                "note": "per step: q, logits, parent, draft tokens, block table, prefix lengths copied in from "
                        "pinned host memory (when pipelined, the next step's copy overlaps this step's compute, "
                        "into a second input set); O, LSE, accepted length, path and bonus copied out; the paged "
                        "KV cache is resident model state; L2 is not flushed in this loop (every step rewrites "
                        "its inputs from the host)"},
    }
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------- CPU oracle legs

def oracle_step(w: wl.Workload, group: int = 0):
    """One oracle verify step with the attention on one kv-head group (its G query heads over
    every sequence and node), scaled to all Hkv groups; the mask and the argmax + acceptance run
    in full.  Returns (wall seconds for the full step, threads, q heads computed)."""
    import oracle
    G = w.G
    g = group % w.Hkv
    t0 = time.perf_counter()
    oracle.build_mask(w.parent)
    t1 = time.perf_counter()
    q = np.ascontiguousarray(w.q[:, g * G:(g + 1) * G])
    kc = np.ascontiguousarray(w.k_cache[:, g:g + 1])
    vc = np.ascontiguousarray(w.v_cache[:, g:g + 1])
    t2 = time.perf_counter()
    _, _, threads = oracle.attn(q, kc, vc, w.block_table, w.prefix_lens, w.parent, G, 1, return_threads=True)
    t3 = time.perf_counter()
    oracle.accept(w.logits, w.draft, w.parent)
    t4 = time.perf_counter()
    full = (t1 - t0) + (t3 - t2) * w.Hkv + (t4 - t3)
    return full, threads, G


def cpu_baseline(w: wl.Workload):
    full, threads, used = oracle_step(w)
    return {"value": w.nb * w.B / full, "unit": UNIT, "cores": threads, "kind": "oracle",
            "host_cores": os.cpu_count(),
            "sample": f"one step of the same workload: mask, attention on kv head 0's {used} query heads over all "
                      f"{w.nb} sequences and {w.B} nodes scaled by {w.Hkv}, argmax + acceptance over all "
                      f"{w.nb * w.B} logits rows; fp64 C oracle, wall clock"}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    w = wl.config(args.config, seed=1234)
    # each step samples one kv-head group (step k takes group k mod Hkv, so Hkv steps cover every
    # head once), which keeps a step to seconds on the host cores
    for k in range(args.warmup):
        oracle_step(w, k)
    times = []
    threads = 0
    used = w.G
    for k in range(args.steps):
        t, threads, used = oracle_step(w, k)
        times.append(t)
    ms = float(np.mean(times)) * 1e3
    v = w.nb * w.B / (ms * 1e-3)
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
           "config": {"workload": wl.CONFIG_NAMES[args.config], "nb": w.nb, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                      "D": w.D, "V": w.V},
           "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                            "sample": f"each step: mask, attention on one kv-head group ({used} of {w.Hq} query "
                                      f"heads, step k takes group k mod {w.Hkv}) scaled by {w.Hkv}, argmax + "
                                      f"acceptance over all rows; fp64 C oracle"},
           "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="measure the headline workload only")
    ap.add_argument("--clock-window", type=float, default=0.4,
                    help="seconds of untimed steps, sampled for clocks, before the timed steps (0 under a profiler)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch.distributed as dist
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

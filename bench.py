#!/usr/bin/env python
"""Benchmark of the paged, quantized MoE expert layer on one GB300.

Workload: the decode-shaped paged layer -- E=256 experts, H=2048, I=512 (3 MiB
of FP8 weights per expert), top-8, CACHE_SLOTS=32 per layer with the LRU page
table, router logits Zipf(1.1)-skewed with 0.7 reuse of a token slot's
previous experts, refills of missed experts from pinned host memory on a side
stream. A stack of L layers (each its own slot pool; one shared working
buffer) is stepped round-robin, so the weights read per step come from HBM,
not L2 (L * 32 slots * 3.16 MB > 129 MB L2).

A step is one layer step: route -> permute -> LRU page table -> refills ->
paged expert FFN -> combine, at T tokens (64 by default; T=1 and T=8 are
reported too). `value` = tokens/s over K timed steps with inputs resident in
HBM; `e2e` = the same through pqe_layer_step_host with pinned host x/logits/y
copied inside every step.

--impl reference times the CPU oracle on the same workload (bounded samples).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

CFG = synth.WORKLOADS["decode"]
METRIC = "MoE-layer tokens/s; % of HBM BW (decode) and FP8 tensor peak (batched)"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="pqe", choices=["pqe", "reference"])
    ap.add_argument("--T", type=int, default=64)
    ap.add_argument("--layers", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the T=1 and T=8 lines")
    ap.add_argument("--no-batched", action="store_true", help="skip the module-batched (T=16384) measurement")
    ap.add_argument("--batched-steps", type=int, default=6)
    ap.add_argument("--workload", default="decode", choices=["decode", "batched", "large", "mixed", "huff", "ram"],
                    help="batched / large / mixed / huff (the decoder alone) / ram (the RAM tier): only that "
                         "measurement (for profiling)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the compressed large-layer (E=512) and mixed-precision (T=4096) measurements")
    ap.add_argument("--overlap-groups", type=int, default=None,
                    help="device pager: refill groups overlapped with the FFN passes (default by T; 0: none)")
    ap.add_argument("--pager", default="both", choices=["host", "device", "both"],
                    help="host: LRU on the host (one read-back per step); device: LRU on the GPU, each layer's step "
                         "replayed from a CUDA graph; both: measure both, the faster is the headline")
    ap.add_argument("--stream-kernel", default="auto", choices=["auto", "cuda", "tc"],
                    help="weight-stream kernel for batches of at most 8 rows: auto (the library's choice), cuda "
                         "(mma.sync on CUDA cores) or tc (tcgen05 on the tensor cores, all-FP8 layers); for A/B runs")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


_FP8_PEAK = {}


def measure_h2d_peak(torch, device, nbytes=1 << 30, reps=5):
    """The host link's ceiling for refills: one pinned-host-to-device copy of
    1 GiB, best of `reps` (GB/s)."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
    del src, dst
    return best


def measure_fp8_peak(torch, device, n=8192, reps=10):
    """Dense e4m3 x e4m3 -> bf16 GEMM through cuBLASLt (torch._scaled_mm),
    n x n x n, burst: the best of `reps` timed calls after warm-up, with fast
    and with regular accumulation, whichever is faster. Stored for
    fp8_peak_tflops(); None when the call is unavailable."""
    try:
        a = (torch.randn(n, n, device=device) * 0.1).to(torch.float8_e4m3fn)
        b = (torch.randn(n, n, device=device) * 0.1).to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=device)
        best = {}
        for fast in (True, False):
            def mm():
                r = torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16,
                                     use_fast_accum=fast)
                return r[0] if isinstance(r, tuple) else r
            for _ in range(3):
                mm()
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                mm()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            best[fast] = 2.0 * n ** 3 / (min(ts) / 1e3) / 1e12
        del a, b
        _FP8_PEAK["tflops"] = max(best.values())
        _FP8_PEAK["kind"] = (f"measured: cuBLASLt e4m3 GEMM {n}^3 burst via torch._scaled_mm (best of {reps}; "
                             f"fast accumulation {best[True]:.0f}, regular {best[False]:.0f} TFLOP/s)")
    except Exception as ex:  # older torch or no FP8 GEMM: the nominal ratio below is used
        _FP8_PEAK["error"] = f"{type(ex).__name__}: {ex}"[:200]
    return _FP8_PEAK


def fp8_peak_tflops():
    """Dense FP8 peak: measured in this run (measure_fp8_peak), else the
    measured bf16 cuBLAS rate x the nominal FP8/bf16 ratio of 2."""
    if "tflops" in _FP8_PEAK:
        return _FP8_PEAK["tflops"], _FP8_PEAK["kind"]
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return 2.0 * float(d["bf16_tflops"]), "measured bf16 x 2 (nominal fp8/bf16 ratio)"
    return 2.0 * 1900.0, "fallback bf16 x 2"


# ---- distributed (replicas only: no data-path collective) -------------------------

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, v: float, device) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- clocks ------------------------------------------------------------------------

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- workload ----------------------------------------------------------------------

def expert_pages_host(pqe, torch, device):
    """All E experts' FP8 pages (synthetic N(0,0.02) weights, quantised by the
    library), pinned on the host: the host tier every layer refills from."""
    E, H, I = CFG.E, CFG.H, CFG.I
    stride = pqe.slot_stride(H, I)
    host = torch.empty((E, stride), dtype=torch.uint8).pin_memory()
    page = torch.zeros(stride, dtype=torch.uint8, device=device)
    for e in range(E):
        w13, w2 = synth.expert_weights(CFG, e)
        pqe.pqe_pack_fp8_page(torch.from_numpy(w13).to(device), torch.from_numpy(w2).to(device), H, I, page)
        host[e].copy_(page)
    torch.cuda.synchronize()
    return host


def make_traces(T, L, n_steps):
    """logits[i] for step i (layer i % L, that layer's trace step i // L)."""
    traces = [synth.RoutingTrace(CFG, T, layer=l) for l in range(L)]
    out = []
    for i in range(n_steps):
        out.append(traces[i % L].step(i // L))
    return out


class Runner:
    def __init__(self, pqe, torch, device, host, L, max_T, device_pager=False, overlap_groups=0):
        E, H, I, k, S = CFG.E, CFG.H, CFG.I, CFG.k, CFG.S
        self.pqe, self.torch, self.device = pqe, torch, device
        self.wb = pqe.alloc_working_buffer(E, H, I, device)
        nbytes = [pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)] * E
        self.layers = [pqe.PagedMoELayer(E, H, I, k, S, E, max_T, host, nbytes, working_buffer=self.wb,
                                         device=device, device_pager=device_pager, overlap_groups=overlap_groups)
                       for _ in range(L)]
        self.stream = torch.cuda.current_stream(device)
        self.side = torch.cuda.Stream(device)

    def close(self):
        for l in self.layers:
            l.close()


class GraphRunner:
    """Device-pager layers replayed from CUDA graphs that each hold a run of up
    to L consecutive steps (one pass over the layers, layer i % L for step i),
    every step captured reading its own HBM-resident inputs (that step's
    logits, one of four x). A timed step is then part of one graph replay,
    route through combine, with no input copies (in a model the layer's inputs
    are already in place); a graph is launched once, so its first-launch cost
    is shared by the steps it holds."""

    def __init__(self, pqe, torch, device, host, L, T, overlap_groups=0, comp=None):
        E, H, I, k, S = CFG.E, CFG.H, CFG.I, CFG.k, CFG.S
        self.pqe, self.torch, self.T = pqe, torch, T
        self.wb = pqe.alloc_working_buffer(E, H, I, device)
        nbytes = [pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)] * E
        if comp is None:
            self.layers = [pqe.PagedMoELayer(E, H, I, k, S, E, T, host, nbytes, working_buffer=self.wb, device=device,
                                             device_pager=True, overlap_groups=overlap_groups) for _ in range(L)]
        else:  # a compressed host tier: (pinned pages, their sizes, code tables on the device)
            pages, sizes, luts = comp
            self.layers = [pqe.PagedMoELayer(E, H, I, k, S, E, T, pages, sizes, compressed=True, luts=luts,
                                             working_buffer=self.wb, device=device, device_pager=True,
                                             overlap_groups=overlap_groups) for _ in range(L)]
        self.stream = torch.cuda.Stream(device)
        # the refills of an overlapped step run on this stream, forked and joined inside each step
        self.side = torch.cuda.Stream(device)
        self.y = [torch.zeros((T, H), dtype=torch.bfloat16, device=device) for _ in range(L)]
        self.graphs = []  # (first step, steps, graph, kernel nodes)

    def capture(self, logits_dev, xs_dev, ranges):
        """Eager steps 0..L-1 (one per layer), then one graph per run of <= L
        steps inside each [a, b) of `ranges`."""
        torch = self.torch
        L = len(self.layers)
        with torch.cuda.stream(self.stream):
            for l, layer in enumerate(self.layers):
                layer.step(xs_dev[l % len(xs_dev)], self.y[l], self.T, logits=logits_dev[l], stream=self.stream,
                           side_stream=self.side)
            torch.cuda.synchronize()
            for a, b in ranges:
                for c in range(a, b, L):
                    n = min(L, b - c)
                    g = torch.cuda.CUDAGraph()
                    n0 = self.pqe.kernel_launches()
                    with torch.cuda.graph(g, stream=self.stream):
                        for i in range(c, c + n):
                            self.layers[i % L].step(xs_dev[i % len(xs_dev)], self.y[i % L], self.T,
                                                    logits=logits_dev[i], stream=self.stream, side_stream=self.side)
                    # launches recorded during the capture = kernel nodes run by each replay
                    self.graphs.append((c, n, g, self.pqe.kernel_launches() - n0))
        torch.cuda.synchronize()

    def replay(self, a, b):
        """Replays the graphs of steps [a, b) (a capture range); returns their kernel nodes."""
        nodes = 0
        with self.torch.cuda.stream(self.stream):
            for c, n, g, k in self.graphs:
                if a <= c < b:
                    g.replay()
                    nodes += k
        return nodes

    def close(self):
        self.graphs.clear()
        for l in self.layers:
            l.close()


def overlap_groups_for(T):
    """Refill groups of an overlapped device-pager step by step size, the best
    measured on the decode-shaped layer: none at T=1 (the FFN passes' fixed
    costs outweigh what they hide), 3 at T=8, 5 at T=64 (2282 -> 2233 us)."""
    return OVERLAP_GROUPS if OVERLAP_GROUPS is not None else (0 if T <= 1 else 3 if T < 32 else 5)


OVERLAP_GROUPS = None  # --overlap-groups


def run_graph(pqe, torch, device, host, T, L, logits_dev, xs_dev, warmup, K, ws, ffn_events=False, comp=None,
              groups=None):
    """Device-pager graph replays of steps L .. L + warmup + K - 1 (layer i % L).
    With ffn_events each layer's FFN is bracketed by event nodes in its graphs
    (after the timed loop they hold the FFN time of that layer's last replay).
    The two nodes add ~11 us to a replayed step, so the headline steps are
    timed without them and the FFN in a second pass."""
    gr = GraphRunner(pqe, torch, device, host, L, T, overlap_groups_for(T) if groups is None else groups, comp)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
    if ffn_events:
        for (a, b), layer in zip(evs, gr.layers):
            a.record(gr.stream)
            b.record(gr.stream)  # creates the events; the graphs record them again
            layer.set_ffn_events(a, b)
    t0 = L + warmup
    gr.capture(logits_dev, xs_dev, [(L, t0), (t0, t0 + K)])
    gr.replay(L, t0)
    torch.cuda.synchronize()
    barrier(ws)
    stats0 = [l.device_stats() for l in gr.layers]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(gr.stream)
    launches = gr.replay(t0, t0 + K)
    e1.record(gr.stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms = e0.elapsed_time(e1)
    stats1 = [l.device_stats() for l in gr.layers]
    d = {k: sum(b[k] - a[k] for a, b in zip(stats0, stats1)) for k in stats0[0]}
    # the FFN of the last replay of each layer: steps L + warmup + K - L .. - 1
    last = [L + warmup + K - L + j for j in range(L)]
    d["ffn_ms_last"] = {i: evs[i % L][0].elapsed_time(evs[i % L][1]) for i in last} if ffn_events else {}
    gr.close()
    return ms, d, launches


def run_timed(r: Runner, T, logits_dev, xs_dev, y, warmup, K, ws, want_ffn=True):
    torch, pqe = r.torch, r.pqe
    L = len(r.layers)
    total = warmup + K
    assert len(logits_dev) >= total
    infos = []
    evs = []
    if want_ffn:
        for _ in range(K):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(r.stream)
            b.record(r.stream)  # creates the events; the library records them again
            evs.append((a, b))
    for i in range(warmup):
        layer = r.layers[i % L]
        layer.set_ffn_events(None, None)
        layer.step(xs_dev[i % len(xs_dev)], y, T, logits=logits_dev[i], stream=r.stream, side_stream=r.side)
    torch.cuda.synchronize()
    barrier(ws)
    launches0 = pqe.kernel_launches()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(r.stream)
    wall0 = time.perf_counter()
    for j in range(K):
        i = warmup + j
        layer = r.layers[i % L]
        if want_ffn:
            layer.set_ffn_events(*evs[j])
        info = layer.step(xs_dev[i % len(xs_dev)], y, T, logits=logits_dev[i], stream=r.stream, side_stream=r.side)
        infos.append((info.n_routed, info.n_miss, info.working_buffer, info.h2d_bytes))
    e1.record(r.stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(ws)
    launches = pqe.kernel_launches() - launches0
    ms = e0.elapsed_time(e1)
    for l in r.layers:
        l.set_ffn_events(None, None)
    ffn_ms = [a.elapsed_time(b) for a, b in evs] if want_ffn else []
    return ms, wall, infos, ffn_ms, launches


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum, ncu) of the
# kernels of one FFN call at T=64 (the tensor-core weight stream, the two GEMM
# launches of the tensor-core batches, the small row passes and the schedule),
# captured one kernel at a time, divided by the algorithmic bytes of the same
# run's calls: 465.6 / 452.6 MB
FFN_DRAM_PER_ALGORITHMIC_BYTE_T64 = 1.03


def routed_experts(logits: np.ndarray, k: int) -> int:
    """Distinct experts in a step's top-k (ties to the lower id, as routed)."""
    return int(np.unique(np.argsort(-logits, axis=1, kind="stable")[:, :k]).size)


def ffn_bytes(n_routed, T):
    """Algorithmic bytes of one moe_paged_ffn call: the routed experts' pages,
    x once, out_perm once."""
    return n_routed * CFG.page_bytes_fp8_with_scales + T * CFG.H * 2 + T * CFG.k * CFG.H * 2


# page bytes incl. fp32 scales (3*H*I + 4*(2I+H))
synth.LayerConfig.page_bytes_fp8_with_scales = property(lambda c: 3 * c.H * c.I + 4 * (2 * c.I + c.H))


def cpu_oracle_sample(host_np, T, logits_list, budget_s=10.0, max_steps=16):
    """The oracle (as it stands) on layer 0's trace steps: routing of all T
    tokens, permutation, LRU step and the FFN of all T tokens; steps are run
    until `budget_s` is spent. Returns (tokens, seconds, threads, steps)."""
    import oracle
    E, H, I, k = CFG.E, CFG.H, CFG.I, CFG.k
    lay = {"w13": 0, "w2": 2 * I * H, "s13": 3 * I * H, "s2": 3 * I * H + 8 * I}
    ex = oracle.ExpertSet(E)
    for e in range(E):
        p = host_np[e]
        ex.set(e, 0, p[lay["w13"]:lay["w13"] + 2 * I * H].reshape(2 * I, H),
               p[lay["s13"]:lay["s13"] + 8 * I].view(np.float32),
               p[lay["w2"]:lay["w2"] + H * I].reshape(H, I), p[lay["s2"]:lay["s2"] + 4 * H].view(np.float32))
    lru = oracle.LRU(E, CFG.S)
    x = synth.activations(CFG, T, 0)
    tokens, t_used, steps = 0, 0.0, 0
    for s, lg in enumerate(logits_list[:max_steps]):
        t0 = time.perf_counter()
        ids, g = oracle.topk_gates(lg, k)
        counts, offsets, perm_src, inv = oracle.permute(ids, E)
        lru.step(counts)
        oracle.moe_ffn(x, ids, g, ex, I)
        t_used += time.perf_counter() - t0
        tokens += T
        steps += 1
        if t_used >= budget_s:
            break
    return tokens, t_used, oracle.num_threads(), steps


# ---- reference arm (the oracle) ----------------------------------------------------------

def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    T, L = args.T, args.layers
    E, H, I = CFG.E, CFG.H, CFG.I
    # pages from the oracle's own quantiser (same bytes as the library's)
    host = np.zeros((E, 3 * H * I + 4 * (2 * I + H)), np.uint8)
    for e in range(E):
        w13, w2 = synth.expert_weights(CFG, e)
        q13, s13 = oracle.quant_e4m3_rows(w13)
        q2, s2 = oracle.quant_e4m3_rows(w2)
        host[e, :2 * I * H] = q13.reshape(-1)
        host[e, 2 * I * H:3 * I * H] = q2.reshape(-1)
        host[e, 3 * I * H:3 * I * H + 8 * I] = s13.view(np.uint8)
        host[e, 3 * I * H + 8 * I:] = s2.view(np.uint8)
    traces = make_traces(T, 1, args.warmup + args.steps)
    # each step: one layer step of the oracle on a bounded token sample
    n_tok = max(1, min(T, 8))
    sub = [lg[:n_tok] for lg in traces]
    _, _, threads, _ = cpu_oracle_sample(host, n_tok, sub[:args.warmup], budget_s=1e9, max_steps=args.warmup)
    tok, secs, threads, steps = cpu_oracle_sample(host, n_tok, sub[args.warmup:], budget_s=1e9,
                                                  max_steps=args.steps)
    v = tok / secs
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"decode-shaped paged MoE layer E=256 H=2048 I=512 top-8 CACHE_SLOTS=32, "
                                   f"T={T}; oracle step on {n_tok} tokens", "T": T},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{steps} layer steps of {n_tok} tokens each"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_batched(pqe, torch, device, host, steps, ws):
    """Module-batched prefill layer: T=16384 tokens in one step, per-expert
    batches of ~512 rows (Zipf-skewed); |U| > CACHE_SLOTS, so every step stages
    the needed non-resident experts into the working buffer. Reports whole
    steps and the FFN alone (FP8 tensor path) against the FP8 peak."""
    cfg3 = synth.WORKLOADS["batched"]
    E, H, I, k, S, T = cfg3.E, cfg3.H, cfg3.I, cfg3.k, cfg3.S, cfg3.T[0]
    nbytes = [pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)] * E
    layer = pqe.PagedMoELayer(E, H, I, k, S, E, T, host, nbytes, device=device)
    stream = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device)
    tr = synth.RoutingTrace(cfg3, T)
    logits = [torch.from_numpy(tr.step(s)).to(device) for s in range(2)]
    x = torch.from_numpy(synth.activations(cfg3, T, 0).view(np.int16)).to(device)
    y = torch.zeros((T, H), dtype=torch.bfloat16, device=device)
    evs = []
    for _ in range(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        b.record(stream)
        evs.append((a, b))
    for i in range(2):  # warm-up
        layer.step(x, y, T, logits=logits[i % 2], stream=stream, side_stream=side)
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    misses = []
    for i in range(steps):
        layer.set_ffn_events(*evs[i])
        info = layer.step(x, y, T, logits=logits[i % 2], stream=stream, side_stream=side)
        misses.append(info.n_miss)
    e1.record(stream)
    torch.cuda.synchronize()
    layer.set_ffn_events(None, None)
    ms = e0.elapsed_time(e1)
    ffn = [a.elapsed_time(b) for a, b in evs]
    flops = 6.0 * T * k * H * I
    peak, kind = fp8_peak_tflops()
    ffn_ms = float(np.mean(ffn))
    tflops = flops / (ffn_ms / 1e3) / 1e12
    layer.close()
    sweep = batch_sweep(pqe, torch, device, host, cfg3, stream, side, peak)
    return {"workload": "module-batched prefill layer (E=256, H=2048, I=512, top-8, T=16384, CACHE_SLOTS=32, "
                        "working buffer)",
            "tokens_per_s": T * steps / (ms / 1e3), "ms_per_step": ms / steps,
            "mean_staged_experts": float(np.mean(misses)),
            "ffn": {"ms": ffn_ms, "tflops": tflops, "peak_tflops": peak, "peak_kind": kind, "frac": tflops / peak,
                    "bound": "tensor", "flops_per_step": flops},
            "batch_size_sweep": sweep}


def batch_sweep(pqe, torch, device, host, cfg, stream, side, peak, Ts=(2048, 4096, 8192, 16384, 32768, 65536),
                steps=4):
    """Module-batch sizing: the FFN of the module-batched layer at accumulated
    batch sizes T from 2048 to 65536 (one layer sized for the largest; the
    token rows of a smaller T are the first T of the largest trace), beside
    the knee the library's sizer puts on the roofline of the measured
    ceilings."""
    E, H, I, k = cfg.E, cfg.H, cfg.I, cfg.k
    bw = peaks()[0]
    Tmax = max(Ts)
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    layer = pqe.PagedMoELayer(E, H, I, k, cfg.S, E, Tmax, host, [nb] * E, device=device)
    tr = synth.RoutingTrace(cfg, Tmax)
    lg_full = [torch.from_numpy(tr.step(s)).to(device) for s in range(2)]
    x_full = torch.from_numpy(synth.activations(cfg, Tmax, 0).view(np.int16)).to(device)
    y_full = torch.zeros((Tmax, H), dtype=torch.bfloat16, device=device)
    out = {"T": [], "ffn_ms": [], "ffn_tflops": [], "ffn_frac_of_fp8_peak": [], "ffn_hbm_gbs": []}
    for T in Ts:
        logits = [l[:T].contiguous() for l in lg_full]
        xs = [x_full[:T]]
        layer.step(xs[0], y_full[:T], T, logits=logits[0], stream=stream, side_stream=side)  # warm-up
        _, ffn, infos = _timed_steps(torch, layer, xs, y_full[:T], T, logits, steps, stream, side)
        f_ms = float(np.mean(ffn))
        routed = float(np.mean([r for r, _, _ in infos]))
        out["T"].append(T)
        out["ffn_ms"].append(f_ms)
        tf = 6.0 * T * k * H * I / (f_ms / 1e3) / 1e12
        out["ffn_tflops"].append(tf)
        out["ffn_frac_of_fp8_peak"].append(tf / peak)
        out["ffn_hbm_gbs"].append((routed * nb + T * H * 2 + T * k * H * 2) / (f_ms / 1e3) / 1e9)
    layer.close()
    best = max(out["ffn_tflops"])
    out["measured_knee_T"] = next(T for T, tf in zip(out["T"], out["ffn_tflops"]) if tf >= 0.9 * best)
    out["model_knee_T"] = pqe.pqe_module_batch_size(E, k, H, I, bw, peak, 64)
    out["note"] = ("measured_knee_T: the smallest swept T within 90% of the best FFN TFLOP/s; model_knee_T: "
                   "pqe_module_batch_size on the measured HBM and FP8 ceilings of this run")
    return out


def _timed_steps(torch, layer, x, y, T, logits, steps, stream, side):
    """Whole layer steps with per-step FFN events; returns (ms total, [ffn ms], [step infos])."""
    evs = []
    for _ in range(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    infos = []
    for i in range(steps):
        layer.set_ffn_events(*evs[i])
        info = layer.step(x[i % len(x)], y, T, logits=logits[i % len(logits)], stream=stream, side_stream=side)
        infos.append((info.n_routed, info.n_miss, info.working_buffer))
    e1.record(stream)
    torch.cuda.synchronize()
    layer.set_ffn_events(None, None)
    return e0.elapsed_time(e1), [a.elapsed_time(b) for a, b in evs], infos


def large_compressed_pages(pqe, torch, device, n_src):
    """n_src distinct experts of the large layer (E=512, H=2560, I=640) as
    Huffman-coded pages in pinned host memory, with their code tables."""
    cfg = synth.WORKLOADS["large"]
    H, I = cfg.H, cfg.I
    LB = pqe.PQE_HUFF_LUT_BYTES
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    bound = pqe.pqe_huff_page_bound(H, I)
    comp = torch.zeros((n_src, bound), dtype=torch.uint8)
    luts_src = torch.zeros((n_src, 2 * LB), dtype=torch.uint8)
    sizes_src = []
    page = torch.zeros(pqe.slot_stride(H, I), dtype=torch.uint8, device=device)
    for j in range(n_src):
        w13, w2 = synth.expert_weights(cfg, j)
        pqe.pqe_pack_fp8_page(torch.from_numpy(w13).to(device), torch.from_numpy(w2).to(device), H, I, page)
        sizes_src.append(pqe.pqe_huff_encode_page(page[:nb].cpu().contiguous(), H, I, comp[j], luts_src[j, :LB],
                                                  luts_src[j, LB:]))
    return comp.pin_memory(), sizes_src, luts_src


def decode_compressed_pages(pqe, torch, host, n_src=32):
    """The decode-shaped layer's host tier as Huffman-coded pages: n_src distinct
    experts encoded (expert e uses page e % n_src), pinned, with code tables."""
    E, H, I = CFG.E, CFG.H, CFG.I
    LB = pqe.PQE_HUFF_LUT_BYTES
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    bound = pqe.pqe_huff_page_bound(H, I)
    comp = torch.zeros((n_src, bound), dtype=torch.uint8)
    luts_src = torch.zeros((n_src, 2 * LB), dtype=torch.uint8)
    sizes_src = [pqe.pqe_huff_encode_page(host[j, :nb].contiguous(), H, I, comp[j], luts_src[j, :LB],
                                          luts_src[j, LB:]) for j in range(n_src)]
    comp = comp.pin_memory()
    return ([comp[e % n_src] for e in range(E)], [sizes_src[e % n_src] for e in range(E)],
            luts_src[torch.arange(E) % n_src].contiguous(), float(np.mean(sizes_src)) / nb)


def run_huff(pqe, torch, device, n_src=32):
    """The decoder alone on the large layer's pages (for profiling)."""
    cfg = synth.WORKLOADS["large"]
    comp, sizes, luts = large_compressed_pages(pqe, torch, device, n_src)
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, cfg.H, cfg.I)
    return huff_decode_rate(pqe, torch, device, comp, sizes, luts, cfg.H, cfg.I, nb)


def run_large(pqe, torch, device, steps_t1=64, steps_big=3, n_src=32):
    """Large paged layer with a compressed host tier (E=512, H=2560, I=640, top-8,
    46 LRU slots): every refill copies a Huffman-coded page and decodes it on the
    GPU. T=1 (decode) and T=4096 whole steps, the FFN against HBM / FP8 peak,
    and the decoder alone on device-resident compressed pages. The host tier
    holds n_src distinct encoded pages (expert e uses page e % n_src), so the
    bytes moved and decoded per step are those of the full layer."""
    cfg = synth.WORKLOADS["large"]
    E, H, I, k, S = cfg.E, cfg.H, cfg.I, cfg.k, cfg.S
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    comp, sizes_src, luts_src = large_compressed_pages(pqe, torch, device, n_src)
    host = [comp[e % n_src] for e in range(E)]
    sizes = [sizes_src[e % n_src] for e in range(E)]
    luts = luts_src[torch.arange(E) % n_src].contiguous().to(device)
    big_T = cfg.T[-1]
    stream = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device)
    out = {"workload": "large paged layer, compressed host tier (E=512, H=2560, I=640, top-8, CACHE_SLOTS=46, "
                       "Huffman-coded FP8 exponents decoded on the GPU after each refill)",
           "mean_compressed_ratio": float(np.mean(sizes_src)) / nb,
           "pager": "device (LRU on the GPU; compressed misses pulled and decoded by a kernel reading the "
                    "step's miss list), eager steps"}
    peak_bw = peaks()[0]
    for T, steps in ((1, steps_t1), (big_T, steps_big)):
        # no refill groups: the decode of compressed pages needs the SMs the FFN
        # passes would take (T=4096: 10.38 ms per step plain, 10.77 with 5 groups)
        groups = OVERLAP_GROUPS if OVERLAP_GROUPS is not None else 0
        layer = pqe.PagedMoELayer(E, H, I, k, S, E, big_T, host, sizes, compressed=True, luts=luts, device=device,
                                  device_pager=True, overlap_groups=groups)
        tr = synth.RoutingTrace(cfg, T)
        n_tr = min(2 * steps + 4, 64)
        logits_np = [tr.step(s) for s in range(n_tr)]
        logits = [torch.from_numpy(l).to(device) for l in logits_np]
        xs = [torch.from_numpy(synth.activations(cfg, T, s % 2).view(np.int16)).to(device) for s in range(2)]
        y = torch.zeros((T, H), dtype=torch.bfloat16, device=device)
        if T > 1:  # the slots first fill with the experts of small steps, as in a serving run
            tr1 = synth.RoutingTrace(cfg, 1)
            x1 = torch.from_numpy(synth.activations(cfg, 1, 0).view(np.int16)).to(device)
            y1 = torch.zeros((1, H), dtype=torch.bfloat16, device=device)
            for i in range(24):
                layer.step(x1, y1, 1, logits=torch.from_numpy(tr1.step(i)).to(device), stream=stream,
                           side_stream=side)
        for i in range(2):  # warm-up
            layer.step(xs[i % 2], y, T, logits=logits[i % n_tr], stream=stream, side_stream=side)
        torch.cuda.synchronize()
        st0 = layer.device_stats()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            layer.step(xs[i % 2], y, T, logits=logits[(2 + i) % n_tr], stream=stream, side_stream=side)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        st1 = layer.device_stats()
        # the FFN call's time: the next steps again with its timing events (one FFN pass per step)
        ffn_logits = [logits[(2 + steps + i) % n_tr] for i in range(steps)]
        _, ffn, _ = _timed_steps(torch, layer, xs, y, T, ffn_logits, steps, stream, side)
        ffn_ms = float(np.mean(ffn))
        routed = float(np.mean([routed_experts(logits_np[(2 + steps + i) % n_tr], k) for i in range(steps)]))
        layer.close()
        rec = {"tokens_per_s": T * steps / (ms / 1e3), "ms_per_step": ms / steps, "steps": steps,
               "overlap_groups": groups,
               "mean_routed_experts": (st1["routed"] - st0["routed"]) / steps,
               "mean_misses": (st1["misses"] - st0["misses"]) / steps,
               "h2d_gb_per_s": (st1["refill_bytes"] - st0["refill_bytes"]) / (ms / 1e3) / 1e9,
               "ffn_ms": ffn_ms}
        # both bounds: the routed pages (plus x and out_perm) against HBM, the FLOPs against
        # the FP8 peak; at T=4096 a batch is ~64 rows per expert, below the FP8 ridge (~290)
        gbs = (routed * (nb + 0.0) + T * H * 2 + T * k * H * 2) / (ffn_ms / 1e3) / 1e9
        tflops = 6.0 * T * k * H * I / (ffn_ms / 1e3) / 1e12
        pk, kind = fp8_peak_tflops()
        rec.update({"ffn_hbm_gbs": gbs, "ffn_frac_of_measured_hbm": gbs / peak_bw, "ffn_tflops": tflops,
                    "ffn_frac_of_fp8_peak": tflops / pk, "fp8_peak_kind": kind,
                    "bound": "hbm" if T * k / max(routed, 1.0) < 290 else "tensor"})
        out["T=%d" % T] = rec
    out["huff_decode"] = huff_decode_rate(pqe, torch, device, comp, sizes_src, luts_src, H, I, nb)
    return out


def run_ram(pqe, torch, device, host, steps=256, L=4, Ts=(1, 8), ram_slots=(256, 128)):
    """The decode-shaped layer (E=256, H=2048, I=512, top-8, 32 VRAM slots per
    layer) with its refills served by a host-RAM tier over a paging file
    (expert-pager article, SSD階層; its Table 2 compares RAM_SLOTS=256 and 128):
    L layers round-robin, each with its own RAM slots; every page is written
    once into one paging file, and a RAM miss is read from it by the reader
    threads (O_DIRECT where the file system allows it). Per RAM_SLOTS and T:
    whole steps, VRAM misses, file reads and bytes per step, and the refill
    latency (the step time above the same steps with every page resident in
    RAM)."""
    E, H, I, k, S = CFG.E, CFG.H, CFG.I, CFG.k, CFG.S
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    path = os.path.join(tempfile.gettempdir(), f"pqe_paging_{os.getpid()}.bin")
    t0 = time.perf_counter()
    offs = pqe.pqe_paging_file_write(path, [host[e] for e in range(E)], [nb] * E)
    write_s = time.perf_counter() - t0
    slot = -(-nb // 4096) * 4096
    wb = pqe.alloc_working_buffer(E, H, I, device)
    stream = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device)
    out = {"workload": "decode-shaped paged layer (E=256, H=2048, I=512, top-8, CACHE_SLOTS=32) with a host-RAM "
                       "tier per layer over a paging file of all experts", "layers_round_robin": L,
           "paging_file_gb": E * slot / 1e9, "paging_file_write_s": write_s, "storage": tempfile.gettempdir()}
    try:
        for S_ram in ram_slots:
            layers, tiers, bufs = [], [], []
            for _ in range(L):
                W_ram = max(Ts) * k  # a step misses at most T*k pages in VRAM
                buf = torch.zeros((S_ram + W_ram) * slot + 4096, dtype=torch.uint8).pin_memory()
                a = (-buf.data_ptr()) % 4096
                ram = buf[a:a + (S_ram + W_ram) * slot]
                tier = pqe.RamTier(path, offs, [nb] * E, S_ram, W_ram, ram, slot, n_threads=8)
                tier.request([1 if e < S_ram else 0 for e in range(E)])  # start with full RAM slots
                tier.wait()
                lay = pqe.PagedMoELayer(E, H, I, k, S, E, max(Ts), host, [nb] * E, working_buffer=wb,
                                        device=device)
                lay.attach_ram_tier(tier)
                layers.append(lay)
                tiers.append(tier)
                bufs.append(buf)
            rec = {}
            for T in Ts:
                lg = [torch.from_numpy(l).to(device) for l in make_traces(T, L, 2 * L + steps)]
                xs = [torch.from_numpy(synth.activations(CFG, T, s).view(np.int16)).to(device) for s in range(2)]
                y = torch.zeros((T, H), dtype=torch.bfloat16, device=device)
                for i in range(2 * L):  # warm-up
                    layers[i % L].step(xs[i % 2], y, T, logits=lg[i], stream=stream, side_stream=side)
                torch.cuda.synchronize()
                st0 = [t.state()[3] for t in tiers]
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                misses = reads = 0
                e0.record(stream)
                for j in range(steps):
                    i = 2 * L + j
                    info = layers[i % L].step(xs[i % 2], y, T, logits=lg[i], stream=stream, side_stream=side)
                    misses += info.n_miss
                    reads += info.n_file_read
                e1.record(stream)
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / steps
                st1 = [t.state()[3] for t in tiers]
                fbytes = sum(b["bytes"] - a["bytes"] for a, b in zip(st0, st1))
                rec[f"T={T}"] = {"ms_per_step": ms, "tokens_per_s": T / (ms / 1e3),
                                 "vram_misses_per_step": misses / steps, "file_reads_per_step": reads / steps,
                                 "file_mb_per_step": fbytes / steps / 1e6,
                                 "file_read_gb_per_s": fbytes / (ms * steps / 1e3) / 1e9 if fbytes else 0.0}
            rec["direct_io"] = tiers[0].state()[3]["direct_io"]
            out[f"RAM_SLOTS={S_ram}"] = rec
            for lay in layers:
                lay.close()
            for t in tiers:
                t.close()
            del bufs
        full = out.get(f"RAM_SLOTS={max(ram_slots)}")
        for S_ram in ram_slots:
            if S_ram != max(ram_slots) and full:
                for T in Ts:
                    r = out[f"RAM_SLOTS={S_ram}"][f"T={T}"]
                    r["refill_latency_ms_per_step"] = r["ms_per_step"] - full[f"T={T}"]["ms_per_step"]
    finally:
        os.unlink(path)
    return out


def run_mixed(pqe, torch, device, steps=256, every=64):
    """Mixed per-expert precision layer (E=256, H=2048, I=512, top-8, T=4096),
    as the PagedWeight commentary's bit-width loop runs it: each expert's
    importance is an EMA of its gate mass (seeded U(0,1) start, alpha 0.9,
    updated every step from the step's routing); every `every` steps the
    experts are re-ranked, the top 25% keep FP8 pages and the rest MXFP4
    pages; an expert whose format changed gets its new host page and its
    resident copy is dropped, so its next use refills it through the pager
    (256 slots: after warm-up every other page stays resident). Reports whole
    steps, the steps that follow a re-rank (they refill the changed pages),
    the sets that changed, and the FFN against HBM (bytes of the routed pages
    in their current format) and the FP8 peak."""
    cfg = synth.WORKLOADS["mixed"]
    E, H, I, k, T = cfg.E, cfg.H, cfg.I, cfg.k, cfg.T[0]
    stride = pqe.slot_stride(H, I)
    n8, n4 = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I), pqe.page_bytes(pqe.PQE_FMT_MXFP4, H, I)
    n_hi = E // 4
    m = synth.importance_init(cfg).astype(np.float64)
    fmt = np.zeros(E, np.uint8)
    pqe.pqe_rank_formats(torch.from_numpy(m), n_hi, torch.from_numpy(fmt))
    host8 = torch.zeros((E, stride), dtype=torch.uint8)
    host4 = torch.zeros((E, -(-n4 // 256) * 256), dtype=torch.uint8)
    page = torch.zeros(stride, dtype=torch.uint8, device=device)
    p4 = torch.zeros(n4, dtype=torch.uint8, device=device)
    nq = 16  # experts whose two pages feed the quality proxy
    q8 = torch.zeros((nq, stride), dtype=torch.uint8, device=device)
    q4 = torch.zeros((nq, n4), dtype=torch.uint8, device=device)
    for e in range(E):
        w13, w2 = synth.expert_weights(cfg, e)
        pqe.pqe_pack_fp8_page(torch.from_numpy(w13).to(device), torch.from_numpy(w2).to(device), H, I, page)
        pqe.pqe_pack_mxfp4_page(page, H, I, p4)
        if e < nq:
            q8[e].copy_(page)
            q4[e].copy_(p4)
        host8[e].copy_(page)
        host4[e, :n4].copy_(p4)
    host8, host4 = host8.pin_memory(), host4.pin_memory()

    def host_page(e):
        return (host8[e], n8) if fmt[e] == pqe.PQE_FMT_FP8 else (host4[e], n4)

    fmt_dev = torch.from_numpy(fmt.copy()).to(device)
    layer = pqe.PagedMoELayer(E, H, I, k, E, 0, T, [host_page(e)[0] for e in range(E)],
                              [host_page(e)[1] for e in range(E)], expert_fmt=fmt_dev, device=device)
    stream = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device)
    tr = synth.RoutingTrace(cfg, T, vectorized=True)
    warm = 3
    lg_np = [tr.step(s) for s in range(warm + steps)]
    logits = [torch.from_numpy(l).to(device) for l in lg_np]
    xs = [torch.from_numpy(synth.activations(cfg, T, s).view(np.int16)).to(device) for s in range(2)]
    y = torch.zeros((T, H), dtype=torch.bfloat16, device=device)
    ids_h = [torch.zeros(T * k, dtype=torch.int32).pin_memory() for _ in range(2)]
    g_h = [torch.zeros(T * k, dtype=torch.float32).pin_memory() for _ in range(2)]
    ids_d = layer.device_view("topk_ids", torch.int32, (T * k,))
    g_d = layer.device_view("topk_w", torch.float32, (T * k,))
    for i in range(warm):  # warm-up: the first step loads every routed page
        layer.step(xs[i % 2], y, T, logits=logits[i], stream=stream, side_stream=side)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ffn = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ffn:
        a.record(stream)
        b.record(stream)
    done = torch.cuda.Event()
    changed, rerank_at, byts, misses = [], [], [], []
    ev[0].record(stream)
    for j in range(steps):
        i = warm + j
        layer.set_ffn_events(*ffn[j])
        info = layer.step(xs[i % 2], y, T, logits=logits[i], stream=stream, side_stream=side)
        misses.append(info.n_miss)
        ids_h[j % 2].copy_(ids_d, non_blocking=True)
        g_h[j % 2].copy_(g_d, non_blocking=True)
        ev[j + 1].record(stream)
        done.record(stream)
        done.synchronize()  # the step's routing on the host for the importance update
        used = np.unique(ids_h[j % 2].numpy())
        byts.append(sum(n8 if fmt[e] == pqe.PQE_FMT_FP8 else n4 for e in used) + T * H * 2 + T * k * H * 2)
        before = fmt.copy()
        if pqe.pqe_importance_step(torch.from_numpy(m), ids_h[j % 2], g_h[j % 2], T, k, E, 0.9, j, every, n_hi,
                                   torch.from_numpy(fmt)):
            moved = np.nonzero(before != fmt)[0]
            for e in moved:  # new page, resident copy dropped: refilled on its next use
                pg, nb = host_page(int(e))
                layer.set_host_page(int(e), pg, nb)
            fmt_dev.copy_(torch.from_numpy(fmt.copy()), non_blocking=False)
            changed.append(int(len(moved)))
            rerank_at.append(j)
    torch.cuda.synchronize()
    layer.set_ffn_events(None, None)
    layer.close()
    step_ms = [ev[j].elapsed_time(ev[j + 1]) for j in range(steps)]
    ffn_ms = [a.elapsed_time(b) for a, b in ffn]
    after = [j + 1 for j in rerank_at if j + 1 < steps]
    gbs = sum(byts) / (sum(ffn_ms) / 1e3) / 1e9
    tflops = 6.0 * T * k * H * I * steps / (sum(ffn_ms) / 1e3) / 1e12
    pk, kind = fp8_peak_tflops()
    quality = quality_proxy_rate(pqe, torch, device, cfg, q8, q4, m[:nq])
    return {"workload": "mixed per-expert precision layer (E=256, H=2048, I=512, top-8, T=4096; importance EMA of "
                        "the gate mass, re-ranked every 64 steps over 256 steps: top 25% FP8 pages, the rest MXFP4)",
            "steps": steps, "rerank_every": every, "n_fp8_experts": int((fmt == 0).sum()),
            "tokens_per_s": T * steps / (sum(step_ms) / 1e3), "ms_per_step": float(np.mean(step_ms)),
            "ms_per_step_after_rerank": [step_ms[j] for j in after],
            "misses_after_rerank": [misses[j] for j in after],
            "ms_per_step_other": float(np.mean([t for j, t in enumerate(step_ms) if j not in after])),
            "reranked_at_step": rerank_at, "fp8_set_changed": changed,
            "ffn_ms": float(np.mean(ffn_ms)), "ffn_hbm_gbs": gbs, "ffn_frac_of_measured_hbm": gbs / peaks()[0],
            "ffn_tflops": tflops, "ffn_frac_of_fp8_peak": tflops / pk, "fp8_peak_kind": kind,
            "note": "each step's routing is read back and folded into the importance EMA on the host before the "
                    "next step is issued",
            "quality_proxy": quality}


def quality_proxy_rate(pqe, torch, device, cfg, q8, q4, m, n=64, reps=4):
    """The 4-bit quality proxy on n sampled tokens per expert, timed per expert,
    and the quality-aware ranking of the sampled experts (score m * q) against
    the plain importance ranking."""
    H, I = cfg.H, cfg.I
    nq = q8.shape[0]
    x = torch.from_numpy(synth.activations(cfg, n, 7).view(np.int16)).to(device)
    ws = torch.zeros(pqe.pqe_quality_workspace_size(n, H, I), dtype=torch.uint8, device=device)
    sums = torch.zeros((nq, 2), dtype=torch.float64, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    for e in range(nq):  # warm-up
        pqe.pqe_expert_quant_error(x, n, q8[e], q4[e], H, I, sums[e], ws, status, stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        for e in range(nq):
            pqe.pqe_expert_quant_error(x, n, q8[e], q4[e], H, I, sums[e], ws, status, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    s = sums.cpu().numpy()
    q = np.sqrt(s[:, 0] / s[:, 1])
    n_hi = nq // 4
    f_plain = torch.zeros(nq, dtype=torch.uint8)
    f_qual = torch.zeros(nq, dtype=torch.uint8)
    pqe.pqe_rank_formats(torch.from_numpy(np.ascontiguousarray(m)), n_hi, f_plain)
    pqe.pqe_rank_formats_quality(torch.from_numpy(np.ascontiguousarray(m)), torch.from_numpy(q), n_hi, f_qual)
    return {"tokens_per_expert": n, "experts": nq, "us_per_expert": e0.elapsed_time(e1) * 1e3 / (reps * nq),
            "rel_err_mean": float(q.mean()), "rel_err_min": float(q.min()), "rel_err_max": float(q.max()),
            "fp8_set_changed": int((f_plain != f_qual).sum().item()) // 2, "status": int(status.item())}


def huff_decode_rate(pqe, torch, device, comp_host, sizes, luts_host, H, I, nb, n_pages=64, reps=5):
    """The GPU decoder alone: n_pages compressed pages already in HBM (copies
    of the distinct host pages; inputs + outputs ~0.6 GB, well above L2)
    decoded into FP8 pages by one fp8_exp_huff_decode_batch launch per call."""
    n_src = len(sizes)
    LB = pqe.PQE_HUFF_LUT_BYTES
    comp = torch.stack([comp_host[j % n_src] for j in range(n_pages)]).to(device)
    luts = torch.stack([luts_host[j % n_src] for j in range(n_pages)]).to(device)
    cb = [sizes[j % n_src] for j in range(n_pages)]
    outp = torch.zeros((n_pages, nb), dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    args = ([comp[j] for j in range(n_pages)], cb, [luts[j, :LB] for j in range(n_pages)],
            [luts[j, LB:] for j in range(n_pages)], H, I, [outp[j] for j in range(n_pages)], status)
    for _ in range(3):  # warm-up
        pqe.fp8_exp_huff_decode_batch(*args, stream=stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        a.record(stream)
        pqe.fp8_exp_huff_decode_batch(*args, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    launch_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    ms = launch_ms / n_pages
    cbm = float(np.mean(cb))
    gbs = (nb + cbm) / (ms / 1e3) / 1e9
    return {"pages_per_launch": n_pages, "ms_per_launch": launch_ms, "ms_per_page": ms,
            "decoded_gb_per_s": nb / (ms / 1e3) / 1e9, "compressed_gb_per_s": cbm / (ms / 1e3) / 1e9,
            "hbm_gb_per_s_in_plus_out": gbs, "frac_of_measured_hbm": gbs / peaks()[0],
            "algorithmic_bytes_per_launch": n_pages * (nb + cbm), "status": int(status.item())}


# ---- main arm ------------------------------------------------------------------------------

def main():
    args = parse_args()
    global OVERLAP_GROUPS
    OVERLAP_GROUPS = args.overlap_groups
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    import torch
    import paged_quantized_expert_gb300 as pqe
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pqe.load()
    pqe.pqe_test_set_stream_kernel({"auto": 0, "cuda": 1, "tc": 2}[args.stream_kernel])
    T, L, K, W = args.T, args.layers, args.steps, max(3, args.warmup)
    if args.workload not in ("huff", "ram"):
        measure_fp8_peak(torch, device)
    if args.workload in ("large", "mixed", "huff"):
        res = {"large": run_large, "mixed": run_mixed, "huff": run_huff}[args.workload](pqe, torch, device)
        if rank == 0:
            print(json.dumps({args.workload: res}))
        return 0
    host = expert_pages_host(pqe, torch, device)
    graph_extra = L if args.pager != "host" else 0
    if args.workload == "ram":
        res = run_ram(pqe, torch, device, host)
        if rank == 0:
            print(json.dumps({"ram": res}))
        return 0
    if args.workload == "batched":
        res = run_batched(pqe, torch, device, host, args.batched_steps, ws)
        if rank == 0:
            print(json.dumps({"batched": res}))
        return 0
    r = Runner(pqe, torch, device, host, L, max(T, 64))
    xs_dev = [torch.from_numpy(synth.activations(CFG, T, s).view(np.int16)).to(device) for s in range(4)]
    logits_np = make_traces(T, L, max(W, 2 * L) + K + graph_extra)  # the e2e leg warms up on 2 L steps at least
    logits_dev = [torch.from_numpy(l).to(device) for l in logits_np]
    y = torch.zeros((T, CFG.H), dtype=torch.bfloat16, device=device)

    clocks = Clocks(local)
    clocks.start()
    ms, wall, infos, ffn_ms, launches = run_timed(r, T, logits_dev, xs_dev, y, W, K, ws)
    clk = clocks.stop()
    ms = max_over_ranks(ws, ms, device)
    host_value, host_ms = ws * T * K / (ms / 1e3), ms / K
    value, pager_used, graph, graph_ffn = host_value, "host", None, {}
    if args.pager != "host":
        r.close()
        clocks_g = Clocks(local)
        clocks_g.start()
        gms, gstats, glaunch = run_graph(pqe, torch, device, host, T, L, logits_dev, xs_dev, W, K, ws)
        clk_g = clocks_g.stop()
        gms = max_over_ranks(ws, gms, device)
        gval = ws * T * K / (gms / 1e3)
        graph = {"tokens_per_s": gval, "ms_per_step": gms / K, "gpu_launches": int(glaunch),
                 "overlap_groups": overlap_groups_for(T),
                 "mean_routed_experts": gstats["routed"] / K, "mean_misses": gstats["misses"] / K,
                 "working_buffer_steps": gstats["working_buffer_steps"],
                 "h2d_gb_per_s": gstats["refill_bytes"] / (gms / 1e3) / 1e9, "clocks": clk_g}
        if args.pager == "device" or gval > host_value:
            value, pager_used, ms, launches, clk = gval, "device", gms, glaunch, clk_g
            # the FFN call's time: a second pass of the same replays with its event nodes
            graph_ffn = run_graph(pqe, torch, device, host, T, L, logits_dev, xs_dev, W, min(K, 128), ws,
                                  ffn_events=True)[1]["ffn_ms_last"]
        r = Runner(pqe, torch, device, host, L, max(T, 64))

    # roofline of the FFN call (w13 + SwiGLU, w2; HBM-bound weight stream), from
    # the run `value` comes from: the host-pager steps (FFN events of every timed
    # step), or the device-pager graph replays (event nodes of each layer's last
    # replay, with those steps' routed experts from their logits)
    peak, peak_kind = peaks()
    if pager_used == "device":
        ffn_steps = sorted(graph_ffn)
        byts = [ffn_bytes(routed_experts(logits_np[i], CFG.k), T) for i in ffn_steps]
        ffn_list = [graph_ffn[i] for i in ffn_steps]
        ffn_source = f"device-pager graph replays (last replay of each of the {L} layers)"
    else:
        byts = [ffn_bytes(n, T) for (n, _, _, _) in infos]
        ffn_list = ffn_ms
        ffn_source = f"host-pager steps ({K} timed steps)"
    ffn_total_ms = sum(ffn_list)
    achieved = sum(byts) / (ffn_total_ms / 1e3) / 1e9 if ffn_total_ms > 0 else None
    # DRAM bytes of one FFN call: the ratio of an ncu capture of its kernels at
    # T=64 to that call's algorithmic bytes, times this run's algorithmic bytes
    traffic = (FFN_DRAM_PER_ALGORITHMIC_BYTE_T64 * float(np.mean(byts))
               if T == 64 and FFN_DRAM_PER_ALGORITHMIC_BYTE_T64 else None)

    # e2e: host buffers through pqe_layer_step_host, on layers with the
    # headline's pager (and its overlap groups); on device-pager layers the call
    # replays its own cached graph of the step's launches between the copies
    x_h = torch.from_numpy(synth.activations(CFG, T, 0).view(np.int16)).pin_memory()
    y_h = torch.zeros((T, CFG.H), dtype=torch.bfloat16).pin_memory()
    lg_h = [torch.from_numpy(l).pin_memory() for l in logits_np]
    Ke = min(K, 128)
    We = max(W, 2 * L) if pager_used == "device" else W
    re = r
    if pager_used == "device":
        r.close()
        re = Runner(pqe, torch, device, host, L, max(T, 64), device_pager=True, overlap_groups=overlap_groups_for(T))
        re.stream = torch.cuda.Stream(device)  # a created stream, as a caller's would be (capturable)
        # two calls per layer at least: the second captures the layer's step graph
        for i in range(We):
            re.layers[i % L].step_host(x_h, y_h, T, logits_host=lg_h[i], stream=re.stream, side_stream=re.side)
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(re.stream)
    for j in range(Ke):
        i = We + j
        re.layers[i % L].step_host(x_h, y_h, T, logits_host=lg_h[i], stream=re.stream, side_stream=re.side)
    e1.record(re.stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ws, e0.elapsed_time(e1), device)
    e2e_value = ws * T * Ke / (e2e_ms / 1e3)
    if re is not r:
        re.close()
        r = Runner(pqe, torch, device, host, L, max(T, 64))

    sweep = {}
    if not args.no_sweep:
        for Ts in (1, 8):
            if Ts == T:
                continue
            lg_s = [torch.from_numpy(l).to(device) for l in make_traces(Ts, L, W + K)]
            xs_s = [torch.from_numpy(synth.activations(CFG, Ts, s).view(np.int16)).to(device) for s in range(4)]
            ys = torch.zeros((Ts, CFG.H), dtype=torch.bfloat16, device=device)
            ms_s, _, inf_s, ffn_s, _ = run_timed(r, Ts, lg_s, xs_s, ys, W, K, ws)
            b_s = [ffn_bytes(n, Ts) for (n, _, _, _) in inf_s]
            rec = {"tokens_per_s": ws * Ts * K / (max_over_ranks(ws, ms_s, device) / 1e3),
                   "ms_per_step": ms_s / K, "pager": "host",
                   "ffn_hbm_gbs": sum(b_s) / (sum(ffn_s) / 1e3) / 1e9 if sum(ffn_s) > 0 else None,
                   "misses_per_step": float(np.mean([m for (_, m, _, _) in inf_s]))}
            if pager_used == "device":
                # the same pager as the headline: graph replays without, then with, the FFN event nodes
                r.close()
                lg_g = [torch.from_numpy(l).to(device) for l in make_traces(Ts, L, W + K + L)]
                gms_s, gst_s, _ = run_graph(pqe, torch, device, host, Ts, L, lg_g, xs_s, W, K, ws)
                gms_s = max_over_ranks(ws, gms_s, device)
                f_s = run_graph(pqe, torch, device, host, Ts, L, lg_g, xs_s, W, min(K, 128), ws,
                                ffn_events=True)[1]["ffn_ms_last"]
                fb = [ffn_bytes(routed_experts(lg_g[i].cpu().numpy(), CFG.k), Ts) for i in sorted(f_s)]
                fm = [f_s[i] for i in sorted(f_s)]
                rec_host = {k: rec[k] for k in ("tokens_per_s", "ms_per_step", "ffn_hbm_gbs")}
                rec = {"tokens_per_s": ws * Ts * K / (gms_s / 1e3), "ms_per_step": gms_s / K, "pager": "device",
                       "overlap_groups": overlap_groups_for(Ts),
                       "ffn_ms": float(np.mean(fm)), "ffn_hbm_gbs": sum(fb) / (sum(fm) / 1e3) / 1e9,
                       "misses_per_step": gst_s["misses"] / K, "host_pager": rec_host}
                r = Runner(pqe, torch, device, host, L, max(T, 64))
            sweep[f"T={Ts}"] = rec

    # the same decode steps with a compressed host tier (device pager, graph replays):
    # the link-bound step moves fewer bytes per refill
    decode_compressed = None
    if not args.no_extra and pager_used == "device":
        r.close()
        pages_c, sizes_c, luts_c, ratio = decode_compressed_pages(pqe, torch, host)
        cms, cst, _ = run_graph(pqe, torch, device, host, T, L, logits_dev, xs_dev, W, K, ws,
                                comp=(pages_c, sizes_c, luts_c.to(device)), groups=0)
        cms = max_over_ranks(ws, cms, device)
        decode_compressed = {"tokens_per_s": ws * T * K / (cms / 1e3), "ms_per_step": cms / K,
                             "compressed_over_fp8_bytes": ratio, "mean_misses": cst["misses"] / K,
                             "h2d_gb_per_s": cst["refill_bytes"] / (cms / 1e3) / 1e9,
                             "note": "the same workload and routing as the headline with Huffman-coded FP8 "
                                     "exponents in the host tier (32 distinct encoded pages), each miss pulled "
                                     "and decoded in one pass; no refill groups"}
        r = Runner(pqe, torch, device, host, L, max(T, 64))

    batched = None
    if not args.no_batched:
        r.close()
        batched = run_batched(pqe, torch, device, host, args.batched_steps, ws)
    large = mixed = ram_tier = None
    if not args.no_extra:
        r.close()
        large = run_large(pqe, torch, device)
        mixed = run_mixed(pqe, torch, device)
        ram_tier = run_ram(pqe, torch, device, host)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tok, secs, threads, steps = cpu_oracle_sample(host.numpy(), T, make_traces(T, 1, 16), budget_s=10.0)
        cpu = {"value": tok / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{steps} layer-0 trace steps x {T} tokens (route, permute, LRU, FFN of every token)"}

    n_routed = [n for (n, _, _, _) in infos]
    misses = [m for (_, m, _, _) in infos]
    h2d = [b for (_, _, _, b) in infos]
    h2d_step = graph["h2d_gb_per_s"] if pager_used == "device" else sum(h2d) / (ms / 1e3) / 1e9
    h2d_peak = measure_h2d_peak(torch, device)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8(e4m3) weights, bf16 activations, fp32 accumulate", "data": "synthetic",
            "config": {"workload": "decode-shaped paged MoE layer (E=256, H=2048, I=512, top-8, "
                                   "CACHE_SLOTS=32 LRU per layer, Zipf(1.1) routing with 0.7 reuse, "
                                   "pinned-host refills)",
                       "T": T, "layers_round_robin": L,
                       "pager": pager_used + (" (LRU on the GPU, each step a CUDA graph replay)"
                                              if pager_used == "device" else " (LRU on the host, eager launches)"),
                       "host_pager": {"tokens_per_s": host_value, "ms_per_step": host_ms},
                       "device_pager_graph": graph,
                       "l2": f"inputs larger than L2: {L} layers x 32 slots x 3.16 MB of weights",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "mean_routed_experts": float(np.mean(n_routed)), "mean_misses": float(np.mean(misses)),
                       "working_buffer_steps": int(sum(w for (_, _, w, _) in infos)),
                       "h2d_gb_per_s": (sum(h2d) / (ms / 1e3) / 1e9), "by_T": sweep},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                         "kernel": "moe_paged_ffn (w13+SwiGLU and w2 weight streams)",
                         "peak_kind": peak_kind,
                         "ffn_ms_per_step": ffn_total_ms / len(ffn_list), "ffn_timing": ffn_source,
                         "algorithmic_bytes_per_step": float(np.mean(byts))},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * CFG.H * 2 + T * CFG.E * 4,
                    "d2h_bytes_per_step": T * CFG.H * 2, "pager": pager_used,
                    "api": "pqe_layer_step_host (pinned host x and logits in, pinned host y out, every step; "
                           "the call's own step graph on device-pager layers)"},
            "gpu_launches": int(launches),
            "fp8_peak": dict(_FP8_PEAK),
            # the step's refills against the host link: bytes refilled per second of
            # whole steps, against a plain pinned-host-to-device copy in this run
            "host_link": {"achieved": h2d_step, "peak": h2d_peak, "unit": "GB/s",
                          "frac": h2d_step / h2d_peak if h2d_peak else None,
                          "peak_kind": "measured: one 1 GiB pinned-host-to-device copy (best of 5), this run",
                          "note": "refill bytes of the timed steps / their whole time: the step is bound by "
                                  "this link, the FFN running beside the refills"},
            "clocks": clk,
            "decode_compressed": decode_compressed,
            "batched": batched,
            "large": large,
            "mixed": mixed,
            "ram_tier": ram_tier,
        }
        print(json.dumps(line))
    r.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

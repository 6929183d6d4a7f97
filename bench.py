"""Benchmark of the NVFP4 MoE layer on GB300.

One step = the whole layer over one batch: route + permute, quantise x into
the routed rows, gate_up grouped GEMM with SiLU-mul + requantisation, down
grouped GEMM with FINALIZE.  Default workload: the prefill layer with
T=16384 tokens, E=256 experts, top-8, H=6144, I=2048 (uniform router logits),
the largest of the layer configurations; the 1024-token decode layer on the
same weights is measured in the same run (the line's decode_c4 entry).

value: tokens/s of the layer with inputs resident in HBM (CUDA events on the
launching stream over exactly --steps steps, after --warmup steps).  The
expert weights (5.4 GB of NVFP4) are far larger than L2 (129 MB), so every
step streams them from HBM; no L2 flush is needed.
e2e: the same through moe_forward with pinned host buffers: every step copies
x and the logits to the device and the output back.
roofline: the gate_up grouped GEMM (the largest kernel).  At prefill it is
bound by the tensor cores: its FLOPs over its event-timed duration against
this GPU's dense NVFP4 MMA rate (the larger of the two probes, both in the
line), with its HBM rate beside it.  At decode (decode_c4) it is bound by
HBM: algorithmic bytes per launch over the duration against the measured
copy bandwidth.
cpu_baseline: the CPU oracle on a bounded sample of the same batch.

--impl reference times the CPU oracle (the reference arm of this repo) on a
bounded sample of the same workload and prints the same JSON line shape.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

T_DEF, E_DEF, K_DEF, H_DEF, I_DEF = 16384, 256, 8, 6144, 2048
DECODE_T_DEF = 1024
METRIC = "MoE-layer tokens/s and grouped-GEMM TFLOPS & HBM GB/s vs roofline, 1 GB300"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=T_DEF)
    ap.add_argument("--experts", type=int, default=E_DEF)
    ap.add_argument("--top-k", type=int, default=K_DEF)
    ap.add_argument("--hidden", type=int, default=H_DEF)
    ap.add_argument("--intermediate", type=int, default=I_DEF)
    ap.add_argument("--zipf", type=float, default=None)
    ap.add_argument("--decode-tokens", type=int, default=DECODE_T_DEF,
                    help="also measure the layer at this many tokens on the same weights (the decode_c4 entry of "
                         "the line; 0 to skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="layer", choices=["layer", "gemm", "dense", "router"],
                    help="layer: the full MoE layer (default); gemm: one grouped GEMM, 256 experts x 32 rows, "
                         "K=6144, N=2048, NONE epilogue; dense: one dense NVFP4 GEMM M=N=K=--dense-size; "
                         "router: the router logits GEMM + routing for --tokens tokens")
    ap.add_argument("--dense-size", type=int, default=16384)
    ap.add_argument("--gated", action="store_true",
                    help="layer workload with the router in front (moe_forward_gated: x and a bf16 gate "
                         "matrix instead of logits)")
    ap.add_argument("--profile-steps", action="store_true",
                    help="no JSON; only the steps run between cudaProfilerStart/Stop (for ncu)")
    return ap.parse_args()


def _code_only(src: str) -> str:
    """C/C++ source with its comments removed and whitespace runs collapsed (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest() -> str:
    """SHA-256 of the code (comments and layout stripped) of the grouped-GEMM source and the headers it
    includes: identifies the measured kernel."""
    import hashlib
    h = hashlib.sha256()
    for rel in ("nvfp4_moe_grouped_gb300/csrc/grouped_gemm.cu", "nvfp4_moe_grouped_gb300/csrc/common.cuh",
                "include/nvfp4_moe.h"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the gate_up GEMM from the committed ncu records, or None when no record is
    for this workload and the current kernel source (a record taken before the kernel changed is stale)."""
    try:
        with open(os.path.join(ROOT, "profiles", "gate_up_dram_traffic.json")) as f:
            doc = json.load(f)
    except Exception:
        return None
    digest = kernel_source_digest()
    for rec in doc.get("records", [doc]):
        if rec.get("workload") == workload and rec.get("kernel_sha256") == digest:
            return rec.get("dram_bytes_per_launch")
    return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1952.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []          # (host time, csv line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi takes a moment to start: wait (bounded) for its first sample
            deadline = time.time() + 5.0
            while not self.lines and time.time() < deadline and self.proc.poll() is None:
                time.sleep(0.005)
        except Exception:
            self.proc = None
        return self

    def start(self):
        """Marks the start of the timed region (host clock)."""
        self.t0 = time.time()

    def stop(self):
        """Marks the end of the timed region (after the closing synchronize)."""
        self.t1 = time.time()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *a):
        if self.proc is not None:
            # one more sample interval so a sample lands after the region ends
            time.sleep(2 * self.interval_ms / 1e3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = "timed region"
        chosen = self.lines
        if self.t0 is not None and self.t1 is not None:
            # a line is printed when its sample is taken: keep those inside the timed region
            chosen = [(t, ln) for t, ln in self.lines if self.t0 <= t <= self.t1]
            if not chosen:
                after = [(t, ln) for t, ln in self.lines if t > self.t1]
                chosen = after[:1]
                window = "first sample after the timed region (region shorter than the sampling interval)"
        for _, ln in chosen:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "window": window}


# ------------------------------------------------------------------ replicas (N > 1)

def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (x itself with one rank): the job's time is its slowest replica's."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    if torch.distributed.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units per second of the whole job: every rank processes units_per_rank in (at most) ms."""
    return world * units_per_rank / (ms / 1e3)


# ------------------------------------------------------------------ setup

def make_layer(T, E, k, H, I, zipf, dev):
    import nvfp4_moe_grouped_gb300 as moe
    from nvfp4_moe_grouped_gb300 import inputs

    x = inputs.activations(T, H)                       # CPU generator, seed 0
    logits = inputs.router_logits(T, E, zipf_s=zipf)   # CPU generator, seed 1
    # full-size weights: drawn on the device with the per-expert seeds, quantised there
    w13f = inputs.expert_weights(E, 2 * I, H, inputs.gate_up_seed_base(), device=dev)
    pw13 = moe.prepare_expert_weights(w13f, gate_up=True)
    del w13f
    w2f = inputs.expert_weights(E, H, I, inputs.down_seed_base(E), device=dev)
    pw2 = moe.prepare_expert_weights(w2f, gate_up=False)
    del w2f
    torch.cuda.empty_cache()
    return x, logits, pw13, pw2


def calibrate_h_scale(fwd, xd, ld, pw13):
    """Static decode multiplier of the intermediate: amax of this batch's h / (6*448)."""
    import nvfp4_moe_grouped_gb300 as moe
    L = fwd.layout
    T, E, k, H, I = fwd.T, fwd.E, fwd.k, fwd.H, fwd.I
    P = L.padded_rows
    r = moe.moe_route_permute(ld, k)
    codes, sf, s = moe.nvfp4_quantize(xd, None, n_items=T * k, src_div=k, dst_row=r.expanded_to_row,
                                      sf_layout=moe.SF_TILED, dst_rows_alloc=P)
    h_f32 = torch.zeros(P, I, dtype=torch.float32, device=xd.device)
    moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw13, r.expert_offsets, moe.EPI_SILU_MUL_QUANT, h_scale=1.0, h_f32=h_f32)
    amax = float(h_f32.abs().max().item())
    del h_f32, codes, sf
    return amax / 2688.0 if amax > 0 else 1.0


def algorithmic_bytes(expert_counts, T, E, k, H, I):
    """Bytes the layer must move: weights of active experts once, activations, intermediates, outputs."""
    active = int((expert_counts > 0).sum())
    R = T * k
    w13 = 2 * I * H // 2 + 2 * I * H // 16
    w2 = H * I // 2 + H * I // 16
    gate_up = active * w13 + R * (H // 2 + H // 16) + R * (I // 2 + I // 16)
    down = active * w2 + R * (I // 2 + I // 16) + T * H * 4 * 2   # FP32 accumulate (read-modify-write)
    layer = gate_up + down + T * H * 2 + T * E * 4 + T * H * 2
    return {"gate_up": gate_up, "down": down, "layer": layer, "active_experts": active}


# ------------------------------------------------------------------ CPU oracle sample

def oracle_sample(x, logits, T, E, k, H, I, n_tokens, h_scale, dev, cache=None):
    """Time the CPU oracle on the first n_tokens tokens of the batch (weights of their experts only).

    `cache` (a dict) keeps the oracle's quantised expert weights between calls: preparing them is model
    setup, untimed either way."""
    import oracle
    from nvfp4_moe_grouped_gb300 import inputs

    xs = x[:n_tokens].float().numpy()
    ls = logits[:n_tokens].numpy()
    ids, _ = oracle.route(ls, k)
    experts = sorted(set(ids.reshape(-1).tolist()))
    if cache is None:
        cache = {}
    wq13, wq2 = cache.setdefault("w13", {}), cache.setdefault("w2", {})
    for e in experts:   # untimed: model preparation (the FP32 weights are redrawn with the same seeds)
        if e in wq13:
            continue
        w13 = inputs.expert_weight(e, 2 * I, H, inputs.gate_up_seed_base(), device=dev).cpu().numpy()
        w2 = inputs.expert_weight(e, H, I, inputs.down_seed_base(E), device=dev).cpu().numpy()
        wq13[e] = oracle.quantize_dynamic(w13)
        wq2[e] = oracle.quantize_dynamic(w2)
    t0 = time.perf_counter()
    # the layer in the method's order, restricted to the sampled tokens; the activations' tensor
    # scale is the whole batch's
    ids, w = oracle.route(ls, k)
    xsc = oracle.tensor_scale_from_amax(oracle.amax(x.float().numpy()))
    xc, xsf = oracle.quantize(xs, xsc)
    out = np.zeros((n_tokens, H))
    for t in range(n_tokens):
        for j in range(k):
            e = int(ids[t, j])
            c13, s13, sc13 = wq13[e]
            y1 = oracle.grouped_gemm(xc[t:t + 1], xsf[t:t + 1], xsc, c13[None], s13[None],
                                     np.array([sc13], np.float32), np.array([0, 1], np.int32), 2 * I, H)
            h = oracle.silu_mul(y1).astype(np.float32)
            hc, hs = oracle.quantize(h, h_scale)
            c2, s2, sc2 = wq2[e]
            y2 = oracle.grouped_gemm(hc, hs, h_scale, c2[None], s2[None], np.array([sc2], np.float32),
                                     np.array([0, 1], np.int32), H, I)
            out[t] += float(w[t, j]) * y2[0]
    dt = time.perf_counter() - t0
    return dt, out


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ arms

def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: bounded samples of the same workload."""
    if rank != 0:
        return
    T, E, k, H, I = args.tokens, args.experts, args.top_k, args.hidden, args.intermediate
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    from nvfp4_moe_grouped_gb300 import inputs
    x = inputs.activations(T, H)
    logits = inputs.router_logits(T, E, zipf_s=args.zipf)
    n_tok = 1
    h_scale = 0.01
    cache = {}
    for _ in range(args.warmup):
        oracle_sample(x, logits, T, E, k, H, I, n_tok, h_scale, dev, cache)
    times = []
    for _ in range(args.steps):
        dt, _ = oracle_sample(x, logits, T, E, k, H, I, n_tok, h_scale, dev, cache)
        times.append(dt)
    tot = sum(times)
    value = n_tok * args.steps / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"moe_layer_T{T}_E{E}_k{k}_H{H}_I{I}" + (f"_zipf{args.zipf}" if args.zipf else "_uniform"),
                       "sample": f"{n_tok} token(s) of the batch per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{n_tok} token(s) per step, {args.steps} steps"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


FP4_PEAK_KIND = ("measured: the larger of this GPU's two dense NVFP4 MMA rate probes (moe_fp4_mma_probe, "
                 "moe_fp4_mma_probe_pair)")


def fp4_peaks(local_rank):
    """This GPU's dense NVFP4 MMA rate from both probes (one CTA per SM with M = 128; CTA pairs with M = 256),
    each timed over about half a second with the SM clock sampled meanwhile; the roofline takes the larger."""
    import nvfp4_moe_grouped_gb300 as moe
    out = {}
    for name, pair in (("cta_m128", False), ("pair_m256", True)):
        moe.fp4_mma_peak_tflops(iters=2000, reps=2, pair=pair)   # warm-up
        with ClockSampler(local_rank) as clk:
            clk.start()
            rate = moe.fp4_mma_peak_tflops(iters=20000, reps=200, pair=pair)
            clk.stop()
        out[name] = {"tflops": rate, "clocks": clk.summary()}
    out["peak_tflops"] = max(out["cta_m128"]["tflops"], out["pair_m256"]["tflops"])
    return out


def measure_layer(args, T, E, k, H, I, x, logits, pw13, pw2, dev, world, local_rank, e2e=True):
    """One layer configuration through moe_forward: eager stage timing (each C-ABI stage bracketed by events on
    the launching stream), the whole layer as one CUDA graph replayed back to back (the headline value, clocks
    sampled meanwhile), and optionally the end-to-end run with pinned host buffers."""
    import ctypes

    import nvfp4_moe_grouped_gb300 as moe

    xd, ld = x.to(dev), logits.to(dev)
    fwd = moe.MoeForward(T, E, k, H, I, dev)
    h_scale = calibrate_h_scale(fwd, xd, ld, pw13)
    L = fwd.layout
    P = L.padded_rows
    R = T * k
    stream = torch.cuda.current_stream()
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    lib = moe._lib.load()
    ptr = lambda name: ctypes.c_void_p(fwd.ws.data_ptr() + getattr(L, name))
    _p = lambda t: ctypes.c_void_p(t.data_ptr())
    _s = lambda: ctypes.c_void_p(stream.cuda_stream)

    def _call(name, st):
        if st != 0:
            raise moe.MoeError(name, st)

    def step(ev=None):
        # the layer as its four C-ABI stages; events between them time each stage on this stream
        _call("moe_route_permute", lib.moe_route_permute(
            _p(ld), T, E, k, ptr("topk_id"), ptr("topk_w"), ptr("expert_offsets"), ptr("perm_to_expanded"),
            ptr("expanded_to_perm"), ptr("expanded_to_row"), ptr("route_ws"),
            lib.moe_route_permute_workspace_size(T, E, k), _s()))
        if ev is not None:
            ev[0].record(stream)
        _call("nvfp4_quantize", lib.nvfp4_quantize(
            _p(xd), 0, T, H, 1, ptr("x_scale"), 1, R, k, ptr("expanded_to_row"), ptr("x_codes"),
            ptr("x_sf"), 1, P, ptr("quant_ws"), lib.nvfp4_quantize_workspace_size(1), _s()))
        if ev is not None:
            ev[1].record(stream)
        ep = moe.EpilogueArgs()
        ep.h_scale = h_scale
        ep.h_scale_out = ptr("h_scale")
        ep.h_codes = ptr("h_codes")
        ep.h_sf = ptr("h_sf")
        _call("moe_grouped_gemm_nvfp4", lib.moe_grouped_gemm_nvfp4(
            ptr("x_codes"), ptr("x_sf"), ptr("x_scale"), _p(pw13.blocked), _p(pw13.scale),
            ptr("expert_offsets"), E, P, 2 * I, H, moe.EPI_SILU_MUL_QUANT, ctypes.byref(ep), None, None, 0, _s()))
        if ev is not None:
            ev[2].record(stream)
        ep = moe.EpilogueArgs()
        ep.perm_to_expanded = ptr("perm_to_expanded")
        ep.topk_w = ptr("topk_w")
        ep.T = T
        ep.k = k
        wsb = lib.moe_grouped_gemm_workspace_size(moe.EPI_FINALIZE, T, k, H)
        _call("moe_grouped_gemm_nvfp4", lib.moe_grouped_gemm_nvfp4(
            ptr("h_codes"), ptr("h_sf"), ptr("h_scale"), _p(pw2.blocked), _p(pw2.scale),
            ptr("expert_offsets"), E, P, H, I, moe.EPI_FINALIZE, ctypes.byref(ep), _p(out), ptr("gemm_ws"), wsb,
            _s()))
        if ev is not None:
            ev[3].record(stream)

    if args.profile_steps:
        prof_step = step
        if moe.forward_kernel_count(T, E, k, H, I) == 1:
            # a layer this small runs as one kernel through moe_forward (not as the four stages): profile that
            def prof_step():
                fwd(xd, ld, pw13, pw2, h_scale, out=out)
        for _ in range(max(1, args.warmup)):
            prof_step()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStart()
        for _ in range(args.steps):
            prof_step()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStop()
        return None

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    counts = np.diff(fwd.view("expert_offsets", torch.int32, (E + 1,)).cpu().numpy())
    ab = algorithmic_bytes(counts, T, E, k, H, I)

    # ---- eager stage calls: per-stage launch times
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    stop.record(stream)
    torch.cuda.synchronize()
    eager_ms = start.elapsed_time(stop)
    prev = [start] + [evs[i][3] for i in range(args.steps - 1)]
    stage_ms = np.zeros(4)
    for i in range(args.steps):
        stage_ms[0] += prev[i].elapsed_time(evs[i][0])
        for j in range(1, 4):
            stage_ms[j] += evs[i][j - 1].elapsed_time(evs[i][j])
    stage_ms /= args.steps

    # ---- the headline region: the whole layer as one CUDA graph, replayed back to back.  The timed graph
    # has no stage-timing event nodes; a second graph with them gives the per-stage split afterwards.
    out_g = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    graph = fwd.graph(xd, ld, pw13, pw2, h_scale, out=out_g, stage_events=False)
    graph_st = fwd.graph(xd, ld, pw13, pw2, h_scale, out=out_g, stage_events=True)
    for _ in range(args.warmup):
        graph.launch()
        graph_st.launch()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    weight_bytes = E * (2 * I * H + H * I) * 9 // 16
    flush = weight_bytes < (256 << 20)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        clk.start()
        if flush:
            # the weights would stay in L2 between steps: write a 256 MB buffer before every step and
            # time each step on its own
            scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for a_, b_ in ev:
                scrub.fill_(1)
                a_.record(stream)
                graph.launch()
                b_.record(stream)
            torch.cuda.synchronize()
            clk.stop()
            ms = sum(a_.elapsed_time(b_) for a_, b_ in ev)
        else:
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(args.steps):
                graph.launch()
            g1.record(stream)
            torch.cuda.synchronize()
            clk.stop()
            ms = g0.elapsed_time(g1)
    if world > 1:
        torch.distributed.barrier()
    graph_st.launch()
    torch.cuda.synchronize()
    graph_last_stages = graph_st.stage_ms()
    ms = max_over_ranks(ms, dev)
    ms_step = ms / args.steps
    res = {"T": T, "ms_step": ms_step, "value": whole_job_rate(T, world, ms_step), "stage_ms": stage_ms,
           "graph_last_stages": graph_last_stages, "eager_ms": eager_ms / args.steps, "ab": ab, "h_scale": h_scale,
           "clocks": clk.summary(), "flush": flush, "weight_bytes": weight_bytes}
    if not e2e:
        return res

    # ---- end to end through the library's host-buffer call (moe_forward_graph_run_host): every step copies
    # its inputs from pinned host memory into the graph's device buffers, replays the layer and copies the
    # output back, all on one stream.  Steps alternate between two streams, each with its own graph, device
    # buffers and workspace, so one step's copies overlap the other's layer, as a serving pipeline runs.
    xh = x.pin_memory()
    lh = logits.pin_memory()
    ohs = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    fwds = [fwd, moe.MoeForward(T, E, k, H, I, dev)]
    xds = [torch.empty_like(xd) for _ in range(2)]
    lds = [torch.empty_like(ld) for _ in range(2)]
    outs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    graphs_e2e = [fwds[b].graph(xds[b], lds[b], pw13, pw2, h_scale, out=outs[b], stage_events=False)
                  for b in range(2)]
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]

    def e2e_step(i):
        b = i & 1
        graphs_e2e[b].run_host(xh, lh, ohs[b], stream=streams[b])

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st_b in streams:
        st_b.wait_stream(stream)
    for i in range(args.steps):
        e2e_step(i)
    for st_b in streams:
        stream.wait_stream(st_b)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    # the output read back is the layer's output for these inputs (the device-timed graph computed it too;
    # FINALIZE's atomics may order the FP32 sums differently, so compare by relative difference)
    ref_out = out_g.float().cpu()
    e2e_rel = float((ohs[(args.steps - 1) & 1].float() - ref_out).norm() / max(float(ref_out.norm()), 1e-30))
    res["e2e"] = {"value": whole_job_rate(T * args.steps, world, e2e_ms), "unit": "tokens/s",
                  "h2d_bytes_per_step": T * H * 2 + T * E * 4, "d2h_bytes_per_step": T * H * 2,
                  "how": "moe_forward_graph_run_host every step: pinned H2D of x and logits, the layer graph, D2H "
                         "of the output, on one stream; steps alternate between two streams (two graphs, buffer "
                         "sets and workspaces), so one step's copies overlap the other's layer",
                  "output_rel_diff_vs_device_run": e2e_rel}
    return res


def layer_roofline(r, k, H, I, fp4, hbm_peak, peak_kind, workload):
    """Roofline of the gate_up GEMM launch of a measured layer: tensor-bound (its FLOPs against the larger
    measured FP4 MMA rate, its HBM rate beside it) where experts see more than 48 routed rows on average,
    HBM-bound (algorithmic bytes against the measured copy bandwidth) otherwise."""
    T = r["T"]
    ab = r["ab"]
    ms = r["stage_ms"][2]
    flops = 2.0 * T * k * 2 * I * H
    hbm = ab["gate_up"] / (ms / 1e3) / 1e9
    if T * k / max(1, ab["active_experts"]) > 48:
        achieved = flops / (ms / 1e3) / 1e12
        return {"bound": "tensor", "kernel": "grouped_gemm gate_up (SiLU-mul + requant epilogue)",
                "achieved": achieved, "peak": fp4["peak_tflops"], "unit": "TFLOP/s",
                "frac": achieved / fp4["peak_tflops"],
                "peak_kind": FP4_PEAK_KIND,
                "traffic": recorded_traffic(workload), "algorithmic_flops_per_launch": flops, "launch_ms": ms,
                "hbm_gbs": hbm, "hbm_frac": hbm / hbm_peak, "algorithmic_bytes_per_launch": ab["gate_up"]}
    return {"bound": "hbm", "kernel": "grouped_gemm gate_up (SiLU-mul + requant epilogue)", "achieved": hbm,
            "peak": hbm_peak, "unit": "GB/s", "frac": hbm / hbm_peak, "peak_kind": peak_kind,
            "traffic": recorded_traffic(workload), "algorithmic_bytes_per_launch": ab["gate_up"], "launch_ms": ms,
            "tflops": flops / (ms / 1e3) / 1e12}


def layer_workload_name(T, E, k, H, I, zipf):
    return f"moe_layer_T{T}_E{E}_k{k}_H{H}_I{I}" + (f"_zipf{zipf}" if zipf else "_uniform")


def run_ours(args, rank, world, local_rank):
    import nvfp4_moe_grouped_gb300 as moe
    from nvfp4_moe_grouped_gb300 import inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    T, E, k, H, I = args.tokens, args.experts, args.top_k, args.hidden, args.intermediate
    x, logits, pw13, pw2 = make_layer(T, E, k, H, I, args.zipf, dev)
    main_r = measure_layer(args, T, E, k, H, I, x, logits, pw13, pw2, dev, world, local_rank, e2e=True)
    if main_r is None:   # --profile-steps: only the profiled steps ran
        return
    # the 1024-token decode layer on the same weights, measured in the same run
    dec = None
    Td = args.decode_tokens
    if Td and Td != T:
        xd4 = inputs.activations(Td, H)
        ld4 = inputs.router_logits(Td, E, zipf_s=args.zipf)
        dec = measure_layer(args, Td, E, k, H, I, xd4, ld4, pw13, pw2, dev, world, local_rank, e2e=False)
    code, where = moe.device_error()
    if code != 0:
        raise RuntimeError(f"device error {code} at {where} during the benchmark")
    if rank != 0:
        return

    hbm_peak, bf16_peak, peak_kind = peaks()
    fp4 = fp4_peaks(local_rank)
    workload = layer_workload_name(T, E, k, H, I, args.zipf)
    roof = layer_roofline(main_r, k, H, I, fp4, hbm_peak, peak_kind, workload)
    stage_ms = main_r["stage_ms"]
    gl = main_r["graph_last_stages"]
    ms_step = main_r["ms_step"]
    flops_layer = 2.0 * T * k * (2 * I * H + H * I)
    cpu = None
    if not args.no_cpu_baseline:
        # a 2-token probe sizes the sample to about 12 s of oracle work (at most 64 tokens); preparing the
        # oracle's copy of each touched expert's weights is model setup and untimed
        cache = {}
        dt2, _ = oracle_sample(x, logits, T, E, k, H, I, 2, main_r["h_scale"], dev, cache)
        n_tok = int(min(T, 64, max(2, math.ceil(12.0 / max(dt2 / 2, 1e-6)))))
        dt, _ = oracle_sample(x, logits, T, E, k, H, I, n_tok, main_r["h_scale"], dev, cache)
        cpu = {"value": n_tok / dt, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"the first {n_tok} tokens of the batch (their {n_tok * k} expert rows), one pass, "
                         f"{dt:.1f} s of oracle work"}
    decode_line = None
    if dec is not None:
        dw = layer_workload_name(Td, E, k, H, I, args.zipf)
        decode_line = {
            "workload": dw, "value": dec["value"], "unit": "tokens/s", "ms_per_step": dec["ms_step"],
            "roofline": layer_roofline(dec, k, H, I, fp4, hbm_peak, peak_kind, dw),
            "stages_ms": {"route_permute": dec["stage_ms"][0], "quantize_x": dec["stage_ms"][1],
                          "gate_up_gemm": dec["stage_ms"][2], "down_gemm_finalize": dec["stage_ms"][3],
                          "source": f"eager stage calls, mean of {args.steps} steps"},
            "hbm_gbs_layer": dec["ab"]["layer"] / (dec["ms_step"] / 1e3) / 1e9,
            "clocks": dec["clocks"]}
    weight_bytes = main_r["weight_bytes"]
    line = {
        "metric": METRIC, "value": main_r["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1xe2m1->f32", "data": "synthetic",
        "config": {"workload": workload,
                   "tokens": T, "experts": E, "top_k": k, "hidden": H, "intermediate": I,
                   "l2": (f"weights ({weight_bytes / 1e9:.3f} GB) below 256 MB: L2 flushed (256 MB write) "
                          f"before each timed step" if main_r["flush"] else
                          f"weights ({weight_bytes / 1e9:.2f} GB) exceed L2 (129 MB); no flush"),
                   "parallelism": f"replicas{world}"},
        "roofline": roof,
        "fp4_mma_probe_tflops": fp4["peak_tflops"],
        "fp4_mma_probes": fp4,
        "stages_ms": {"route_permute": stage_ms[0], "quantize_x": stage_ms[1], "gate_up_gemm": stage_ms[2],
                      "down_gemm_finalize": stage_ms[3], "source": f"eager stage calls, mean of {args.steps} steps"},
        "graph_last_step_stages_ms": {"route_permute": gl[0], "quantize_x": gl[1], "gate_up_gemm": gl[2],
                                      "down_gemm_finalize": gl[3], "layer": gl[4]},
        "eager_ms_per_step": main_r["eager_ms"],
        "timing": "value: CUDA-graph replays of the whole layer (moe_forward_graph_launch, no stage-timing nodes) "
                  "back to back; roofline.launch_ms: the gate_up GEMM launch inside eager stage calls timed with "
                  "events on the launching stream",
        "gemm_tflops": {"gate_up": 2.0 * T * k * 2 * I * H / (stage_ms[2] / 1e3) / 1e12,
                        "down": 2.0 * T * k * H * I / (stage_ms[3] / 1e3) / 1e12,
                        "layer": flops_layer / (ms_step / 1e3) / 1e12},
        "hbm_gbs_layer": main_r["ab"]["layer"] / (ms_step / 1e3) / 1e9,
        "active_experts": main_r["ab"]["active_experts"],
        "e2e": main_r["e2e"],
        "decode_c4": decode_line,
        # per step: routing (1 or 3), amax + quantiser, gate_up GEMM, down GEMM, FP32 -> BF16; or the
        # single-launch layer for small shapes
        "gpu_launches": moe.forward_kernel_count(T, E, k, H, I) * args.steps,
        "clocks": main_r["clocks"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_gemm(args, rank, world, local_rank):
    """One grouped GEMM at the decode shape: 256 experts x exactly 32 rows, K=6144, N=2048, NONE."""
    import nvfp4_moe_grouped_gb300 as moe
    from nvfp4_moe_grouped_gb300 import inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    E, rows, N, K = 256, 32, 2048, 6144
    R = E * rows
    offs = torch.arange(0, R + 1, rows, dtype=torch.int32)
    pad = torch.arange(0, E + 1, dtype=torch.int64) * 128
    dst = (pad[:-1, None] + torch.arange(rows)[None, :]).reshape(-1).to(torch.int32)
    x = inputs.activations(R, K)
    codes, sf, s = moe.nvfp4_quantize(x.to(dev), None, dst_row=dst.to(dev), sf_layout=moe.SF_TILED,
                                      dst_rows_alloc=E * 128)
    wf = inputs.expert_weights(E, N, K, 100, device=dev)
    pw = moe.prepare_expert_weights(wf, gate_up=False)
    del wf
    torch.cuda.empty_cache()
    offs_d = offs.to(dev)
    out = torch.zeros(E * 128, N, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, offs_d, moe.EPI_NONE, out=out)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    if args.profile_steps:
        torch.cuda.cudart().cudaProfilerStart()
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStop()
        return
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        clk.start()
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        clk.stop()
    ms = a.elapsed_time(b) / args.steps
    w_bytes = E * N * (K // 2 + K // 16)
    alg = w_bytes + R * (K // 2 + K // 16) + R * N * 2
    flops = 2.0 * R * N * K
    hbm_peak, _, peak_kind = peaks()
    gbs = alg / (ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "grouped-GEMM TFLOPS & HBM GB/s vs roofline (NVFP4, NONE epilogue)", "value": gbs,
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e2m1xe2m1->f32",
            "data": "synthetic",
            "config": {"workload": "grouped_gemm_E256_rows32_K6144_N2048_none",
                       "l2": "weights (1.81 GB) exceed L2; no flush"},
            "tflops": flops / (ms / 1e3) / 1e12,
            "roofline": {"bound": "hbm", "kernel": "grouped_gemm NONE", "achieved": gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": gbs / hbm_peak, "peak_kind": peak_kind, "traffic": None,
                         "algorithmic_bytes_per_launch": alg, "launch_ms": ms},
            "gpu_launches": args.steps, "clocks": clk.summary()}), flush=True)


def cublaslt_reference(M, N, K, iters, peak_tflops):
    """The same dense FP4 GEMM through cuBLASLt's block-scaled e2m1 matmul (a library timing reference built
    beside the layer's library; operands hold a fixed pattern, only the time is used)."""
    import ctypes
    from nvfp4_moe_grouped_gb300 import build as nb
    if not os.path.exists(nb.REF_LIB):
        return {"status": "reference library not built"}
    lib = ctypes.CDLL(nb.REF_LIB)
    fn = lib.nvfp4_cublaslt_gemm_time
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_float), ctypes.c_char_p, ctypes.c_int]
    ms = ctypes.c_float(0.0)
    msg = ctypes.create_string_buffer(256)
    rc = fn(M, N, K, 3, iters, ctypes.byref(ms), msg, 256)
    if rc != 0:
        return {"status": msg.value.decode(errors="replace")}
    tf = 2.0 * M * N * K / (ms.value / 1e3) / 1e12
    return {"library": "cuBLASLt block-scaled e2m1 x e2m1 (VEC16_UE4M3 scales), FP32 accumulate, bf16 out",
            "ms": ms.value, "tflops": tf, "frac_of_fp4_peak": tf / peak_tflops, "status": "ok",
            "timing": f"{iters} back-to-back calls after 3 warm-up calls, CUDA events"}


def run_dense(args, rank, world, local_rank):
    """One dense NVFP4 GEMM, M = N = K = --dense-size (a 'very large matrices' measurement), BF16 out,
    against this GPU's measured dense FP4 MMA rate."""
    import nvfp4_moe_grouped_gb300 as moe
    from nvfp4_moe_grouped_gb300 import inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    M = N = K = args.dense_size
    alloc = (M + 127) // 128 * 128
    x = inputs.activations(M, K, seed=0, device=dev)
    codes, sf, s = moe.nvfp4_quantize(x, None, sf_layout=moe.SF_TILED, dst_rows_alloc=alloc)
    del x
    wf = inputs.expert_weights(1, N, K, 900, device=dev)
    pw = moe.prepare_expert_weights(wf, gate_up=False)
    del wf
    torch.cuda.empty_cache()
    out = torch.zeros(alloc, N, dtype=torch.bfloat16, device=dev)
    in_bytes = alloc * (K // 2 + K // 16) + N * (K // 2 + K // 16)
    l2_flush = in_bytes < (256 << 20)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if l2_flush else None
    stream = torch.cuda.current_stream()

    def step():
        moe.dense_gemm_nvfp4(codes, sf, s, pw, M, out=out)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    if args.profile_steps:
        torch.cuda.cudart().cudaProfilerStart()
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStop()
        return
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        clk.start()
        for a, b in evs:
            if flush is not None:
                flush.fill_(1)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        clk.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    flops = 2.0 * M * N * K
    tf = flops / (ms / 1e3) / 1e12
    fp4 = fp4_peaks(local_rank) if rank == 0 else None
    if rank == 0:
        peak_fp4 = fp4["peak_tflops"]
        del codes, sf, pw, out
        torch.cuda.empty_cache()
        ref = cublaslt_reference(M, N, K, max(3, args.steps), peak_fp4)
        print(json.dumps({
            "metric": "dense NVFP4 GEMM TFLOPS vs dense FP4 peak", "value": tf, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e2m1xe2m1->f32",
            "data": "synthetic",
            "config": {"workload": f"dense_gemm_M{M}_N{N}_K{K}_bf16out",
                       "l2": ("256 MB written between timed launches (inputs fit in L2)" if l2_flush
                              else f"inputs ({in_bytes / 2**20:.0f} MB) exceed L2; no flush")},
            "roofline": {"bound": "tensor", "kernel": "grouped_gemm NONE (one group)", "achieved": tf,
                         "peak": peak_fp4, "unit": "TFLOP/s", "frac": tf / peak_fp4,
                         "peak_kind": FP4_PEAK_KIND,
                         "traffic": None, "algorithmic_flops_per_launch": flops, "launch_ms": ms},
            "fp4_mma_probes": fp4, "cublaslt_reference": ref,
            "gpu_launches": args.steps, "clocks": clk.summary()}), flush=True)


def run_gated(args, rank, world, local_rank):
    """The layer with the router in front (moe_forward_gated), as one CUDA graph, beside the same layer fed
    precomputed logits."""
    import nvfp4_moe_grouped_gb300 as moe
    from nvfp4_moe_grouped_gb300 import inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    T, E, k, H, I = args.tokens, args.experts, args.top_k, args.hidden, args.intermediate
    x, logits, pw13, pw2 = make_layer(T, E, k, H, I, args.zipf, dev)
    xd, ld = x.to(dev), logits.to(dev)
    wg = inputs.router_gate(E, H, device=dev)
    fwd = moe.MoeForward(T, E, k, H, I, dev, gated=True)
    h_scale = calibrate_h_scale(moe.MoeForward(T, E, k, H, I, dev), xd, ld, pw13)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(1, args.warmup)):
        fwd.gated(xd, wg, pw13, pw2, h_scale, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd.gated(xd, wg, pw13, pw2, h_scale, out=out, stream=torch.cuda.current_stream())
    plain = fwd.graph(xd, ld, pw13, pw2, h_scale, out=torch.empty_like(out), stage_events=False)
    for _ in range(max(1, args.warmup)):
        g.replay()
        plain.launch()
    torch.cuda.synchronize()
    weight_bytes = E * (2 * I * H + H * I) * 9 // 16
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if weight_bytes < (256 << 20) else None

    def timed(launch):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            if flush is not None:
                flush.fill_(1)
            a.record(stream)
            launch()
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / args.steps

    with ClockSampler(local_rank) as clk:
        clk.start()
        ms = timed(g.replay)
        clk.stop()
    ms_plain = timed(plain.launch)
    ms = max_over_ranks(ms, dev)
    counts = np.diff(fwd.view("expert_offsets", torch.int32, (E + 1,)).cpu().numpy())
    ab = algorithmic_bytes(counts, T, E, k, H, I)
    layer_bytes = ab["layer"] - T * E * 4 + E * H * 2   # the gate matrix is read instead of the logits
    hbm_peak, _, peak_kind = peaks()
    gbs = layer_bytes / (ms / 1e3) / 1e9
    if T * k / max(1, ab["active_experts"]) > 48:
        # compute-bound regime (as for the layer workload): the whole graph's expert-GEMM FLOPs against the
        # measured dense FP4 MMA rate
        fp4_peak = fp4_peaks(local_rank)["peak_tflops"]
        flops = 2.0 * T * k * (2 * I * H + H * I)
        tf = flops / (ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": "whole layer with the router (one CUDA graph)", "achieved": tf,
                "peak": fp4_peak, "unit": "TFLOP/s", "frac": tf / fp4_peak,
                "peak_kind": FP4_PEAK_KIND, "traffic": None,
                "algorithmic_flops_per_launch": flops, "launch_ms": ms, "hbm_gbs": gbs}
    else:
        roof = {"bound": "hbm", "kernel": "whole layer with the router (one CUDA graph)", "achieved": gbs,
                "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak, "peak_kind": peak_kind,
                "traffic": None, "algorithmic_bytes_per_launch": layer_bytes, "launch_ms": ms}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": whole_job_rate(T, world, ms), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e2m1xe2m1->f32 (router bf16xbf16->f32)",
            "data": "synthetic",
            "config": {"workload": f"moe_layer_gated_T{T}_E{E}_k{k}_H{H}_I{I}" + (f"_zipf{args.zipf}" if args.zipf
                                                                                  else "_uniform"),
                       "l2": "weights exceed L2; no flush" if flush is None else "256 MB written between steps"},
            "roofline": roof,
            "same_layer_fed_logits_ms": ms_plain,
            # router (logits GEMM + top-k), scan, scatter, quantiser, gate_up, down, FP32->BF16 per step
            "gpu_launches": 7 * args.steps, "clocks": clk.summary()}), flush=True)


def run_router(args, rank, world, local_rank):
    """The router: logits GEMM x . w_gate^T (bf16, tcgen05) + top-k routing and permutation."""
    import nvfp4_moe_grouped_gb300 as moe
    from nvfp4_moe_grouped_gb300 import inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    T, E, k, H = args.tokens, args.experts, args.top_k, args.hidden
    x = inputs.activations(T, H, seed=0, device=dev)
    wg = inputs.router_gate(E, H, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # inputs fit in L2
    r, _ = moe.moe_router(x, wg, k, want_logits=False)
    ws = torch.empty(moe._lib.load().moe_router_workspace_size(T, E, H, k), dtype=torch.uint8, device=dev)
    for _ in range(max(1, args.warmup)):
        moe.moe_router(x, wg, k, want_logits=False, out=r, ws=ws)
    torch.cuda.synchronize()
    if args.profile_steps:
        torch.cuda.cudart().cudaProfilerStart()
        for _ in range(args.steps):
            moe.moe_router(x, wg, k, want_logits=False, out=r, ws=ws)
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStop()
        return
    # the call as one CUDA graph, so host-side marshalling between launches is not timed
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe.moe_router(x, wg, k, want_logits=False, out=r, ws=ws, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step():
        graph.replay()

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        clk.start()
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        clk.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    alg = T * H * 2 + E * H * 2 + 2 * T * E * 4 + T * k * (4 + 4 + 4 * 3) + (E + 1) * 4
    gbs = alg / (ms / 1e3) / 1e9
    hbm_peak, _, peak_kind = peaks()
    if rank == 0:
        print(json.dumps({
            "metric": "router (logits GEMM + top-k + permutation) tokens/s", "value": T / (ms / 1e3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16xbf16->f32",
            "data": "synthetic",
            "config": {"workload": f"router_T{T}_E{E}_k{k}_H{H}",
                       "l2": "256 MB written between timed calls (inputs fit in L2)"},
            "roofline": {"bound": "hbm", "kernel": "router (3 launches: logits GEMM + top-k, scan, scatter)", "achieved": gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": gbs / hbm_peak, "peak_kind": peak_kind, "traffic": None,
                         "algorithmic_bytes_per_launch": alg, "launch_ms": ms},
            "gpu_launches": 3 * args.steps, "clocks": clk.summary()}), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    try:
        if args.workload == "layer" and args.gated:
            run_gated(args, rank, world, local_rank)
        elif args.workload == "gemm":
            run_gemm(args, rank, world, local_rank)
        elif args.workload == "dense":
            run_dense(args, rank, world, local_rank)
        elif args.workload == "router":
            run_router(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the GB300 MoE expert layer (libmoe.so).

Workloads (all inputs seeded and synthetic, shapes of the pages' model:
H=2048, 256 routed experts, top-8, one shared expert, I=512, int4 g64):
  prefill32k   (default) a 32768-token prompt in 4096-token chunks through 40
               pre-norm MoE layers (the library's chunk loop,
               moe_prefill_stack), centred weight generator; tokens/s.  The
               default run adds, from the same process, the same prompt with
               the literal generator, decode40, layer4096 and layer2048
               ("extras" in the JSON line; --no-extras leaves them out).
  decode40     one token at a time through a stack of 40 MoE layers with
               RMSNorm + residual between layers; metric: HBM GB/s of the
               bytes a token must stream (router + 9 experts per layer).
  layer256     one layer, T=256
  layer512zipf one layer, T=512, Zipf(1.1)-skewed routing
  layer2048    one layer, T=2048
  layer4096    one layer, T=4096
The prefill workloads report tokens/s and R_gemm, the grouped gate/up and
down GEMMs' time against the slower of their FLOPs at the bf16 peak and their
packed bytes at the HBM bandwidth.

One JSON line is printed by rank 0.  ``--impl reference`` times the CPU
oracle (the only reference this project has) on a bounded sample of the
same workload.  Multi-GPU runs are independent replicas (one process per
GPU, no collective on the data path): value = units of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

H, E, K_TOP, I_DIM, G = 2048, 256, 8, 512, 64
EXPERT_BYTES = 3 * (H * I_DIM // 2) + 3 * 2 * 2 * (H * I_DIM // G)   # 1,769,472
GATEUP_BYTES = 2 * (H * I_DIM // 2) + 2 * 2 * 2 * (H * I_DIM // G)   # 1,179,648
ROUTER_BYTES = E * H * 4                                              # 2,097,152

# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu
# capture of the current kernels (profiles/*.md give the commands); None
# where no capture of that workload exists.  Update with every kernel change.
TRAFFIC = {
    # gate/up + down, one launch each (the roofline kernel pair of the prefill lines)
    "layer256": 475_237_376,      # profiles/grouped_experts_tc_layer256.md
    "layer4096": 784_453_120,     # profiles/grouped_experts_tc_layer4096.md
    "prefill32k": 784_453_120,    # every 4096-token chunk-layer is the layer4096 launch pair
    "decode40": 127_976_576,      # decode_layer_kernel, 7 layers; profiles/decode_layer_decode40.md
    "gdn2k": 36_231_706,          # gdn_scan_kernel, profiles/gdn_scan_gdn2k.md
    "attn32k": 67_307_776,        # attn_block_kernel, profiles/attn_block_attn128k.md
    "attn128k": 268_621_926,      # attn_block_kernel, profiles/attn_block_attn128k.md
}
METRIC = "MoE-layer prefill tokens/s & % of roofline (T=256–32K); T=1 HBM GB/s"

STACK = 7  # layers per launch of the stacked decode kernel

WORKLOADS = {
    "decode40": dict(T=1, layers=40, chunk=1, zipf=False, centred=False,
                     desc="T=1 decode through 40 MoE layers (H=2048, E=256, top-8 + 1 shared, I=512, int4 g64), "
                          "RMSNorm + residual between layers, 64 distinct tokens cycled"),
    "layer256": dict(T=256, layers=1, chunk=256, zipf=False, centred=False, desc="one MoE layer, T=256"),
    "layer512zipf": dict(T=512, layers=1, chunk=512, zipf=True, centred=False,
                         desc="one MoE layer, T=512, Zipf(1.1) expert-bias skew"),
    "layer2048": dict(T=2048, layers=1, chunk=2048, zipf=False, centred=False, desc="one MoE layer, T=2048"),
    "layer4096": dict(T=4096, layers=1, chunk=4096, zipf=False, centred=False, desc="one MoE layer, T=4096"),
    "prefill32k": dict(T=32768, layers=40, chunk=4096, zipf=False, centred=True,
                       desc="32768-token prompt, 8 chunks of 4096 through 40 MoE layers (centred weights), "
                            "one fixed workspace"),
    "gdn2k": dict(T=2048, layers=1, chunk=2048, zipf=False, centred=False, Hk=16, Hv=32, dk=128, dv=128,
                  desc="Gated DeltaNet scan of one 2048-token sequence from an empty state (16 key heads, "
                       "32 value heads, dk = dv = 128), 6 distinct input sets cycled"),
    "attn32k": dict(T=1, L=32768, layers=1, chunk=1, zipf=False, centred=False, Hq=16, Hkv=2, D=256, sets=4,
                    desc="decode attention, one query token over a 32768-position KV cache (16 query heads, "
                         "2 KV heads, head dim 256, bf16), 4 distinct caches cycled"),
    "attn128k": dict(T=1, L=131072, layers=1, chunk=1, zipf=False, centred=False, Hq=16, Hkv=2, D=256, sets=2,
                     desc="decode attention, one query token over a 131072-position KV cache (16 query heads, "
                          "2 KV heads, head dim 256, bf16), 2 distinct caches cycled"),
}
ATTN_METRIC = "decode attention GB/s of KV cache streamed (T=1, 16 query / 2 KV heads, D=256); % of HBM"
GDN_SETS = 6
GDN_METRIC = "Gated DeltaNet scan tokens/s (one sequence, T=2048, 32 value heads); % of FP32 FMA peak"
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # SMs x FP32 lanes x 2 flops (FMA) x max SM clock
DEFAULT_STEPS = {"decode40": 2000, "layer256": 200, "layer512zipf": 200, "layer2048": 100, "layer4096": 50,
                 "prefill32k": 8, "gdn2k": 1500, "attn32k": 40000, "attn128k": 16000}  # >= ~1 s timed: clock samples
DEFAULT_WARMUP = {"decode40": 50, "layer256": 10, "layer512zipf": 10, "layer2048": 5, "layer4096": 5,
                  "prefill32k": 3, "gdn2k": 3, "attn32k": 10, "attn128k": 5}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default="prefill32k", choices=sorted(WORKLOADS))
    ap.add_argument("--tile-rows", type=int, default=128, choices=[128, 64],
                    help="token rows per grouped-GEMM tile (64: MOE_FLAG_TILE_ROWS_64)")
    ap.add_argument("--generator", default=None, choices=["centred", "literal"],
                    help="weight generator of a prefill workload (default: the workload's own)")
    ap.add_argument("--no-extras", action="store_true",
                    help="prefill32k: leave out the literal-generator, decode and single-layer lines")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--experts", default="tc", choices=["tc", "simt"], help="grouped GEMM kernels")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (profiling aid; the reported workloads use the default)")
    a = ap.parse_args()
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.workload] if a.impl == "ours" else 5
    if a.warmup is None:
        a.warmup = DEFAULT_WARMUP[a.workload] if a.impl == "ours" else 1
    a.warmup = max(a.warmup, 3) if a.impl == "ours" else a.warmup
    return a


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0:  # sampling is running before the timed region starts
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def gpu_id(device):
    """nvidia-smi id of a torch device (its UUID when torch exposes it)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device.index or 0)


# ------------------------------------------------------------------ inputs

class WeightCache:
    """Packed weights of the stack's layers on the device, generated on the
    host once per (seed, layer, generator) and shared by the workloads of one
    run; each layer also gets the router's bf16 parts (moe_router_split) once."""

    def __init__(self, device):
        self.device = device
        self.layers = {}

    def get(self, seed, layer, centred):
        import torch
        import bit_grouped_expert_gb300 as moe
        import synthetic as syn
        key = (seed, layer, bool(centred))
        if key not in self.layers:
            W = syn.experts(seed, E + 1, H, I_DIM, layer=layer, centred=centred)
            W["router"] = syn.router(seed, E, H, layer=layer)
            out = {}
            for n, a in W.items():
                a = np.ascontiguousarray(a)
                if a.dtype == np.uint16:
                    a = a.view(np.int16)
                elif a.dtype == np.uint32:
                    a = a.view(np.int32)
                out[n] = torch.from_numpy(a).to(self.device)
            out["router_split"] = torch.empty(moe.moe_router_split_bytes(E, H), dtype=torch.uint8, device=self.device)
            moe.moe_router_split(out["router"], E, H, out["router_split"])
            self.layers[key] = out
        return self.layers[key]


def as_dev(a, device):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


# ------------------------------------------------------------------ our arm

def gemm_flops(rows):
    """Expert FLOPs of the grouped gate/up and down GEMMs for `rows` token
    rows (pairs + shared rows): 2 matrices x 2 flops x H x I, and 2 x H x I."""
    return 4 * rows * H * I_DIM, 2 * rows * H * I_DIM


def run_ours(args, wl, rank, world, device, cache=None, steps=None, warmup=None, e2e_on=True, name=None):
    import torch
    import bit_grouped_expert_gb300 as moe
    import synthetic as syn

    torch.cuda.set_device(device)
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    name = args.workload if name is None else name
    cache = cache or WeightCache(device)
    T, L, chunk = wl["T"], wl["layers"], wl["chunk"]
    flags = moe.MOE_FLAG_SIMT_EXPERTS if args.experts == "simt" else 0
    if args.tile_rows == 64:
        flags |= moe.MOE_FLAG_TILE_ROWS_64
    if L > 1:
        flags |= moe.MOE_FLAG_PRENORM  # stacks: out = r + MoE(RMSNorm(r)), in place
    plan = moe.moe_plan(moe.make_config(H, E, K_TOP, I_DIM, 1, G), chunk, flags)
    ws = torch.zeros(moe.moe_workspace_bytes(plan), dtype=torch.uint8, device=device)
    moe.moe_workspace_init(plan, ws)
    seed = args.seed + 1000 * rank
    weights = [cache.get(seed, l, wl["centred"]) for l in range(L)]
    cws = [moe.make_weights(w) for w in weights]
    bias = as_dev(syn.zipf_bias(seed, E), device) if wl["zipf"] else None

    n_in = 64 if T == 1 else 1
    x_host = syn.activations(seed, max(T, n_in), H)
    if T == 1:
        tokens = as_dev(x_host[:n_in], device).reshape(n_in, 1, H)
        x_in = torch.empty((1, H), dtype=torch.int16, device=device)
    else:
        x_in = as_dev(x_host, device)
    r = torch.empty((T if T > 1 else 1, H), dtype=torch.int16, device=device)
    out = torch.empty((T, H), dtype=torch.int16, device=device)

    stream = torch.cuda.Stream(device=device)
    launches = [0]

    # Timed kernels.  Decode: the decode kernel, which runs up to STACK layers
    # per cooperative launch (the 2nd and 4th launches of a step are
    # bracketed).  Prefill: the grouped gate/up and down GEMMs, N_EV launches
    # of each per step (the stacks: spread over the chunks and layers).
    N_EV = 4
    if T == 1 and L > 1:
        groups = [(l0, min(L, l0 + STACK)) for l0 in range(0, L, STACK)]
        prof_groups = [j for j in (1, 3) if j < len(groups) and groups[j][1] - groups[j][0] == STACK] or [0]
        layers_per_launch = groups[prof_groups[0]][1] - groups[prof_groups[0]][0]
        kerns = [moe.MOE_KERNEL_DECODE_LAYER]
        n_ev = len(prof_groups)
    else:
        layers_per_launch = 1
        kerns = [moe.MOE_KERNEL_GATEUP, moe.MOE_KERNEL_DOWN]
        n_ev = N_EV if L > 1 else 1  # a single layer launches each kernel once per step
    ev = {kn: ([torch.cuda.Event(enable_timing=True) for _ in range(n_ev)],
               [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]) for kn in kerns}
    profiling = [False]

    def stack(j):
        on = profiling[0] and j in prof_groups
        kn = kerns[0]
        if on:
            i = prof_groups.index(j)
            moe.moe_profile_events(kn, ev[kn][0][i:i + 1], ev[kn][1][i:i + 1])
        l0, l1 = groups[j]
        moe.moe_decode_stack(plan, r, cws[l0:l1], None, ws, stream=stream)
        launches[0] += moe.moe_last_launch_count()
        if on:
            moe.moe_profile_events(kn)

    def body(xb=x_in, ob=out):
        launches[0] = 0
        if T == 1 and L > 1:
            # the residual stream through the whole stack, one call per group
            r.copy_(xb)
            for j in range(len(groups)):
                stack(j)
            ob.copy_(r)
            return
        if profiling[0]:
            for kn in kerns:
                moe.moe_profile_events(kn, ev[kn][0], ev[kn][1])
                if L > 1:  # 4 of the step's chunk-layers: (0, 0), (2, 1), (4, 2), (6, 3)
                    moe.moe_profile_stride(kn, (T // chunk) * L // n_ev + 1)
        if L == 1:
            moe.moe_forward(plan, xb, None, T, cws[0], bias, ob, ws, stream=stream)
            launches[0] += moe.moe_last_launch_count()
        else:  # the library's chunk loop over the whole prompt
            r.copy_(xb)
            moe.moe_prefill_stack(plan, r, T, cws, None, ws, stream=stream)
            launches[0] += moe.moe_last_launch_count()
            ob.copy_(r)
        if profiling[0]:
            for kn in kerns:
                moe.moe_profile_events(kn)

    # warm the path once eagerly, then capture one step into a CUDA graph
    with torch.cuda.stream(stream):
        if T == 1:
            x_in.copy_(tokens[0])
        body()
    torch.cuda.synchronize()
    for a, b in ev.values():  # create the CUDA events now, outside the capture
        for e in a + b:
            e.record(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    profiling[0] = True
    with torch.cuda.graph(graph, stream=stream):
        body()
    profiling[0] = False
    per_step_launches = launches[0]
    # a second copy of the step on its own input and output buffers, for the
    # double-buffered end-to-end loop
    x_in2, out2 = torch.empty_like(x_in), torch.empty_like(out)
    graph2 = None
    if e2e_on:
        graph2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph2, stream=stream):
            body(x_in2, out2)

    def step(i):
        if T == 1:
            x_in.copy_(tokens[i % n_in])
        graph.replay()

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id(device)) as clk:
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(steps):
                step(i)
            t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    kern_ms, dom_err = {}, None
    try:
        for kn, (a, b) in ev.items():
            kern_ms[kn] = sum(x.elapsed_time(y) for x, y in zip(a, b)) / len(a)
    except Exception as ex:  # noqa: BLE001 - reported in the JSON line
        kern_ms, dom_err = {}, f"{type(ex).__name__}: {ex}"[:300]
    if world > 1:
        ms = max_over_ranks(ms, device)

    # bytes / flops of the workload
    st = moe.moe_device_status(plan, ws)
    touched = E + 1
    if T > 1:
        v = moe.moe_route_view(plan, ws, min(T, chunk))
        counts = moe.workspace_tensor(ws, v.counts_d, E, torch.int32).cpu().numpy()
        touched = int((counts > 0).sum()) + 1  # of the last chunk the step routed
    result = {}
    pk = peaks()
    if T == 1:
        bytes_tok = L * (ROUTER_BYTES + 9 * EXPERT_BYTES + 3 * H * 2)
        gbs = bytes_tok * steps / (ms * 1e-3) / 1e9 * world
        result.update(value=gbs, unit="GB/s", higher_is_better=True)
        dk = kerns[0]
        if dk in kern_ms:
            dom_bytes = layers_per_launch * (ROUTER_BYTES + 9 * EXPERT_BYTES + 3 * H * 2)
            achieved = dom_bytes / (kern_ms[dk] * 1e-3) / 1e9
            roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": TRAFFIC.get(name),
                        "kernel": (f"decode kernel, {layers_per_launch} layers per launch (RMSNorm+router+top-k+9 "
                                   "experts+combine each)"),
                        "kernel_ms": round(kern_ms[dk], 5), "peak_src": pk["src"]}
        else:
            roofline = {"error": dom_err}
    else:
        tps = T * steps / (ms * 1e-3) * world
        result.update(value=tps, unit="tokens/s", higher_is_better=True)
        rows = (K_TOP + 1) * chunk
        f_gu, f_dn = gemm_flops(rows)
        b_gu = touched * GATEUP_BYTES + chunk * H * 2
        b_dn = touched * (EXPERT_BYTES - GATEUP_BYTES)
        if moe.MOE_KERNEL_GATEUP in kern_ms and moe.MOE_KERNEL_DOWN in kern_ms:
            t_gu, t_dn = kern_ms[moe.MOE_KERNEL_GATEUP] * 1e-3, kern_ms[moe.MOE_KERNEL_DOWN] * 1e-3
            tflops = pk["bf16_tflops_sustained"] if L > 1 else pk["bf16_tflops"]
            # R_gemm: the two grouped GEMMs against the slower of their FLOPs at
            # the bf16 peak and their packed bytes at the HBM bandwidth
            t_flops = (f_gu + f_dn) / (tflops * 1e12)
            t_bytes = (b_gu + b_dn) / (pk["hbm_gbs"] * 1e9)
            if t_flops >= t_bytes:
                achieved, peak, unit, bound = (f_gu + f_dn) / (t_gu + t_dn) / 1e12, tflops, "TFLOP/s", "tensor"
            else:
                achieved, peak, unit, bound = (b_gu + b_dn) / (t_gu + t_dn) / 1e9, pk["hbm_gbs"], "GB/s", "hbm"
            roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                        "frac": round(achieved / peak, 4), "traffic": TRAFFIC.get(name),
                        "kernel": "grouped gate/up + SwiGLU and grouped down (tcgen05), per chunk-layer",
                        "kernel_ms": round((t_gu + t_dn) * 1e3, 5),
                        "gateup_ms": round(t_gu * 1e3, 5), "down_ms": round(t_dn * 1e3, 5),
                        "gateup_frac": round(max(f_gu / (tflops * 1e12), b_gu / (pk["hbm_gbs"] * 1e9)) / t_gu, 4),
                        "down_frac": round(max(f_dn / (tflops * 1e12), b_dn / (pk["hbm_gbs"] * 1e9)) / t_dn, 4),
                        "peak_src": pk["src"],
                        "peak_kind": "sustained (kernel timed inside a long step)" if L > 1 else "burst"}
        else:
            roofline = {"error": dom_err}

    result.update(ms_per_step=ms / steps, roofline=roofline, clocks=clk.summary(),
                  gpu_launches=per_step_launches * steps, device_status=st,
                  touched_experts=touched if T > 1 else None)
    if not e2e_on:
        return result

    # end to end: every step copies its input from pinned host memory to the
    # device, runs, and copies its output back to pinned host memory.  Two
    # buffer sets alternate, so step i's copies (on their own streams) overlap
    # the neighbouring steps' compute; the clock stops when the last output
    # has reached the host.
    in_rows = 1 if T == 1 else T
    host_in = torch.from_numpy(np.ascontiguousarray(x_host[:in_rows]).view(np.int16)).pin_memory()
    host_out = [torch.empty((T, H), dtype=torch.int16).pin_memory() for _ in range(2)]
    xs, outs, graphs = (x_in, x_in2), (out, out2), (graph, graph2)
    h2d, d2h = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = min(steps, 200 if T == 1 else max(3, steps))
    torch.cuda.synchronize()
    t_e = time.perf_counter()
    for i in range(e2e_steps):
        b = i & 1
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(done[b])  # step i-2 has consumed this input buffer
            xs[b][:in_rows].copy_(host_in, non_blocking=True)
            in_ready[b].record(h2d)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_read[b])  # step i-2's output has been copied out
        with torch.cuda.stream(stream):
            graphs[b].replay()
            done[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(done[b])
            host_out[b].copy_(outs[b], non_blocking=True)
            out_read[b].record(d2h)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t_e
    if T == 1:
        e2e_val = bytes_tok * e2e_steps / e2e_s / 1e9 * world
    else:
        e2e_val = T * e2e_steps / e2e_s * world
    result["e2e"] = {"value": e2e_val, "unit": result["unit"], "h2d_bytes_per_step": in_rows * H * 2,
                     "d2h_bytes_per_step": T * H * 2}
    result["dtype"] = "int4-g64 weights, bf16 activations, fp32 accumulate"
    return result


def run_default_extras(args, rank, world, device, cache):
    """The other halves of the metric, measured in the same process after the
    headline prefill line: the 32K prompt with the literal weight generator,
    T=1 decode through 40 layers, and one layer at T=4096 and T=2048."""
    out = {}
    for name, gen, steps, warmup in (("prefill32k_literal", False, 3, 3), ("decode40", None, 2000, 50),
                                     ("layer4096", None, 50, 5), ("layer2048", None, 100, 5)):
        wl = dict(WORKLOADS[name.split("_")[0]])
        if gen is not None:
            wl["centred"] = gen
        res = run_ours(args, wl, rank, world, device, cache=cache, steps=steps, warmup=warmup, e2e_on=False,
                       name=name)
        keep = {k: res[k] for k in ("value", "unit", "ms_per_step", "roofline", "clocks", "touched_experts",
                                    "device_status") if k in res}
        keep["workload"] = (wl["desc"] + (" [literal weight generator]" if gen is False else ""))
        keep["steps"], keep["warmup"] = steps, warmup
        out[name] = keep
        torch_sync()
    return out


def torch_sync():
    import torch
    torch.cuda.synchronize()


def run_gdn(args, wl, rank, world, device):
    """The Gated DeltaNet scan: each step scans one 2048-token sequence from
    an empty state (state reset + scan, one captured graph per input set)."""
    import torch
    import __graft_entry__
    import bit_grouped_expert_gb300 as moe
    import synthetic as syn

    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.set_device(device)
    T, Hk, Hv, dk, dv = wl["T"], wl["Hk"], wl["Hv"], wl["dk"], wl["dv"]
    seed = args.seed + 1000 * rank
    host = [syn.gdn_inputs(seed + i, T, Hk, Hv, dk, dv) for i in range(GDN_SETS)]
    sets = [{n: as_dev(a, device) for n, a in h.items()} for h in host]
    outs = [torch.empty((T, Hv, dv), dtype=torch.int16, device=device) for _ in range(GDN_SETS)]
    stream = torch.cuda.Stream(device=device)
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def body(i, prof=None):
        d = sets[i]
        d["state"].zero_()
        if prof is not None:
            moe.moe_profile_events(moe.MOE_KERNEL_GDN_SCAN, ev_a[prof:prof + 1], ev_b[prof:prof + 1])
        moe.gdn_scan(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["state"], outs[i], T, Hk, Hv, dk, dv,
                     stream=stream)
        if prof is not None:
            moe.moe_profile_events(moe.MOE_KERNEL_GDN_SCAN)

    with torch.cuda.stream(stream):
        body(0)
    torch.cuda.synchronize()
    for e in ev_a + ev_b:
        e.record(stream)
    torch.cuda.synchronize()
    graphs = []
    for i in range(GDN_SETS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body(i, prof=(i - 1) // 2 if i in (1, 3) else None)  # sets 1 and 3 time the scan kernel
        graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % GDN_SETS].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id(device)) as clk:
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(args.steps):
                graphs[i % GDN_SETS].replay()
            t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    if world > 1:  # the slowest rank's time
        ms = max_over_ranks(ms, device)
    dom_ms = sum(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)) / 2
    tps = T * args.steps / (ms * 1e-3) * world
    flops = 7.0 * Hv * dk * dv * T  # per sequence: u (2), state update (3), output (2) per state element per token
    achieved = flops / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "alu", "achieved": round(achieved, 3), "peak": round(FP32_PEAK_TFLOPS, 1),
                "unit": "TFLOP/s", "frac": round(achieved / FP32_PEAK_TFLOPS, 4),
                "traffic": TRAFFIC.get(args.workload), "kernel": "gdn_scan_kernel (state in registers)",
                "kernel_ms": round(dom_ms, 5),
                "peak_src": "derived: 152 SMs x 128 FP32 lanes x 2 flops x 2070 MHz"}
    # end to end: each step copies its inputs from pinned host memory, scans,
    # and copies the outputs back.  Two buffer sets alternate, so a step's
    # copies (on their own streams) overlap the neighbouring steps' scans.
    pinned = [{n: torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if a.dtype == np.uint16 else a.dtype))
               .pin_memory() for n, a in h.items() if n != "state"} for h in host[:2]]
    host_o = [torch.empty((T, Hv, dv), dtype=torch.int16).pin_memory() for _ in range(2)]
    h2d = sum(a.numel() * a.element_size() for a in pinned[0].values())
    s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = min(args.steps, 50)
    torch.cuda.synchronize()
    te = time.perf_counter()
    for i in range(e2e_steps):
        b = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(done[b])  # step i-2's scan has read this input set
            for n, a in pinned[b].items():
                sets[b][n].copy_(a, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_read[b])  # step i-2's output has been copied out
        with torch.cuda.stream(stream):
            graphs[b].replay()
            done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            host_o[b].copy_(outs[b], non_blocking=True)
            out_read[b].record(s_out)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - te
    e2e = {"value": T * e2e_steps / e2e_s * world, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": T * Hv * dv * 2}
    return {"metric": GDN_METRIC, "value": tps, "unit": "tokens/s", "higher_is_better": True,
            "ms_per_step": ms / args.steps, "roofline": roofline, "e2e": e2e, "clocks": clk.summary(),
            "gpu_launches": args.steps, "dtype": "bf16 q/k/v/o, fp32 alpha/beta/state and sums",
            "config_extra": {"l2": f"{GDN_SETS} distinct input sets of {h2d / 1e6:.0f} MB cycled (larger than L2 "
                                   "together)", "experts": None}}


def run_attn(args, wl, rank, world, device):
    """Decode attention: each step is one query token against a KV cache of
    wl["L"] positions (the caches cycle so that each step reads its cache from
    HBM)."""
    import torch
    import __graft_entry__
    import bit_grouped_expert_gb300 as moe
    import synthetic as syn

    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.set_device(device)
    L, Hq, Hkv, D, n_sets = wl["L"], wl["Hq"], wl["Hkv"], wl["D"], wl["sets"]
    seed = args.seed + 1000 * rank
    host = [syn.attn_inputs(seed + i, L, Hq, Hkv, D) for i in range(n_sets)]
    sets = [{n: as_dev(a, device) for n, a in h.items()} for h in host]
    ws = torch.zeros(moe.attn_decode_workspace_bytes(L, Hq, D), dtype=torch.uint8, device=device)
    outs = [torch.empty((Hq, D), dtype=torch.int16, device=device) for _ in range(n_sets)]
    stream = torch.cuda.Stream(device=device)
    # the block pass is timed in one or two of the caches' graphs, so that most
    # steps run without event nodes between the pass and its combine kernel
    prof_sets = [1] if n_sets == 2 else [1, 2]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in prof_sets]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in prof_sets]

    def body(i, prof=None):
        d = sets[i]
        if prof is not None:
            moe.moe_profile_events(moe.MOE_KERNEL_ATTN_DECODE, ev_a[prof:prof + 1], ev_b[prof:prof + 1])
        moe.attn_decode(d["q"], d["k"], d["v"], L, Hq, Hkv, D, ws, outs[i], stream=stream)
        if prof is not None:
            moe.moe_profile_events(moe.MOE_KERNEL_ATTN_DECODE)

    with torch.cuda.stream(stream):
        body(0)
    torch.cuda.synchronize()
    for e in ev_a + ev_b:
        e.record(stream)
    torch.cuda.synchronize()
    graphs = []
    for i in range(n_sets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body(i, prof=prof_sets.index(i) if i in prof_sets else None)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % n_sets].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id(device)) as clk:
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(args.steps):
                graphs[i % n_sets].replay()
            t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    if world > 1:  # the slowest rank's time
        ms = max_over_ranks(ms, device)
    dom_ms = sum(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)) / len(prof_sets)
    kv_bytes = 2 * L * Hkv * D * 2
    gbs = kv_bytes * args.steps / (ms * 1e-3) / 1e9 * world
    pk = peaks()
    achieved = kv_bytes / (dom_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": TRAFFIC.get(args.workload),
                "kernel": "attn_block_kernel (one block of positions per SM, 8 query heads per KV row read)",
                "kernel_ms": round(dom_ms, 5), "peak_src": pk["src"]}
    # end to end: every step copies the query in from pinned host memory and
    # the output back, both captured with the attention call into one graph
    # per buffer set (the copies are 8 KB; a step is tens of microseconds, so
    # per-step stream bookkeeping on the host would cost more than the step)
    host_q = torch.from_numpy(np.ascontiguousarray(host[0]["q"]).view(np.int16)).pin_memory()
    host_o = [torch.empty((Hq, D), dtype=torch.int16).pin_memory() for _ in range(2)]
    e2e_graphs = []
    for b in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            sets[b]["q"].copy_(host_q, non_blocking=True)
            body(b)
            host_o[b].copy_(outs[b], non_blocking=True)
        e2e_graphs.append(g)
    e2e_steps = min(args.steps, 2000)
    torch.cuda.synchronize()
    te = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            e2e_graphs[i & 1].replay()
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - te
    e2e = {"value": kv_bytes * e2e_steps / e2e_s / 1e9 * world, "unit": "GB/s", "h2d_bytes_per_step": Hq * D * 2,
           "d2h_bytes_per_step": Hq * D * 2}
    return {"metric": ATTN_METRIC, "value": gbs, "unit": "GB/s", "higher_is_better": True,
            "ms_per_step": ms / args.steps, "roofline": roofline, "e2e": e2e, "clocks": clk.summary(),
            "gpu_launches": 2 * args.steps, "dtype": "bf16 q/K/V/o, fp32 scores and sums, bf16 weights for P.V",
            "config_extra": {"l2": f"{n_sets} distinct caches of {kv_bytes / 1e6:.0f} MB cycled (larger than L2 "
                                   "together)", "experts": None, "kv_positions": L}}


def attn_oracle_sample(wl, seed, target_s=None):
    """The oracle on a prefix of the cache: as many positions as take about
    target_s seconds (all of them at most); GB/s of K and V read."""
    from oracle.attn import decode_attention
    import synthetic as syn
    L, Hq, Hkv, D = wl["L"], wl["Hq"], wl["Hkv"], wl["D"]
    n = min(L, 4096)
    while True:
        d = syn.attn_inputs(seed, n, Hq, Hkv, D)
        t = time.perf_counter()
        decode_attention(d["q"], d["k"], d["v"])
        dt = time.perf_counter() - t
        if target_s is None or dt >= 0.5 * target_s or n >= L:
            break
        n = min(L, max(2 * n, int(n * target_s / max(dt, 1e-3))))
    return dt, 2 * n * Hkv * D * 2 / 1e9, "GB/s", f"one query over the first {n} cache positions (GB of K and V read)"


def gdn_oracle_sample(wl, seed, target_s=None):
    """The oracle scan over the first tokens of one sequence (all heads):
    64 tokens, or as many as take about target_s seconds."""
    from oracle.gdn import gdn_scan as oracle_scan
    import synthetic as syn
    T = wl["T"]
    d = syn.gdn_inputs(seed, T, wl["Hk"], wl["Hv"], wl["dk"], wl["dv"])
    n = 64
    while True:
        t = time.perf_counter()
        oracle_scan(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["state"], t_end=n)
        dt = time.perf_counter() - t
        if target_s is None or dt >= 0.5 * target_s or n >= T:
            break
        n = min(T, max(2 * n, int(n * target_s / max(dt, 1e-3))))
    return dt, float(n), "tokens/s", f"the first {n} tokens of one sequence through the scan (all 32 heads)"


# ------------------------------------------------------------------ oracle (CPU)

def oracle_sample(wl, seed, target_s=None):
    """Run the CPU oracle on a bounded sample of the workload: one token (T=1)
    or 64 tokens (32 for stacks) through one layer, or, with target_s, as many
    tokens as take about target_s seconds (at most 256 single tokens, or the
    workload's T).  Returns (seconds, units, unit, description)."""
    import oracle as orc
    import synthetic as syn
    T = wl["T"]
    d = orc.Dims()
    W = syn.experts(seed, E + 1, H, I_DIM, layer=0, centred=wl["centred"])
    W["router"] = syn.router(seed, E, H, layer=0)
    if T == 1:
        xs = syn.activations(seed, 256, H)
        n, dt = 0, 0.0
        while n < 256:
            t = time.perf_counter()
            orc.moe_layer(d, xs[n:n + 1], W)
            dt += time.perf_counter() - t
            n += 1
            if target_s is None or dt >= target_s:
                break
        units = n * (ROUTER_BYTES + 9 * EXPERT_BYTES + 3 * H * 2) / 1e9
        return dt, units, "GB/s", (f"{n} token(s) one at a time through 1 layer "
                                   "(GB of router + 9 experts streamed per second)")
    bias = syn.zipf_bias(seed, E) if wl["zipf"] else None
    n_tok = 32 if wl["layers"] > 1 else 64
    while True:
        x = syn.activations(seed, n_tok, H)
        t = time.perf_counter()
        orc.moe_layer(d, x, W, bias=bias)
        dt = time.perf_counter() - t
        if target_s is None or dt >= 0.5 * target_s or n_tok >= T:
            break
        n_tok = min(T, max(2 * n_tok, int(n_tok * target_s / max(dt, 1e-3))))
    # tokens/s of the workload: one layer of the sample, scaled to all layers
    units = n_tok / wl["layers"]
    desc = f"{n_tok} tokens through one layer" if wl["layers"] == 1 else \
        f"{n_tok} tokens through 1 of {wl['layers']} layers, extrapolated to the {wl['layers']}-layer stack"
    return dt, units, "tokens/s", desc


def cpu_baseline(wl, seed):
    import oracle as orc
    orc.build()
    sample = gdn_oracle_sample if "Hv" in wl else attn_oracle_sample if "Hkv" in wl else oracle_sample
    dt, units, unit, desc = sample(wl, seed, target_s=10.0)
    # the scan and attention oracles are numpy (the attention's matrix products may use BLAS threads)
    cores = 1 if "Hv" in wl else (os.cpu_count() or 1) if "Hkv" in wl else orc.num_threads()
    return {"value": units / dt, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc,
            "seconds": round(dt, 3)}


def run_reference(args, wl):
    import oracle as orc
    import synthetic as syn
    orc.build()
    syn.build()
    sample = gdn_oracle_sample if "Hv" in wl else attn_oracle_sample if "Hkv" in wl else oracle_sample
    for i in range(args.warmup):
        sample(wl, args.seed + i)
    steps = args.steps
    tot, units, unit, desc = 0.0, 0.0, None, None
    for i in range(steps):
        dt, u, unit, desc = sample(wl, args.seed + 100 + i)
        tot += dt
        units += u
    val = units / tot
    return {"value": val, "unit": unit, "higher_is_better": True, "ms_per_step": tot / steps * 1e3,
            "cpu_baseline": {"value": val, "unit": unit,
                             "cores": 1 if "Hv" in wl else (os.cpu_count() or 1) if "Hkv" in wl else orc.num_threads(),
                             "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "dtype": "fp64 oracle (bf16 rounding points of the layer)"}


# ------------------------------------------------------------------ main

def main():
    args = parse()
    wl = dict(WORKLOADS[args.workload])
    if args.layers is not None:
        wl["layers"] = args.layers
        wl["desc"] += f" [profiling override: {args.layers} layers]"
    if args.generator is not None:
        wl["centred"] = args.generator == "centred"
        wl["desc"] += f" [{args.generator} weight generator]"
    if args.tile_rows != 128:
        wl["desc"] += f" [{args.tile_rows}-row tiles]"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    base = {"metric": GDN_METRIC if "Hv" in wl else ATTN_METRIC if "Hkv" in wl else METRIC, "n_gpus": args.gpus if world == 1 else world, "steps": args.steps,
            "warmup": args.warmup, "scaling": "weak", "vs_baseline": None, "data": "synthetic",
            "config": {"workload": f"{args.workload}: {wl['desc']}", "tokens_per_step": wl["T"],
                       "layers": wl["layers"], "chunk": wl["chunk"], "tile_rows": args.tile_rows,
                       "generator": ("centred" if wl.get("centred") else "literal") if "Hv" not in wl and "Hkv" not in wl
                       else None,
                       "parallelism": "replicas" if world > 1 else "1 GPU",
                       "l2": (f"{GDN_SETS} distinct input sets cycled (~50 MB each, larger than L2 together)"
                              if "Hv" in wl else f"{wl.get('sets')} distinct KV caches cycled" if "Hkv" in wl
                              else "inputs larger than L2 (packed weights >= 455 MB per layer)"),
                       "experts": args.experts}}
    if args.impl == "reference":
        if rank != 0:
            return
        res = run_reference(args, wl)
        line = {**base, **res, "impl": "reference"}
        print(json.dumps(line))
        return
    import torch
    device = torch.device("cuda", local)
    if world > 1:
        torch.cuda.set_device(device)
        torch.distributed.init_process_group("nccl")
    if "Hv" in wl or "Hkv" in wl:
        res = (run_gdn if "Hv" in wl else run_attn)(args, wl, rank, world, device)
        extras = None
    else:
        import __graft_entry__
        if rank == 0:
            __graft_entry__.build()
        if world > 1:
            torch.distributed.barrier()
        cache = WeightCache(device)
        res = run_ours(args, wl, rank, world, device, cache=cache)
        extras = None
        if args.workload == "prefill32k" and not args.no_extras and args.layers is None and args.generator is None:
            extras = run_default_extras(args, rank, world, device, cache)
        del cache
    if rank == 0:
        extra = res.pop("config_extra", {})
        line = {**base, **res}
        line["config"] = {**line["config"], **extra}
        if extras:
            line["extras"] = extras
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(wl, args.seed)
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

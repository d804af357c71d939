"""Benchmark of the fused GEMM + on-chip epilogue path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama|rmsproj|lnproj|swiglu|fp8swiglu|dgrad|wgrad|skinny]
                    [--impl coda|reference] [--profile-steps]

Default workload: the LLaMA-7B-like non-attention block at 16384 tokens (d 4096,
ffn 11008): commuted RMSNorm -> QKV projection, out-projection + residual,
commuted RMSNorm -> SwiGLU up-projection, down-projection + residual; four fused
GEMM+epilogue calls, bf16 in, fp32 accumulate, 6.63 TFLOP per step.  The other
workloads are the single calls of the same family (the commuted-RMSNorm
projection, the SwiGLU up-projection with dropout, the dgrad, ...).
One step = one pass of the fused path over the synthetic batch.  Prints one
JSON line (rank 0): fused TFLOP/s, the roofline of the fused GEMM kernel, the
same chain run unfused through the library's own kernels, DRAM bytes fused vs
unfused, an end-to-end figure through host buffers, clocks, and the fp64
oracle timed on the host cores as the CPU baseline.

--profile-steps runs, after the warm-up, one fused step and then one unfused
step, each between full L2 flushes and each followed by a read-only pass over
a 256 MiB buffer, and exits: under ncu (one metric group, --cache-control none)
every kernel of a step is captured in order, and the read-only pass after it
writes back exactly the step's outputs still dirty in L2, so the step's DRAM
bytes are its kernels' reads and writes plus that pass's writes.

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the
launching stream, with a 256 MiB device write and a 256 MiB read between steps
so every step reads its operands from HBM and starts with no dirty L2 lines.
Under torchrun each rank runs an independent replica (the path has no
cross-GPU exchange); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_NCORES = len(os.sched_getaffinity(0))
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_NCORES))

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "fused GEMM+epilogue TFLOP/s and % of GB300 bf16 roofline; DRAM bytes vs unfused"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20

DESCRIPTIONS = {
    "rmsproj": "commuted RMSNorm projection D = rsqrt(mean(X^2)+1e-6)*(X@(gamma*W)), X[4096,2048], W[2048,8192]",
    "lnproj": "commuted LayerNorm projection D = r*(X@(gamma*W) - mu*colsum(gamma*W)) + beta@W, X[4096,2048], "
              "W[2048,8192]",
    "swiglu": "SwiGLU up-projection [G|U] = X[8192,4096] @ W[4096,22016], SiLU(G)*U, dropout p=0.1",
    "dgrad": "dgrad dX = (dY[8192,4096] @ W[16384,4096]^T) * GELU'(Z), rows sum(dX*Xhat), sum(dX)",
    "skinny": "decode-sized MLP up-projection: rmsnorm(X[128,4096]) @ W[4096,22016] (commuted), SiLU(G)*U; X "
              "arrives with its row sums of squares (the out-projection's residual epilogue emits them)",
    "wgrad": "weight gradient dW[11008,4096] = up[16384,11008]^T @ dY[16384,4096] / 8 + dW (in place), "
             "row sums of squares",
    "fp8swiglu": "SwiGLU up-projection in FP8 E4M3: X[8192,4096] quantised per row each step, W[22016,4096] "
                 "per channel once, dequantised in the epilogue, SiLU(G)*U",
    "mxfp8swiglu": "SwiGLU up-projection in MXFP8 (E4M3 codes, an E8M0 scale per 32 elements of K applied by the "
                   "tensor cores): X[8192,4096] quantised each step, W[22016,4096] once, SiLU(G)*U",
    "llama": "LLaMA-7B-like non-attention block, 16384 tokens, d=4096, ffn=11008 (4 fused GEMMs): commuted "
             "RMSNorm->QKV, out-proj+residual, commuted RMSNorm->SwiGLU up-proj, down-proj+residual; one layer of "
             "a stack: the norms' row sums of squares come from the preceding residual epilogues (the input's "
             "with the input, the next layer's emitted by the down-projection)",
}
DEFAULT_STEPS = {"rmsproj": 3000, "lnproj": 3000, "swiglu": 300, "dgrad": 300, "llama": 60, "skinny": 3000, "wgrad": 300, "fp8swiglu": 300,
                 "mxfp8swiglu": 300}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str):
    """DRAM bytes of the fused and unfused steps and of the dominant kernel from
    the committed ncu summary, or None when the kernel sources changed since
    that capture."""
    from gemm_epilogue_transformer_tmem_gb300.traffic import kernel_hash
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"coda_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ timing
def timed_loop(calls, steps, warmup, flush, stream, counter=None, sync_each=False):
    """Run `steps` steps; returns (per-call total ms list, total ms, kernels the
    library launched during the timed steps per `counter`, or None).  Every
    call is bracketed by events on `stream`; the L2 flush runs outside them.
    sync_each: the host waits for each step before queueing the next (as a
    caller that reads the step's result back does)."""
    for _ in range(warmup):
        flush()
        for c in calls:
            c()
    torch.cuda.synchronize()
    count0 = counter() if counter else None
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
           for _ in range(steps)]
    for i in range(steps):
        flush()
        for j, c in enumerate(calls):
            evs[i][j][0].record(stream)
            c()
            evs[i][j][1].record(stream)
        if sync_each:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    launched = (counter() - count0) if counter else None
    per_call = [0.0] * len(calls)
    for i in range(steps):
        for j in range(len(calls)):
            per_call[j] += evs[i][j][0].elapsed_time(evs[i][j][1])
    return per_call, sum(per_call), launched


def fused_calls(step):
    return [step.fused]


# ------------------------------------------------------------- CPU oracle
class OracleSample:
    """The fp64 oracle on a row sample of a workload, inputs generated once.
    calibrate() picks the row count for about `target_s` seconds per run."""

    def __init__(self, workload: str):
        from gemm_epilogue_transformer_tmem_gb300 import inputs
        from oracle import coda_oracle as O
        self.w, self.I, self.O = workload, inputs, O
        gen = dict(rmsproj=inputs.make_rmsproj, lnproj=inputs.make_lnproj, swiglu=inputs.make_swiglu,
                   dgrad=inputs.make_dgrad, llama=inputs.make_llama_block, skinny=inputs.make_skinny,
                   wgrad=inputs.make_wgrad, fp8swiglu=inputs.make_swiglu, mxfp8swiglu=inputs.make_swiglu)[workload]
        self.t = {k: O.to_f64(v) for k, v in gen(0).items()}
        self.Mmax = dict(llama=self.t["X"].shape[0] if "X" in self.t else 0,
                         wgrad=self.t["dW_old"].shape[0] if "dW_old" in self.t else 0).get(
            workload, next(iter(self.t.values())).shape[0])
        self.rows = 32
        if workload == "fp8swiglu":   # weight preparation, outside the timed sample
            w8, self.sw = O.quantize_rows_e4m3(self.t["W"].T)
            self.w8 = O.e4m3_decode(w8)
        if workload == "mxfp8swiglu":   # weight preparation, outside the timed sample
            self.wmx = O.dequantize_mx(*O.quantize_mx_e4m3(self.t["W"].T))

    def run(self, rows: int):
        """Returns (seconds, flops) of the oracle on the first `rows` rows."""
        I, O, t = self.I, self.O, self.t
        r = slice(0, rows)
        t0 = time.perf_counter()
        if self.w == "rmsproj":
            O.run_chain(t["X"][r], t["W"], [("RMS_ROWSCALE", 0, I.EPS_RMS)], norm_gamma=t["gamma"])
            fl = 2 * rows * t["W"].shape[0] * t["W"].shape[1]
        elif self.w == "lnproj":
            O.run_chain(t["X"][r], t["W"], [("LN_ROWSCALE", 0, I.EPS_LN)], norm_gamma=t["gamma"],
                        norm_beta=t["beta"])
            fl = 2 * rows * t["W"].shape[0] * t["W"].shape[1]
        elif self.w == "wgrad":
            # rows of dW = features of up: the sample takes the first `rows` of them
            O.run_chain(t["up"][:, r].T, t["dY"], [("SCALE", 0, I.WGRAD_SCALE), ("RESIDUAL", 0, 1.0),
                                                   ("ROW_SUMSQ", 0)], residual_t=t["dW_old"][r])
            fl = 2 * rows * t["dY"].shape[0] * t["dY"].shape[1]
        elif self.w == "fp8swiglu":
            # per-row E4M3 quantisation of the sample rows (W's output channels were
            # quantised once, as weight preparation), then the dequantised GEMM and SwiGLU
            x8, sx = O.quantize_rows_e4m3(t["X"][r])
            O.run_chain(O.e4m3_decode(x8), self.w8, [("ROW_SCALE", 0), ("COL_SCALE_F32",), ("SWIGLU",)],
                        b_layout="nk", row_vecs={0: sx}, col_scale_f32=self.sw)
            fl = 2 * rows * t["W"].shape[0] * t["W"].shape[1]
        elif self.w == "mxfp8swiglu":
            # MXFP8 quantisation of the sample rows (W quantised once, as weight
            # preparation), the product of the dequantised operands, SwiGLU
            xa = O.dequantize_mx(*O.quantize_mx_e4m3(t["X"][r]))
            O.run_chain(xa, self.wmx, [("SWIGLU",)], b_layout="nk")
            fl = 2 * rows * t["W"].shape[0] * t["W"].shape[1]
        elif self.w == "skinny":
            O.run_chain(t["X"][r], t["W"], [("RMS_ROWSCALE", None, I.EPS_RMS), ("SWIGLU",)],
                        norm_gamma=t["gamma"])
            fl = 2 * rows * t["W"].shape[0] * t["W"].shape[1]
        elif self.w == "swiglu":
            O.run_chain(t["X"][r], t["W"], [("SWIGLU",), ("DROPOUT", 0, I.DROPOUT_P)])
            fl = 2 * rows * t["W"].shape[0] * t["W"].shape[1]
        elif self.w == "dgrad":
            O.run_chain(t["dY"][r], t["W"], [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1)],
                        b_layout="nk", z=t["Z"][r], xhat=t["Xhat"][r])
            fl = 2 * rows * t["W"].shape[0] * t["W"].shape[1]
        else:
            eps = I.EPS_RMS
            X = t["X"][r]
            O.run_chain(X, t["W_qkv"], [("RMS_ROWSCALE", None, eps)], norm_gamma=t["gamma_attn"])
            h = O.run_chain(t["attn_out"][r], t["W_o"], [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)], residual_t=X)["D"]
            up = O.run_chain(h, t["W_up"], [("RMS_ROWSCALE", None, eps), ("SWIGLU",)],
                             norm_gamma=t["gamma_mlp"])["D"]
            O.run_chain(up, t["W_down"], [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)], residual_t=h)
            d, f = t["W_o"].shape[0], t["W_down"].shape[0]
            fl = 2 * rows * d * (3 * d + d + 2 * f) + 2 * rows * f * d
        return time.perf_counter() - t0, fl

    def calibrate(self, target_s: float) -> int:
        """Grow the row sample towards target_s of CPU work; once it covers the
        whole workload, repeat the whole workload instead (self.reps)."""
        self.reps = 1
        dt, _ = self.run(self.rows)
        while dt < target_s / 3 and self.rows < self.Mmax:
            grow = max(2.0, min(16.0, 0.8 * target_s / max(dt, 1e-3)))
            self.rows = min(self.Mmax, int(self.rows * grow))
            dt, _ = self.run(self.rows)
        if self.rows >= self.Mmax and dt < target_s / 2:
            self.reps = max(1, int(round(target_s / max(dt, 1e-3))))
        return self.rows

    def run_sample(self):
        """(seconds, flops) of the calibrated sample: `rows` rows, `reps` times."""
        tot_t, tot_f = 0.0, 0
        for _ in range(self.reps):
            dt, fl = self.run(self.rows)
            tot_t += dt
            tot_f += fl
        return tot_t, tot_f

    def describe(self) -> str:
        if self.reps > 1:
            return f"fp64 oracle on the whole workload ({self.rows} rows), repeated {self.reps} times"
        return f"fp64 oracle on the first {self.rows} rows of the workload"


def aggregate_ms(total_ms: float, dist, device) -> float:
    """Max over ranks of the timed region (each rank ran its own replica)."""
    if dist is None:
        return total_ms
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# -------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama", choices=sorted(DESCRIPTIONS))
    ap.add_argument("--impl", default="coda", choices=["coda", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-library", action="store_true")
    ap.add_argument("--tile-order", default="static", choices=["static", "dynamic"],
                    help="tile order of grids with more tiles than clusters (library knob; default static)")
    ap.add_argument("--tail-helpers", default="on", choices=["on", "off"],
                    help="non-epilogue warps share each CTA's last-tile epilogue (library knob; default on)")
    ap.add_argument("--split-k", default="auto", choices=["auto", "off", "force"],
                    help="split over K for single-CTA problems (library knob; default auto)")
    ap.add_argument("--raster", default="auto", choices=["auto", "rows", "cols"],
                    help="tile order of the persistent grid (library knob; default auto)")
    ap.add_argument("--raster-group", type=int, default=0, help="blocks per raster group (0: the library's)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="llama only: tokens per step (default 16384); smaller values make the small cases an "
                         "ncu capture needs")
    ap.add_argument("--profile-steps", action="store_true",
                    help="one fused and one unfused step between L2 flushes, for an ncu capture; no JSON line")
    args = ap.parse_args()
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[args.workload]
    warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, steps, warmup, world, rank)

    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist

    import __graft_entry__ as entry
    entry.build()
    from gemm_epilogue_transformer_tmem_gb300 import coda, workloads
    coda.set_split_k(args.split_k)
    coda.set_tile_scheduler(args.tile_order)
    coda.set_tail_helpers(args.tail_helpers == "on")
    coda.set_raster(args.raster, args.raster_group)

    dev = torch.device("cuda", local)
    if args.tokens is not None and args.workload != "llama":
        raise SystemExit("--tokens applies to the llama workload only")
    step = (workloads.BUILDERS[args.workload](dev=dev) if args.tokens is None
            else workloads.build_llama(dev=dev, tokens=args.tokens))
    stream = torch.cuda.current_stream()
    # L2 flush between steps: write a buffer larger than L2, then read another
    # one, so the timed step starts with a cold L2 that holds no dirty lines
    # (a write alone leaves ~126 MB to be written back during the next step,
    # which takes HBM bandwidth from it)
    flush_buf = torch.empty((L2_FLUSH_BYTES // 4,), dtype=torch.float32, device=dev)
    flush_rd = torch.ones((L2_FLUSH_BYTES // 4,), dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        flush_buf.zero_()
        torch.sum(flush_rd, dim=0, out=flush_out)

    if args.profile_steps:
        for _ in range(warmup):
            flush()
            step.fused()
        for call in (step.fused, step.unfused):
            flush()
            call()
            # read-only pass: evicts the step's dirty lines (its writes) and writes nothing itself
            torch.sum(flush_rd, dim=0, out=flush_out)
        torch.cuda.synchronize()
        st, info = coda.check_device_error()
        if st != 0:
            raise RuntimeError(f"device error {st}: {info}")
        print(f"profile steps done: {args.workload}", flush=True)
        return

    # ---- fused step, device-resident inputs
    sampler = ClockSampler(local) if rank == 0 else None
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # a step of several calls is timed call by call (events between them), so
    # that the roofline of its dominant call is measured on that call alone
    calls = [c for _, c, _ in step.parts] if step.parts else [step.fused]
    per_call, total_ms, launches = timed_loop(calls, steps, warmup, flush, stream, coda.launch_count)
    clocks = sampler.stop() if sampler else None
    plan = coda.last_plan()      # how the step's last GEMM call ran
    st, info = coda.check_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st}: {info}")
    total_ms = aggregate_ms(total_ms, pg, dev)
    if pg:
        pg.barrier()
    ms = total_ms / steps
    value = world * step.flops / (ms * 1e-3) / 1e12

    # ---- unfused chain through the library's own kernels
    unfused = None
    if not args.no_unfused:
        u_steps = max(steps // 2, 3)
        _, u_total, u_launched = timed_loop([step.unfused], u_steps, warmup, flush, stream, coda.launch_count)
        u_ms = u_total / u_steps
        unfused = {"ms_per_step": round(u_ms, 5), "value": round(step.flops / (u_ms * 1e-3) / 1e12, 2),
                   "unit": UNIT, "kernels_per_step": u_launched / u_steps,
                   "speedup_fused": round(u_ms / ms, 3)}

    # ---- the same unfused chain with cuBLAS's GEMM (torch.matmul) in place of the library's own
    unfused_lib = None
    if not args.no_unfused and not args.no_library and step.unfused_library is not None and rank == 0:
        try:
            ul_steps = max(steps // 2, 3)
            _, ul_total, _ = timed_loop([step.unfused_library], ul_steps, warmup, flush, stream)
            ul_ms = ul_total / ul_steps
            unfused_lib = {"what": "the unfused chain with torch.matmul (cuBLAS) for its GEMMs, the library's "
                                   "separate kernels for the other steps",
                           "ms_per_step": round(ul_ms, 5), "value": round(step.flops / (ul_ms * 1e-3) / 1e12, 2),
                           "unit": UNIT, "speedup_fused": round(ul_ms / ms, 3)}
        except RuntimeError as exc:
            unfused_lib = {"unavailable": str(exc).splitlines()[0][:200]}

    # ---- the step's GEMMs alone through torch.matmul (cuBLAS): a reference point
    library = None
    if not args.no_library and step.library is not None and rank == 0:
        try:
            l_steps = max(steps // 2, 3)
            _, l_total, _ = timed_loop([step.library], l_steps, warmup, flush, stream)
            l_ms = l_total / l_steps
            library = {"what": "torch.matmul (cuBLAS) of the step's GEMMs on the same operands, no epilogue",
                       "ms_per_step": round(l_ms, 5), "value": round(step.flops / (l_ms * 1e-3) / 1e12, 2),
                       "unit": UNIT, "fused_step_vs_library_gemm": round(l_ms / ms, 3)}
        except RuntimeError as exc:
            library = {"unavailable": str(exc).splitlines()[0][:200]}

    # ---- end to end through host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e and rank == 0:
        hin = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v.cpu())
               for k, v in step.host_inputs.items()}
        hout = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in step.host_outputs.items()}
        e2e_steps = max(steps // 10, 3)

        def e2e_call():
            if step.e2e is not None:     # the step overlaps its copies with its own calls
                step.e2e(hin, hout)
                return
            for k, v in hin.items():
                step.host_inputs[k].copy_(v, non_blocking=True)
            step.fused()
            for k, v in hout.items():
                v.copy_(step.host_outputs[k], non_blocking=True)

        # the host reads each step's result back before it queues the next
        _, e_total, _ = timed_loop([e2e_call], e2e_steps, 3, flush, stream, sync_each=True)
        e_ms = e_total / e2e_steps
        e2e = {"value": round(step.flops / (e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
               "ms_per_step": round(e_ms, 5),
               "copies": ("overlapped with the step's calls on two side streams (events order them), in "
                          "blocks of tokens where the step is the LLaMA block"
                          if step.e2e is not None else "host-to-device, step, device-to-host on the launching stream")
                         + "; the host waits for each step's read-back before the next step",
               "h2d_bytes_per_step": int(sum(v.numel() * v.element_size() for v in hin.values())),
               "d2h_bytes_per_step": int(sum(v.numel() * v.element_size() for v in hout.values()))}

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    call_s = sum(per_call) / steps * 1e-3
    dom_name, dom_flops, dom_s = args.workload, step.flops, call_s
    if step.parts:
        i = max(range(len(step.parts)), key=lambda j: step.parts[j][2])
        dom_name, dom_flops, dom_s = step.parts[i][0], step.parts[i][2], per_call[i] / steps * 1e-3
    traffic = load_traffic(args.workload)
    if step.bound == "hbm":
        # the weight stream bounds the step: algorithmic bytes against the measured copy bandwidth
        peak = float(peaks["hbm_gbs"])
        achieved = step.fused_bytes / call_s / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "peak_source": f"HBM copy, of {peak_src}"}
    else:
        # the fused kernels are timed in short bursts between L2 flushes: burst peak
        # (FP8 operands: the measured bf16 peak times the nominal FP8 / bf16 ratio 2)
        peak = float(peaks["bf16_tflops"]) * step.peak_scale
        achieved = dom_flops / dom_s / 1e12
        src = "bf16 burst" if step.peak_scale == 1.0 else f"bf16 burst x {step.peak_scale:g} (nominal fp8/bf16)"
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 4), "peak_source": f"{src}, of {peak_src}"}
    roofline.update(kernel=f"{dom_name}: the fused GEMM call" + (", timed alone within the step" if step.parts else
                                                                 " (with its finishing kernels)"),
                    traffic=traffic.get("dominant_kernel_bytes", traffic.get("bytes_per_launch")) if traffic else None,
                    algorithmic_bytes=step.parts_bytes.get(dom_name, step.fused_bytes) if step.parts else
                    step.fused_bytes)
    if step.parts:
        roofline["calls"] = {n: {"ms": round(per_call[j] / steps, 5),
                                 "tflops": round(fl / (per_call[j] / steps * 1e-3) / 1e12, 2)}
                             for j, (n, _, fl) in enumerate(step.parts)}

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        osm = OracleSample(args.workload)
        osm.calibrate(12.0)
        dt, fl = osm.run_sample()
        cpu = {"value": round(fl / dt / 1e12, 6), "unit": UNIT, "cores": _NCORES, "kind": "oracle",
               "sample": f"{osm.describe()} ({dt:.1f} s)"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}" +
                               (f" (run at {args.tokens} tokens, not 16384)" if args.tokens else ""),
                   "flops_per_step": step.flops,
                   "l2": "flushed between steps outside the timed events: a 256 MiB device write, then a "
                         "256 MiB read, so no dirty lines are written back inside the timed region",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "weight_prep": "gamma folded into W once per weight version, not in the step",
                   "plan_of_last_gemm": plan},
        "roofline": roofline,
        "dram_bytes": {"fused_algorithmic": step.fused_bytes, "unfused_algorithmic": step.unfused_bytes,
                       "fused_measured": traffic.get("fused_step_bytes") if traffic else None,
                       "unfused_measured": traffic.get("unfused_step_bytes") if traffic else None,
                       "measured_by": traffic.get("source") if traffic else None},
        "unfused": unfused,
        "unfused_cublas": unfused_lib,
        "library_gemm": library,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def reference_arm(args, steps, warmup, world, rank):
    """The fp64 oracle timed on the host cores as the reference implementation."""
    if rank != 0:
        return
    osm = OracleSample(args.workload)
    per_step = max(0.5, min(10.0, 150.0 / (steps + warmup)))
    rows = osm.calibrate(per_step)
    vals = []
    for i in range(warmup + steps):
        dt, fl = osm.run_sample()
        if i >= warmup:
            vals.append((fl / dt / 1e12, dt))
    value = statistics.median(v for v, _ in vals)
    ms = statistics.median(dt for _, dt in vals) * 1e3
    info = (rows,)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                   "sample": f"{osm.describe()} per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": _NCORES, "kind": "oracle",
                         "sample": f"{osm.describe()} per step"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

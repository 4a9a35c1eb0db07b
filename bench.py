#!/usr/bin/env python3
"""Benchmark of the fine-grained FP8 hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fp8q|reference]

One step = one FP8 Fprop pass of the dense FFN up-projection
(tokens 4096, hidden 7168 -> 18432): quantize X (BF16 4096x7168, 1x128
groups), quantize W (BF16 18432x7168, 128x128 blocks), block-scaled FP8 GEMM
with FP32 promotion every 128 K and BF16 output.  `value` is GEMM TFLOP/s
over the whole step (inputs resident in HBM; 323 MB of BF16 inputs per step
exceed the 126 MB L2, so no flush is needed).  The JSON line also carries:
  roofline      the GEMM kernel against the FP8 dense peak (the measured BF16
                matmul peak x 2, the nominal FP8:BF16 ratio)
  e2e           the same metric through the C ABI with host buffers: pinned
                H2D copies of X and W, the three kernels, D2H of Y per step
  breakdown     activation quantization 16384x7168 (GB/s vs HBM), Wgrad
                2048x7168x8192 and the 256-expert MoE grouped GEMM (TFLOP/s)
  cpu_baseline  the CPU oracle on a bounded sample of the same step
  clocks        NVML samples of SM clock and throttle reasons while timing
`--impl reference` times the CPU oracle (the reference of this build) on a
bounded sample of each step instead.  Under torchrun every rank runs an
independent replica (no collective on the data path); value sums ranks.
"""
import argparse
import hashlib
import json
import os
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FPROP = dict(M=4096, N=18432, K=7168)
ACT = dict(T=16384, H=7168)
WGRAD = dict(T=8192, Dout=2048, Din=7168)
MOE = dict(T=8192, H=7168, E=256, N=2048, topk=8)
METRIC = "FP8 blockscaled GEMM TFLOP/s (% B300 dense FP8 peak); quantize GB/s (% HBM)"
FP8_PER_BF16 = 2.0  # nominal dense ratio: 4.5 PFLOP/s FP8 / 2.25 PFLOP/s BF16


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="fp8q", choices=["fp8q", "reference"])
    p.add_argument("--no-breakdown", action="store_true", help="time the Fprop step only")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


def kernel_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fine_grained_fp8_quantize_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu capture, if it was taken of
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_sha()
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(tok.split("=", 1) for tok in line.split())
            if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("sources") == sha:
                return float(kv["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """Polls NVML (SM clock, max clock, throttle reasons) in a thread."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle"}

    def __init__(self, index):
        self.samples = []
        self.reasons = 0
        self.ok = False
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.ok = True
        except Exception:
            self.max_mhz = None
        self._stop = threading.Event()

    def _run(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                get = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                    nv.nvmlDeviceGetCurrentClocksThrottleReasons
                self.reasons |= get(self.h)
            except Exception:
                pass
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": len(self.samples)}
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": float(np.median(self.samples)), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(self.samples)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def gpu_arm(args, rank, world, dist):
    import torch

    import fine_grained_fp8_quantize_b300 as f
    import synth

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    stream = torch.cuda.current_stream()
    pk = peaks()
    M, N, K = FPROP["M"], FPROP["N"], FPROP["K"]
    flops = 2.0 * M * N * K

    X, W = synth.fprop_inputs(device="cuda", seed=2 + 1000 * rank)
    qx = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    sx = torch.empty(K // 128, M, dtype=torch.float32, device="cuda")
    qw = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    sw = torch.empty(N // 128, K // 128, dtype=torch.float32, device="cuda")
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")

    def step(ev=None):
        f.fp8q_quantize_act(X, qx, sx)
        f.fp8q_quantize_weight(W, qw, sw)
        if ev is not None:
            ev[0].record(stream)
        f.fp8q_gemm(qx, sx, qw, sw, Y)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = f.fp8q_get_device_status()
    if st != 0:
        raise RuntimeError("device status after warm-up: %s" % f.fp8q_status_string(st))

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    with sampler:
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = t0.elapsed_time(t1)
    gemm_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    if dist:
        tt = torch.tensor([ms], dtype=torch.float64, device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    st = f.fp8q_get_device_status()
    if st != 0:
        raise RuntimeError("device status after timing: %s" % f.fp8q_status_string(st))

    ms_step = ms / args.steps
    value = world * flops * args.steps / (ms * 1e-3) / 1e12
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    peak_fp8 = pk["bf16"] * FP8_PER_BF16
    roofline = {
        "kernel": "gemm_kernel<bf16 out, 128x128 B scales>",
        "bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": round(peak_fp8, 1), "unit": "TFLOP/s",
        "frac": round(gemm_tflops / peak_fp8, 4),
        "peak_note": "%s BF16 matmul burst %.1f TFLOP/s x 2 (nominal FP8:BF16); frac vs sustained x2 = %.4f"
                     % (pk["src"], pk["bf16"], gemm_tflops / (pk["bf16_sus"] * FP8_PER_BF16)),
        "gemm_ms": round(gemm_ms, 4), "flops_per_launch": flops,
        "traffic": recorded_traffic("gemm_kernel", "fprop_4096x18432x7168"),
    }

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32 accumulate, bf16 out",
        "data": "synthetic (seeded SplitMix64 + Box-Muller; X N(0,1) with 0.1% x1e3, W N(0,0.02^2))",
        "config": {"workload": "fprop 4096x18432x7168: quantize X 1x128 + quantize W 128x128 + block-scaled "
                               "FP8 GEMM, BF16 out", "M": M, "N": N, "K": K, "global_batch": M * world,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": "inputs larger than L2 (323 MB BF16 per step), no flush"},
        "roofline": roofline,
        "gpu_launches": 3 * args.steps,
        "clocks": sampler.summary(),
    }

    if rank == 0 and not args.no_e2e:
        out["e2e"] = e2e_fprop(args, f, torch, X, W)
    if rank == 0 and not args.no_breakdown:
        out["breakdown"] = breakdown(args, f, torch, synth, pk)
    if rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline_fprop(X, W, budget_s=15.0)
    return out


def e2e_fprop(args, f, torch, X, W):
    """Fprop through the C ABI with host buffers: per step pinned H2D of X and
    W, quantize X, quantize W, GEMM, D2H of Y; CUDA events around it all."""
    M, N, K = FPROP["M"], FPROP["N"], FPROP["K"]
    hX = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    hW = torch.empty(W.shape, dtype=W.dtype, pin_memory=True)
    hX.copy_(X)
    hW.copy_(W)
    hY = torch.empty(M, N, dtype=torch.bfloat16, pin_memory=True)
    dX = torch.empty_like(X)
    dW = torch.empty_like(W)
    qx = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    sx = torch.empty(K // 128, M, dtype=torch.float32, device="cuda")
    qw = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    sw = torch.empty(N // 128, K // 128, dtype=torch.float32, device="cuda")
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        dX.copy_(hX, non_blocking=True)
        dW.copy_(hW, non_blocking=True)
        f.fp8q_quantize_act(dX, qx, sx)
        f.fp8q_quantize_weight(dW, qw, sw)
        f.fp8q_gemm(qx, sx, qw, sw, Y)
        hY.copy_(Y, non_blocking=True)

    steps = max(3, min(args.steps, 20))
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 3),
            "steps": steps, "h2d_bytes_per_step": X.numel() * 2 + W.numel() * 2,
            "d2h_bytes_per_step": M * N * 2}


def _time(fn, iters, torch, warm=3):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def breakdown(args, f, torch, synth, pk):
    res = {}
    iters = max(5, min(args.steps, 50))
    # -- activation quantization, 16384 x 7168, 1x128 rows + 128x1 transposed copy
    T, H = ACT["T"], ACT["H"]
    X = synth.act_quant_inputs(device="cuda")
    q_row = torch.empty(T, H, dtype=torch.uint8, device="cuda")
    s_row = torch.empty(H // 128, T, dtype=torch.float32, device="cuda")
    q_colT = torch.empty(H, T, dtype=torch.uint8, device="cuda")
    s_col = torch.empty(T // 128, H, dtype=torch.float32, device="cuda")
    ms = _time(lambda: f.fp8q_quantize_act(X, q_row, s_row, q_colT, s_col), iters, torch)
    nbytes = T * H * 2 + 2 * T * H + 2 * (T * H // 128) * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    res["act_quant_16384x7168"] = {
        "ms": round(ms, 4), "GB/s": round(gbs, 1), "bytes": nbytes,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(gbs / pk["hbm"], 4), "frac_of_8TBs_nominal": round(gbs / 8000.0, 4),
                     "traffic": recorded_traffic("quant_tile_kernel", "act_16384x7168")}}
    del X, q_row, s_row, q_colT, s_col

    # -- Wgrad: dW = dY^T X, 128x1 groups along 8192 tokens, FP32 out
    dY, Xw = synth.wgrad_inputs(device="cuda")
    Tt, Do, Di = WGRAD["T"], WGRAD["Dout"], WGRAD["Din"]
    qdy = torch.empty(Do, Tt, dtype=torch.uint8, device="cuda")
    sdy = torch.empty(Tt // 128, Do, dtype=torch.float32, device="cuda")
    qx = torch.empty(Di, Tt, dtype=torch.uint8, device="cuda")
    sx = torch.empty(Tt // 128, Di, dtype=torch.float32, device="cuda")
    dW = torch.empty(Do, Di, dtype=torch.float32, device="cuda")
    f.fp8q_quantize_act(dY, None, None, qdy, sdy)
    f.fp8q_quantize_act(Xw, None, None, qx, sx)
    ms_g = _time(lambda: f.fp8q_gemm_ex(qdy, sdy, qx, sx, dW, 1), iters, torch)
    ms_all = _time(lambda: (f.fp8q_quantize_act(dY, None, None, qdy, sdy), f.fp8q_quantize_act(Xw, None, None, qx, sx),
                            f.fp8q_gemm_ex(qdy, sdy, qx, sx, dW, 1)), iters, torch)
    fl = 2.0 * Do * Di * Tt
    res["wgrad_2048x7168x8192"] = {
        "gemm_ms": round(ms_g, 4), "gemm_TFLOP/s": round(fl / ms_g / 1e9, 1),
        "step_ms": round(ms_all, 4), "step_TFLOP/s": round(fl / ms_all / 1e9, 1),
        "frac_of_fp8_peak": round(fl / ms_g / 1e9 / (pk["bf16"] * FP8_PER_BF16), 4)}
    del dY, Xw, qdy, sdy, qx, sx, dW

    # -- MoE grouped GEMM: 8192 tokens, 256 experts (top-8), 7168 -> 2048, BF16 out
    off, src = synth.moe_routing()
    counts = off[1:] - off[:-1]
    active = [int(e) for e in np.flatnonzero(counts)]
    E, Nn, Kk = MOE["E"], MOE["N"], MOE["H"]
    Xm, Wm = synth.moe_inputs(device="cuda", experts=active)
    qw, sw = f.quantize_weight(Wm.view(E * Nn, Kk))
    qw = qw.view(E, Nn, Kk)
    sw = sw.view(E, Nn // 128, Kk // 128)
    src_d = torch.from_numpy(src.astype(np.int32)).cuda()
    off_d = torch.from_numpy(off.astype(np.int32)).cuda()
    R = len(src)
    qa = torch.empty(R, Kk, dtype=torch.uint8, device="cuda")
    sa = torch.empty(Kk // 128, R, dtype=torch.float32, device="cuda")
    Cm = torch.empty(R, Nn, dtype=torch.bfloat16, device="cuda")
    f.fp8q_quantize_act_gather(Xm, src_d, qa, sa)
    ms_g = _time(lambda: f.fp8q_grouped_gemm(qa, sa, qw, sw, Cm, off_d), iters, torch)
    ms_all = _time(lambda: (f.fp8q_quantize_act_gather(Xm, src_d, qa, sa),
                            f.fp8q_grouped_gemm(qa, sa, qw, sw, Cm, off_d)), iters, torch)
    fl = 2.0 * R * Nn * Kk
    wbytes = len(active) * Nn * Kk
    gbytes = R * Kk + R * (Kk // 128) * 4 + wbytes + R * Nn * 2
    t_comp = fl / (pk["bf16"] * FP8_PER_BF16 * 1e12)
    t_mem = gbytes / (pk["hbm"] * 1e9)
    res["moe_grouped_256x(7168->2048)"] = {
        "active_experts": len(active), "rows": R, "gemm_ms": round(ms_g, 4),
        "gemm_TFLOP/s": round(fl / ms_g / 1e9, 1), "step_ms": round(ms_all, 4),
        "bound": "tensor" if t_comp > t_mem else "hbm",
        "roofline_frac": round(max(t_comp, t_mem) / (ms_g * 1e-3), 4),
        "min_bytes": gbytes}
    return res


def cpu_baseline_fprop(X, W, budget_s=15.0):
    """The CPU oracle as it stands on a bounded sample of the Fprop step:
    quantize R rows of X and all of W, then compute R full output rows."""
    import oracle
    import synth
    M, N, K = FPROP["M"], FPROP["N"], FPROP["K"]
    xb = synth.bf16_bits(X)
    wb = synth.bf16_bits(W)
    R = 8
    t = time.perf_counter()
    rows = np.arange(0, M, M // R)[:R]
    qx, sx = oracle.quantize_act_rows(xb[rows])
    qw, sw = oracle.quantize_weight(wb)
    mi = np.repeat(np.arange(R), N)
    ni = np.tile(np.arange(N), R)
    oracle.gemm_points(qx, sx, qw, sw, mi, ni)
    dt = time.perf_counter() - t
    fl = 2.0 * R * N * K
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d of 4096 rows of the fprop step (quantize those rows, quantize all of W, %d full output "
                      "rows); %.1f s" % (R, R, dt)}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def reference_arm(args):
    import oracle
    import synth
    import torch
    M, N, K = FPROP["M"], FPROP["N"], FPROP["K"]
    R = 4
    X = synth.matrix(2, 1, R, K, 1.0, entry_frac=1e-3, entry_scale=1e3)   # rows of the fprop X
    W = synth.matrix(2, 2, N, K, 0.02)
    xb, wb = synth.bf16_bits(X), synth.bf16_bits(W)
    mi = np.repeat(np.arange(R), N)
    ni = np.tile(np.arange(N), R)

    def step():
        qx, sx = oracle.quantize_act_rows(xb)
        qw, sw = oracle.quantize_weight(wb)
        oracle.gemm_points(qx, sx, qw, sw, mi, ni)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t) / args.steps
    fl = 2.0 * R * N * K
    v = fl / dt / 1e12
    sample = "%d of 4096 rows of the fprop step per step (quantize them and all of W, %d full output rows)" % (R, R)
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 exact / f32 promotion order (CPU)",
            "data": "synthetic", "config": {"workload": "fprop 4096x18432x7168 (bounded row sample)",
                                            "M": M, "N": N, "K": K},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(reference_arm(args)))
        return 0
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    out = gpu_arm(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

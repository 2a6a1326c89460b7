"""Benchmark of the fused linear-layer hot path on one GB300 (or N replicas).

One step = one pass of the whole path over one batch of synthetic input:
  1. forward   D = relu(X W^T + b) with the bit-packed mask (RELU_AUX_BIAS),
               W[11008, 4096], X[8192, 4096]          (tcgen05 GEMM, fused epilogue)
  2. backward  dZ = dY * mask, bgrad = sum_tokens dZ  (DRELU_BGRAD stream)
  3. weight gradient dW = dZ^T X                      (tcgen05 GEMM, NONE epilogue)
  4. decode    y = gelu(W2 x + b2), W2[4096, 4096], one token (GEMV, GELU_BIAS)
The LLaMA-7B-like MLP and the hidden-4096 decode projection stand in for the
pages' workloads (nvmath-python RELU_AUX_BIAS / DRELU_BGRAD, ops-nn decode).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (the path has no
exchange step); the time is the max over ranks, the value sums all ranks.
Prints one JSON line on rank 0.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM+bias+act TFLOP/s & % FP16 tensor peak; M=1 GEMV/bgrad HBM GB/s"
T_TOK, D_IN, D_OUT, D_DEC = 8192, 4096, 11008, 4096
WORKLOAD = ("LLaMA-7B-like MLP training step (fwd RELU_AUX_BIAS 11008x8192x4096 + DRELU_BGRAD "
            "dY[8192,11008] + dW 11008x4096x8192) + decode GEMV GELU_BIAS 4096x1x4096")


# Timing-only cases for the other workload configs: key -> (workload key, unfused?)
CONFIG_CASES = {
    "cfg_c1": ("c1", False), "cfg_c2_bias": ("c2_bias", False),
    "cfg_c2_relu_bias": ("c2_relu_bias", False), "cfg_c2_gelu_bias": ("c2_gelu_bias", False),
    "cfg_c2_gelu_bias_unfused": ("c2_gelu_bias", True),
    "cfg_c3_T512": ("c3_T512", False), "cfg_c3_T512_unfused": ("c3_T512", True),
    "cfg_c3_T2048": ("c3_T2048", False), "cfg_c3_T2048_unfused": ("c3_T2048", True),
    "cfg_c5": ("c5", False), "cfg_c5_unfused": ("c5", True),
    # backward GEMM dH = G W2^T (11008 x 8192 x 4096) with DRELU_BGRAD fused
    # in its epilogue, vs. the GEMM followed by the standalone DRELU_BGRAD
    "cfg_bwd_gemm_drelu": ("bwd", False), "cfg_bwd_gemm_drelu_unfused": ("bwd", True),
    # the same workloads with bfloat16 operands, bias and output
    "cfg_c4_fwd": ("c4_fwd", False), "cfg_c4_fwd_bf16": ("c4_fwd", False, "bf16"),
    "cfg_c4_dw_bf16": ("c4_dw", False, "bf16"), "cfg_c3_T1_bf16": ("c3_T1", False, "bf16"),
    "cfg_c5_bf16": ("c5", False, "bf16"),
    # the forward's shape with other epilogues (what each epilogue costs)
    "cfg_c4_fwd_none": ("c4_fwd", False, "f16", "none"), "cfg_c4_fwd_bias": ("c4_fwd", False, "f16", "bias"),
    "cfg_c4_fwd_gelu": ("c4_fwd", False, "f16", "gelu_bias"),
}


# Timing-only cases of the later rows: name -> (kind, params)
ROW_CASES = {}
for _T in (1, 2048, 8192):
    for _n in ("rmsnorm", "layernorm"):
        for _u in (False, True):
            ROW_CASES[f"norm_{_n}_T{_T}" + ("_unfused" if _u else "")] = ("norm", dict(T=_T, norm=_n, unfused=_u))
ROW_CASES.update({
    "gelu_aux_fwd": ("gelu_aux", dict(unfused=False)), "gelu_aux_fwd_unfused": ("gelu_aux", dict(unfused=True)),
    "dgelu": ("dgelu", dict(K=0, unfused=False)),
    "drelu_rows": ("drelu_rows", dict()),
    "dw_drelu": ("dw_drelu", dict(unfused=False)), "dw_drelu_unfused": ("dw_drelu", dict(unfused=True)),
    "bwd_gemm_dgelu": ("dgelu", dict(K=D_IN, unfused=False)),
    "bwd_gemm_dgelu_unfused": ("dgelu", dict(K=D_IN, unfused=True)),
})


def kernel_source_hash(files=("gemm_epilogues_gb300/csrc/ge_gemm.cu", "gemm_epilogues_gb300/csrc/ge_gemm_kernel.cuh",
                               "gemm_epilogues_gb300/csrc/ge_ptx.cuh", "gemm_epilogues_gb300/csrc/ge_internal.h",
                               "gemm_epilogues_gb300/csrc/ge_api.cu")) -> str:
    """Hash of the GEMM kernel's code and of the planner that picks its tile
    order (which moves its DRAM traffic): comments and blank lines are left
    out, so a change of wording alone does not invalidate a capture."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in src.splitlines()]
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def captured_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    capture in profiles/traffic.json, or None when the GEMM sources changed
    since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("gemm_source_hash") != kernel_source_hash():
        return None
    return t.get("per_launch_bytes", {}).get(kernel)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "tflops": float(p["bf16_tflops"]),
                "tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "tflops": 1900.0, "tflops_sustained": 1700.0, "source": "fallback"}


def choose_tensor_peak(peaks, timed_s: float, clocks):
    """The measured tensor peak a kernel timed in a region of `timed_s`
    seconds is held to: the sustained figure (a seconds-long loop under the
    power cap) only when the region lasted at least a second and the clock
    record saw the power cap; otherwise the burst figure.
    Returns (peak, sustained?, power cap seen?)."""
    capped = bool(clocks) and "sw_power_cap" in (clocks.get("reasons") or [])
    sustained = timed_s >= 1.0 and capped
    return (peaks["tflops_sustained"] if sustained else peaks["tflops"]), sustained, capped


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 100):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU side

_ORACLE_INPUTS = {}


def oracle_sample_rate(rows: int = 256, threads: int | None = None):
    """The oracle (fp64 CPU) on a bounded sample of the forward GEMM: `rows`
    tokens of X against the whole W. Returns (TFLOP/s, seconds, threads)."""
    import numpy as np
    import torch
    from gemm_epilogues_gb300.inputs import f16_tensor
    from oracle import oracle
    oracle.build()
    threads = threads or os.cpu_count() or 1
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    if rows not in _ORACLE_INPUTS:  # generated once, outside the timed call
        _ORACLE_INPUTS[rows] = (bits(f16_tensor((D_OUT, D_IN), 3001, "normal", 1 / 64)),
                                bits(f16_tensor((rows, D_IN), 3002)),
                                bits(f16_tensor((D_OUT,), 3003, "normal", math.sqrt(0.02))))
    W, X, b = _ORACLE_INPUTS[rows]
    t0 = time.perf_counter()
    oracle.linear_forward(W, X, b, "relu_aux_bias", D_OUT, rows, D_IN,
                          a_major="k", b_major="k", d_layout="col", threads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * D_OUT * rows * D_IN
    return flops / dt / 1e12, dt, threads


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle as it stands, timed on the host cores,
    same metric and unit, each step a bounded sample of the workload."""
    if rank != 0:
        return
    rows = 64
    for _ in range(args.warmup):
        oracle_sample_rate(rows)
    times = []
    thr = None
    for _ in range(args.steps):
        _, dt, thr = oracle_sample_rate(rows)
        times.append(dt)
    flops = 2.0 * D_OUT * rows * D_IN
    value = flops * len(times) / sum(times) / 1e12
    sample = f"forward GEMM on {rows} of {T_TOK} tokens (all 11008 outputs, K=4096) per step"
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU side

def run_config(args, rank):
    """Time one workload config (fused or the unfused three-kernel sequence):
    `steps` launches after `warmup`, each after a read-only L2 flush."""
    import torch
    import gemm_epilogues_gb300 as ge
    from gemm_epilogues_gb300.inputs import pages_workloads
    key, unfused, *rest = CONFIG_CASES[args.case]
    dtype = rest[0] if rest else "f16"
    if key == "bwd":
        return run_bwd_gemm_drelu(args, rank, unfused)
    w = pages_workloads()[key]
    w.dtype = dtype
    if len(rest) > 1:
        w.epilogue = rest[1]
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    A, B, bias = w.make(dev)
    major = {"k": ge.GE_K_MAJOR, "m": ge.GE_MN_MAJOR, "n": ge.GE_MN_MAJOR}
    L = ge.make_layout(major[w.a_major], major[w.b_major], ge.GE_D_ROW if w.d_layout == "row" else ge.GE_D_COL)
    plan = ge.Plan(w.M, w.N, w.K, ge.EPILOGUE_BY_NAME[w.epilogue], L,
                   dtype=ge.GE_BF16 if dtype == "bf16" else ge.GE_F16)
    D = torch.empty(w.d_shape(), dtype=A.dtype, device=dev)
    aux = torch.empty(max(plan.aux_bytes // 4, 1), dtype=torch.int32, device=dev)
    bias_arg = bias if w.epilogue != "none" else None
    aux_arg = aux if w.epilogue == "relu_aux_bias" else None
    flush_buf = torch.ones((256 << 20) // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    run = plan.execute_unfused if unfused else plan.execute
    times = []
    for i in range(args.warmup + args.steps):
        torch.sum(flush_buf, dim=0, out=flush_out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(A, B, bias_arg, D, aux_arg, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    assert ge.ge_get_last_device_error(plan.handle) == ge.GE_OK
    ms = sum(times) / len(times)
    tflops = w.flops / (ms * 1e-3) / 1e12
    line = {"case": args.case, "workload": w.name, "dtype": dtype, "unfused": unfused, "path": plan.path,
            "tile_n": plan.tile_n, "ms": ms, "min_ms": min(times), "tflops": tflops,
            "frac_of_peak": tflops / peaks["tflops"],
            "gbs_algorithmic": w.algorithmic_bytes() / (ms * 1e-3) / 1e9}
    plan.free()
    if rank == 0:
        print(json.dumps(line), flush=True)


def _time_flushed(run, steps, warmup, dev):
    """Device time of `run()` per call (ms list): CUDA events on the current
    stream around each call, after a read-only pass over 2x L2."""
    import torch
    flush_buf = torch.ones((256 << 20) // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    times = []
    for i in range(warmup + steps):
        torch.sum(flush_buf, dim=0, out=flush_out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1))
    return times


def run_row_case(args, rank):
    """The later rows at the pages' shapes: MatMul + bias + residual + norm
    over a LLaMA-7B attention output projection (4096 x T x 4096), the
    GELU_AUX_BIAS forward and the DGELU_BGRAD backward of the MLP
    (11008 x 8192 x 4096), fused or by separate kernels."""
    import torch
    import gemm_epilogues_gb300 as ge
    from gemm_epilogues_gb300.inputs import f16_tensor
    kind, prm = ROW_CASES[args.case]
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    line = {"case": args.case}
    if kind == "norm":
        M, N, K = D_DEC, prm["T"], D_DEC
        W = f16_tensor((M, K), 7001, "normal", 1 / 64, dev)
        X = f16_tensor((N, K), 7002, "normal", 1.0, dev)
        b = f16_tensor((M,), 7003, "normal", 0.1, dev)
        R = f16_tensor((N, M), 7004, "normal", 1.0, dev)
        g = f16_tensor((M,), 7005, "normal", 1.0, dev)
        be = f16_tensor((M,), 7006, "normal", 0.1, dev)
        H = torch.empty((N, M), dtype=torch.float16, device=dev)
        Y = torch.empty((N, M), dtype=torch.float16, device=dev)
        plan = ge.Plan(M, N, K, ge.EPILOGUE_BY_NAME[prm["norm"]],
                       ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL))
        run = lambda: plan.execute_norm(W, X, b, R, g, be, H, Y, 1e-5, stream, unfused=prm["unfused"])
        flops = 2.0 * M * N * K
        alg_bytes = 2 * (M * K + N * K + 3 * M * N) + 2 * 3 * M
        line["workload"] = f"out-proj {M}x{N}x{K} + bias + residual + {prm['norm']}"
    elif kind == "gelu_aux":
        M, N, K = D_OUT, T_TOK, D_IN
        W = f16_tensor((M, K), 7011, "normal", 1 / 64, dev)
        X = f16_tensor((N, K), 7012, "normal", 1.0, dev)
        b = f16_tensor((M,), 7013, "normal", 0.1, dev)
        Y = torch.empty((N, M), dtype=torch.float16, device=dev)
        Z = torch.empty((N, M), dtype=torch.float16, device=dev)
        plan = ge.Plan(M, N, K, ge.GE_EPI_GELU_AUX_BIAS, ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL))
        fn = plan.execute_unfused if prm["unfused"] else plan.execute
        run = lambda: fn(W, X, b, Y, Z, stream)
        flops = 2.0 * M * N * K
        alg_bytes = 2 * (M * K + N * K + 2 * M * N) + 2 * M
        line["workload"] = f"MLP fwd GELU_AUX_BIAS {M}x{N}x{K}"
    elif kind == "dw_drelu":
        # Weight gradient of the MLP layer from the incoming dY: fused (the
        # ReLU backward applied to the GEMM's A operand, bgrad in the same
        # pass) or the two-kernel flow (standalone DRELU_BGRAD storing dZ,
        # then the dW GEMM on it)
        M, N, K = D_OUT, D_IN, T_TOK
        dY = f16_tensor((K, M), 7041, "normal", 1.0, dev)
        Xw = f16_tensor((K, N), 7042, "normal", 1.0, dev)
        ld_aux = (M + 127) // 128 * 4
        gen = torch.Generator(device=dev)
        gen.manual_seed(7043)
        aux = torch.randint(-2**31, 2**31 - 1, (K * ld_aux,), generator=gen, device=dev, dtype=torch.int32)
        dW = torch.empty((M, N), dtype=torch.float16, device=dev)
        bgrad = torch.empty(M, dtype=torch.float32, device=dev)
        L = ge.make_layout(ge.GE_MN_MAJOR, ge.GE_MN_MAJOR, ge.GE_D_ROW)
        if prm["unfused"]:
            plan = ge.Plan(M, N, K, ge.GE_EPI_NONE, L)
            drelu = ge.Plan(M, K, 0, ge.GE_EPI_DRELU_BGRAD, ge.make_layout(d=ge.GE_D_COL))
            dZ = torch.empty_like(dY)

            def run():
                drelu.execute(dY, None, bgrad, dZ, aux, stream)
                plan.execute(dZ, Xw, None, dW, None, stream)
        else:
            plan = ge.Plan(M, N, K, ge.GE_EPI_DW_DRELU_BGRAD, L)
            drelu = None
            run = lambda: plan.execute(dY, Xw, bgrad, dW, aux, stream)
        flops = 2.0 * M * N * K
        alg_bytes = 2 * (M * K + K * N + M * N) + 4 * K * ld_aux + 4 * M
        line["workload"] = f"dW {M}x{N}x{K} from dY with the ReLU backward + bgrad"
    elif kind == "drelu_rows":
        # DRELU_BGRAD with a row-major D: dY[11008 features][8192 tokens], the
        # bias gradient a sum along each stored row
        M, N = D_OUT, T_TOK
        dY = f16_tensor((M, N), 7031, "normal", 1.0, dev)
        ld_aux = (N + 127) // 128 * 4
        gen = torch.Generator(device=dev)
        gen.manual_seed(7032)
        aux = torch.randint(-2**31, 2**31 - 1, (M * ld_aux,), generator=gen, device=dev, dtype=torch.int32)
        dZ = torch.empty((M, N), dtype=torch.float16, device=dev)
        bgrad = torch.empty(M, dtype=torch.float32, device=dev)
        plan = ge.Plan(M, N, 0, ge.GE_EPI_DRELU_BGRAD, ge.make_layout(d=ge.GE_D_ROW))
        run = lambda: plan.execute(dY, None, bgrad, dZ, aux, stream)
        flops = 0.0
        alg_bytes = 4 * M * N + 4 * M * ld_aux + 4 * M
        line["workload"] = f"DRELU_BGRAD row-major dY[{M},{N}]"
        drelu = None
    else:  # dgelu: standalone (K = 0) or as the backward GEMM's epilogue
        M, N = D_OUT, T_TOK
        K = prm["K"]
        Z = f16_tensor((N, M), 7021, "normal", 2.0, dev)
        dZ = torch.empty((N, M), dtype=torch.float16, device=dev)
        bgrad = torch.empty(M, dtype=torch.float32, device=dev)
        if K == 0:
            dY = f16_tensor((N, M), 7022, "normal", 1.0, dev)
            plan = ge.Plan(M, N, 0, ge.GE_EPI_DGELU_BGRAD, ge.make_layout(d=ge.GE_D_COL))
            run = lambda: plan.execute(dY, None, bgrad, dZ, Z, stream)
            flops = 0.0
            alg_bytes = 6 * M * N + 4 * M
            line["workload"] = f"DGELU_BGRAD dY[{N},{M}]"
            drelu = None
        else:
            G = f16_tensor((N, K), 7023, "normal", 1.0, dev)
            W2 = f16_tensor((M, K), 7024, "normal", 1 / 64, dev)
            Kl = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
            plan = ge.Plan(M, N, K, ge.GE_EPI_NONE if prm["unfused"] else ge.GE_EPI_DGELU_BGRAD, Kl)
            if prm["unfused"]:
                drelu = ge.Plan(M, N, 0, ge.GE_EPI_DGELU_BGRAD, ge.make_layout(d=ge.GE_D_COL))

                def run():
                    plan.execute(W2, G, None, dZ, None, stream)
                    drelu.execute(dZ, None, bgrad, dZ, Z, stream)
            else:
                drelu = None
                run = lambda: plan.execute(W2, G, bgrad, dZ, Z, stream)
            flops = 2.0 * M * N * K
            alg_bytes = 2 * (M * K + N * K + 2 * M * N) + 4 * M
            line["workload"] = f"backward GEMM {M}x{N}x{K} + DGELU_BGRAD"
    times = _time_flushed(run, args.steps, args.warmup, dev)
    assert ge.ge_get_last_device_error(plan.handle) == ge.GE_OK
    ms = sum(times) / len(times)
    line.update({"ms": ms, "min_ms": min(times), "gbs_algorithmic": alg_bytes / (ms * 1e-3) / 1e9,
                 "hbm_frac_of_peak": alg_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]})
    if flops:
        line.update({"tflops": flops / (ms * 1e-3) / 1e12, "frac_of_peak": flops / (ms * 1e-3) / 1e12 / peaks["tflops"]})
    plan.free()
    if kind in ("dgelu", "drelu_rows", "dw_drelu") and drelu is not None:
        drelu.free()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_bwd_gemm_drelu(args, rank, unfused):
    """dH[8192 tokens, 11008] = G[8192, 4096] W2[11008, 4096]^T masked by the
    forward ReLU mask: fused (one GEMM with the DRELU_BGRAD epilogue) or
    unfused (GEMM with no epilogue, then the standalone DRELU_BGRAD pass)."""
    import torch
    import gemm_epilogues_gb300 as ge
    from gemm_epilogues_gb300.inputs import f16_tensor
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    M, N, K = D_OUT, T_TOK, D_IN
    G = f16_tensor((N, K), 6001, "normal", 1.0, dev)
    W2 = f16_tensor((M, K), 6002, "normal", 1 / 64, dev)
    ld_aux = (M + 127) // 128 * 4
    g = torch.Generator(device=dev)
    g.manual_seed(6003)
    aux = torch.randint(-2**31, 2**31 - 1, (N * ld_aux,), generator=g, device=dev, dtype=torch.int32)
    dZ = torch.empty((N, M), dtype=torch.float16, device=dev)
    bgrad = torch.empty(M, dtype=torch.float32, device=dev)
    Kl = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    gemm = ge.Plan(M, N, K, ge.GE_EPI_NONE if unfused else ge.GE_EPI_DRELU_BGRAD, Kl)
    drelu = ge.Plan(M, N, 0, ge.GE_EPI_DRELU_BGRAD, ge.make_layout(d=ge.GE_D_COL)) if unfused else None
    flush_buf = torch.ones((256 << 20) // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    times = []
    for i in range(args.warmup + args.steps):
        torch.sum(flush_buf, dim=0, out=flush_out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if unfused:
            gemm.execute(W2, G, None, dZ, None, stream)
            drelu.execute(dZ, None, bgrad, dZ, aux, stream)
        else:
            gemm.execute(W2, G, bgrad, dZ, aux, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    assert ge.ge_get_last_device_error(gemm.handle) == ge.GE_OK
    ms = sum(times) / len(times)
    flops = 2.0 * M * N * K
    line = {"case": args.case, "workload": "backward GEMM 11008x8192x4096 + DRELU_BGRAD",
            "unfused": unfused, "ms": ms, "min_ms": min(times), "tflops": flops / ms / 1e9,
            "frac_of_peak": flops / ms / 1e9 / peaks["tflops"]}
    gemm.free()
    if drelu:
        drelu.free()
    if rank == 0:
        print(json.dumps(line), flush=True)


# Every workload config, timed alone: key -> (workload key, dtype)
CONFIG_TABLE = (("cfg_c1", "c1"), ("cfg_c2_bias", "c2_bias"), ("cfg_c2_relu_bias", "c2_relu_bias"),
                ("cfg_c2_gelu_bias", "c2_gelu_bias"), ("cfg_c3_T1", "c3_T1"), ("cfg_c3_T512", "c3_T512"),
                ("cfg_c3_T2048", "c3_T2048"), ("cfg_c4_fwd", "c4_fwd"), ("cfg_c4_bwd", "c4_bwd"),
                ("cfg_c4_dw", "c4_dw"), ("cfg_c5", "c5"))
# configs whose launch lasts microseconds: their per-launch event time holds
# the launch and event overhead, so the device time is also taken from CUDA
# graph replays
_MICRO = ("cfg_c1", "cfg_c2_bias", "cfg_c2_relu_bias", "cfg_c2_gelu_bias", "cfg_c3_T1", "cfg_c3_T512",
          "cfg_c3_T2048")


def _pct(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, max(0, int(math.ceil(q * len(xs))) - 1))]


def _graph_device_ms(run, flush_fn, reps, rounds=5):
    """Device time of one `run()` from CUDA graph replays: a graph of `reps`
    (flush, run) pairs minus a graph of `reps` flushes, per run; the median of
    `rounds` replays. None if capture fails."""
    import torch
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):  # warm the captured calls outside capture
            flush_fn()
            run()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g_both, g_flush = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_both):
            for _ in range(reps):
                flush_fn()
                run()
        with torch.cuda.graph(g_flush):
            for _ in range(reps):
                flush_fn()
        torch.cuda.synchronize()
    except Exception:
        torch.cuda.synchronize()
        return None
    stream = torch.cuda.current_stream()
    out = []
    for _ in range(rounds):
        t = []
        for g in (g_both, g_flush):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g.replay()  # warm
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            t.append(e0.elapsed_time(e1))
        out.append((t[0] - t[1]) / reps)
    del g_both, g_flush
    return statistics.median(out)


def run_config_table(dev, peaks, flush, keep_cpu_inputs=False, gpu_index=0):
    """Every workload config alone on this GPU: per-launch CUDA-event times
    after an L2 flush (median and p90 over >= 50 launches after 10 warm-ups;
    the 17.6-TFLOP config 5 over 10), the SM clock and throttle reasons
    sampled during each config's timed launches, the roofline of each config
    (the faster of the burst tensor peak and its bytes at the copy rate; a
    tensor-bound config also gets its fraction of the sustained peak), the
    same engine's unfused three-kernel sequence, and for microsecond launches
    the device time from graph replays. Returns (entries, cpu_inputs) where
    cpu_inputs are host copies of the inputs the oracle baselines use."""
    import torch
    import gemm_epilogues_gb300 as ge
    from gemm_epilogues_gb300.inputs import f16_tensor, pages_workloads, sample_rows
    stream = torch.cuda.current_stream()
    works = pages_workloads()
    major = {"k": ge.GE_K_MAJOR, "m": ge.GE_MN_MAJOR, "n": ge.GE_MN_MAJOR}
    tpk = peaks["tflops"] * 1e12  # burst: each config is timed alone, briefly
    hbm = peaks["hbm_gbs"] * 1e9
    out, cpu_in = {}, {}

    last_clocks = {}

    def timed(fn, warm, reps, sample=False):
        ts = []
        cs = ClockSampler(gpu_index, 20) if sample else None
        for i in range(warm + reps):
            if cs is not None and i == warm:
                cs.start()
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= warm:
                ts.append(e0.elapsed_time(e1))
        if cs is not None:
            last_clocks.clear()
            last_clocks.update(cs.stop())
        return ts

    for key, wk in CONFIG_TABLE:
        big = key == "cfg_c5"
        warm, reps = (3, 10) if big else (10, 50)
        if wk == "c4_bwd":
            # DRELU_BGRAD on dY[8192 tokens, 11008]: mask words drawn at random
            M, N = D_OUT, T_TOK
            dY = f16_tensor((N, M), 3004, "normal", 1.0, dev)
            ld_aux = (M + 127) // 128 * 4
            gen = torch.Generator(device=dev)
            gen.manual_seed(3005)
            aux = torch.randint(-2**31, 2**31 - 1, (N * ld_aux,), generator=gen, device=dev, dtype=torch.int32)
            dZ = torch.empty_like(dY)
            bgrad = torch.empty(M, dtype=torch.float32, device=dev)
            plan = ge.Plan(M, N, 0, ge.GE_EPI_DRELU_BGRAD, ge.make_layout(d=ge.GE_D_COL))
            run = lambda: plan.execute(dY, None, bgrad, dZ, aux, stream)
            ts = timed(run, warm, reps, sample=True)
            assert ge.ge_get_last_device_error(plan.handle) == ge.GE_OK
            nbytes = 2 * N * M * 2 + 4 * N * ld_aux + 4 * M
            med = statistics.median(ts)
            out[key] = {"workload": f"DRELU_BGRAD dY[{N},{M}] + mask -> dZ, fp32 bgrad[{M}]", "path": "drelu",
                        "ms": med, "p90_ms": _pct(ts, 0.9), "reps": reps, "gbs": nbytes / (med * 1e-3) / 1e9,
                        "algorithmic_bytes": nbytes, "bound": "hbm",
                        "frac_of_roofline": nbytes / hbm / (med * 1e-3), "roofline_gbs": peaks["hbm_gbs"],
                        "clocks": dict(last_clocks)}
            if keep_cpu_inputs:
                cpu_in[key] = (dY.cpu(), aux.cpu(), M, N, ld_aux)
            plan.free()
            del dY, aux, dZ, bgrad
            continue
        w = works[wk]
        A, B, bias = w.make(dev)
        L = ge.make_layout(major[w.a_major], major[w.b_major],
                           ge.GE_D_ROW if w.d_layout == "row" else ge.GE_D_COL)
        plan = ge.Plan(w.M, w.N, w.K, ge.EPILOGUE_BY_NAME[w.epilogue], L)
        if plan.path == ge.GE_PATH_GEMV:
            plan.set_attr(ge.GE_ATTR_STATIC_A, 1)  # decode weights: never written upstream
        D = torch.empty(w.d_shape(), dtype=A.dtype, device=dev)
        aux = torch.empty(max(plan.aux_bytes // 4, 1), dtype=torch.int32, device=dev)
        bias_arg = bias if w.epilogue != "none" else None
        aux_arg = aux if w.epilogue == "relu_aux_bias" else None
        # (the stream is looked up at each call: graph capture runs on its own)
        run = lambda: plan.execute(A, B, bias_arg, D, aux_arg, torch.cuda.current_stream())
        ts = timed(run, warm, reps, sample=True)
        assert ge.ge_get_last_device_error(plan.handle) == ge.GE_OK
        med = statistics.median(ts)
        flops, nbytes = w.flops, w.algorithmic_bytes()
        t_roof = max(flops / tpk, nbytes / hbm)
        path, tile_n, pair, split = plan.config
        e = {"workload": w.name, "path": {ge.GE_PATH_GEMV: "gemv", ge.GE_PATH_TC_GEMM: "tcgen05"}.get(path, path),
             "tile_n": tile_n, "pair": pair, "split": split,
             "ms": med, "p90_ms": _pct(ts, 0.9), "min_ms": min(ts), "reps": reps,
             "tflops": flops / (med * 1e-3) / 1e12, "gbs": nbytes / (med * 1e-3) / 1e9,
             "flops": flops, "algorithmic_bytes": nbytes,
             "bound": "hbm" if nbytes / hbm > flops / tpk else "tensor",
             "roofline_tflops": flops / t_roof / 1e12, "frac_of_roofline": t_roof / (med * 1e-3),
             "frac_of_tensor_peak": flops / (med * 1e-3) / tpk,
             "clocks": dict(last_clocks)}
        if e["bound"] == "tensor":
            e["frac_of_sustained_peak"] = flops / (med * 1e-3) / (peaks["tflops_sustained"] * 1e12)
        if key in _MICRO:
            g = _graph_device_ms(run, flush.zero_, 20)
            if g is not None and g > 0:
                e["graph_device_ms"] = g
                e["graph_frac_of_roofline"] = t_roof / (g * 1e-3)
        if w.epilogue != "none":
            urun = lambda: plan.execute_unfused(A, B, bias_arg, D, aux_arg, torch.cuda.current_stream())
            uts = timed(urun, 2 if big else 5, 5 if big else 30)
            assert ge.ge_get_last_device_error(plan.handle) == ge.GE_OK
            e["unfused_ms"] = statistics.median(uts)
            e["fused_speedup"] = e["unfused_ms"] / med
        out[key] = e
        if keep_cpu_inputs:
            # inputs of the oracle baseline: whole problems up to config 3,
            # 256 sampled stored rows of D for the others
            if wk in ("c4_fwd", "c4_dw", "c5"):
                rows_total = w.N if w.d_layout == "col" else w.M
                idx = torch.as_tensor(sample_rows(rows_total, 256), device=dev)
                if wk == "c4_fwd":  # stored rows = tokens = rows of X
                    cpu_in[key] = ("sample", A.cpu(), B.index_select(0, idx).cpu(), bias.cpu(), w, rows_total)
                elif wk == "c4_dw":  # stored rows = features = columns of the M-major A
                    cpu_in[key] = ("sample", A.index_select(1, idx).contiguous().cpu(), B.cpu(),
                                   None, w, rows_total)
                else:  # stored rows = rows of A
                    cpu_in[key] = ("sample", A.index_select(0, idx).cpu(), B.cpu(),
                                   bias.index_select(0, idx).cpu(), w, rows_total)
            else:
                cpu_in[key] = ("full", A.cpu(), B.cpu(), bias.cpu(), w, None)
        plan.free()
        del A, B, bias, D, aux
        torch.cuda.empty_cache()
    return out, cpu_in


def oracle_config_baselines(cpu_in):
    """The oracle (fp64, the host's cores) on each config: whole problems for
    configs 1-3 and the DRELU_BGRAD pass, 256 sampled rows of D for the
    config-4 GEMMs and config 5 (the rate scaled to the whole problem by the
    ratio of rows, which the oracle's row-parallel loop makes linear)."""
    import numpy as np
    import torch
    from oracle import oracle
    oracle.build()
    thr = os.cpu_count() or 1
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    out = {}
    for key, v in cpu_in.items():
        if key == "cfg_c4_bwd":
            dY, aux, M, N, ld_aux = v
            dyb, auxw = bits(dY), aux.numpy().view(np.uint32)
            t0 = time.perf_counter()
            oracle.drelu_bgrad(dyb, auxw, M, N, d_layout="col", ld_aux=ld_aux)
            dt = time.perf_counter() - t0
            nbytes = 2 * N * M * 2 + 4 * N * ld_aux + 4 * M
            out[key] = {"gbs": nbytes / dt / 1e9, "s": dt, "sample": "whole problem", "threads": 1}
            continue
        kind, A, B, bias, w, rows_total = v
        Ab, Bb = bits(A), bits(B)
        bb = None if bias is None else bits(bias)
        M, N = w.M, w.N
        if kind == "sample":  # the sampled stored rows of D
            if w.d_layout == "col":
                N = B.shape[0] if w.b_major == "k" else B.shape[1]
            else:
                M = A.shape[1] if w.a_major == "m" else A.shape[0]
        n_s = N if w.d_layout == "col" else M
        t0 = time.perf_counter()
        oracle.linear_forward(Ab, Bb, bb, w.epilogue, M, N, w.K, a_major=w.a_major, b_major=w.b_major,
                              d_layout=w.d_layout, threads=thr)
        dt = time.perf_counter() - t0
        flops = 2.0 * M * N * w.K
        e = {"tflops": flops / dt / 1e12, "s": dt, "threads": thr,
             "sample": "whole problem" if kind == "full" else f"{n_s} of {rows_total} stored rows of D"}
        if kind == "sample":
            e["extrapolated_s"] = dt * rows_total / n_s
        out[key] = e
    return out


def run_ours(args, world, rank, local):
    import torch
    import gemm_epilogues_gb300 as ge
    from gemm_epilogues_gb300.inputs import f16_tensor

    ge.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    stream = torch.cuda.current_stream()

    # weights and inputs, resident in HBM
    W = f16_tensor((D_OUT, D_IN), 3001, "normal", 1 / 64, dev)
    X = f16_tensor((T_TOK, D_IN), 3002, "normal", 1.0, dev)
    b = f16_tensor((D_OUT,), 3003, "normal", math.sqrt(0.02), dev)
    dY = f16_tensor((T_TOK, D_OUT), 3004, "normal", 1.0, dev)
    W2 = f16_tensor((D_DEC, D_DEC), 2001, "normal", 1 / 64, dev)
    b2 = f16_tensor((D_DEC,), 2003, "normal", math.sqrt(0.02), dev)
    x1 = f16_tensor((1, D_DEC), 2002, "normal", 1.0, dev)

    K_, MN = ge.GE_K_MAJOR, ge.GE_MN_MAJOR
    fwd = ge.Plan(D_OUT, T_TOK, D_IN, ge.GE_EPI_RELU_AUX_BIAS, ge.make_layout(K_, K_, ge.GE_D_COL))
    bwd = ge.Plan(D_OUT, T_TOK, 0, ge.GE_EPI_DRELU_BGRAD, ge.make_layout(d=ge.GE_D_COL))
    dwp = ge.Plan(D_OUT, D_IN, T_TOK, ge.GE_EPI_NONE, ge.make_layout(MN, MN, ge.GE_D_ROW))
    dec = ge.Plan(D_DEC, 1, D_DEC, ge.GE_EPI_GELU_BIAS, ge.make_layout(K_, K_, ge.GE_D_COL))
    assert dec.path == ge.GE_PATH_GEMV
    dec.set_attr(ge.GE_ATTR_STATIC_A, 1)  # decode weights are never written by earlier work

    def _launches(p):  # kernels one execute launches: the GEMM, and the fixup of a split-K tail
        path, _, _, split = p.config
        return 2 if path == ge.GE_PATH_TC_GEMM and split > 1 else 1

    launches_per_step = _launches(fwd) + 1 + _launches(dwp) + 1  # + DRELU_BGRAD + GEMV

    Y = torch.empty((T_TOK, D_OUT), dtype=torch.float16, device=dev)
    aux = torch.empty(fwd.aux_bytes // 4, dtype=torch.int32, device=dev)
    dZ = torch.empty_like(dY)
    bgrad = torch.empty(D_OUT, dtype=torch.float32, device=dev)
    dW = torch.empty((D_OUT, D_IN), dtype=torch.float16, device=dev)
    y1 = torch.empty((1, D_DEC), dtype=torch.float16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size if hasattr(
        torch.cuda.get_device_properties(dev), "L2_cache_size") else 128 << 20
    # L2 flush between timed launches: a read-only pass over 2x L2 leaves L2
    # full of clean lines (a memset would leave dirty lines whose write-back
    # then competes with the next kernel's reads).
    flush_buf = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    class _Flush:
        @staticmethod
        def zero_():
            torch.sum(flush_buf, dim=0, out=flush_out)

    flush = _Flush()

    names = ["fwd_gemm_relu_aux_bias", "drelu_bgrad", "dw_gemm", "decode_gemv_gelu_bias"]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fwd.execute(W, X, b, Y, aux, stream)
        if ev is not None:
            ev[1].record(stream)
        bwd.execute(dY, None, bgrad, dZ, aux, stream)
        if ev is not None:
            ev[2].record(stream)
        dwp.execute(dZ, X, None, dW, None, stream)
        if ev is not None:
            ev[3].record(stream)
        dec.execute(W2, x1, b2, y1, None, stream)
        if ev is not None:
            ev[4].record(stream)

    if args.case != "step":
        # Profiling mode: only one kernel of the step, `steps` times after
        # `warmup` launches (each launch preceded by the L2 flush).
        if args.case == "chain":  # the 32-layer decode stack of the bench line
            Wc = [f16_tensor((D_DEC, D_DEC), 2200 + i, "normal", 1 / 64, dev) for i in range(32)]
            bc = [f16_tensor((D_DEC,), 2300 + i, "normal", math.sqrt(0.02), dev) for i in range(32)]
            Yc = torch.empty((32, 1, D_DEC), dtype=torch.float16, device=dev)
            chain = ge.Plan(D_DEC, 1, D_DEC, ge.GE_EPI_GELU_BIAS, ge.make_layout(K_, K_, ge.GE_D_COL))
        one = {"fwd": lambda: fwd.execute(W, X, b, Y, aux, stream),
               "chain": lambda: chain.execute_chain(Wc, bc, x1, Yc, stream),
               "fwd_unfused": lambda: fwd.execute_unfused(W, X, b, Y, aux, stream),
               "bwd": lambda: bwd.execute(dY, None, bgrad, dZ, aux, stream),
               "dw": lambda: dwp.execute(dZ, X, None, dW, None, stream),
               "gemv": lambda: dec.execute(W2, x1, b2, y1, None, stream)}[args.case]
        times = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            one()
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                times.append(e0.elapsed_time(e1))
        for p in (fwd, bwd, dwp, dec):
            assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        if rank == 0:
            print(json.dumps({"case": args.case, "ms": sum(times) / len(times), "min_ms": min(times),
                              "launches": args.steps}), flush=True)
        return

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    for p in (fwd, bwd, dwp, dec):
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()  # L2 flushed between timed steps, outside the events
        step(evs[k])
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    for p in (fwd, bwd, dwp, dec):
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK

    per = {n: [] for n in names}
    tot = []
    for e in evs:
        for i, n in enumerate(names):
            per[n].append(e[i].elapsed_time(e[i + 1]))
        tot.append(e[0].elapsed_time(e[4]))
    ms_step_local = sum(tot) / len(tot)
    ms_step = reduce_max(ms_step_local, world)

    flops_gemm = 2.0 * D_OUT * T_TOK * D_IN
    flops_dec = 2.0 * D_DEC * D_DEC
    flops_step = 2 * flops_gemm + flops_dec
    value = flops_step * world / (ms_step * 1e-3) / 1e12

    aux_bytes = fwd.aux_bytes
    bytes_fwd = 2 * (D_OUT * D_IN + T_TOK * D_IN + T_TOK * D_OUT) + 2 * D_OUT + aux_bytes
    bytes_bwd = 2 * T_TOK * D_OUT * 2 + aux_bytes + 4 * D_OUT
    bytes_dw = 2 * (T_TOK * D_OUT + T_TOK * D_IN + D_OUT * D_IN)
    bytes_dec = 2 * (D_DEC * D_DEC + D_DEC + D_DEC + D_DEC)
    mean = {n: sum(v) / len(v) for n, v in per.items()}
    kern = {
        "fwd_gemm_relu_aux_bias": {"ms": mean[names[0]], "tflops": flops_gemm / mean[names[0]] / 1e9},
        "drelu_bgrad": {"ms": mean[names[1]], "gbs": bytes_bwd / mean[names[1]] / 1e6},
        "dw_gemm": {"ms": mean[names[2]], "tflops": flops_gemm / mean[names[2]] / 1e9},
        "decode_gemv_gelu_bias": {"ms": mean[names[3]], "gbs": bytes_dec / mean[names[3]] / 1e6},
    }
    for k in ("fwd_gemm_relu_aux_bias", "dw_gemm"):
        kern[k]["frac_of_peak"] = kern[k]["tflops"] / peaks["tflops"]
        kern[k]["frac_of_sustained_peak"] = kern[k]["tflops"] / peaks["tflops_sustained"]
    for k in ("drelu_bgrad", "decode_gemv_gelu_bias"):
        kern[k]["frac_of_peak"] = kern[k]["gbs"] / peaks["hbm_gbs"]
    kern["fwd_gemm_relu_aux_bias"]["algorithmic_bytes"] = bytes_fwd
    kern["drelu_bgrad"]["algorithmic_bytes"] = bytes_bwd
    kern["dw_gemm"]["algorithmic_bytes"] = bytes_dw
    kern["decode_gemv_gelu_bias"]["algorithmic_bytes"] = bytes_dec
    # What two events around one tiny launch (a one-element fill) read on
    # this stream: the part of a single microsecond-scale launch's time that
    # is launch and event overhead rather than the kernel's work.
    tiny = torch.empty(1, dtype=torch.float32, device=dev)
    floor = []
    with torch.cuda.stream(stream):
        for _ in range(25):
            flush.zero_()
            f0 = torch.cuda.Event(enable_timing=True)
            f1 = torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            tiny.zero_()
            f1.record(stream)
            f1.synchronize()
            floor.append(f0.elapsed_time(f1))
    kern["decode_gemv_gelu_bias"]["event_launch_floor_ms"] = sorted(floor[5:])[len(floor[5:]) // 2]
    dominant = max(("fwd_gemm_relu_aux_bias", "dw_gemm"), key=lambda k: kern[k]["ms"])
    achieved = kern[dominant]["tflops"]
    # Which measured peak applies follows from this run's own clock record:
    # the sustained figure (a seconds-long loop under the power cap) only
    # when the timed region itself lasted seconds and the power cap was seen
    # in it; otherwise the burst figure.
    timed_s = sum(tot) * 1e-3
    peak, sustained, capped = choose_tensor_peak(peaks, timed_s, clk)
    traffic = captured_traffic(dominant)
    roofline = {"bound": "tensor", "kernel": dominant, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, from the "
                                   "committed capture of the same kernel source" if traffic else
                                   "none: the kernel source changed since the last capture"),
                "peak_source": (f"{peaks['source']} bf16 {'sustained' if sustained else 'burst'} "
                                f"(fp16 tensor rate = bf16; timed region {timed_s:.3f} s, "
                                f"sw_power_cap {'seen' if capped else 'not seen'})"),
                "burst_peak": peaks["tflops"], "sustained_peak": peaks["tflops_sustained"],
                "frac_of_burst": achieved / peaks["tflops"],
                "frac_of_sustained": achieved / peaks["tflops_sustained"]}

    # ---- baselines and the back-to-back decode measurement (outside the step)
    # (1) the unfused three-kernel sequence on the forward's inputs
    ut = []
    for i in range(8):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fwd.execute_unfused(W, X, b, Y, aux, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            ut.append(e0.elapsed_time(e1))
    fwd.execute(W, X, b, Y, aux, stream)  # leave the fused result in Y
    unf_ms = sum(ut) / len(ut)
    kern["fwd_unfused_baseline"] = {"ms": unf_ms, "tflops": flops_gemm / unf_ms / 1e9,
                                    "frac_of_peak": flops_gemm / unf_ms / 1e9 / peaks["tflops"],
                                    "fused_speedup": unf_ms / kern["fwd_gemm_relu_aux_bias"]["ms"]}
    # (2) decode GEMV launched back to back over 8 weight copies (268 MB, more
    # than L2), the pattern of a decode step through several layers
    # The launches are captured in a CUDA graph so the host (Python + ctypes)
    # does not pace them; one plan per weight copy keeps the pointer checks
    # out of the capture.
    W2s = [W2] + [f16_tensor((D_DEC, D_DEC), 2100 + i, "normal", 1 / 64, dev) for i in range(7)]
    decs = [ge.Plan(D_DEC, 1, D_DEC, ge.GE_EPI_GELU_BIAS, ge.make_layout(K_, K_, ge.GE_D_COL)) for _ in W2s]
    for pl in decs:
        pl.set_attr(ge.GE_ATTR_STATIC_A, 1)
    for pl, Wi in zip(decs, W2s):
        pl.execute(Wi, x1, b2, y1, None, stream)
    torch.cuda.synchronize()
    rounds = 6
    graph_ok = True
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for pl, Wi in zip(decs, W2s):
                pl.execute(Wi, x1, b2, y1, None, cs)
        g.replay()
        torch.cuda.synchronize()
    except Exception:
        graph_ok = False
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(rounds):
        if graph_ok:
            g.replay()
        else:
            for pl, Wi in zip(decs, W2s):
                pl.execute(Wi, x1, b2, y1, None, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    b2b_ms = e0.elapsed_time(e1) / (rounds * len(W2s))
    for pl in decs:
        assert ge.ge_get_last_device_error(pl.handle) == ge.GE_OK
        pl.free()
    kern["decode_gemv_back_to_back"] = {"ms": b2b_ms, "gbs": bytes_dec / b2b_ms / 1e6,
                                        "frac_of_peak": bytes_dec / b2b_ms / 1e6 / peaks["hbm_gbs"],
                                        "launches": rounds * len(W2s), "weights": "8 x 33.5 MB rotating",
                                        "cuda_graph": graph_ok}
    del W2s
    # (3) a stack of decode projections in one launch (ge_execute_chain):
    # 32 layers of 4096 x 4096 (1.07 GB of weights, far more than L2), each
    # layer's output the next layer's input, L2 flushed before each launch
    CH = 32
    Wc = [f16_tensor((D_DEC, D_DEC), 2200 + i, "normal", 1 / 64, dev) for i in range(CH)]
    bc = [f16_tensor((D_DEC,), 2300 + i, "normal", math.sqrt(0.02), dev) for i in range(CH)]
    Yc = torch.empty((CH, 1, D_DEC), dtype=torch.float16, device=dev)
    chain = ge.Plan(D_DEC, 1, D_DEC, ge.GE_EPI_GELU_BIAS, ge.make_layout(K_, K_, ge.GE_D_COL))
    ct = _time_flushed(lambda: chain.execute_chain(Wc, bc, x1, Yc, stream), 10, 3, dev)
    assert ge.ge_get_last_device_error(chain.handle) == ge.GE_OK
    chain.free()
    ch_ms = statistics.median(ct) / CH
    kern["decode_gemv_chain"] = {"ms": ch_ms, "gbs": bytes_dec / ch_ms / 1e6,
                                 "frac_of_peak": bytes_dec / ch_ms / 1e6 / peaks["hbm_gbs"],
                                 "layers_per_launch": CH, "launches": len(ct),
                                 "launch_ms_median": statistics.median(ct),
                                 "weights": f"{CH} x 33.5 MB, one cooperative launch, L2 flushed before each"}
    del Wc, bc, Yc
    assert ge.ge_get_last_device_error(dec.handle) == ge.GE_OK
    assert ge.ge_get_last_device_error(fwd.handle) == ge.GE_OK

    # ---- end to end through the public API: host buffers, copies timed.
    # Every step copies its inputs (X, dY, x) from pinned host memory and reads
    # its results (dW, bgrad, y) back. The copies of step i+1's inputs and the
    # read-back of step i's results run on their own streams while step i
    # computes (double-buffered device inputs and outputs), so the step is
    # bound by max(compute, copies) instead of their sum.
    bias_fwd = b
    Xh = X.cpu().pin_memory()
    dYh = dY.cpu().pin_memory()
    x1h = x1.cpu().pin_memory()
    e_steps = max(3, min(args.steps, 50))
    dWh = [torch.empty(dW.shape, dtype=dW.dtype).pin_memory() for _ in range(2)]
    bgh = [torch.empty(bgrad.shape, dtype=bgrad.dtype).pin_memory() for _ in range(2)]
    y1h = [torch.empty(y1.shape, dtype=y1.dtype).pin_memory() for _ in range(2)]
    Xd = [torch.empty_like(X) for _ in range(2)]
    dYd = [torch.empty_like(dY) for _ in range(2)]
    x1d = [torch.empty_like(x1) for _ in range(2)]
    dWd = [dW, torch.empty_like(dW)]
    bgd = [bgrad, torch.empty_like(bgrad)]
    y1d = [y1, torch.empty_like(y1)]
    h2d_s = torch.cuda.Stream()
    d2h_s = torch.cuda.Stream()

    def run_e2e(nsteps):
        h2d_s.wait_stream(stream)  # copies start after the timing event
        in_ready = [torch.cuda.Event() for _ in range(2)]
        in_free = [torch.cuda.Event() for _ in range(2)]
        out_ready = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):
            in_free[b].record(stream)
            out_free[b].record(d2h_s)

        def issue_h2d(i):
            b = i & 1
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(in_free[b])
                Xd[b].copy_(Xh, non_blocking=True)
                dYd[b].copy_(dYh, non_blocking=True)
                x1d[b].copy_(x1h, non_blocking=True)
                in_ready[b].record(h2d_s)

        issue_h2d(0)
        for i in range(nsteps):
            b = i & 1
            if i + 1 < nsteps:
                issue_h2d(i + 1)
            stream.wait_event(in_ready[b])
            stream.wait_event(out_free[b])
            fwd.execute(W, Xd[b], bias_fwd, Y, aux, stream)
            bwd.execute(dYd[b], None, bgd[b], dZ, aux, stream)
            dwp.execute(dZ, Xd[b], None, dWd[b], None, stream)
            dec.execute(W2, x1d[b], b2, y1d[b], None, stream)
            in_free[b].record(stream)
            out_ready[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(out_ready[b])
                dWh[b].copy_(dWd[b], non_blocking=True)
                bgh[b].copy_(bgd[b], non_blocking=True)
                y1h[b].copy_(y1d[b], non_blocking=True)
                out_free[b].record(d2h_s)
        stream.wait_stream(d2h_s)

    h2d = Xh.numel() * 2 + dYh.numel() * 2 + x1h.numel() * 2
    d2h = dWh[0].numel() * 2 + bgh[0].numel() * 4 + y1h[0].numel() * 2
    run_e2e(2)
    torch.cuda.synchronize()
    # three timed runs of e_steps steps each; the median is reported, so one
    # host-side stall (the copies are issued from Python) does not decide it
    e2e_runs = []
    for _ in range(3):
        barrier(world)
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        run_e2e(e_steps)
        ev1.record(stream)
        torch.cuda.synchronize()
        e2e_runs.append(ev0.elapsed_time(ev1) / e_steps)
    barrier(world)
    e2e_ms = reduce_max(sorted(e2e_runs)[1], world)
    e2e_value = flops_step * world / (e2e_ms * 1e-3) / 1e12
    # results of the last step reached the host and equal the device values
    last = (e_steps - 1) & 1
    assert torch.equal(dWh[last], dWd[last].cpu()) and torch.equal(bgh[last], bgd[last].cpu())

    # The same copies with no compute: the host link's own time per step
    # (both directions at once), the floor under the end-to-end number.
    def run_copies(nsteps):
        h2d_s.wait_stream(stream)
        d2h_s.wait_stream(stream)
        for i in range(nsteps):
            b = i & 1
            with torch.cuda.stream(h2d_s):
                Xd[b].copy_(Xh, non_blocking=True)
                dYd[b].copy_(dYh, non_blocking=True)
                x1d[b].copy_(x1h, non_blocking=True)
            with torch.cuda.stream(d2h_s):
                dWh[b].copy_(dWd[b], non_blocking=True)
                bgh[b].copy_(bgd[b], non_blocking=True)
                y1h[b].copy_(y1d[b], non_blocking=True)
        stream.wait_stream(h2d_s)
        stream.wait_stream(d2h_s)

    run_copies(1)
    torch.cuda.synchronize()
    ev0.record(stream)
    run_copies(e_steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    link_ms = reduce_max(ev0.elapsed_time(ev1) / e_steps, world)

    # ---- every workload config alone (one GPU; replicas skip it)
    configs, cfg_cpu_in = None, {}
    if world == 1 and not args.no_configs:
        configs, cfg_cpu_in = run_config_table(dev, peaks, flush, keep_cpu_inputs=not args.no_cpu_baseline,
                                               gpu_index=local)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rows = 4096
        rate, dt, thr = oracle_sample_rate(rows)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"forward GEMM on {rows} of {T_TOK} tokens (all 11008 outputs, K=4096), "
                         f"{dt:.1f} s wall"}
        if cfg_cpu_in:
            cpu["configs"] = oracle_config_baselines(cfg_cpu_in)
            cfg_cpu_in = None

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f16 (fp32 accumulate)", "data": "synthetic",
                "config": {"workload": WORKLOAD, "tokens": T_TOK, "d_in": D_IN, "d_out": D_OUT,
                           "decode_hidden": D_DEC, "l2": "flushed between timed steps (read-only pass over 2x L2)",
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "kernels": kern, "configs": configs, "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "overlap": "inputs of step i+1 copied and results of step i read back on "
                                   "their own streams while step i computes",
                        "copies_only_ms_per_step": link_ms,
                        "runs_ms_per_step": e2e_runs, "of_runs": "median"},
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clk}
        print(json.dumps(line), flush=True)
    for p in (fwd, bwd, dwp, dec):
        p.free()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the table of every workload config")
    ap.add_argument("--case", default="step",
                    choices=["step", "fwd", "bwd", "dw", "gemv", "fwd_unfused", "chain"] + sorted(CONFIG_CASES)
                    + sorted(ROW_CASES),
                    help="time one kernel of the step alone, or one of the workload configs")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.case in CONFIG_CASES:
            run_config(args, rank)
        elif args.case in ROW_CASES:
            run_row_case(args, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

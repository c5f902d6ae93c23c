"""Throughput of the fused dense layer on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one call of the hot path over one batch of synthetic input. The
default workload is the fused RMSNorm -> linear layer in fp16 with
x[512, 4096], gamma[4096], eps 1e-6 and W[4096, 4096], no bias (the shape of
the LLMBoost fused_rmsnorm_linear benchmark). Inputs rotate over enough copies
to exceed the 129 MB L2 between steps, so every step reads its operands from
HBM.

--impl ours (default): the CUDA path through the C ABI; `value` is device
throughput with inputs resident in HBM; `e2e` repeats it through the same
call with pinned host buffers, host<->device copies inside the timed region.
--impl reference: the float64 CPU oracle on the host cores, one bounded
sample of the workload per step.

With torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); the time is the maximum over ranks and the
value counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-kernel TFLOP/s & % of GB300 tensor peak; GB/s vs HBM at decode shapes"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The pages' own number for this exact workload: fused RMSNorm -> Linear,
# [512,4096] x [4096,4096] fp16, 0.208 ms on an A30 (LLMBoost benchmark table).
PAGE_FUSED_MS = 0.208


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
WORKLOADS = {
    "rmsnorm_gemm_f16_512x4096x4096": dict(kind="norm", norm="rms", dtype="f16", M=512, N=4096, K=4096, eps=1e-6),
    "gemm_bias_gelu_f16_512x1024x1024": dict(kind="pattern", pattern="gemm_bias_gelu", dtype="f16", M=512, N=1024,
                                             K=1024),
    "swiglu_ffn_bf16_4096x4096x11008": dict(kind="swiglu", dtype="bf16", M=4096, D=4096, F=11008, eps=1e-6),
}


def parse_workload(name: str) -> dict:
    """A named workload, or kind:args: pattern:<name>:<dt>:M:N:K, norm:<rms|layer>:<dt>:M:N:K,
    swiglu:<dt>:M:D:F, multi:<rms|layer>:<dt>:M:K:N1,N2,.. (one norm, several weights),
    biasin:<dt>:M:N:K:<act> (input-bias prologue), rmsnorm:<dt>:M:K (standalone RMSNorm)."""
    if name in WORKLOADS:
        return dict(WORKLOADS[name], name=name)
    parts = name.split(":")
    if parts[0] == "multi":
        _, nm, dt, M, K, Ns = parts
        return dict(kind="multi", norm=nm, dtype=dt, M=int(M), K=int(K), Ns=[int(n) for n in Ns.split(",")],
                    eps=1e-6 if nm == "rms" else 1e-5, name=name)
    if parts[0] == "biasin":
        _, dt, M, N, K, act = parts
        return dict(kind="biasin", dtype=dt, M=int(M), N=int(N), K=int(K), act=act, name=name)
    if parts[0] == "rmsnorm":
        _, dt, M, K = parts
        return dict(kind="rmsnorm", dtype=dt, M=int(M), K=int(K), eps=1e-6, name=name)
    if parts[0] == "layer":
        _, dt, M, D, Dkv, F = parts[:6]
        L = int(parts[6]) if len(parts) > 6 else 4
        return dict(kind="layer", dtype=dt, M=int(M), D=int(D), Dkv=int(Dkv), F=int(F), L=L, eps=1e-6, name=name)
    if parts[0] == "pattern":
        _, pat, dt, M, N, K = parts
        return dict(kind="pattern", pattern=pat, dtype=dt, M=int(M), N=int(N), K=int(K), name=name)
    if parts[0] == "norm":
        _, nm, dt, M, N, K = parts
        return dict(kind="norm", norm=nm, dtype=dt, M=int(M), N=int(N), K=int(K), eps=1e-6 if nm == "rms" else 1e-5,
                    name=name)
    if parts[0] == "swiglu":
        _, dt, M, D, F = parts
        return dict(kind="swiglu", dtype=dt, M=int(M), D=int(D), F=int(F), eps=1e-6, name=name)
    raise SystemExit(f"unknown workload {name}")


def describe(w: dict) -> str:
    if w["kind"] == "norm":
        nm = "rmsnorm_gemm" if w["norm"] == "rms" else "layernorm_gemm"
        return f"{nm} {w['dtype']}: x[{w['M']},{w['K']}] gamma[{w['K']}] eps={w['eps']:g} W[{w['N']},{w['K']}], no bias"
    if w["kind"] == "pattern":
        return f"{w['pattern']} {w['dtype']}: A[{w['M']},{w['K']}] W[{w['N']},{w['K']}]"
    if w["kind"] == "multi":
        nm = "rmsnorm" if w["norm"] == "rms" else "layernorm"
        ws = ", ".join(f"W{i}[{n},{w['K']}]" for i, n in enumerate(w["Ns"]))
        return f"{nm} feeding {len(w['Ns'])} weights {w['dtype']}: x[{w['M']},{w['K']}] eps={w['eps']:g}, {ws}"
    if w["kind"] == "biasin":
        return (f"input-bias prologue {w['dtype']}: act={w['act']}((A[{w['M']},{w['K']}] + b_in[{w['K']}]) "
                f"W[{w['N']},{w['K']}]^T + bias)")
    if w["kind"] == "rmsnorm":
        return f"standalone rmsnorm {w['dtype']}: x[{w['M']},{w['K']}] gamma[{w['K']}] eps={w['eps']:g}"
    if w["kind"] == "layer":
        return (f"{w['L']} chained decoder layers, dense part, {w['dtype']}: M={w['M']} D={w['D']} Dkv={w['Dkv']} "
                f"F={w['F']} (RMSNorm+QKV, attention output projection + residual, RMSNorm+SwiGLU FFN + residual; "
                f"the attention output is a fixed input)")
    return (f"swiglu_ffn {w['dtype']}: x[{w['M']},{w['D']}] RMSNorm, Wg/Wu[{w['F']},{w['D']}], "
            f"Wd[{w['D']},{w['F']}], + x")


def roofline_of(flops: float, nbytes: float, per_launch_ms: float, peaks: dict, peak_src: str, traffic):
    """Roofline record of one step: bound by tensor throughput or by HBM bandwidth,
    whichever the step's arithmetic intensity puts it under (the ridge point of
    the measured peaks), with both fractions reported."""
    tensor_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    secs = per_launch_ms / 1e3
    tflops = flops / secs / 1e12
    gbs = nbytes / secs / 1e9
    ridge = tensor_peak * 1e12 / (hbm_peak * 1e9)  # flop per byte
    common = {"traffic": traffic, "algorithmic_bytes": nbytes, "tflops": tflops, "tensor_frac": tflops / tensor_peak,
              "hbm_gbs": gbs, "hbm_frac": gbs / hbm_peak, "intensity": flops / nbytes}
    if flops / nbytes < ridge:
        return {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                "peak_source": f"hbm_gbs (copy) of {peak_src}", **common}
    return {"bound": "tensor", "achieved": tflops, "peak": tensor_peak, "unit": "TFLOP/s", "frac": tflops / tensor_peak,
            "peak_source": f"bf16_tflops (burst, fp16 dense rate equal) of {peak_src}", **common}


def flops_per_step(w: dict) -> float:
    """2MNK plus the epilogue / prologue element ops (norm 3 per input element,
    row scale 1 per output, bias 1, gelu 8, silu 4, relu 1, residual 1, SwiGLU product 1)."""
    if w["kind"] == "swiglu":
        M, D, F = w["M"], w["D"], w["F"]
        return 6.0 * M * D * F + 3 * M * D + 2 * M * F + 4 * M * F + M * F + M * D
    if w["kind"] == "multi":
        M, K = w["M"], w["K"]
        return sum(2.0 * M * N * K + M * N for N in w["Ns"]) + 3 * M * K
    if w["kind"] == "rmsnorm":
        return 4.0 * w["M"] * w["K"]  # square-accumulate (2), scale by 1/rms and by gamma (2)
    if w["kind"] == "layer":
        M, D, Dkv, F = w["M"], w["D"], w["Dkv"], w["F"]
        return w["L"] * (2.0 * M * D * (D + 2 * Dkv) + 3 * M * D + M * (D + 2 * Dkv)  # RMSNorm + QKV
                         + 2.0 * M * D * D + 2 * M * D                                 # output projection, residual
                         + 6.0 * M * D * F + 3 * M * D + 2 * M * F + 4 * M * F + M * F + M * D)  # FFN
    M, N, K = w["M"], w["N"], w["K"]
    f = 2.0 * M * N * K
    if w["kind"] == "biasin":
        acts = {"none": 0, "gelu": 8, "silu": 4, "relu": 1}
        return f + M * K + M * N * (1 + acts[w["act"]])
    if w["kind"] == "norm":
        return f + 3 * M * K + M * N
    p = w["pattern"]
    f += M * N * (("bias" in p) + 8 * ("gelu" in p) + 4 * ("silu" in p) + ("relu" in p) + ("residual" in p))
    return f


def bytes_per_step(w: dict) -> float:
    """Algorithmic HBM bytes: every operand read once, the output written once."""
    e = 2
    if w["kind"] == "swiglu":
        M, D, F = w["M"], w["D"], w["F"]
        return e * (M * D + D + 2 * F * D + 2 * M * F + D * F + M * D + M * D)
    if w["kind"] == "multi":
        M, K = w["M"], w["K"]
        return e * (M * K + K * (2 if w["norm"] == "layer" else 1) + sum(N * K + M * N for N in w["Ns"]))
    if w["kind"] == "rmsnorm":
        return e * (2 * w["M"] * w["K"] + w["K"])
    if w["kind"] == "layer":
        M, D, Dkv, F = w["M"], w["D"], w["Dkv"], w["F"]
        weights = D * (D + 2 * Dkv) + D * D + 3 * D * F + 2 * D
        acts = M * D + M * (D + 2 * Dkv) + M * D + M * D + 2 * M * F + M * D  # x, q/k/v, attn, h, h_ffn w+r, out
        return e * w["L"] * (weights + acts)  # the layers share one set of weights, read once per layer
    M, N, K = w["M"], w["N"], w["K"]
    b = e * (M * K + N * K + M * N)
    if w["kind"] == "biasin":
        return b + e * (K + N)
    if w["kind"] == "norm":
        b += e * K * (2 if w["norm"] == "layer" else 1)
    else:
        p = w["pattern"]
        b += e * N * ("bias" in p) + e * M * N * ("residual" in p)
    return b


def make_inputs(w: dict):
    from gemm_epilogue_tma_gb300 import synthetic as syn
    if w["kind"] == "norm":
        return syn.norm_gemm_inputs(w["M"], w["N"], w["K"], w["norm"], w["dtype"])
    if w["kind"] == "pattern":
        return syn.gemm_inputs(w["M"], w["N"], w["K"], w["pattern"], w["dtype"])
    if w["kind"] == "multi":
        t = syn.multi_inputs(w["M"], w["Ns"], w["K"], w["norm"], w["dtype"])
        return {k: v for k, v in t.items() if not k.startswith("bias")}  # the timed calls use no output bias
    if w["kind"] == "biasin":
        t = syn.input_bias_inputs(w["M"], w["N"], w["K"], w["dtype"])
        t.pop("residual")
        return t
    if w["kind"] == "rmsnorm":
        t = syn.norm_gemm_inputs(w["M"], 8, w["K"], "rms", w["dtype"])
        return {"x": t["x"], "gamma": t["gamma"]}
    if w["kind"] == "layer":
        return syn.layer_inputs(w["M"], w["D"], w["Dkv"], w["F"], w["dtype"])
    return syn.swiglu_inputs(w["M"], w["D"], w["F"], w["dtype"])


def out_shapes(w: dict):
    """Shapes of the tensors one step writes."""
    if w["kind"] == "multi":
        return [(w["M"], N) for N in w["Ns"]]
    if w["kind"] == "swiglu":
        return [(w["M"], w["D"])]
    if w["kind"] == "rmsnorm":
        return [(w["M"], w["K"])]
    if w["kind"] == "layer":  # the last layer's out, then per layer q, k, v, h, out
        M, D, Dkv = w["M"], w["D"], w["Dkv"]
        return [(M, D)] + [(M, D), (M, Dkv), (M, Dkv), (M, D), (M, D)] * w["L"]
    return [(w["M"], w["N"])]


def e2e_input_keys(w: dict, t: dict):
    """Inputs copied host to device each end-to-end step: a decoder layer's
    activations (its weights stay resident), else every input."""
    if w["kind"] == "layer":
        return ["x", "attn"]
    return [k for k, v in t.items() if v is not None]


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Host-only translation units: changing them does not change any kernel.
HOST_ONLY_SOURCES = ("fl_host.cu", "fl_noalloc.cu")


def kernel_sources_hash(files=None) -> str:
    """Hash of device-code sources: the named files of csrc/ (the kernel a
    traffic record was taken on, its headers and its instantiation unit), or
    every kernel source when none are named."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_epilogue_tma_gb300", "csrc")
    names = sorted(files) if files else [n for n in sorted(os.listdir(csrc))
                                         if n.endswith((".cu", ".cuh", ".h")) and n not in HOST_ONLY_SOURCES]
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the sources of the
    captured kernel are unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    rec = d.get(workload)
    if not rec or rec.get("sources") != kernel_sources_hash(rec.get("files")):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float, load0: float = None):
        """Samples from the busy replays run just before the timed region
        through its end ([load0, t1]: the GPU under the same load the whole
        time), else inside the timed region [t0, t1], and only failing that
        the whole run."""
        inside, window = [], "timed_region"
        if load0 is not None:
            inside = [s for (t, s) in self.samples if load0 <= t <= t1 + 0.05]
            window = "load_before_and_during_timed_region"
        if not inside:
            inside = [s for (t, s) in self.samples if t0 <= t <= t1 + 0.05]
            window = "timed_region"
        if not inside:
            inside = [s for (_, s) in self.samples]
            window = "whole_run"
        mhz, maxmhz, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in inside:
            try:
                mhz.append(float(s[1]))
                maxmhz.append(float(s[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, s[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxmhz), "reasons": sorted(reasons),
                "samples": len(mhz), "window": window}


def dist_setup():
    """Rank, world size, and a process group when launched by torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int) -> float:
    """Maximum of a per-rank float over the process group (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_cores_used() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_step(w: dict, f64: dict, row0: int, rows: int):
    """The float64 oracle on rows [row0, row0+rows) of the workload (rows are independent)."""
    import oracle
    sl = slice(row0, row0 + rows)
    if w["kind"] == "norm":
        return oracle.norm_gemm(f64["x"][sl], f64["gamma"], f64.get("beta"), f64["W"], None, w["eps"], w["norm"])
    if w["kind"] == "pattern":
        r = f64.get("residual")
        return oracle.gemm_epilogue(f64["A"][sl], f64["W"], f64.get("bias"), None if r is None else r[sl],
                                    w["pattern"])
    if w["kind"] == "multi":
        return [oracle.norm_gemm(f64["x"][sl], f64["gamma"], f64.get("beta"), f64[f"W{i}"], None, w["eps"], w["norm"])
                for i in range(len(w["Ns"]))]
    if w["kind"] == "biasin":
        return oracle.input_bias_gemm(f64["A"][sl], f64["bias_in"], f64["W"], f64["bias"], None, w["act"])
    if w["kind"] == "rmsnorm":
        return oracle.rms_norm(f64["x"][sl], f64["gamma"], w["eps"])
    if w["kind"] == "layer":
        x, a = f64["x"][sl], f64["attn"][sl]
        qkv = [oracle.norm_gemm(x, f64["gamma_attn"], None, f64[W], None, w["eps"], "rms") for W in ("Wq", "Wk", "Wv")]
        h = oracle.linear(a, f64["Wo"]) + x
        return qkv, oracle.swiglu_ffn(h, f64["gamma_ffn"], f64["Wg"], f64["Wu"], f64["Wd"], None, w["eps"], w["dtype"])
    return oracle.swiglu_ffn(f64["x"][sl], f64["gamma"], f64["Wg"], f64["Wu"], f64["Wd"], None, w["eps"], w["dtype"])


def rows_of(w):
    return w["M"]


def flops_of_rows(w, rows):
    return flops_per_step(w) * rows / rows_of(w)


def cpu_baseline(w: dict, seconds: float = 10.0, rows_per_call: int = 16) -> dict:
    """The oracle as it stands, timed on a bounded sample of the workload's rows."""
    from gemm_epilogue_tma_gb300 import synthetic as syn
    t = make_inputs(w)
    f64 = {k: syn.as_f64(v) for k, v in t.items() if v is not None}
    M = rows_of(w)
    rows_per_call = min(rows_per_call, M)
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_step(w, f64, done % max(1, M - rows_per_call + 1), rows_per_call)
        done += rows_per_call
        el = time.perf_counter() - t0
        if el >= seconds or done >= 64 * M:
            break
    tf = flops_of_rows(w, done) / el / 1e12
    return {"value": tf, "unit": "TFLOP/s", "cores": cpu_cores_used(), "kind": "oracle",
            "sample": f"{done} rows of {M} ({rows_per_call} per call) in {el:.1f} s, float64 NumPy"}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_reference(args, w: dict, rank: int, world: int):
    if rank != 0:
        return
    from gemm_epilogue_tma_gb300 import synthetic as syn
    t = make_inputs(w)
    f64 = {k: syn.as_f64(v) for k, v in t.items() if v is not None}
    M = rows_of(w)
    rows = 1  # one row of the workload per step keeps --steps K within minutes
    for i in range(args.warmup):
        oracle_step(w, f64, i % M, rows)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(w, f64, i % M, rows)
    el = time.perf_counter() - t0
    value = flops_of_rows(w, rows * args.steps) / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w), "name": w["name"], "sample_rows_per_step": rows,
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores_used(), "kind": "oracle",
                         "sample": f"{rows} row of {M} per step, float64 NumPy oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w: dict, rank: int, world: int, local: int):
    import torch

    import gemm_epilogue_tma_gb300 as fl

    torch.cuda.set_device(local)
    fl.lib()
    fl.set_option("tile_n", args.tile_n)
    fl.set_option("variant", args.variant)
    fl.set_option("split_k", args.split_k)
    # the benchmark's weights are never written: the small-M kernel may stage
    # them before its programmatic dependency on the previous step resolves
    fl.set_option("weight_preload", 0 if args.no_weight_preload else 1)
    fl.set_option("launch_cache", 0 if args.no_launch_cache else 1)
    dev = torch.device("cuda", local)
    t = make_inputs(w)
    set_bytes = sum(v.numel() * v.element_size() for v in t.values() if v is not None)
    shapes = out_shapes(w)
    out_bytes = sum(a * b * 2 for a, b in shapes)
    # enough input copies to exceed the L2 three times over between reuses
    # (capped for tiny workloads, whose copies then stay in L2: said in config)
    nsets = min(256, max(2, int(3 * L2_BYTES // (set_bytes + out_bytes)) + 1))
    sets = []
    for _ in range(nsets):
        g = {k: (v.to(dev) if v is not None else None) for k, v in t.items()}
        g["outs"] = [torch.empty(sh, dtype=t[next(iter(t))].dtype, device=dev) for sh in shapes]
        g["out"] = g["outs"][0]
        if w["kind"] == "layer":
            # L layers chained through their outputs (layer l reads layer l-1's
            # out as x), sharing the weights and the attention stand-in
            o = g["outs"]
            base = {k: v for k, v in g.items() if k not in ("outs", "out", "x")}
            g["layers"], x = [], g["x"]
            for l in range(w["L"]):
                q, k_, v_, h, out_l = o[1 + 5 * l: 6 + 5 * l]
                g["layers"].append(fl.DecoderLayer(eps=w["eps"], x=x, out=out_l, q=q, k=k_, v=v_, h=h, bias_o=None,
                                                   **base))
                x = out_l
            g["out"] = g["outs"][0] = x
        if w["kind"] == "swiglu":
            g["ws"] = torch.empty(fl.swiglu_ffn_workspace_size(w["M"], w["F"], w["dtype"]), dtype=torch.uint8,
                                  device=dev)
        sets.append(g)
    n_out = len(shapes)

    def step(g, stream=None):
        if w["kind"] == "layer":
            for layer in g["layers"]:
                for half in (0, 1):
                    layer.issue(half, stream=stream)
        elif w["kind"] == "multi" and args.separate:
            for i in range(n_out):
                fl.norm_gemm(g["x"], g["gamma"], g[f"W{i}"], beta=g.get("beta"), out=g["outs"][i], eps=w["eps"],
                             norm=w["norm"], stream=stream)
        elif w["kind"] == "multi":
            fl.norm_gemm_multi(g["x"], g["gamma"], [g[f"W{i}"] for i in range(n_out)], beta=g.get("beta"),
                               outs=g["outs"], eps=w["eps"], norm=w["norm"], stream=stream)
        elif w["kind"] == "biasin":
            fl.input_bias_gemm(g["A"], g["bias_in"], g["W"], bias=g["bias"], out=g["out"], act=w["act"],
                               stream=stream)
        elif w["kind"] == "rmsnorm":
            fl.rms_norm(g["x"], g["gamma"], out=g["out"], eps=w["eps"], stream=stream)
        elif w["kind"] == "norm":
            fl.norm_gemm(g["x"], g["gamma"], g["W"], beta=g.get("beta"), out=g["out"], eps=w["eps"],
                         norm=w["norm"], stream=stream)
        elif w["kind"] == "pattern":
            fl.gemm_epilogue(g["A"], g["W"], bias=g.get("bias"), residual=g.get("residual"), out=g["out"],
                             pattern=w["pattern"], stream=stream)
        else:
            fl.swiglu_ffn(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], out=g["out"], eps=w["eps"],
                          workspace=g["ws"], stream=stream)

    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local) if rank == 0 else None
    for i in range(args.warmup):
        step(sets[i % nsets])
    torch.cuda.synchronize()
    fl.device_status()
    # this library's kernels per step, as its own launch counter reports them
    n0 = fl.kernel_launches()
    step(sets[0])
    launches_per_step = fl.kernel_launches() - n0
    torch.cuda.synchronize()

    # The timed loop replays CUDA graphs of the same library calls (one step
    # per input copy), so the host launch path does not throttle short kernels.
    def capture(n):
        if n == 0 or args.no_graph:
            return None
        if args.library_capture:
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                gr = fl.Graph.capture(lambda: [step(sets[j % nsets], stream=side) for j in range(n)], stream=side)
            stream.wait_stream(side)
            gr.replay = gr.launch
            return gr
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(n):
                step(sets[j % nsets])
        return g

    full = capture(nsets)
    rest = capture(args.steps % nsets)
    reps = args.steps // nsets

    def timed_steps():
        if args.no_graph:
            for i in range(args.steps):
                step(sets[i % nsets])
            return
        for _ in range(reps):
            full.replay()
        if rest is not None:
            rest.replay()

    if not args.no_graph:
        full.replay()
        torch.cuda.synchronize()
    # Busy replays right before the timed region (untimed), long enough for
    # the clock sampler to see the GPU under this load even when the timed
    # region itself is shorter than one sampling interval.
    load0 = time.time()
    while time.time() - load0 < args.load_seconds:
        if args.no_graph:
            for i in range(nsets):
                step(sets[i % nsets])
        else:
            full.replay()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    ev0.record(stream)
    timed_steps()
    enqueue_s = time.time() - wall0  # host time to issue the K steps (stream calls: the launch path's cost)
    ev1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    fl.device_status()
    ms_max = max_over_ranks(ms, world)
    clocks = sampler.summary(wall0, wall1, load0) if sampler else None
    if sampler:
        sampler.stop()

    # end to end through the same call: pinned host inputs in, result back to
    # pinned host, every step. Steps are pipelined the way a serving loop runs
    # them: two device buffer sets; step i's inputs go up on a copy stream into
    # set i % 2 while the compute stream runs step i - 1, and its result comes
    # back on a third stream once its kernels are done (set i % 2 is refilled
    # only after step i - 2's result has been read back).
    host = {k: t[k].pin_memory() for k in e2e_input_keys(w, t)}
    # the step's result read back: a layer stack's last output, else every output
    d2h_shapes = shapes[:1] if w["kind"] == "layer" else shapes
    houts = [torch.empty(sh, dtype=sets[0]["out"].dtype).pin_memory() for sh in d2h_shapes]
    gsets = [sets[0], sets[1 % nsets]]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    e2e_steps = max(3, min(args.steps, 200))
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n, start_event):
        up_s.wait_event(start_event)
        for i in range(n):
            b = i % 2
            g = gsets[b]
            if i >= 2:
                up_s.wait_event(ev_free[b])  # step i - 2's result is back: set b is free
            with torch.cuda.stream(up_s):
                for k, v in host.items():
                    if v is not None:
                        g[k].copy_(v, non_blocking=True)
                ev_in[b].record(up_s)
            stream.wait_event(ev_in[b])
            step(g)
            ev_out[b].record(stream)
            down_s.wait_event(ev_out[b])
            with torch.cuda.stream(down_s):
                for ho, o in zip(houts, g["outs"]):
                    ho.copy_(o, non_blocking=True)
                ev_free[b].record(down_s)
        stream.wait_stream(down_s)
        stream.wait_stream(up_s)

    warm = torch.cuda.Event()
    warm.record(stream)
    e2e_run(3, warm)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    fl.device_status()

    if rank != 0:
        return
    flops = flops_per_step(w)
    value = flops * args.steps * world / (ms_max / 1e3) / 1e12
    per_launch_ms = ms / args.steps
    peaks, peak_src = load_peaks()
    traffic = recorded_traffic(w["name"])
    roofline = roofline_of(flops, bytes_per_step(w), per_launch_ms, peaks, peak_src, traffic)
    vs = None
    if w["name"] == "rmsnorm_gemm_f16_512x4096x4096":
        vs = value / world / (flops / (PAGE_FUSED_MS / 1e3) / 1e12)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": vs, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": describe(w), "name": w["name"],
                   "l2": f"inputs rotate over {nsets} copies ({nsets * (set_bytes + out_bytes) / 2**20:.0f} MiB "
                         + ("> 129 MB L2)" if nsets * (set_bytes + out_bytes) > L2_BYTES else
                            "< 129 MB L2: the operands are L2-resident)"),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": ("stream calls" if args.no_graph
                              else f"CUDA graphs of {nsets} steps of library calls, replayed"
                              + (" (captured with fl_capture_begin / fl_capture_end)" if args.library_capture
                                 else "")),
                   "weights": "read-only; " + ("read after the previous step" if args.no_weight_preload else
                                               "the split-K kernel stages its first weight tiles before the "
                                               "programmatic dependency resolves; the other kernels only "
                                               "prefetch them into L2"),
                   "vs_baseline_ref": "A30 fused RMSNorm->Linear 0.208 ms (LLMBoost page), other hardware",
                   "host_enqueue_us_per_step": enqueue_s * 1e6 / args.steps},
        "roofline": roofline,
        "e2e": {"value": flops * e2e_steps * world / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": sum(a * b * 2 for a, b in d2h_shapes)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, seconds=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="rmsnorm_gemm_f16_512x4096x4096")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tile-n", type=int, default=0, help="force the CTA tile width (128/256; 0 = auto)")
    ap.add_argument("--variant", type=int, default=0, help="force 1 = tile kernel, 2 = small-M split-K kernel")
    ap.add_argument("--split-k", type=int, default=0, help="force the K split of the small-M kernel")
    ap.add_argument("--no-graph", action="store_true", help="time plain stream calls instead of graph replays")
    ap.add_argument("--library-capture", action="store_true",
                    help="capture the replayed graphs with the library's fl_capture_begin / fl_capture_end")
    ap.add_argument("--no-launch-cache", action="store_true",
                    help="prepare every call afresh (FL_OPT_LAUNCH_CACHE off): host cost without the cache")
    ap.add_argument("--separate", action="store_true",
                    help="multi workloads: one fl_norm_gemm call per weight instead of one fl_norm_gemm_multi call")
    ap.add_argument("--load-seconds", type=float, default=0.3,
                    help="untimed busy replays right before the timed region, sampled for the clock record")
    ap.add_argument("--no-weight-preload", action="store_true",
                    help="read weights only after the previous step (FL_OPT_WEIGHT_PRELOAD off)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    w = parse_workload(args.workload)
    if w["kind"] == "layer":
        # a decode step through a layer stack: captured with the library's own
        # capture calls (fl_capture_begin / fl_capture_end)
        args.library_capture = True
    rank, world, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, w, rank, world)
        else:
            run_ours(args, w, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark of the 2:4 sparse hot path on one GB300: prune + compress of the
weights, then the sparse x dense product for a batch of activations.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all] [--impl {st24,reference}]

One pass of a workload = prune_compress of every weight of the workload, then
st24_spmm of every weight with every activation width of the workload.  A
timed step is `passes_per_step` such passes (chosen so the timed region lasts
a few seconds and the clock sampler sees it under load).  Inputs are seeded
synthetic tensors (st24_inputs).  The timed region is K steps replayed as CUDA
graphs on one stream, bracketed by a barrier and a synchronize.

The default (`--workload all`) prints ONE JSON line whose headline is the
largest workload (fp8-e4m3 28672x8192 with N in {1, 64, 512, 4096, 8192}, plus
prune/compress of the bf16 weight), with the decode, prefill and int8
workloads, the listing's dense-vs-unstructured demo and the transposed product
as sub-records under "workloads", each with its own value, roofline, clocks,
end-to-end figure and CPU baseline.  ``--impl reference`` times the CPU oracle
on a bounded sample of the headline workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import st24_inputs as inputs  # noqa: E402

METRIC = "2:4 SpMM TFLOP/s and % of sparse tensor peak / HBM roofline on 1 GB300"
UNIT = "TFLOP/s"

# Workloads: element type, output type, weight shapes [(M, K)], activation widths, layers,
# weight std, beta, per-row scale.  `layers` distinct weights of each shape per pass, so each
# product is launched behind another product (as in a model's layer stack), not behind a graph
# boundary, and every pass streams more weight bytes than L2 holds.
WORKLOADS = {
    "fp8": dict(ab="e4m3", c="bf16", shapes=[(28672, 8192)], Ns=list(inputs.FP8_NS), layers=2, a_std=0.02,
                beta=0.0, scale=False, extra_prune_bf16=(28672, 8192),
                desc="fp8-e4m3 2:4 SpMM: 2 distinct 28672x8192 weights N(0,0.02), N in {1,64,512,4096,8192}, "
                     "bf16 out; prune/compress of the bf16 28672x8192 weight"),
    "decode_bf16": dict(ab="bf16", c="bf16", shapes=[(4096, 4096)], Ns=list(inputs.DECODE_NS), layers=16,
                        a_std=0.02, beta=0.0, scale=False,
                        desc="decode-shaped bf16 2:4 SpMM: 16 distinct 4096x4096 weights N(0,0.02), "
                             "activations N(0,1) for N in {1,8,16,32}, bf16 out"),
    "prefill_bf16": dict(ab="bf16", c="bf16", shapes=list(inputs.PREFILL_SHAPES), Ns=[4096], layers=2,
                         a_std=0.02, beta=1.0, scale=False,
                         desc="prefill-shaped bf16 2:4 SpMM: 2 x (11008x4096 and 4096x11008) distinct weights, "
                              "N=4096, beta=1 with C N(0,1), bf16 out"),
    "int8": dict(ab="s8", c="bf16", shapes=[(8192, 8192)], Ns=list(inputs.INT8_NS), layers=4, a_std=1.0,
                 beta=0.0, scale=True,
                 desc="int8 2:4 SpMM: 4 distinct 8192x8192 weights uniform [-127,127], N in {16,2048}, "
                      "int32 accumulate, per-row fp32 scale, bf16 out"),
    # The chapter's listing timed dense against 75%-unstructured-sparse weights run as dense (no
    # faster) at 4096^3; re-measured here with the 2:4 product beside both (context, not a target).
    "demo_bf16": dict(ab="bf16", c="bf16", shapes=[(4096, 4096)], Ns=[4096], layers=8, a_std=1.0, beta=0.0,
                      scale=False, unstructured_context=0.75,
                      desc="the listing's 4096^3 demo in bf16: 2:4 SpMM of 8 distinct 4096x4096 weights, "
                           "N=4096, beside dense and 75%-unstructured-zero dense matmuls"),
    # The transposed use of the compressed weights dX = dY * W (retraining after the prune), at the
    # prefill shapes: a dense contraction over M read from the compressed form (tensor-bound).
    "transposed_bf16": dict(ab="bf16", c="bf16", shapes=list(inputs.PREFILL_SHAPES), Ns=[4096], layers=2,
                            a_std=0.02, beta=0.0, scale=False, op="spmm_t",
                            desc="transposed use dX = dY * W of 2 x (11008x4096 and 4096x11008) compressed bf16 "
                                 "weights, dY of N=4096 rows, bf16 out"),
}
HEADLINE = "fp8"
SUB_WORKLOADS = ["decode_bf16", "prefill_bf16", "int8", "demo_bf16", "transposed_bf16"]


def flops_per_pass(w):
    return sum(2.0 * M * K * N for (M, K) in w["shapes"] for N in w["Ns"]) * w["layers"]


def spmm_bytes(w):
    """Algorithmic HBM bytes of all SpMM launches of one pass (compressed A, B, C, scale)."""
    return sum(launch_bytes(w, M, K, N) for (M, K) in w["shapes"] for N in w["Ns"]) * w["layers"]


def prune_bytes(w):
    es = inputs.ELEM_SIZE[w["ab"]]
    return sum(M * K * es + M * K // 2 * es + M * K // 8 for (M, K) in w["shapes"]) * w["layers"]


def groups(w):
    """(activation index, shape index) pairs, one captured graph and one timing each."""
    return [(ni, si) for ni in range(len(w["Ns"])) for si in range(len(w["shapes"]))]


def launch_bytes(w, M, K, N):
    """Algorithmic HBM bytes of one product: compressed A and metadata, B, C (read too when beta != 0), scale.
    For the transposed use: compressed A, dY (N x M) and dX (N x K)."""
    es = inputs.ELEM_SIZE[w["ab"]]
    cs = inputs.ELEM_SIZE[w["c"]]
    if w.get("op") == "spmm_t":
        return M * K // 2 * es + M * K // 8 + M * N * es + K * N * cs * (2 if w["beta"] else 1)
    return M * K // 2 * es + M * K // 8 + K * N * es + M * N * cs * (2 if w["beta"] else 1) + \
        (4 * M if w["scale"] else 0)


def n_spmm(w):
    return len(w["shapes"]) * len(w["Ns"]) * w["layers"]


def n_prune(w):
    return len(w["shapes"]) * w["layers"]


def kernel_source_hash():
    """sha256 of the CUDA sources and the C header (identifies the kernels a traffic figure belongs to)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(f for f in glob.glob(os.path.join(ROOT, "structured_sparse_gemm_gb300", "csrc", "*"))
                   if os.path.isfile(f)) + [os.path.join(ROOT, "include", "st24.h")]
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + fh.read())
    return h.hexdigest()


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` on `workload` from an ncu capture recorded in
    profiles/traffic.json, or None when absent or taken on kernels that have changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[workload][kernel]
    except Exception:
        return None
    return rec["dram_bytes_per_launch"] if rec.get("source_sha256") == kernel_source_hash() else None


def max_over_ranks(value: float, world: int, device="cuda") -> float:
    """The largest of every rank's value: the job's step time is its slowest replica's."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_replica_step: float, ms_step: float) -> float:
    """Whole-job throughput: every replica's work over the slowest replica's step time."""
    return world * flops_per_replica_step / (ms_step * 1e-3) / 1e12


def passes_for(target_s: float, steps: int, pass_ms: float) -> int:
    """Passes per timed step so that `steps` steps last about `target_s` seconds (at least 1)."""
    if pass_ms <= 0 or steps <= 0:
        return 1
    return max(1, int(math.ceil(target_s * 1e3 / (steps * pass_ms))))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def mma_sp_peak_tops(kind: int) -> float | None:
    """Dense-equivalent TOPS of back-to-back register-only mma.sp (kind 0: int8
    m16n8k64, 1: bf16 m16n8k32), measured now on this GPU by the library's
    peak probe; None if it cannot run."""
    import ctypes
    import structured_sparse_gemm_gb300 as st
    try:
        lib = ctypes.CDLL(st._build_lib.PEAK_LIB)
        lib.st24peak_mma_sp.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
        out = ctypes.c_double(0.0)
        return out.value if lib.st24peak_mma_sp(kind, ctypes.byref(out)) == 0 else None
    except OSError:
        return None


_MMA_SP_PEAK = {}


def tensor_peak(ab: str, bf16_dense: float, bf16_sustained: float, long_region: bool, dense_op: bool = False):
    """2:4-sparse tensor peak (dense-equivalent TFLOP/s) of an element type, and where it comes from.

    16-bit: twice the measured dense bf16 peak; e4m3: twice that again (the nominal
    fp8/bf16 ratio); int8: the measured mma.sp rate (tcgen05 has no int8 kind here).
    A timed region of seconds runs under the power cap, so it is compared with the
    sustained dense figure; a short one with the burst figure."""
    dense = bf16_sustained if long_region else bf16_dense
    which = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    if dense_op:   # a dense contraction (the transposed use of the compressed weight)
        return dense, f"measured dense bf16 (MEASURED_PEAKS.json {which}): a dense MMA"
    if ab in ("bf16", "f16"):
        return 2.0 * dense, f"2 x measured dense bf16 (MEASURED_PEAKS.json {which})"
    if ab == "e4m3":
        return 4.0 * dense, f"4 x measured dense bf16 (MEASURED_PEAKS.json {which}; sparse x2, fp8/bf16 nominal x2)"
    if "s8" not in _MMA_SP_PEAK:
        _MMA_SP_PEAK["s8"] = mma_sp_peak_tops(0)
    t = _MMA_SP_PEAK["s8"]
    if t is None:
        return None, "unavailable"
    return t, "measured live: register-only mma.sp m16n8k64 s8 loop (csrc/peak/peak_mma_sp.cu)"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)   # the first sample lands before the timed work starts
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        return summarize_clock_lines(getattr(self, "lines", []))


def summarize_clock_lines(lines):
    """Median SM clock over the samples taken under load (power above 1.3x the smallest
    sample, or all samples if none qualifies), the maximum clock, and the throttle reasons
    seen active in any sample."""
    rows = []
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [x.strip() for x in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm, mx = float(parts[1]), float(parts[2])
        except ValueError:
            continue
        try:
            pw = float(parts[3])
        except ValueError:
            pw = None
        rows.append((sm, mx, pw, [nm for nm, v in zip(names, parts[5:9]) if v.lower() == "active"]))
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
    pws = [r[2] for r in rows if r[2] is not None]
    floor = min(pws) if pws else None
    load = [r for r in rows if floor is not None and r[2] is not None and r[2] > 1.3 * floor + 20.0] or rows
    reasons = sorted({nm for r in rows for nm in r[3]})
    return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": rows[-1][1], "reasons": reasons,
            "samples": len(rows), "samples_under_load": len(load) if load is not rows else 0,
            "power_w_max": max(pws) if pws else None}


# ---------------------------------------------------------------- the GPU arm
def build_workload(w, dev, seed=0):
    """Weights, activations and outputs of one workload, resident on `dev`."""
    import structured_sparse_gemm_gb300 as st

    layers = []
    for li in range(w["layers"]):
        for si, (M, K) in enumerate(w["shapes"]):
            g = inputs.generator(seed + 1000 * li + si)
            A = inputs.draw(w["ab"], (M, K), w["a_std"], g).to(dev)
            values = torch.empty((M, K // 2), dtype=A.dtype, device=dev)
            meta = torch.empty((M, K // 8), dtype=torch.uint8, device=dev)
            scale = inputs.row_scale(M, g).to(dev) if w["scale"] else None
            acts = []
            t = w.get("op") == "spmm_t"
            for N in w["Ns"]:
                # X is the product's right operand ([N, K]; dY [N, M] for the transposed use), Y its output
                X = inputs.draw(w["ab"], (N, M if t else K), 1.0, g).to(dev)
                Y = inputs.draw(w["c"], (N, K if t else M), 1.0, g).to(dev) if w["beta"] else \
                    torch.empty((N, K if t else M), dtype=inputs.TORCH_DTYPE[w["c"]], device=dev)
                ws_bytes = 0 if t else st.st24_spmm_workspace_bytes(w["ab"], w["c"], M, N, K)
                ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
                acts.append((X, Y, ws))
            layers.append(dict(A=A, values=values, meta=meta, scale=scale, acts=acts, M=M, K=K, si=si))
    return layers


def prune_phase(layers, stream=None):
    import structured_sparse_gemm_gb300 as st
    for L in layers:
        st.st24_prune_compress(L["A"], L["values"], L["meta"], stream=stream)


def product(w, L, X, Y, ws, stream=None, kernel="auto", fixed_a=True):
    """One product of the workload through the public API: st24_spmm, or st24_spmm_t for the transposed use."""
    import structured_sparse_gemm_gb300 as st
    if w.get("op") == "spmm_t":
        st.st24_spmm_t(L["values"], L["meta"], X, Y, K=L["K"], beta=w["beta"], stream=stream)
    else:
        st.st24_spmm(L["values"], L["meta"], X, Y, K=L["K"], beta=w["beta"], row_scale=L["scale"],
                     workspace=ws, stream=stream, kernel=kernel, fixed_a=fixed_a)


def spmm_phase(layers, w, stream=None, kernel="auto", only=None, fixed_a=True):
    """The products of one pass.  Run inside a captured graph, after the prune
    graph has completed, so the weights are fixed for the whole phase
    (ST24_SPMM_FIXED_A)."""
    for ni in range(len(w["Ns"])):
        for L in layers:
            if only is not None and (ni, L["si"]) != only:
                continue
            X, Y, ws = L["acts"][ni]
            product(w, L, X, Y, ws, stream=stream, kernel=kernel, fixed_a=fixed_a)


def time_launches(fn, stream, reps=10, warm=3):
    """Mean device time in microseconds of fn() (launched on `stream`), over `reps` calls."""
    for _ in range(warm):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps * 1e3


def extra_prune_timings(w, stream, dev):
    """Prune/compress timings on the bf16 weight the fp8 one is cast from (timed apart from the step):
    2:4 prune+compress, the fused per-row quantisation to e4m3, and the N:M patterns."""
    import structured_sparse_gemm_gb300 as st
    M, K = w["extra_prune_bf16"]
    Wb = inputs.prune_weight_bf16(M, K).to(dev)
    out = {"shape": [M, K]}
    vb = torch.empty((M, K // 2), dtype=torch.bfloat16, device=dev)
    mb = torch.empty((M, K // 8), dtype=torch.uint8, device=dev)
    us = time_launches(lambda: st.st24_prune_compress(Wb, vb, mb, stream=stream), stream)
    nbytes = M * K * 2 + M * K // 2 * 2 + M * K // 8
    out["prune_compress_bf16"] = {"us_per_launch": us, "GB/s": nbytes / (us * 1e-6) / 1e9, "bytes": nbytes}
    vq = torch.empty((M, K // 2), dtype=torch.float8_e4m3fn, device=dev)
    sq = torch.empty(M, dtype=torch.float32, device=dev)
    us = time_launches(lambda: st.st24_quantize_prune_compress(Wb, vq, mb, sq, stream=stream), stream)
    nbytes = M * K * 2 + M * K // 2 + M * K // 8 + 4 * M
    out["quantize_prune_compress_bf16_to_e4m3"] = {"us_per_launch": us, "GB/s": nbytes / (us * 1e-6) / 1e9,
                                                   "bytes": nbytes}
    del vq, sq
    for (n, m) in [(1, 4), (2, 8), (1, 8)]:
        us = time_launches(lambda: st.st24_prune_compress_nm(Wb, vb, mb, n, m, stream=stream), stream)
        nbytes = M * K * 2 + M * K // 2 * 2 + M * K // 8
        out[f"prune_compress_nm_{n}of{m}_bf16"] = {"us_per_launch": us, "GB/s": nbytes / (us * 1e-6) / 1e9,
                                                   "bytes": nbytes}
    del vb, mb
    # 4:8 as two 2:4 forms (values M x K, metadata M x 2 K/8)
    v2 = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    m2 = torch.empty((M, K // 4), dtype=torch.uint8, device=dev)
    us = time_launches(lambda: st.st24_prune_compress_nm2(Wb, v2, m2, 4, 8, stream=stream), stream)
    nbytes = M * K * 2 + M * K * 2 + M * K // 4
    out["prune_compress_nm2_4of8_bf16"] = {"us_per_launch": us, "GB/s": nbytes / (us * 1e-6) / 1e9, "bytes": nbytes}
    del Wb, v2, m2
    return out


def run_gpu(args, w, rank, world, target_s):
    import structured_sparse_gemm_gb300 as st

    dev = torch.device("cuda", torch.cuda.current_device())
    st.load()
    layers = build_workload(w, dev, seed=rank)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        # eager warm-up (also sets kernel attributes before capture)
        prune_phase(layers)
        spmm_phase(layers, w, kernel=args.kernel, fixed_a=args.fixed_a)
        stream.synchronize()
        # one graph for the prune phase, one per (activation width, shape) for the products
        g_prune = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_prune, stream=stream):
            prune_phase(layers)
        g_spmm = []
        for grp in groups(w):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                spmm_phase(layers, w, kernel=args.kernel, only=grp, fixed_a=args.fixed_a)
            g_spmm.append(g)

    def one_pass():
        g_prune.replay()
        for g in g_spmm:
            g.replay()

    # warm-up passes; their time sizes the timed steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        one_pass()
        e0.record(stream)
        for _ in range(max(args.warmup, 1)):
            one_pass()
        e1.record(stream)
    torch.cuda.synchronize()
    pass_ms = e0.elapsed_time(e1) / max(args.warmup, 1)
    R = passes_for(target_s, args.steps, pass_ms)
    if world > 1:
        R = int(max_over_ranks(float(R), world, "cuda"))
    if st.st24_device_status() != 0:
        raise RuntimeError("device status after warm-up")

    nG = len(groups(w))
    # per pass: start, after prune, after each product group
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 + nG)] for _ in range(args.steps * R)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            for k in range(args.steps * R):
                ev[k][0].record(stream)
                g_prune.replay()
                ev[k][1].record(stream)
                for ni, g in enumerate(g_spmm):
                    g.replay()
                    ev[k][2 + ni].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    status = st.st24_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    passes = args.steps * R
    total_ms = ev[0][0].elapsed_time(ev[-1][-1])
    prune_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / passes
    spmm_ms = sum(e[1].elapsed_time(e[-1]) for e in ev) / passes
    per_group_ms = [sum(e[1 + gi].elapsed_time(e[2 + gi]) for e in ev) / passes for gi in range(nG)]
    extra = extra_prune_timings(w, stream, dev) if w.get("extra_prune_bf16") else None
    return dict(total_ms=total_ms, passes_per_step=R, pass_ms=total_ms / passes, prune_ms=prune_ms, spmm_ms=spmm_ms,
                per_group_ms=per_group_ms, clocks=clk.summary(), extra_prune=extra, layers=layers, stream=stream)


def run_e2e(args, w, layers, stream):
    """Same pass through the public API with host inputs: H2D of the weights and
    activations, prune+compress, SpMM, D2H of the outputs, all timed."""
    import structured_sparse_gemm_gb300 as st

    host = []
    h2d = d2h = 0
    for L in layers:
        hA = torch.empty(L["A"].shape, dtype=L["A"].dtype, pin_memory=True)
        hA.copy_(L["A"].cpu())
        hX = []
        for (X, Y, ws) in L["acts"]:
            t = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
            t.copy_(X.cpu())
            hX.append((t, torch.empty(Y.shape, dtype=Y.dtype, pin_memory=True)))
            h2d += t.numel() * t.element_size()
            d2h += Y.numel() * Y.element_size()
        h2d += hA.numel() * hA.element_size()
        host.append((hA, hX))

    # Uploads run on their own stream, layer by layer, so each layer's weight
    # copy overlaps the work already queued (the previous layers' prune and
    # the previous step's products): the host link, not the GPU, bounds a step.
    copy_stream = torch.cuda.Stream(device=stream.device)
    copied = [torch.cuda.Event() for _ in layers]
    pruned = [torch.cuda.Event() for _ in layers]
    products_done = torch.cuda.Event()
    first = [True]

    def step():
        for i, (L, (hA, hX)) in enumerate(zip(layers, host)):
            with torch.cuda.stream(copy_stream):
                if not first[0]:
                    copy_stream.wait_event(pruned[i])         # the last step's prune has read A
                L["A"].copy_(hA, non_blocking=True)
                if not first[0]:
                    copy_stream.wait_event(products_done)     # the last step's products have read X
                for (X, Y, ws), (hx, hy) in zip(L["acts"], hX):
                    X.copy_(hx, non_blocking=True)
                copied[i].record(copy_stream)
        first[0] = False
        with torch.cuda.stream(stream):
            for i, L in enumerate(layers):
                stream.wait_event(copied[i])
                st.st24_prune_compress(L["A"], L["values"], L["meta"])
                pruned[i].record(stream)
            for ni in range(len(w["Ns"])):
                for li, L in enumerate(layers):
                    X, Y, ws = L["acts"][ni]
                    # The weights pruned by the kernel just before the first
                    # product may still be in flight: that product waits.
                    fixed = args.fixed_a and not (ni == 0 and li == 0 and len(layers) == 1)
                    product(w, L, X, Y, ws, fixed_a=fixed)
            products_done.record(stream)
            for L, (hA, hX) in zip(layers, host):
                for (X, Y, ws), (hx, hy) in zip(L["acts"], hX):
                    hy.copy_(Y, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)    # no timed upload starts before the timed region
    for _ in range(args.steps):
        step()
    e1.record(stream)             # each step ends with its outputs' download on `stream`
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    del host
    return ms, h2d, d2h


# ---------------------------------------------------------------- dense context
def _dense_op(ab: str, dev):
    """(operand dtype, fn(X, W, out) -> None, label) of torch's dense product for an element type,
    or None for a shape the op rejects: bf16 matmul for 16-bit inputs, _scaled_mm for e4m3,
    _int_mm for int8 (context only, not this library's path)."""
    if ab in ("bf16", "f16"):
        dt = inputs.TORCH_DTYPE[ab]
        return dt, (lambda X, W, out: torch.matmul(X, W.t(), out=out)), f"torch.matmul {ab}", dt
    if ab == "e4m3":
        one = torch.ones((), dtype=torch.float32, device=dev)
        return (torch.float8_e4m3fn,
                (lambda X, W, out: out.copy_(torch._scaled_mm(X, W.t(), scale_a=one, scale_b=one,
                                                              out_dtype=torch.bfloat16))),
                "torch._scaled_mm e4m3 -> bf16", torch.bfloat16)
    return torch.int8, (lambda X, W, out: torch._int_mm(X, W.t(), out=out)), "torch._int_mm int8 -> int32", torch.int32


def dense_context(w, dev, zero_fraction: float = 0.0, reps: int = 20):
    """torch's dense product of the unpruned shapes (context only), like for like with the sparse
    pass: `layers` distinct random weights per shape (so they stream from HBM), every activation
    width, each (shape, N) group captured in one CUDA graph.  With zero_fraction, weights with that
    fraction of unstructured zeros, multiplied by the same dense kernel.  Per group: microseconds per
    product, or the error the op raised for that shape."""
    dt, fn, label, out_dt = _dense_op(w["ab"], dev)
    transposed = w.get("op") == "spmm_t"
    if transposed:   # dX = dY @ W: W [M, K] is the right operand as stored
        fn = lambda X, W, out: torch.matmul(X, W, out=out)   # noqa: E731
        label = "torch.matmul bf16 (dY @ W)"
    res = {"op": label, "groups": []}
    total_us = 0.0
    complete = True
    for (M, K) in w["shapes"]:
        Ws = []
        for _ in range(w["layers"]):
            W = torch.randn(M, K, device=dev, dtype=torch.float32)
            if zero_fraction:
                W = W * (torch.rand(M, K, device=dev) >= zero_fraction)
            Ws.append(W.to(dt) if dt != torch.int8 else W.mul(40).clamp(-127, 127).to(torch.int8))
            del W
        for N in w["Ns"]:
            X = torch.randn(N, M if transposed else K, device=dev, dtype=torch.float32)
            X = X.to(dt) if dt != torch.int8 else X.mul(40).clamp(-127, 127).to(torch.int8)
            outs = [torch.empty((N, K if transposed else M), dtype=out_dt, device=dev) for _ in Ws]
            try:
                for W, o in zip(Ws, outs):
                    fn(X, W, o)
                torch.cuda.synchronize()
            except Exception as e:   # e.g. _int_mm needs N > 16, _scaled_mm N % 16 == 0
                res["groups"].append({"M": M, "K": K, "N": N, "error": str(e).splitlines()[0][:120]})
                complete = False
                continue
            s = torch.cuda.Stream(device=dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                for W, o in zip(Ws, outs):   # warm the op's workspace outside capture
                    fn(X, W, o)
                s.synchronize()
                with torch.cuda.graph(g, stream=s):
                    for W, o in zip(Ws, outs):
                        fn(X, W, o)
            us = time_launches(g.replay, s, reps=reps) / len(Ws)
            total_us += us * len(Ws)
            res["groups"].append({"M": M, "K": K, "N": N, "us_per_launch": us,
                                  "tflops": 2.0 * M * K * N / (us * 1e-6) / 1e12})
            del outs, X
        del Ws
    res["ms_per_pass"] = total_us * 1e-3 if complete else None
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- the oracle (CPU baseline)
def oracle_sample(w, budget_s: float):
    """Time the CPU oracle on a bounded sample of the workload: prune+compress of
    the first weight, then its product with the activation widths in order,
    repeated until about `budget_s` seconds of CPU work have been done."""
    import oracle

    M, K = w["shapes"][0]
    g = inputs.generator(0)
    A = inputs.raw(inputs.draw(w["ab"], (M, K), w["a_std"], g)).numpy()
    # rows of the weight in the sample: all of them unless one SpMM pass would blow the budget
    rows = M if M * K * max(w["Ns"]) <= 4e9 else max(128, int(4e9 // (K * max(w["Ns"]))) // 128 * 128)
    sub = A[:rows]
    transposed = w.get("op") == "spmm_t"
    # the product's right operand for those rows: X [N, K], or dY [N, rows] for the transposed use
    Xs = [inputs.raw(inputs.draw(w["ab"], (N, rows if transposed else K), 1.0, g)).numpy() for N in w["Ns"]]
    flops, reps = 0.0, 0
    t0 = time.perf_counter()
    while True:
        _, _, ov, om = oracle.prune_compress(w["ab"], sub)
        for N, X in zip(w["Ns"], Xs):
            if transposed:
                oracle.spmm_t(w["ab"], w["c"], ov, om, X, K)
            else:
                oracle.spmm(w["ab"], w["c"], ov, om, X, K)
            flops += 2.0 * rows * K * N
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    what = "transposed product dY * W" if transposed else "SpMM"
    return flops, dt, oracle.default_threads(), (
        f"{reps} x (prune+compress of {rows}x{K} weight rows and {what} for N in {w['Ns']})")


# ---------------------------------------------------------------- one workload's record
def roofline_of(w, r, per_group, tpeak, tpeak_src, hbm, hbm_src, name):
    """Roofline of the dominant kernel: the products or the prune, by share of the pass.  For the
    products: the launches of the bound that takes most of their time, aggregated (algorithmic
    bytes or flops over their summed time)."""
    if r["spmm_ms"] >= r["prune_ms"]:
        by_bound = {}
        for g in per_group:
            by_bound.setdefault(g["bound"], []).append(g)
        bound = max(by_bound, key=lambda b: sum(g["us_per_launch"] * g["launches_per_step"] for g in by_bound[b]))
        sel = by_bound[bound]
        t_s = sum(g["us_per_launch"] * g["launches_per_step"] for g in sel) * 1e-6
        n_l = sum(g["launches_per_step"] for g in sel)
        label = "st24_spmm " + ", ".join(f"{g['M']}x{g['K']} N={g['N']}" for g in sel)
        if bound == "tensor":
            fl = sum(2.0 * g["M"] * g["K"] * g["N"] * g["launches_per_step"] for g in sel)
            rf = {"bound": "tensor", "achieved": fl / t_s / 1e12, "peak": tpeak, "unit": "TFLOP/s",
                  "frac": fl / t_s / 1e12 / tpeak, "peak_source": tpeak_src, "flops_per_launch": fl / n_l}
        else:
            nb = sum(g["bytes_per_launch"] * g["launches_per_step"] for g in sel)
            rf = {"bound": "hbm", "achieved": nb / t_s / 1e9, "peak": hbm, "unit": "GB/s",
                  "frac": nb / t_s / 1e9 / hbm, "peak_source": hbm_src, "bytes_per_launch": nb / n_l}
        rf.update({"traffic": measured_traffic(name, "st24_spmm"), "kernel": label, "avg_launch_us": t_s * 1e6 / n_l})
        return rf
    gbs = prune_bytes(w) / (r["prune_ms"] * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
            "traffic": measured_traffic(name, "st24_prune_compress"), "kernel": "st24_prune_compress",
            "peak_source": hbm_src, "bytes_per_launch": prune_bytes(w) / n_prune(w),
            "avg_launch_us": r["prune_ms"] * 1e3 / n_prune(w)}


def measure(name, args, rank, world, target_s, cpu_budget_s):
    """Everything measured for one workload: the timed steps, per-kernel figures, the roofline of the
    dominant kernel, the end-to-end pass, the dense context and the CPU oracle baseline."""
    w = WORKLOADS[name]
    r = run_gpu(args, w, rank, world, target_s)
    R = r["passes_per_step"]
    pass_ms = max_over_ranks(r["pass_ms"], world, "cuda")
    ms_step = pass_ms * R
    flops = flops_per_pass(w)
    value = job_tflops(world, flops, pass_ms)
    hbm, bf16_peak, bf16_sus, peak_kind = peaks()
    long_region = args.steps * ms_step >= 1000.0
    tpeak, tpeak_src = tensor_peak(w["ab"], bf16_peak, bf16_sus, long_region, dense_op=w.get("op") == "spmm_t")
    hbm_src = f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback"

    # Every (shape, N) product group: its bound is the one its arithmetic
    # intensity meets first (flops / tensor peak vs bytes / HBM peak).
    per_group = []
    for gi, (ni, si) in enumerate(groups(w)):
        (M, K), N = w["shapes"][si], w["Ns"][ni]
        us = r["per_group_ms"][gi] * 1e3 / w["layers"]
        nbytes = launch_bytes(w, M, K, N)
        fl = 2.0 * M * K * N
        tensor_bound = tpeak is not None and fl / (tpeak * 1e12) > nbytes / (hbm * 1e9)
        g = {"M": M, "K": K, "N": N, "launches_per_step": w["layers"], "us_per_launch": us,
             "bytes_per_launch": nbytes, "GB/s": nbytes / (us * 1e-6) / 1e9,
             "tflops_dense_equiv": fl / (us * 1e-6) / 1e12, "tflops_actual": fl / 2 / (us * 1e-6) / 1e12,
             "bound": "tensor" if tensor_bound else "hbm"}
        g["frac"] = g["tflops_dense_equiv"] / tpeak if tensor_bound else g["GB/s"] / hbm
        g["share_of_pass"] = r["per_group_ms"][gi] / r["pass_ms"]
        per_group.append(g)
    prune_gbs = prune_bytes(w) / (r["prune_ms"] * 1e-3) / 1e9
    rec = {"workload": w["desc"], "name": name, "value": value, "unit": UNIT, "ms_per_step": ms_step,
           "passes_per_step": R, "ms_per_pass": pass_ms, "steps": args.steps, "dtype": w["ab"],
           "gpu_launches": args.steps * R * (n_spmm(w) + n_prune(w)), "clocks": r["clocks"],
           "roofline": roofline_of(w, r, per_group, tpeak, tpeak_src, hbm, hbm_src, name),
           "kernels": {"prune_compress": {"launches_per_pass": n_prune(w),
                                          "us_per_launch": r["prune_ms"] * 1e3 / n_prune(w),
                                          "GB/s": prune_gbs, "frac_hbm": prune_gbs / hbm},
                       "spmm": {"launches_per_pass": n_spmm(w), "us_per_launch": r["spmm_ms"] * 1e3 / n_spmm(w),
                                "GB/s": spmm_bytes(w) / (r["spmm_ms"] * 1e-3) / 1e9,
                                "tflops_dense_equiv": flops / (r["spmm_ms"] * 1e-3) / 1e12,
                                "tensor_peak_tflops": tpeak, "tensor_peak_source": tpeak_src,
                                "groups": per_group}},
           "config": {"name": name, "kernel": args.kernel, "shapes": w["shapes"], "Ns": w["Ns"],
                      "layers": w["layers"], "ab": w["ab"], "out": w["c"], "fixed_a": args.fixed_a,
                      "l2": "inputs larger than L2: every pass streams all weights (dense and compressed) from HBM"}}
    if r.get("extra_prune"):
        ep = dict(r["extra_prune"])
        shape = ep.pop("shape")
        for k, v in ep.items():
            v["frac_hbm"] = v["GB/s"] / hbm
            v["shape"] = shape
            rec["kernels"][k] = v
    if rank == 0 and not args.no_e2e:
        e2e_ms, h2d, d2h = run_e2e(args, w, r["layers"], r["stream"])
        rec["e2e"] = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                      "note": "one pass per step through the public API, host buffers, copies timed"}
    dev = r["layers"][0]["A"].device
    del r["layers"]
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_context:
        dc = dense_context(w, dev)
        rec["context"] = {"dense": dc, "dense_ms_per_pass": dc["ms_per_pass"],
                          "sparse_spmm_ms_per_pass": r["spmm_ms"]}
        if w.get("unstructured_context"):
            rec["context"]["dense_75pct_unstructured_zeros"] = dense_context(w, dev, w["unstructured_context"])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, dt, threads, sample = oracle_sample(w, cpu_budget_s)
        rec["cpu_baseline"] = {"value": f / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                               "sample": sample}
    torch.cuda.empty_cache()
    return rec


# Small cases that launch one kernel family a few times and exit: what the
# profiler captures (the last launches are the steady-state ones).
KERNEL_CASES = {
    "fp8_pair": "st24_spmm e4m3 28672x8192, N = 4096, one weight: 3 launches of the CTA-pair kernel",
    "prefill_pair": "st24_spmm bf16 11008x4096 and 4096x11008, N = 4096, beta = 1: 3 launches of each, alternating",
    "transposed_pair": "st24_spmm_t bf16 11008x4096 weight, N = 4096, beta = 1: 3 launches of the CTA-pair kernel",
    "decode_narrow": "st24_spmm bf16 4096x4096, N = 16, 4 weights: 2 rounds of 4 launches of the narrow kernel",
    "prune_bf16": "st24_prune_compress and st24_prune_compress_nm2 (4:8) of a bf16 28672x8192 weight: twice each",
    "fp8_groups": "st24_spmm e4m3 28672x8192 at N = 512, 4096 and 8192 (the tensor-bound groups), one weight: two rounds",
    "fp8_narrow": "st24_spmm e4m3 28672x8192 at N = 1 and 64 (the HBM-bound groups), one weight: two rounds",
    "decode_mix": "st24_spmm bf16 4096x4096 at N = 1, 16 and 32, one weight each: two rounds",
    "int8_mix": "st24_spmm int8 8192x8192 at N = 16 and 2048, row scales, bf16 out: two rounds",
    "demo_pair": "st24_spmm bf16 4096x4096, N = 4096: 3 launches",
    "transposed_both": "st24_spmm_t bf16 11008x4096 and 4096x11008 weights, N = 4096: two rounds",
}


def run_kernel_case(name):
    import structured_sparse_gemm_gb300 as st
    dev = torch.device("cuda", 0)
    st.load()
    g = inputs.generator(0)

    def compressed(ab, M, K):
        W = inputs.draw(ab, (M, K), 0.02, g).to(dev)
        v = torch.empty((M, K // 2), dtype=W.dtype, device=dev)
        m = torch.empty((M, K // 8), dtype=torch.uint8, device=dev)
        st.st24_prune_compress(W, v, m)
        return v, m

    def product(ab, M, K, N, beta, vm=None):
        v, m = vm if vm is not None else compressed(ab, M, K)
        X = inputs.draw(ab, (N, K), 1.0, g).to(dev)
        Y = inputs.draw("bf16", (N, M), 1.0, g).to(dev)
        scale = inputs.row_scale(M, g).to(dev) if ab == "s8" else None
        ws = torch.zeros(max(st.st24_spmm_workspace_bytes(ab, "bf16", M, N, K), 16), dtype=torch.uint8, device=dev)
        return lambda: st.st24_spmm(v, m, X, Y, K=K, beta=beta, row_scale=scale, workspace=ws, fixed_a=True)

    def transposed(M, K, N):
        v, m = compressed("bf16", M, K)
        dY = inputs.draw("bf16", (N, M), 1.0, g).to(dev)
        dX = inputs.draw("bf16", (N, K), 1.0, g).to(dev)
        return lambda: st.st24_spmm_t(v, m, dY, dX, K=K, beta=1.0)

    if name == "fp8_pair":
        calls = [product("e4m3", 28672, 8192, 4096, 0.0)] * 3
    elif name == "prefill_pair":
        a, b = product("bf16", 11008, 4096, 4096, 1.0), product("bf16", 4096, 11008, 4096, 1.0)
        calls = [a, b] * 3
    elif name == "transposed_pair":
        calls = [transposed(11008, 4096, 4096)] * 3
    elif name == "transposed_both":
        calls = [transposed(11008, 4096, 4096), transposed(4096, 11008, 4096)] * 2
    elif name == "decode_narrow":
        calls = [product("bf16", 4096, 4096, 16, 0.0) for _ in range(4)] * 2
    elif name == "decode_mix":
        calls = [product("bf16", 4096, 4096, n, 0.0) for n in (1, 16, 32)] * 2
    elif name == "fp8_groups":
        vm = compressed("e4m3", 28672, 8192)
        calls = [product("e4m3", 28672, 8192, n, 0.0, vm) for n in (512, 4096, 8192)] * 2
    elif name == "fp8_narrow":
        vm = compressed("e4m3", 28672, 8192)
        calls = [product("e4m3", 28672, 8192, n, 0.0, vm) for n in (1, 64)] * 2
    elif name == "int8_mix":
        vm = compressed("s8", 8192, 8192)
        calls = [product("s8", 8192, 8192, n, 0.0, vm) for n in (16, 2048)] * 2
    elif name == "demo_pair":
        calls = [product("bf16", 4096, 4096, 4096, 0.0)] * 3
    else:   # prune_bf16
        W = inputs.prune_weight_bf16().to(dev)
        M, K = W.shape
        v = torch.empty((M, K // 2), dtype=W.dtype, device=dev)
        m = torch.empty((M, K // 8), dtype=torch.uint8, device=dev)
        v2 = torch.empty((M, K), dtype=W.dtype, device=dev)
        m2 = torch.empty((M, K // 4), dtype=torch.uint8, device=dev)
        calls = [lambda: st.st24_prune_compress(W, v, m), lambda: st.st24_prune_compress_nm2(W, v2, m2, 4, 8)] * 2
    torch.cuda.synchronize()
    for c in calls:
        c()
    torch.cuda.synchronize()
    if st.st24_device_status() != 0:
        raise RuntimeError("device status set")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(WORKLOADS),
                    help="all = the headline workload plus every other one as a sub-record")
    ap.add_argument("--impl", default="st24", choices=["st24", "reference"])
    ap.add_argument("--target-s", type=float, default=6.0,
                    help="seconds the headline workload's timed region should last (sets passes per step)")
    ap.add_argument("--sub-target-s", type=float, default=1.5,
                    help="the same for each sub-workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-context", action="store_true", help="skip the dense torch context runs")
    ap.add_argument("--kernel", default="auto", choices=["auto", "tcgen05", "mma_sp", "mma_sp_direct"],
                    help="SpMM kernel family (auto = what st24_spmm picks)")
    ap.add_argument("--no-fixed-a", dest="fixed_a", action="store_false",
                    help="do not declare the weights fixed (ST24_SPMM_FIXED_A) to the products")
    ap.add_argument("--kernel-case", choices=sorted(KERNEL_CASES),
                    help="run one small profiling case (a few launches of one kernel family) and exit")
    args = ap.parse_args()
    if args.kernel_case:
        run_kernel_case(args.kernel_case)
        return
    head = HEADLINE if args.workload == "all" else args.workload
    subs = SUB_WORKLOADS if args.workload == "all" else []
    w = WORKLOADS[head]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    config = {"workload": w["desc"], "name": head, "kernel": args.kernel, "shapes": w["shapes"], "Ns": w["Ns"],
              "layers": w["layers"], "ab": w["ab"], "out": w["c"], "fixed_a": args.fixed_a,
              "l2": "inputs larger than L2: every pass streams all weights (dense and compressed) from HBM"}

    if args.impl == "reference":
        if rank != 0:
            return
        per_step, flops, threads, sample = [], 0.0, 1, ""
        for _ in range(args.warmup):
            oracle_sample(w, 0.0)
        for _ in range(args.steps):
            f, dt, threads, sample = oracle_sample(w, 4.0)
            per_step.append(dt)
            flops += f
        tot = sum(per_step)
        value = flops / tot / 1e12
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w["ab"],
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    rec = measure(head, args, rank, world, args.target_s, 8.0)
    config["passes_per_step"] = rec["passes_per_step"]
    line = {"metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w["ab"], "data": "synthetic", "config": config,
            "gpu_launches": rec["gpu_launches"], "clocks": rec["clocks"], "roofline": rec["roofline"],
            "kernels": rec["kernels"]}
    for k in ("e2e", "context", "cpu_baseline"):
        if k in rec:
            line[k] = rec[k]
    if subs:
        line["workloads"] = {s: measure(s, args, rank, world, args.sub_target_s, 4.0) for s in subs}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

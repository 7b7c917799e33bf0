"""Benchmark of the 2:4 sparse hot path on one GB300: prune + compress of the
weights, then the sparse x dense product for a batch of activations.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl {st24,reference}]

One step = prune_compress of every weight of the workload, then st24_spmm of
every weight with every activation width of the workload.  Inputs are seeded
synthetic tensors (st24_inputs).  The timed region is K steps replayed as CUDA
graphs on one stream, bracketed by a barrier and a synchronize.  Prints one JSON
line.  ``--impl reference`` times the CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
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

# Workloads: (name, element type, output type, weight shapes [(M, K)], activation widths, layers,
#             weight std, beta, per-row scale).  `layers` distinct weights of each shape per step,
#             so each product is launched behind another product (as in a model's layer stack),
#             not behind a graph boundary, and every step streams its weights from HBM.
WORKLOADS = {
    "decode_bf16": dict(ab="bf16", c="bf16", shapes=[(4096, 4096)], Ns=list(inputs.DECODE_NS), layers=16,
                        a_std=0.02, beta=0.0, scale=False,
                        desc="decode-shaped bf16 2:4 SpMM: 16 distinct 4096x4096 weights N(0,0.02), "
                             "activations N(0,1) for N in {1,8,16,32}, bf16 out"),
    "prefill_bf16": dict(ab="bf16", c="bf16", shapes=list(inputs.PREFILL_SHAPES), Ns=[4096], layers=2,
                         a_std=0.02, beta=1.0, scale=False,
                         desc="prefill-shaped bf16 2:4 SpMM: 2 x (11008x4096 and 4096x11008) distinct weights, "
                              "N=4096, beta=1 with C N(0,1), bf16 out"),
    "int8": dict(ab="s8", c="bf16", shapes=[(8192, 8192)], Ns=list(inputs.INT8_NS), layers=2, a_std=1.0,
                 beta=0.0, scale=True,
                 desc="int8 2:4 SpMM: 2 distinct 8192x8192 weights uniform [-127,127], N in {16,2048}, "
                      "int32 accumulate, per-row fp32 scale, bf16 out"),
    # The chapter's listing timed dense against 75%-unstructured-sparse weights run as dense (no
    # faster) at 4096^3; re-measured here with the 2:4 product beside both (context, not a target).
    "demo_bf16": dict(ab="bf16", c="bf16", shapes=[(4096, 4096)], Ns=[4096], layers=8, a_std=1.0, beta=0.0,
                      scale=False, unstructured_context=0.75,
                      desc="the listing's 4096^3 demo in bf16: 2:4 SpMM of 8 distinct 4096x4096 weights, "
                           "N=4096, beside dense and 75%-unstructured-zero dense matmuls"),
    "fp8": dict(ab="e4m3", c="bf16", shapes=[(28672, 8192)], Ns=list(inputs.FP8_NS), layers=2, a_std=0.02,
                beta=0.0, scale=False, extra_prune_bf16=(28672, 8192),
                desc="fp8-e4m3 2:4 SpMM: 2 distinct 28672x8192 weights N(0,0.02), N in {1,64,512,4096,8192}, "
                     "bf16 out"),
}


def flops_per_step(w):
    return sum(2.0 * M * K * N for (M, K) in w["shapes"] for N in w["Ns"]) * w["layers"]


def spmm_bytes(w):
    """Algorithmic HBM bytes of all SpMM launches of one step (compressed A, B, C, scale)."""
    return sum(launch_bytes(w, M, K, N) for (M, K) in w["shapes"] for N in w["Ns"]) * w["layers"]


def prune_bytes(w):
    es = inputs.ELEM_SIZE[w["ab"]]
    return sum(M * K * es + M * K // 2 * es + M * K // 8 for (M, K) in w["shapes"]) * w["layers"]


def groups(w):
    """(activation index, shape index) pairs, one captured graph and one timing each."""
    return [(ni, si) for ni in range(len(w["Ns"])) for si in range(len(w["shapes"]))]


def launch_bytes(w, M, K, N):
    """Algorithmic HBM bytes of one product: compressed A and metadata, B, C (read too when beta != 0), scale."""
    es = inputs.ELEM_SIZE[w["ab"]]
    cs = inputs.ELEM_SIZE[w["c"]]
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


def tensor_peak(ab: str, bf16_dense: float):
    """2:4-sparse tensor peak (dense-equivalent TFLOP/s) of an element type, and where it comes from.

    16-bit: twice the measured dense bf16 peak; e4m3: twice that again (the nominal
    fp8/bf16 ratio); int8: the measured mma.sp rate (tcgen05 has no int8 kind here)."""
    if ab in ("bf16", "f16"):
        return 2.0 * bf16_dense, "2 x measured dense bf16 (MEASURED_PEAKS.json bf16_tflops)"
    if ab == "e4m3":
        return 4.0 * bf16_dense, "4 x measured dense bf16 (sparse x2, fp8/bf16 nominal x2)"
    t = mma_sp_peak_tops(0)
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
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


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
            for N in w["Ns"]:
                X = inputs.draw(w["ab"], (N, K), 1.0, g).to(dev)
                Y = inputs.draw(w["c"], (N, M), 1.0, g).to(dev) if w["beta"] else \
                    torch.empty((N, M), dtype=inputs.TORCH_DTYPE[w["c"]], device=dev)
                ws_bytes = st.st24_spmm_workspace_bytes(w["ab"], w["c"], M, N, K)
                ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
                acts.append((X, Y, ws))
            layers.append(dict(A=A, values=values, meta=meta, scale=scale, acts=acts, M=M, K=K, si=si))
    return layers


def prune_phase(layers, stream=None):
    import structured_sparse_gemm_gb300 as st
    for L in layers:
        st.st24_prune_compress(L["A"], L["values"], L["meta"], stream=stream)


def spmm_phase(layers, w, stream=None, kernel="auto", only=None, fixed_a=True):
    """The products of one step.  Run inside a captured graph, after the prune
    graph has completed, so the weights are fixed for the whole phase
    (ST24_SPMM_FIXED_A)."""
    import structured_sparse_gemm_gb300 as st
    for ni in range(len(w["Ns"])):
        for L in layers:
            if only is not None and (ni, L["si"]) != only:
                continue
            X, Y, ws = L["acts"][ni]
            st.st24_spmm(L["values"], L["meta"], X, Y, K=L["K"], beta=w["beta"], row_scale=L["scale"],
                         workspace=ws, stream=stream, kernel=kernel, fixed_a=fixed_a)


def run_gpu(args, w, rank, world):
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
        # one graph for the prune phase, one per activation width for the products
        g_prune = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_prune, stream=stream):
            prune_phase(layers)
        g_spmm = []
        for grp in groups(w):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                spmm_phase(layers, w, kernel=args.kernel, only=grp, fixed_a=args.fixed_a)
            g_spmm.append(g)
    for _ in range(args.warmup):
        g_prune.replay()
        for g in g_spmm:
            g.replay()
    torch.cuda.synchronize()
    if st.st24_device_status() != 0:
        raise RuntimeError("device status after warm-up")

    nG = len(groups(w))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 + nG)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                ev[k][0].record(stream)
                g_prune.replay()
                ev[k][1].record(stream)
                for ni, g in enumerate(g_spmm):
                    g.replay()
                    ev[k][2 + ni].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    extra = None
    if w.get("extra_prune_bf16"):
        # prune/compress of the bf16 weight the fp8 one is cast from (timed apart from the step)
        M, K = w["extra_prune_bf16"]
        Wb = inputs.prune_weight_bf16(M, K).to(layers[0]["A"].device)
        vb = torch.empty((M, K // 2), dtype=torch.bfloat16, device=Wb.device)
        mb = torch.empty((M, K // 8), dtype=torch.uint8, device=Wb.device)
        for _ in range(3):
            st.st24_prune_compress(Wb, vb, mb, stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                st.st24_prune_compress(Wb, vb, mb, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        nbytes = M * K * 2 + M * K // 2 * 2 + M * K // 8
        extra = {"shape": [M, K], "us_per_launch": us, "GB/s": nbytes / (us * 1e-6) / 1e9, "bytes": nbytes}
        del vb, mb
        # the same weight quantised per row to e4m3, then pruned and compressed, in one pass
        vq = torch.empty((M, K // 2), dtype=torch.float8_e4m3fn, device=Wb.device)
        mq = torch.empty((M, K // 8), dtype=torch.uint8, device=Wb.device)
        sq = torch.empty(M, dtype=torch.float32, device=Wb.device)
        for _ in range(3):
            st.st24_quantize_prune_compress(Wb, vq, mq, sq, stream=stream)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                st.st24_quantize_prune_compress(Wb, vq, mq, sq, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        nbytes = M * K * 2 + M * K // 2 + M * K // 8 + 4 * M
        extra["quantize_e4m3"] = {"us_per_launch": us, "GB/s": nbytes / (us * 1e-6) / 1e9, "bytes": nbytes}
        del vq, mq, sq
        # the same weight pruned 2:8 (kept in the 2:4 form)
        vn = torch.empty((M, K // 2), dtype=torch.bfloat16, device=Wb.device)
        mn = torch.empty((M, K // 8), dtype=torch.uint8, device=Wb.device)
        for _ in range(3):
            st.st24_prune_compress_nm(Wb, vn, mn, 2, 8, stream=stream)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                st.st24_prune_compress_nm(Wb, vn, mn, 2, 8, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        nbytes = M * K * 2 + M * K // 2 * 2 + M * K // 8
        extra["nm_2of8"] = {"us_per_launch": us, "GB/s": nbytes / (us * 1e-6) / 1e9, "bytes": nbytes}
        del Wb, vn, mn
    total_ms = ev[0][0].elapsed_time(ev[-1][-1])
    prune_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    spmm_ms = sum(e[1].elapsed_time(e[-1]) for e in ev)
    per_group_ms = [sum(e[1 + gi].elapsed_time(e[2 + gi]) for e in ev) / args.steps for gi in range(nG)]
    status = st.st24_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    return dict(total_ms=total_ms, prune_ms=prune_ms, spmm_ms=spmm_ms, per_group_ms=per_group_ms, clocks=clk.summary(),
                extra_prune=extra,
                layers=layers, stream=stream)


def run_e2e(args, w, layers, stream):
    """Same step through the public API with host inputs: H2D of the weights and
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
                    st.st24_spmm(L["values"], L["meta"], X, Y, K=L["K"], beta=w["beta"], row_scale=L["scale"],
                                 workspace=ws, fixed_a=fixed)
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
    return ms, h2d, d2h


def dense_context(w, dev, zero_fraction: float = 0.0):
    """torch.matmul of the unpruned shapes (context only; bf16/f16 dense, int8/fp8 via bf16);
    with zero_fraction, of weights with that fraction of unstructured zeros (a dense kernel)."""
    times = []
    for (M, K) in w["shapes"]:
        W = torch.randn(M, K, device=dev, dtype=torch.bfloat16)
        if zero_fraction:
            W = W * (torch.rand(M, K, device=dev) >= zero_fraction)
        for N in w["Ns"]:
            X = torch.randn(N, K, device=dev, dtype=torch.bfloat16)
            for _ in range(3):
                X @ W.t()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(10):
                X @ W.t()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / 10)
    return sum(times) * w["layers"]


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
    Xs = [inputs.raw(inputs.draw(w["ab"], (N, K), 1.0, g)).numpy() for N in w["Ns"]]
    flops, reps = 0.0, 0
    t0 = time.perf_counter()
    while True:
        _, _, ov, om = oracle.prune_compress(w["ab"], sub)
        for N, X in zip(w["Ns"], Xs):
            oracle.spmm(w["ab"], w["c"], ov, om, X, K)
            flops += 2.0 * rows * K * N
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return flops, dt, oracle.default_threads(), (
        f"{reps} x (prune+compress of {rows}x{K} weight rows and SpMM for N in {w['Ns']})")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode_bf16", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="st24", choices=["st24", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kernel", default="auto", choices=["auto", "tcgen05", "mma_sp", "mma_sp_direct"],
                    help="SpMM kernel family (auto = what st24_spmm picks)")
    ap.add_argument("--no-fixed-a", dest="fixed_a", action="store_false",
                    help="do not declare the weights fixed (ST24_SPMM_FIXED_A) to the products")
    args = ap.parse_args()
    w = WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    config = {"workload": w["desc"], "name": args.workload, "kernel": args.kernel, "shapes": w["shapes"], "Ns": w["Ns"],
              "layers": w["layers"], "ab": w["ab"], "out": w["c"], "fixed_a": args.fixed_a,
              "l2": "inputs larger than L2: every step streams all weights (dense and compressed) from HBM"}

    if args.impl == "reference":
        if rank != 0:
            return
        per_step, flops, threads, sample = [], 0.0, 1, ""
        for _ in range(args.warmup):
            oracle_sample(w, 0.0)
        for _ in range(args.steps):
            f, dt, threads, sample = oracle_sample(w, 8.0)
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
    r = run_gpu(args, w, rank, world)
    ms_step = max_over_ranks(r["total_ms"] / args.steps, world, "cuda")
    flops = flops_per_step(w)
    value = job_tflops(world, flops, ms_step)
    hbm, bf16_peak, bf16_sus, peak_kind = peaks()

    spmm_launch_ms = r["spmm_ms"] / args.steps / n_spmm(w)
    prune_launch_ms = r["prune_ms"] / args.steps / n_prune(w)
    spmm_gbs = spmm_bytes(w) / (r["spmm_ms"] / args.steps * 1e-3) / 1e9
    prune_gbs = prune_bytes(w) / (r["prune_ms"] / args.steps * 1e-3) / 1e9
    tpeak, tpeak_src = tensor_peak(w["ab"], bf16_peak)
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
        g["share_of_step"] = r["per_group_ms"][gi] / (r["total_ms"] / args.steps)
        per_group.append(g)

    # The dominant kernel (the products or the prune, by share of the step).
    # For the products: the launches of the bound that takes most of their
    # time, aggregated (algorithmic bytes or flops over their summed time).
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
            roofline = {"bound": "tensor", "achieved": fl / t_s / 1e12, "peak": tpeak, "unit": "TFLOP/s",
                        "frac": fl / t_s / 1e12 / tpeak, "peak_source": tpeak_src, "flops_per_launch": fl / n_l}
        else:
            nb = sum(g["bytes_per_launch"] * g["launches_per_step"] for g in sel)
            roofline = {"bound": "hbm", "achieved": nb / t_s / 1e9, "peak": hbm, "unit": "GB/s",
                        "frac": nb / t_s / 1e9 / hbm, "peak_source": hbm_src, "bytes_per_launch": nb / n_l}
        roofline.update({"traffic": measured_traffic(args.workload, "st24_spmm"), "kernel": label,
                         "avg_launch_us": t_s * 1e6 / n_l})
    else:
        roofline = {"bound": "hbm", "achieved": prune_gbs, "peak": hbm, "unit": "GB/s", "frac": prune_gbs / hbm,
                    "traffic": measured_traffic(args.workload, "st24_prune_compress"),
                    "kernel": "st24_prune_compress", "peak_source": hbm_src,
                    "bytes_per_launch": prune_bytes(w) / n_prune(w), "avg_launch_us": prune_launch_ms * 1e3}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w["ab"], "data": "synthetic", "config": config,
            "gpu_launches": args.steps * (n_spmm(w) + n_prune(w)),
            "clocks": r["clocks"], "roofline": roofline,
            "kernels": {"prune_compress": {"launches_per_step": n_prune(w), "us_per_launch": prune_launch_ms * 1e3,
                                           "GB/s": prune_gbs, "frac_hbm": prune_gbs / hbm},
                        "spmm": {"launches_per_step": n_spmm(w), "us_per_launch": spmm_launch_ms * 1e3,
                                 "GB/s": spmm_gbs,
                                 "tflops_dense_equiv": flops / (r["spmm_ms"] / args.steps * 1e-3) / 1e12,
                                 "tensor_peak_tflops": tpeak, "tensor_peak_source": tpeak_src,
                                 "groups": per_group}}}
    if r.get("extra_prune"):
        ep = dict(r["extra_prune"])
        q = ep.pop("quantize_e4m3", None)
        nm = ep.pop("nm_2of8", None)
        if nm:
            nm["frac_hbm"] = nm["GB/s"] / hbm
            nm["shape"] = ep["shape"]
            line["kernels"]["prune_compress_nm_2of8_bf16"] = nm
        ep["frac_hbm"] = ep["GB/s"] / hbm
        line["kernels"]["prune_compress_bf16"] = ep
        if q:
            q["frac_hbm"] = q["GB/s"] / hbm
            q["shape"] = ep["shape"]
            line["kernels"]["quantize_prune_compress_bf16_to_e4m3"] = q
    if rank == 0 and not args.no_e2e:
        e2e_ms, h2d, d2h = run_e2e(args, w, r["layers"], r["stream"])
        line["e2e"] = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
    if rank == 0:
        line["context"] = {"dense_torch_matmul_ms_per_step": dense_context(w, r["layers"][0]["A"].device)}
        if w.get("unstructured_context"):
            line["context"]["dense_matmul_75pct_unstructured_zeros_ms_per_step"] = dense_context(
                w, r["layers"][0]["A"].device, w["unstructured_context"])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, dt, threads, sample = oracle_sample(w, 10.0)
        line["cpu_baseline"] = {"value": f / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": sample}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

"""SpMM on the GPU against the oracle, element by element.

Small and ragged shapes are compared in full; the full-size workloads are
compared on sampled outputs the oracle computes one by one, plus properties
that hold at any size (determinism, workspace reuse)."""
import numpy as np
import pytest
import torch

import oracle
import st24_inputs as inputs
import structured_sparse_gemm_gb300 as st
from helpers import assert_close, bits, decode_out

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def gpu_run(case, out=None, repeat=1, ws=None, kernel="auto"):
    """Prune+compress A and run the product on the GPU through the C ABI."""
    Ad = case.A.to(DEV)
    values, meta = st.compress(Ad)
    X = case.X.to(DEV)
    tdt = inputs.TORCH_DTYPE[case.c]
    outs = []
    for _ in range(repeat):
        Y = case.C_in.to(DEV).to(tdt) if case.C_in is not None else torch.full(
            (case.N, case.M), 3, dtype=torch.int32 if case.c == "s32" else torch.float32, device=DEV).to(tdt)
        scale = case.scale.to(DEV) if case.scale is not None else None
        wsz = st.st24_spmm_workspace_bytes(case.ab, case.c, case.M, case.N, case.K)
        w = ws if ws is not None else (torch.zeros(max(wsz, 1), dtype=torch.uint8, device=DEV) if wsz else None)
        st.st24_spmm(values, meta, X, Y, K=case.K, alpha=case.alpha, beta=case.beta, row_scale=scale, workspace=w,
                     kernel=kernel)
        torch.cuda.synchronize()
        outs.append(Y)
    assert st.st24_device_status() == 0
    return values, meta, outs


def oracle_full(case):
    _, _, ov, om = oracle.prune_compress(case.ab, bits(case.A))
    Cin = bits(case.C_in.to(inputs.TORCH_DTYPE[case.c])) if case.C_in is not None else None
    out, acc = oracle.spmm(case.ab, case.c, ov, om, bits(case.X), case.K, alpha=case.alpha, beta=case.beta,
                           C_in=Cin, scale=None if case.scale is None else case.scale.numpy())
    return (acc.astype(np.float64) if case.c == "s32" else out)


def check_full(case, kernel="auto"):
    _, _, (Y,) = gpu_run(case, kernel=kernel)
    assert_close(decode_out(Y), oracle_full(case), case.ab, case.c, case.name)


def sample_points(M, N, count, seed=0):
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, count)) + [0, M - 1, min(127, M - 1), min(128, M - 1)] * 2
    cols = list(rng.integers(0, N, count)) + [0, N - 1] * 4
    return np.array(rows, np.int64), np.array(cols, np.int64)


def check_sampled(case, count=2048, kernel="auto"):
    values, meta, (Y,) = gpu_run(case, kernel=kernel)
    rows, cols = sample_points(case.M, case.N, count)
    # the oracle samples from its own compressed form of the same input
    _, _, ov, om = oracle.prune_compress(case.ab, bits(case.A))
    Cin = bits(case.C_in.to(inputs.TORCH_DTYPE[case.c])) if case.C_in is not None else None
    ref, acc = oracle.spmm_sampled(case.ab, case.c, ov, om, bits(case.X), case.K, rows, cols, alpha=case.alpha,
                                   beta=case.beta, C_in=Cin,
                                   scale=None if case.scale is None else case.scale.numpy())
    got = decode_out(Y)[cols, rows]
    full_scale = decode_out(Y)
    assert_close(got, acc.astype(np.float64) if case.c == "s32" else ref, case.ab, case.c, case.name)
    assert np.isfinite(full_scale).all()
    # and the GPU's compressed form is the oracle's
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)


# ---- small / ragged shapes, compared in full ------------------------------------

KERNELS = ["tcgen05", "mma_sp"]


def kernels_for(ab):
    return ["mma_sp"] if ab == "s8" else KERNELS


@pytest.mark.parametrize("kernel", KERNELS)
def test_small_f16_workload(kernel):
    check_full(inputs.small_f16(), kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("ab", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("c", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(200, 37, 384), (129, 1, 128), (64, 130, 512), (300, 64, 256), (384, 200, 1280)])
def test_ragged(kernel, ab, c, M, N, K):
    if kernel not in kernels_for(ab):
        pytest.skip("no int8 tcgen05 kind on sm_103a")
    # int8 sums reach ~1e5 and overflow f16 unless scaled, as the int8 workload is (1/127 per row)
    case = inputs.spmm_case(ab, c, M, N, K, a_std=0.02 if ab == "e4m3" else 1.0, seed=M + N + K,
                            with_scale=(ab == "s8"))
    check_full(case, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("ab", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("N,c", [(48, "bf16"), (300, "bf16"), (300, "f32"), (300, "f16")])
def test_alpha_beta_scale(kernel, ab, N, c):
    # N = 300 runs the wide-tile path (two 256 x 224 tiles per pair row, ragged) with C staged per chunk
    if kernel not in kernels_for(ab):
        pytest.skip("no int8 tcgen05 kind on sm_103a")
    case = inputs.spmm_case(ab, c, 257, N, 640, alpha=0.5, beta=-0.75, with_scale=True,
                            a_std=0.02 if ab == "e4m3" else 1.0, seed=11)
    check_full(case, kernel=kernel)


# The register-direct family (16-bit inputs, N <= 32): ragged rows, every
# split of K over a cluster (1, 2, 4, 8 CTAs), several 512-K rounds per CTA,
# K ranges that end inside a round, and each B width it stages (8, 16, 32).
DIRECT_SHAPES = [(129, 1, 128), (200, 5, 384), (300, 16, 640), (64, 32, 512), (385, 24, 1280),
                 (130, 17, 4224), (1000, 9, 8192), (77, 8, 2048)]


@pytest.mark.parametrize("ab", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("c", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,K", DIRECT_SHAPES)
def test_direct_ragged(ab, c, M, N, K):
    case = inputs.spmm_case(ab, c, M, N, K, a_std=0.02 if ab == "e4m3" else 1.0, seed=M + N + K,
                            with_scale=(ab == "s8"))
    check_full(case, kernel="mma_sp_direct")


@pytest.mark.parametrize("ab", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("N,c", [(1, "bf16"), (13, "f16"), (32, "f32")])
def test_direct_alpha_beta_scale(ab, N, c):
    case = inputs.spmm_case(ab, c, 257, N, 640, alpha=0.5, beta=-0.75, with_scale=True,
                            a_std=0.02 if ab == "e4m3" else 1.0, seed=11)
    check_full(case, kernel="mma_sp_direct")


@pytest.mark.parametrize("kernel", ["mma_sp", "mma_sp_direct"])
@pytest.mark.parametrize("N", [1, 16, 32])
def test_int8_large_sums_exact(kernel, N):
    """int8 -> int32 stays bit-exact when the sums need 26 bits (beyond fp32's
    24): weights and activations all large and mostly of one sign, K = 8192."""
    g = inputs.generator(77)
    A = torch.randint(100, 128, (256, 8192), generator=g).to(torch.int8)
    A[:, ::61] = -128
    X = torch.randint(96, 128, (N, 8192), generator=g).to(torch.int8)
    case = inputs.SpmmCase(f"int8 large sums N={N}", "s8", "s32", 256, N, 8192, 1.0, 0.0, A, X, None, None)
    _, _, (Y,) = gpu_run(case, kernel=kernel)
    ref = oracle_full(case)
    assert np.abs(ref).max() > 2 ** 25
    assert np.array_equal(decode_out(Y).astype(np.int64), ref.astype(np.int64))


@pytest.mark.parametrize("ab,N,K", [("bf16", 4, 1024), ("bf16", 5, 1024), ("bf16", 64, 1024), ("bf16", 65, 1024),
                                    ("e4m3", 64, 1024), ("e4m3", 64, 1152), ("e4m3", 65, 1024), ("f16", 1, 1024)])
def test_auto_at_the_family_boundaries(ab, N, K):
    # 16-bit inputs: N <= 4 runs the register-direct kernel (one wave), 5..64
    # the narrow tcgen05 one, 65 and up the wide tcgen05 one; e4m3 with N <= 64
    # runs the narrow one when K is a multiple of 256, else the wide one
    check_full(inputs.spmm_case(ab, "bf16", 512, N, K, a_std=0.02, seed=N))


def test_direct_rejects_wide_n():
    with pytest.raises(st.St24Error) as e:
        gpu_run(inputs.spmm_case("bf16", "bf16", 128, 33, 256), kernel="mma_sp_direct")
    assert e.value.status == 2


@pytest.mark.parametrize("kernel,ab,N", [("tcgen05", "bf16", 100), ("tcgen05", "e4m3", 300), ("mma_sp", "f16", 24),
                                         ("mma_sp", "s8", 100), ("mma_sp_direct", "bf16", 24),
                                         ("mma_sp_direct", "e4m3", 9)])
@pytest.mark.parametrize("pad_c", [8, 3])
def test_strided_b_and_c(kernel, ab, N, pad_c):
    """B and C as views into wider buffers (ldb = K + 64, ldc = M + pad_c): the
    product reads and writes through the strides and leaves the padding alone."""
    M, K = 200, 512
    c = "s32" if ab == "s8" else "bf16"
    case = inputs.spmm_case(ab, c, M, N, K, a_std=0.02 if ab == "e4m3" else 1.0, seed=3,
                            beta=0.0 if ab == "s8" else 0.5)
    values, meta = st.compress(case.A.to(DEV))
    Xw = torch.zeros((N, K + 64), dtype=case.X.dtype, device=DEV)
    Xw[:, :K] = case.X.to(DEV)
    tdt = inputs.TORCH_DTYPE[c]
    Yw = torch.full((N, M + pad_c), 7, dtype=tdt, device=DEV)
    if case.C_in is not None:
        Yw[:, :M] = case.C_in.to(DEV).to(tdt)
    wsz = st.st24_spmm_workspace_bytes(ab, c, M, N, K)
    ws = torch.zeros(max(wsz, 1), dtype=torch.uint8, device=DEV)
    st.st24_spmm(values, meta, Xw[:, :K], Yw[:, :M], K=K, beta=case.beta, workspace=ws, kernel=kernel)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    assert bool((Yw[:, M:] == 7).all())
    assert_close(decode_out(Yw[:, :M].contiguous()), oracle_full(case), ab, c, case.name + " strided")


@pytest.mark.parametrize("N", [8, 200])
def test_int8_int32_bit_exact(N):
    case = inputs.spmm_case("s8", "s32", 384, N, 1024, seed=N)
    check_full(case)


def test_k_equals_zero():
    Y = torch.randn(5, 7, device=DEV)
    Y0 = Y.clone()
    X = torch.empty((5, 0), dtype=torch.bfloat16, device=DEV)
    v = torch.empty((7, 0), dtype=torch.bfloat16, device=DEV)
    e = torch.empty((7, 0), dtype=torch.uint8, device=DEV)
    st.st24_spmm(v, e, X, Y, K=0, beta=2.0)
    torch.cuda.synchronize()
    assert torch.equal(Y, 2.0 * Y0)


def test_deterministic_and_workspace_reuse():
    # the one-CTA tcgen05 kernel splits decode tiles over K through the workspace
    case = inputs.decode_bf16(32)
    wsz = st.st24_spmm_workspace_bytes("bf16", "bf16", case.M, case.N, case.K)
    assert wsz > 0
    ws = torch.zeros(wsz, dtype=torch.uint8, device=DEV)
    _, _, outs = gpu_run(case, repeat=3, ws=ws, kernel="tcgen05")
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    # the per-tile counters (the workspace's last bytes) are back at zero after each call
    assert int(ws[-256:].sum()) == 0


# ---- the workloads at their full sizes -------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS + ["mma_sp_direct"])
@pytest.mark.parametrize("N", inputs.DECODE_NS)
def test_decode_bf16_full(kernel, N):
    check_full(inputs.decode_bf16(N), kernel=kernel)


@pytest.mark.parametrize("kernel,N", [(k, n) for k in KERNELS for n in (1, 32, 200)] +
                         [("mma_sp_direct", 1), ("mma_sp_direct", 32)])
def test_fixed_weights_back_to_back(kernel, N):
    """Products over several weights enqueued back to back with ST24_SPMM_FIXED_A
    (weight tiles loaded while the previous product still runs) equal the same
    products without it, bit for bit, and the first one matches the oracle."""
    cases = [inputs.spmm_case("bf16", "bf16", 1024, N, 2048, seed=40 + i) for i in range(4)]
    layers = []
    for c in cases:
        values, meta = st.compress(c.A.to(DEV))
        layers.append((values, meta, c.X.to(DEV)))
    torch.cuda.synchronize()
    wsz = st.st24_spmm_workspace_bytes("bf16", "bf16", 1024, N, 2048)
    ws = torch.zeros(max(wsz, 1), dtype=torch.uint8, device=DEV)   # one workspace shared by the chain
    outs = {}
    for fixed in (False, True):
        Ys = [torch.empty((N, 1024), dtype=torch.bfloat16, device=DEV) for _ in layers]
        for _ in range(2):
            for (values, meta, X), Y in zip(layers, Ys):
                st.st24_spmm(values, meta, X, Y, K=2048, workspace=ws, kernel=kernel, fixed_a=fixed)
        torch.cuda.synchronize()
        outs[fixed] = Ys
    assert st.st24_device_status() == 0
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)
    assert_close(decode_out(outs[True][0]), oracle_full(cases[0]), "bf16", "bf16", "fixed weights")


def test_kernel_families_agree():
    # the two kernel families compute the same sums; on one k-block per tile they agree closely
    case = inputs.spmm_case("bf16", "f32", 512, 96, 2048, seed=5)
    _, _, (Ya,) = gpu_run(case, kernel="tcgen05")
    _, _, (Yb,) = gpu_run(case, kernel="mma_sp")
    ref = oracle_full(case)
    assert_close(decode_out(Ya), ref, "bf16", "f32", "tcgen05")
    assert_close(decode_out(Yb), ref, "bf16", "f32", "mma_sp")


def test_tcgen05_rejects_int8():
    case = inputs.spmm_case("s8", "s32", 128, 16, 256, seed=1)
    with pytest.raises(st.St24Error) as e:
        gpu_run(case, kernel="tcgen05")
    assert e.value.status == 2


@pytest.mark.slow
@pytest.mark.parametrize("M,K", inputs.PREFILL_SHAPES)
def test_prefill_bf16_sampled(M, K):
    check_sampled(inputs.prefill_bf16(M, K))


@pytest.mark.slow
@pytest.mark.parametrize("N", inputs.INT8_NS)
def test_int8_sampled(N):
    check_sampled(inputs.int8(N))


@pytest.mark.slow
def test_int8_int32_full_size_sampled():
    check_sampled(inputs.int8(2048, out="s32"))


@pytest.mark.slow
@pytest.mark.parametrize("N", inputs.FP8_NS)
def test_fp8_sampled(N):
    check_sampled(inputs.fp8(N), count=1024)


@pytest.mark.slow
@pytest.mark.parametrize("N", [64, 4096])
def test_fp8_sampled_mma_sp(N):
    check_sampled(inputs.fp8(N), count=512, kernel="mma_sp")


@pytest.mark.slow
def test_prefill_bf16_sampled_mma_sp():
    check_sampled(inputs.prefill_bf16(4096, 11008), count=512, kernel="mma_sp")


# Few, long output tiles: the CTA pairs split them over K and finish them
# through the workspace (the last contributor sums the partials); more tiles
# run as whole tiles in data-parallel waves.  Both schedules, with beta, on
# 224- and 128-column tiles with two accumulators and (e4m3, N = 449..512)
# 256-column tiles with one.
@pytest.mark.parametrize("ab", ["bf16", "e4m3"])
@pytest.mark.parametrize("M,N,K", [(256, 200, 32768), (512, 448, 16384), (1024, 1000, 2048), (1000, 500, 4096),
                                   (256, 480, 65536)])
def test_pair_schedules(ab, M, N, K):
    case = inputs.spmm_case(ab, "bf16", M, N, K, a_std=0.02 if ab == "e4m3" else 1.0, seed=M + N, beta=0.5)
    check_sampled(case, count=1024, kernel="tcgen05")


# e4m3 256-column tiles with beta = 0 run with one more stage and no C
# staging (outputs by direct stores): whole tiles and tiles split over K.
@pytest.mark.parametrize("M,N,K", [(1000, 500, 4096), (256, 480, 65536)])
def test_wide_tiles_beta0(M, N, K):
    case = inputs.spmm_case("e4m3", "bf16", M, N, K, a_std=0.02, seed=M + N + K + 1)
    check_sampled(case, count=1024, kernel="tcgen05")

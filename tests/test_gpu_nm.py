"""N:M prune + compress on the GPU against the oracle, bit for bit: one 2:4 form
(1:4, 1:8, 2:8) and the product of that form through st24_spmm; two 2:4 forms
side by side (4:8, 3:8, ...) and their product in one accumulator
(ST24_SPMM_TWO_FORMS) on every kernel family that takes it."""
import numpy as np
import pytest
import torch

import oracle
import st24_inputs as inputs
import structured_sparse_gemm_gb300 as st
from helpers import assert_close, bits, decode_out

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PATTERNS = [(1, 4), (1, 8), (2, 8), (2, 4)]


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("n,m", PATTERNS)
@pytest.mark.parametrize("M,K", [(37, 96), (5, 8), (130, 4104), (513, 2048)])
def test_matches_oracle(dt, n, m, M, K):
    W = inputs.draw(dt, (M, K), 0.02 if dt == "e4m3" else 1.0, inputs.generator(M + K + n + m))
    values, meta = st.compress_nm(W.to(DEV), n, m)
    torch.cuda.synchronize()
    _, ov, om = oracle.prune_compress_nm(dt, n, m, bits(W))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)


def test_k_ending_in_half_a_metadata_byte():
    # 1:4 with K % 8 == 4: the last 4 elements of a row fill half a metadata byte
    W = inputs.draw("bf16", (9, 12), 1.0, inputs.generator(1))
    values, meta = st.compress_nm(W.to(DEV), 1, 4)
    _, ov, om = oracle.prune_compress_nm("bf16", 1, 4, bits(W))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)


def test_tie_heavy_rows():
    vals = np.random.default_rng(2).choice([-2, -1, 0, 1, 2], size=(64, 256))
    W = torch.tensor(vals, dtype=torch.bfloat16)
    for n, m in PATTERNS:
        values, meta = st.compress_nm(W.to(DEV), n, m)
        _, ov, om = oracle.prune_compress_nm("bf16", n, m, bits(W))
        assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
        assert np.array_equal(meta.cpu().numpy(), om)


@pytest.mark.parametrize("n,m", [(1, 4), (2, 8)])
@pytest.mark.parametrize("N", [8, 300])
def test_product_of_nm_form(n, m, N):
    # the 2:4 form of an N:M-pruned weight multiplies like any compressed weight
    M, K = 384, 1024
    W = inputs.draw("bf16", (M, K), 0.02, inputs.generator(5))
    values, meta = st.compress_nm(W.to(DEV), n, m)
    X = inputs.draw("bf16", (N, K), 1.0, inputs.generator(6))
    Y = torch.empty((N, M), dtype=torch.float32, device=DEV)
    ws = torch.zeros(max(st.st24_spmm_workspace_bytes("bf16", "f32", M, N, K), 1), dtype=torch.uint8, device=DEV)
    st.st24_spmm(values, meta, X.to(DEV), Y, K=K, workspace=ws)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    pruned, ov, om = oracle.prune_compress_nm("bf16", n, m, bits(W))
    ref, _ = oracle.spmm("bf16", "f32", ov, om, bits(X), K)
    assert_close(decode_out(Y), ref, "bf16", "f32", f"{n}:{m} N={N}")
    # and the compressed-form product is the dense product of the N:M-pruned weight
    dense, _ = oracle.gemm_dense("bf16", "f32", pruned, bits(X))
    assert np.allclose(dense, ref, rtol=0, atol=1e-9 * np.abs(ref).max())


# ---- up to four kept per subgroup (4:8, 3:8, ...) as two 2:4 forms ---------------

PATTERNS2 = [(4, 8), (3, 8), (2, 8), (1, 4), (4, 4)]


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("n,m", PATTERNS2)
@pytest.mark.parametrize("M,K", [(37, 96), (5, 8), (130, 4104), (513, 2048)])
def test_two_forms_match_oracle(dt, n, m, M, K):
    if K % m:
        pytest.skip("K must be a multiple of m")
    W = inputs.draw(dt, (M, K), 0.02 if dt == "e4m3" else 1.0, inputs.generator(M + K + n + m))
    values, meta = st.compress_nm2(W.to(DEV), n, m)
    torch.cuda.synchronize()
    _, ov, om = oracle.prune_compress_nm2(dt, n, m, bits(W))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)


def test_two_forms_tie_heavy_rows():
    vals = np.random.default_rng(3).choice([-2, -1, 0, 1, 2], size=(64, 256))
    W = torch.tensor(vals, dtype=torch.bfloat16)
    for n, m in PATTERNS2:
        values, meta = st.compress_nm2(W.to(DEV), n, m)
        _, ov, om = oracle.prune_compress_nm2("bf16", n, m, bits(W))
        assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
        assert np.array_equal(meta.cpu().numpy(), om)


def _two_form_product(ab, c, M, N, K, kernel, seed, beta=0.0):
    W = inputs.draw(ab, (M, K), 0.02 if ab == "e4m3" else 1.0, inputs.generator(seed))
    X = inputs.draw(ab, (N, K), 1.0, inputs.generator(seed + 1))
    values, meta = st.compress_nm2(W.to(DEV), 4, 8)
    tdt = inputs.TORCH_DTYPE[c]
    C_in = inputs.draw(c, (N, M), 1.0, inputs.generator(seed + 2)) if beta else None
    Y = C_in.to(DEV).to(tdt) if beta else torch.zeros((N, M), dtype=tdt, device=DEV)
    scale = inputs.row_scale(M, inputs.generator(seed + 3)).to(DEV) if ab == "s8" and c != "s32" else None
    wsz = st.st24_spmm_workspace_bytes(ab, c, M, N, 2 * K)
    ws = torch.zeros(max(wsz, 16), dtype=torch.uint8, device=DEV)
    st.st24_spmm(values, meta, X.to(DEV), Y, K=K, beta=beta, row_scale=scale, workspace=ws, kernel=kernel,
                 two_forms=True)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    # the oracle's own two forms, multiplied as the M x 2K matrix [form 0 | form 1] by B stacked twice
    _, ov, om = oracle.prune_compress_nm2(ab, 4, 8, bits(W))
    X2 = np.concatenate([bits(X), bits(X)], axis=1)
    ref, acc = oracle.spmm(ab, c, ov, om, X2, 2 * K, beta=beta,
                           C_in=None if C_in is None else bits(C_in.to(tdt)),
                           scale=None if scale is None else scale.cpu().numpy())
    return decode_out(Y), (acc.astype(np.float64) if c == "s32" else ref)


@pytest.mark.parametrize("kernel,ab,N", [("auto", "bf16", 1), ("auto", "bf16", 16), ("auto", "bf16", 300),
                                         ("tcgen05_narrow", "f16", 40), ("tcgen05", "bf16", 100),
                                         ("mma_sp", "bf16", 24), ("auto", "e4m3", 1), ("auto", "e4m3", 64),
                                         ("auto", "e4m3", 520), ("tcgen05", "e4m3", 16)])
@pytest.mark.parametrize("M,K", [(300, 512), (130, 1024)])
def test_two_form_product(kernel, ab, N, M, K):
    got, ref = _two_form_product(ab, "bf16", M, N, K, kernel, seed=M + N)
    assert_close(got, ref, ab, "bf16", f"4:8 {kernel} {ab} {M}x{N}x{K}")


@pytest.mark.parametrize("N,c", [(16, "s32"), (300, "bf16")])
def test_two_form_product_int8(N, c):
    got, ref = _two_form_product("s8", c, 256, N, 1024, "auto", seed=N)
    assert_close(got, ref, "s8", c, f"4:8 int8 N={N}")


def test_two_form_product_beta():
    got, ref = _two_form_product("bf16", "bf16", 300, 48, 768, "auto", seed=9, beta=0.5)
    assert_close(got, ref, "bf16", "bf16", "4:8 beta")


def test_two_form_product_is_the_pruned_product():
    # the two-form result equals the dense product of the 4:8-pruned weight
    M, N, K = 128, 32, 512
    W = inputs.draw("bf16", (M, K), 1.0, inputs.generator(4))
    X = inputs.draw("bf16", (N, K), 1.0, inputs.generator(5))
    values, meta = st.compress_nm2(W.to(DEV), 4, 8)
    Y = torch.empty((N, M), dtype=torch.float32, device=DEV)
    st.st24_spmm(values, meta, X.to(DEV), Y, K=K, two_forms=True)
    torch.cuda.synchronize()
    pruned, _, _ = oracle.prune_compress_nm2("bf16", 4, 8, bits(W))
    dense, _ = oracle.gemm_dense("bf16", "f32", pruned, bits(X))
    assert_close(decode_out(Y), dense, "bf16", "f32", "4:8 vs dense")


@pytest.mark.slow
@pytest.mark.parametrize("N", [1, 4096])
def test_two_form_fp8_full_size_sampled(N):
    M, K = 28672, 8192
    W = inputs.draw("e4m3", (M, K), 0.02, inputs.generator(0))
    X = inputs.draw("e4m3", (N, K), 1.0, inputs.generator(1))
    values, meta = st.compress_nm2(W.to(DEV), 4, 8)
    Y = torch.empty((N, M), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(max(st.st24_spmm_workspace_bytes("e4m3", "bf16", M, N, 2 * K), 16), dtype=torch.uint8,
                     device=DEV)
    st.st24_spmm(values, meta, X.to(DEV), Y, K=K, workspace=ws, two_forms=True)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    _, ov, om = oracle.prune_compress_nm2("e4m3", 4, 8, bits(W))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)
    rng = np.random.default_rng(0)
    rows = np.concatenate([rng.integers(0, M, 512), [0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 512), [0, N - 1]])
    X2 = np.concatenate([bits(X), bits(X)], axis=1)
    ref, _ = oracle.spmm_sampled("e4m3", "bf16", ov, om, X2, 2 * K, rows, cols)
    assert_close(decode_out(Y)[cols, rows], ref, "e4m3", "bf16", f"4:8 fp8 N={N} sampled")


# ---- special values and strides on the lanes kernel ---------------------------

def _special_weight(dt, M, K, seed):
    g = torch.Generator().manual_seed(seed)
    if dt == "s8":
        # int8 -128 (|-128| = 128) sends its pieces unit by unit; the rest stay on lanes
        vals = torch.tensor([-128, -127, -1, 0, 1, 127], dtype=torch.int8)
        W = vals[torch.randint(0, len(vals), (M, K), generator=g)]
        W[: M // 2] = torch.where(W[: M // 2] == -128, torch.tensor(-127, dtype=torch.int8), W[: M // 2])
        return W
    vals = torch.tensor([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, float("nan"), float("inf")])
    if dt == "e4m3":
        vals = vals[:8]   # no infinity in e4m3
    W = vals[torch.randint(0, len(vals), (M, K), generator=g)].to(inputs.TORCH_DTYPE[dt])
    if dt != "e4m3":
        W[: M // 2] = torch.where(torch.isnan(W[: M // 2].float()), torch.zeros((), dtype=W.dtype), W[: M // 2])
        raw = inputs.raw(W)   # NaNs with different payloads tie with each other
        raw[M - 1, 0:8] = torch.tensor([0x7FC1, 0x7FC3, 0x3C00, 0x7FC2, 0, 0x7FC5, 0x7FC4, 1],
                                       dtype=torch.int32).to(raw.dtype)
    return W


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("n,m", [(1, 4), (2, 8), (1, 8)])
def test_special_values(dt, n, m):
    W = _special_weight(dt, 96, 512, n + m)
    values, meta = st.compress_nm(W.to(DEV), n, m)
    _, ov, om = oracle.prune_compress_nm(dt, n, m, bits(W))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("n,m", [(4, 8), (3, 8), (3, 4)])
def test_two_forms_special_values(dt, n, m):
    W = _special_weight(dt, 96, 512, 10 + n + m)
    values, meta = st.compress_nm2(W.to(DEV), n, m)
    _, ov, om = oracle.prune_compress_nm2(dt, n, m, bits(W))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("two", [False, True])
def test_padded_row_stride(dt, two):
    # rows 16-byte aligned but longer than K: the lanes kernel reads row by row
    M, K, pad = 70, 1024, 64
    full = inputs.draw(dt, (M, K + pad), 0.02 if dt == "e4m3" else 1.0, inputs.generator(7))
    Wd = full.to(DEV)[:, :K]
    assert Wd.stride(0) == K + pad
    n, m = (4, 8) if two else (2, 8)
    fn, ref = (st.compress_nm2, oracle.prune_compress_nm2) if two else (st.compress_nm, oracle.prune_compress_nm)
    values, meta = fn(Wd, n, m)
    _, ov, om = ref(dt, n, m, bits(full[:, :K].contiguous()))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)


@pytest.mark.parametrize("two", [False, True])
def test_odd_piece_count(two):
    # a piece count that is not a multiple of the 64 a warp takes per round: the last
    # lanes hold one piece or none
    M, K = 3, 40   # 15 pieces of bf16
    W = inputs.draw("bf16", (M, K), 1.0, inputs.generator(11))
    n, m = (3, 8) if two else (1, 8)
    fn, ref = (st.compress_nm2, oracle.prune_compress_nm2) if two else (st.compress_nm, oracle.prune_compress_nm)
    values, meta = fn(W.to(DEV), n, m)
    _, ov, om = ref("bf16", n, m, bits(W))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)

"""The narrow-N tcgen05 kernel family (N <= 64; f16, bf16, e4m3) against the
oracle: ragged shapes compared in full (rows past a 128-row tile, a last
8-bit k-block that is half past K, every MMA width 16/32/48/64 and N inside
each), the epilogue's alpha / beta / per-row scale, strided operands, the
decode workload at full size, fixed weights back to back, determinism and
the fp8 workload at full size on sampled outputs."""
import numpy as np
import pytest
import torch

import st24_inputs as inputs
import structured_sparse_gemm_gb300 as st
from helpers import assert_close, decode_out
from test_gpu_spmm import check_full, check_sampled, gpu_run, oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
K_NARROW = "tcgen05_narrow"


@pytest.mark.parametrize("ab", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("c", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(129, 1, 128), (200, 7, 384), (300, 16, 640), (64, 17, 512), (385, 33, 1280),
                                   (130, 48, 4224), (1000, 64, 8192), (77, 40, 2048), (5000, 3, 1152)])
def test_narrow_ragged(ab, c, M, N, K):
    case = inputs.spmm_case(ab, c, M, N, K, a_std=0.02 if ab == "e4m3" else 1.0, seed=M + N + K)
    if ab == "e4m3" and K % 256:
        # 8-bit values are streamed in 128-byte chunks of 256 K: other K are not taken
        with pytest.raises(st.St24Error) as e:
            gpu_run(case, kernel=K_NARROW)
        assert e.value.status == 2
        return
    check_full(case, kernel=K_NARROW)


@pytest.mark.parametrize("ab", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("N,c", [(1, "bf16"), (13, "f16"), (32, "f32"), (64, "bf16")])
def test_narrow_alpha_beta_scale(ab, N, c):
    case = inputs.spmm_case(ab, c, 257, N, 768 if ab == "e4m3" else 640, alpha=0.5, beta=-0.75, with_scale=True,
                            a_std=0.02 if ab == "e4m3" else 1.0, seed=11)
    check_full(case, kernel=K_NARROW)


@pytest.mark.parametrize("N", inputs.DECODE_NS)
def test_narrow_decode_bf16_full(N):
    check_full(inputs.decode_bf16(N), kernel=K_NARROW)


@pytest.mark.parametrize("ab,N", [("bf16", 24), ("e4m3", 9), ("f16", 64)])
@pytest.mark.parametrize("pad_c", [8, 3])
def test_narrow_strided_b_and_c(ab, N, pad_c):
    M, K = 200, 512
    case = inputs.spmm_case(ab, "bf16", M, N, K, a_std=0.02 if ab == "e4m3" else 1.0, seed=3, beta=0.5)
    values, meta = st.compress(case.A.to(DEV))
    Xw = torch.zeros((N, K + 64), dtype=case.X.dtype, device=DEV)
    Xw[:, :K] = case.X.to(DEV)
    Yw = torch.full((N, M + pad_c), 7, dtype=torch.bfloat16, device=DEV)
    Yw[:, :M] = case.C_in.to(DEV).to(torch.bfloat16)
    wsz = st.st24_spmm_workspace_bytes(ab, "bf16", M, N, K)
    ws = torch.zeros(max(wsz, 1), dtype=torch.uint8, device=DEV)
    st.st24_spmm(values, meta, Xw[:, :K], Yw[:, :M], K=K, beta=case.beta, workspace=ws, kernel=K_NARROW)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    assert bool((Yw[:, M:] == 7).all())
    assert_close(decode_out(Yw[:, :M].contiguous()), oracle_full(case), ab, "bf16", case.name + " strided")


@pytest.mark.parametrize("N", [1, 16, 32, 64])
def test_narrow_fixed_weights_back_to_back(N):
    """Back-to-back products over four weights with ST24_SPMM_FIXED_A (the next
    product's weight stages load while the previous one runs) equal the same
    products without it, bit for bit, and the first matches the oracle."""
    cases = [inputs.spmm_case("bf16", "bf16", 1024, N, 2048, seed=40 + i) for i in range(4)]
    layers = []
    for c in cases:
        values, meta = st.compress(c.A.to(DEV))
        layers.append((values, meta, c.X.to(DEV)))
    torch.cuda.synchronize()
    wsz = st.st24_spmm_workspace_bytes("bf16", "bf16", 1024, N, 2048)
    ws = torch.zeros(max(wsz, 1), dtype=torch.uint8, device=DEV)
    outs = {}
    for fixed in (False, True):
        Ys = [torch.empty((N, 1024), dtype=torch.bfloat16, device=DEV) for _ in layers]
        for _ in range(2):
            for (values, meta, X), Y in zip(layers, Ys):
                st.st24_spmm(values, meta, X, Y, K=2048, workspace=ws, kernel=K_NARROW, fixed_a=fixed)
        torch.cuda.synchronize()
        outs[fixed] = Ys
    assert st.st24_device_status() == 0
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)
    assert_close(decode_out(outs[True][0]), oracle_full(cases[0]), "bf16", "bf16", "fixed weights")


def test_narrow_deterministic_and_workspace_reuse():
    case = inputs.decode_bf16(32)
    wsz = st.st24_spmm_workspace_bytes("bf16", "bf16", case.M, case.N, case.K)
    ws = torch.zeros(max(wsz, 1), dtype=torch.uint8, device=DEV)
    _, _, outs = gpu_run(case, repeat=3, ws=ws, kernel=K_NARROW)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert int(ws[-256:].sum()) == 0   # the tile counters are back at zero


def test_narrow_rejects_int8_and_wide_n():
    with pytest.raises(st.St24Error) as e:
        gpu_run(inputs.spmm_case("s8", "s32", 128, 16, 256, seed=1), kernel=K_NARROW)
    assert e.value.status == 2
    with pytest.raises(st.St24Error) as e:
        gpu_run(inputs.spmm_case("bf16", "bf16", 128, 65, 256, seed=1), kernel=K_NARROW)
    assert e.value.status == 2


@pytest.mark.slow
@pytest.mark.parametrize("N", [1, 64])
def test_narrow_fp8_sampled(N):
    check_sampled(inputs.fp8(N), count=1024, kernel=K_NARROW)

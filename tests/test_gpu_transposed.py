"""The transposed use of a compressed weight, dX = alpha * dY * A + beta * dX
(st24_spmm_t), on the GPU against the oracle: ragged shapes in full (rows of
A past a 64-row stage, N past a tile, every output type), the epilogue, strided
operands, the decode-shaped weight in full, the prefill-shaped weights at full
size on sampled outputs, determinism, and the argument checks."""
import numpy as np
import pytest
import torch

import oracle
import st24_inputs as inputs
import structured_sparse_gemm_gb300 as st
from helpers import assert_close, bits, decode_out

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def make(ab, c, M, N, K, *, alpha=1.0, beta=0.0, a_std=1.0, seed=0):
    """Weight A [M, K], dY [N, M] and dX_in [N, K] (seeded)."""
    g = inputs.generator(seed)
    A = inputs.draw(ab, (M, K), a_std, g)
    dY = inputs.draw(ab, (N, M), 1.0, g)
    C_in = inputs.draw(c, (N, K), 1.0, g) if beta != 0.0 else None
    return A, dY, C_in


def run_gpu(ab, c, A, dY, C_in, alpha, beta, values=None, meta=None):
    if values is None:
        values, meta = st.compress(A.to(DEV))
    N, K, M = dY.shape[0], A.shape[1], dY.shape[1]
    dX = (C_in.to(DEV) if C_in is not None else torch.full((N, K), 3.0, device=DEV)).to(inputs.TORCH_DTYPE[c])
    # dY's row stride must be a multiple of 16 bytes: pad rows of a ragged M
    ldb = (M + 7) // 8 * 8
    dYd = torch.zeros((N, ldb), dtype=dY.dtype, device=DEV)
    dYd[:, :M] = dY.to(DEV)
    st.st24_spmm_t(values, meta, dYd[:, :M], dX, K=K, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    return dX


def reference(ab, c, A, dY, C_in, alpha, beta):
    _, _, ov, om = oracle.prune_compress(ab, bits(A))
    out, _ = oracle.spmm_t(ab, c, ov, om, bits(dY), A.shape[1], alpha=alpha, beta=beta,
                           C_in=None if C_in is None else bits(C_in.to(inputs.TORCH_DTYPE[c])))
    return out


@pytest.mark.parametrize("ab", ["f16", "bf16"])
@pytest.mark.parametrize("c", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(64, 16, 128), (200, 37, 384), (130, 64, 256), (77, 130, 512), (300, 300, 1280),
                                   (1000, 257, 256), (64, 1, 128)])
def test_transposed_ragged(ab, c, M, N, K):
    A, dY, _ = make(ab, c, M, N, K, seed=M + N + K)
    got = run_gpu(ab, c, A, dY, None, 1.0, 0.0)
    assert_close(decode_out(got), reference(ab, c, A, dY, None, 1.0, 0.0), ab, c, f"spmm_t {M}x{N}x{K}")


@pytest.mark.parametrize("ab,c,N", [("bf16", "bf16", 48), ("f16", "f32", 300), ("bf16", "f16", 256)])
def test_transposed_alpha_beta(ab, c, N):
    A, dY, C_in = make(ab, c, 257, N, 640, alpha=0.5, beta=-0.75, seed=11)
    got = run_gpu(ab, c, A, dY, C_in, 0.5, -0.75)
    assert_close(decode_out(got), reference(ab, c, A, dY, C_in, 0.5, -0.75), ab, c, "spmm_t alpha beta")


@pytest.mark.parametrize("pad", [8, 3])
def test_transposed_strided(pad):
    M, N, K = 200, 70, 512
    A, dY, C_in = make("bf16", "bf16", M, N, K, beta=0.5, seed=3)
    values, meta = st.compress(A.to(DEV))
    dYw = torch.zeros((N, M + 56), dtype=torch.bfloat16, device=DEV)   # ldb = M + 56 (a multiple of 8)
    dYw[:, :M] = dY.to(DEV)
    dXw = torch.full((N, K + pad), 7, dtype=torch.bfloat16, device=DEV)
    dXw[:, :K] = C_in.to(DEV)
    st.st24_spmm_t(values, meta, dYw[:, :M], dXw[:, :K], K=K, beta=0.5)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    assert bool((dXw[:, K:] == 7).all())
    assert_close(decode_out(dXw[:, :K].contiguous()), reference("bf16", "bf16", A, dY, C_in, 1.0, 0.5),
                 "bf16", "bf16", "spmm_t strided")


@pytest.mark.parametrize("N", [1, 32])
def test_transposed_decode_weight_full(N):
    A, dY, _ = make("bf16", "bf16", 4096, N, 4096, a_std=0.02, seed=N)
    got = run_gpu("bf16", "bf16", A, dY, None, 1.0, 0.0)
    assert_close(decode_out(got), reference("bf16", "bf16", A, dY, None, 1.0, 0.0), "bf16", "bf16", "decode weight")


@pytest.mark.slow
@pytest.mark.parametrize("M,K", inputs.PREFILL_SHAPES)
def test_transposed_prefill_sampled(M, K):
    N = 4096
    A, dY, _ = make("bf16", "bf16", M, N, K, a_std=0.02, seed=5)
    got = decode_out(run_gpu("bf16", "bf16", A, dY, None, 1.0, 0.0))
    rng = np.random.default_rng(0)
    ks = np.concatenate([rng.integers(0, K, 768), [0, K - 1, 127, 128]])
    ns = np.concatenate([rng.integers(0, N, 768), [0, N - 1, 255, 256]])
    _, _, ov, om = oracle.prune_compress("bf16", bits(A))
    ref, _ = oracle.spmm_t_sampled("bf16", "bf16", ov, om, bits(dY), K, ks, ns)
    assert_close(got[ns, ks], ref, "bf16", "bf16", f"spmm_t {M}x{N}x{K} sampled")
    assert np.isfinite(got).all()


def test_transposed_deterministic():
    A, dY, _ = make("bf16", "f32", 1024, 200, 1024, seed=9)
    values, meta = st.compress(A.to(DEV))
    a = run_gpu("bf16", "f32", A, dY, None, 1.0, 0.0, values, meta)
    b = run_gpu("bf16", "f32", A, dY, None, 1.0, 0.0, values, meta)
    assert torch.equal(a, b)


def test_transposed_rejects():
    A, dY, _ = make("bf16", "bf16", 64, 8, 192, seed=1)   # K % 128 != 0
    with pytest.raises(st.St24Error) as e:
        run_gpu("bf16", "bf16", A, dY, None, 1.0, 0.0)
    assert e.value.status == 2
    A, dY, _ = make("s8", "bf16", 64, 8, 128, seed=1)     # int8 is not taken
    with pytest.raises(st.St24Error) as e:
        run_gpu("s8", "bf16", A, dY, None, 1.0, 0.0)
    assert e.value.status == 2

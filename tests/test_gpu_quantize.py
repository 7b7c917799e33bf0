"""Quantise + prune + compress on the GPU against the oracle (bit-exact codes,
metadata and scales), and the dequantised product through st24_spmm."""
import numpy as np
import pytest
import torch

import oracle
import st24_inputs as inputs
import structured_sparse_gemm_gb300 as st
from helpers import assert_close, bits, decode_out

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TDT = {"e4m3": torch.float8_e4m3fn, "s8": torch.int8}


def weight(src, M, K, seed):
    """Rows N(0, 1) with per-row magnitudes spread over e^N(0, 1), one zero row,
    one row with a single non-zero."""
    g = inputs.generator(seed)
    W = torch.randn(M, K, generator=g) * torch.exp(torch.randn(M, 1, generator=g))
    if M > 2:
        W[1] = 0
        W[2] = 0
        W[2, K // 3] = -0.75
    return W.to(inputs.TORCH_DTYPE[src])


def check(W_host, src, dst, W_dev=None):
    Wd = W_host.to(DEV) if W_dev is None else W_dev
    values, meta, scales = st.quantize_compress(Wd, TDT[dst])
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    _, ov, om, osc = oracle.quantize_prune_compress(src, dst, bits(W_host))
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta.cpu().numpy(), om)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), osc.view(np.uint32))
    return values, meta, scales


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("dst", ["e4m3", "s8"])
@pytest.mark.parametrize("M,K", [(1, 16), (37, 96), (130, 4096), (65, 16384), (9, 16400), (300, 8192)])
def test_matches_oracle(src, dst, M, K):
    # K = 16384 is the largest row held in registers; 16400 takes the two-pass path
    check(weight(src, M, K, seed=M + K), src, dst)


@pytest.mark.parametrize("dst", ["e4m3", "s8"])
def test_strided_rows(dst):
    W = weight("bf16", 50, 512, seed=4)
    Ww = torch.zeros((50, 512 + 64), dtype=torch.bfloat16, device=DEV)
    Ww[:, :512] = W.to(DEV)
    check(W, "bf16", dst, W_dev=Ww[:, :512])


def test_fp8_workload_weight_sampled_rows():
    # the fp8 workload's 28672 x 8192 weight, quantised on the GPU; sampled rows
    # against the oracle (rows are independent)
    W = inputs.prune_weight_bf16(28672, 8192)
    values, meta, scales = st.quantize_compress(W.to(DEV), torch.float8_e4m3fn)
    torch.cuda.synchronize()
    rows = np.array(sorted(set([0, 1, 28671] + list(np.random.default_rng(3).integers(0, 28672, 61)))))
    _, ov, om, osc = oracle.quantize_prune_compress("bf16", "e4m3", bits(W[rows]))
    assert np.array_equal(bits(values[rows]).view(np.uint8), ov.view(np.uint8))
    assert np.array_equal(meta[rows].cpu().numpy(), om)
    assert np.array_equal(scales[rows].cpu().numpy(), osc)


@pytest.mark.parametrize("dst", ["e4m3", "s8"])
@pytest.mark.parametrize("N", [1, 24, 300])
def test_dequantised_product(dst, N):
    # quantise the weight, multiply by 8-bit activations with the row scales:
    # the product equals the oracle's product of the same codes and scales
    M, K = 257, 1024
    W = weight("bf16", M, K, seed=N)
    values, meta, scales = check(W, "bf16", dst)
    X = inputs.draw(dst, (N, K), 1.0, inputs.generator(N + 1))
    Y = torch.empty((N, M), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(max(st.st24_spmm_workspace_bytes(dst, "bf16", M, N, K), 1), dtype=torch.uint8, device=DEV)
    st.st24_spmm(values, meta, X.to(DEV), Y, K=K, row_scale=scales, workspace=ws)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    _, ov, om, osc = oracle.quantize_prune_compress("bf16", dst, bits(W))
    ref, _ = oracle.spmm(dst, "bf16", ov, om, bits(X), K, scale=osc)
    assert_close(decode_out(Y), ref, dst, "bf16", f"quantised {dst} N={N}")

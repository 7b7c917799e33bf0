"""N:M prune + compress (1:4, 1:8, 2:8) on the GPU against the oracle, bit for bit,
and the product of its 2:4 form through st24_spmm."""
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

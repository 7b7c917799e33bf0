"""Prune/compress and decompress on the GPU against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import st24_inputs as inputs
import structured_sparse_gemm_gb300 as st
from helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_compress(W_cpu: torch.Tensor, ldw_pad: int = 0):
    M, K = W_cpu.shape
    if ldw_pad:
        big = torch.zeros((M, K + ldw_pad), dtype=W_cpu.dtype)
        big[:, :K] = W_cpu
        Wd = big.to(DEV)[:, :K]
    else:
        Wd = W_cpu.to(DEV)
    values = torch.empty((M, K // 2), dtype=W_cpu.dtype, device=DEV)
    meta = torch.empty((M, (K // 4 + 1) // 2), dtype=torch.uint8, device=DEV)
    st.st24_prune_compress(Wd, values, meta)
    torch.cuda.synchronize()
    return values, meta


def check(W_cpu, ldw_pad=0):
    dt = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float8_e4m3fn: "e4m3", torch.int8: "s8"}[W_cpu.dtype]
    pruned, _, ov, om = oracle.prune_compress(dt, bits(W_cpu))
    values, meta = run_compress(W_cpu, ldw_pad)
    assert np.array_equal(bits(values).view(np.uint8), ov.view(np.uint8)), "values differ"
    assert np.array_equal(meta.cpu().numpy(), om), "metadata differs"
    # decompress of the GPU's compressed form == oracle prune
    M, K = W_cpu.shape
    back = torch.full((M, K), 7, dtype=torch.int8, device=DEV).view(W_cpu.dtype) if W_cpu.element_size() == 1 \
        else torch.full((M, K), 7, dtype=torch.int16, device=DEV).view(W_cpu.dtype)
    st.st24_decompress(values, meta, back)
    torch.cuda.synchronize()
    assert np.array_equal(bits(back).view(np.uint8), pruned.view(np.uint8)), "decompress differs"


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("M,K", [(1, 32), (37, 256), (130, 1024), (64, 4096)])
def test_fast_path(dt, M, K):
    W = inputs.draw(dt, (M, K), 0.02 if dt in ("e4m3", "bf16") else 1.0, inputs.generator(M * 7 + K))
    check(W)


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("M,K,pad", [(5, 4, 0), (9, 12, 0), (33, 100, 0), (17, 64, 3), (40, 256, 8)])
def test_general_path_ragged_and_strided(dt, M, K, pad):
    W = inputs.draw(dt, (M, K), 0.5, inputs.generator(M + K + pad))
    check(W, ldw_pad=pad)


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
def test_ties_zeros_nan(dt):
    g = torch.Generator().manual_seed(1)
    M, K = 64, 512
    if dt == "s8":
        W = torch.randint(-3, 4, (M, K), generator=g).to(torch.int8)
        W[0, :8] = torch.tensor([-128, 127, 5, -127, 0, 0, 0, 0], dtype=torch.int8)
    else:
        vals = torch.tensor([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, float("nan"), float("inf")])
        if dt == "e4m3":
            vals = vals[:8]  # no infinity in e4m3
        W = vals[torch.randint(0, len(vals), (M, K), generator=g)].to(inputs.TORCH_DTYPE[dt])
        if dt != "e4m3":
            # NaNs with different payloads tie with each other
            raw = inputs.raw(W)
            raw[1, 0:4] = torch.tensor([0x7FC1, 0x7FC3, 0x3C00, 0x7FC2], dtype=torch.int32).to(raw.dtype)
    check(W)


def test_int8_extremes():
    # |-128| = 128 does not fit the 8-bit lanes of the fast selection: pieces holding a -128 take the
    # 16-bit lanes, the others the 8-bit ones; both must follow the same tie and magnitude rule
    g = torch.Generator().manual_seed(3)
    vals = torch.tensor([-128, -127, -1, 0, 1, 127], dtype=torch.int8)
    W = vals[torch.randint(0, len(vals), (96, 1024), generator=g)]
    W[:48, :512] = torch.where(W[:48, :512] == -128, torch.tensor(-127, dtype=torch.int8), W[:48, :512])
    check(W)


def test_empty_is_noop():
    W = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    st.st24_prune_compress(W, torch.empty(0, device=DEV), torch.empty(0, device=DEV))


@pytest.mark.slow
def test_full_size_bf16_weight():
    # The 28672 x 8192 bf16 weight the prune/compress benchmark times.
    check(inputs.prune_weight_bf16())


def test_deterministic_repeat():
    W = inputs.draw("e4m3", (256, 2048), 0.02, inputs.generator(3))
    a = run_compress(W)
    b = run_compress(W)
    assert torch.equal(a[0].view(torch.uint8), b[0].view(torch.uint8)) and torch.equal(a[1], b[1])

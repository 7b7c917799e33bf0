"""st24_spmm_noalloc: the SpMM entry point for callers that cannot allocate.

Callers such as plugins inside a runtime that owns all device memory, or code
running during a global-mode stream capture, cannot cudaMalloc a workspace;
st24_spmm_noalloc keeps the split-K scratch in a fixed 16 MiB array owned by
the library.  These tests call it through the C ABI and compare it with
st24_spmm given a workspace of its own, on two calls in a row (the array keeps
the previous call's contents between them).  The file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import st24_inputs as inputs
import structured_sparse_gemm_gb300 as st
from helpers import assert_close, decode_out
from test_gpu_spmm import oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def prepare(case):
    values, meta = st.compress(case.A.to(DEV))
    X = case.X.to(DEV)
    scale = case.scale.to(DEV) if case.scale is not None else None
    return values, meta, X, scale


def out_like(case):
    return torch.zeros((case.N, case.M), dtype=inputs.TORCH_DTYPE[case.c], device=DEV)


def call_noalloc(case, values, meta, X, Y, scale):
    lib = st.load()
    stream = torch.cuda.current_stream().cuda_stream
    return lib.st24_spmm_noalloc(st.dtype_code(case.ab), st.dtype_code(case.c), case.M, case.N, case.K,
                                 ctypes.c_float(case.alpha), values.data_ptr(), meta.data_ptr(), X.data_ptr(),
                                 X.stride(0), ctypes.c_float(case.beta), Y.data_ptr(), Y.stride(0),
                                 None if scale is None else scale.data_ptr(), stream)


# Shapes whose automatic kernel choice splits tiles through the scratch: the
# warp-level int8 kernel with a stream-K tail (more tiles than SMs) and with
# every tile split over K (few tiles), and fp8 with K not a multiple of 256
# (the one-CTA tcgen05 kernel).
CASES = [
    inputs.spmm_case("s8", "bf16", 28672, 16, 4096, with_scale=True, seed=2, name="int8 28672x16x4096"),
    inputs.spmm_case("s8", "s32", 1000, 16, 4096, seed=5, name="int8 1000x16x4096"),
    inputs.spmm_case("e4m3", "f32", 1000, 40, 2176, a_std=0.02, seed=4, name="e4m3 1000x40x2176"),
]


@pytest.mark.parametrize("case", CASES, ids=["int8_N16_streamk", "int8_N16_split", "e4m3_ragged_tcgen05"])
def test_noalloc_matches_spmm_twice(case):
    values, meta, X, scale = prepare(case)
    # the existing entry point needs a workspace for these shapes ...
    with pytest.raises(st.St24Error) as e:
        st.st24_spmm(values, meta, X, out_like(case), K=case.K, alpha=case.alpha, beta=case.beta, row_scale=scale)
    assert e.value.status == 6   # ST24_ERR_WORKSPACE: so the no-allocation call really uses its scratch
    # ... and computes the reference result with one of its own
    ref = out_like(case)
    ws_bytes = st.st24_spmm_workspace_bytes(case.ab, case.c, case.M, case.N, case.K)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    st.st24_spmm(values, meta, X, ref, K=case.K, alpha=case.alpha, beta=case.beta, row_scale=scale, workspace=ws)
    torch.cuda.synchronize()
    expect = oracle_full(case)
    for _ in range(2):
        Y = out_like(case)
        assert call_noalloc(case, values, meta, X, Y, scale) == 0
        torch.cuda.synchronize()
        assert torch.equal(Y, ref)   # same kernels, same order of the split-K sums
        assert_close(decode_out(Y), expect, case.ab, case.c, case.name)
    assert st.st24_device_status() == 0


def test_noalloc_rejects_more_than_its_scratch():
    # N = 4096 on a 512 x 32768 weight: 2 x 19 tiles of 256 x 224, fewer than the CTA pairs and
    # long, so each is split two ways over K, and the 76 pairs' partial tiles need ~35 MB
    case = inputs.spmm_case("bf16", "bf16", 512, 4096, 32768, a_std=0.02, seed=1)
    assert st.st24_spmm_workspace_bytes("bf16", "bf16", 512, 4096, 32768) > 16 << 20
    values, meta, X, scale = prepare(case)
    Y = out_like(case)
    assert call_noalloc(case, values, meta, X, Y, scale) == 6   # ST24_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(Y)) == 0                    # nothing was launched

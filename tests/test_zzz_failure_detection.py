"""Failure detection without a GPU fault: a kernel whose bounded wait runs out
reports ST24_ERR_TIMEOUT through the device status word, the word is cleared
once read, and the context keeps working (runs last: it leaves the word clean)."""
import time

import pytest
import torch

import st24_inputs as inputs
import structured_sparse_gemm_gb300 as st
from helpers import assert_close, bits, decode_out

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TIMEOUT = 5   # ST24_ERR_TIMEOUT


def test_bounded_wait_reports_and_clears():
    assert st.st24_device_status() == 0
    t0 = time.time()
    st.st24_selftest_wait_timeout()
    assert st.st24_device_status() == TIMEOUT   # synchronises: the wait gave up and the kernel returned
    assert 0.5 < time.time() - t0 < 60
    assert st.st24_device_status() == 0         # read once, cleared
    # the context is still usable: a product right after matches the oracle
    case = inputs.spmm_case("bf16", "f32", 256, 8, 512, a_std=0.02, seed=9)
    values, meta = st.compress(case.A.to(DEV))
    Y = torch.zeros((case.N, case.M), dtype=torch.float32, device=DEV)
    st.st24_spmm(values, meta, case.X.to(DEV), Y, K=case.K)
    torch.cuda.synchronize()
    assert st.st24_device_status() == 0
    _, _, ov, om = oracle.prune_compress("bf16", bits(case.A))
    ref, _ = oracle.spmm("bf16", "f32", ov, om, bits(case.X), case.K)
    assert_close(decode_out(Y), ref, "bf16", "f32", "after the timeout")

"""Failure detection without a GPU fault: every mbarrier wait in the kernels
is bounded.  A test hook (DMT_BMM_TEST_STALL_MMA=1, read when the plan is
created) makes the MMA thread wait on a barrier phase that nothing completes;
with a 50 ms limit (DMT_BMM_WAIT_TIMEOUT_MS) the kernel must record
BMM_ERR_DEVICE_TIMEOUT, stop every role, drain its own copies and MMAs, free
Tensor Memory and return, leaving the context usable for the next run."""
import time

import numpy as np
import pytest
import torch

from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

from bmm_harness import check_full, desc_for, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pair", ["0", "1"])
def test_expired_wait_is_reported_and_the_next_run_is_clean(pair, monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p = wl.Problem(batch=2, M=512, N=512, K=512, transB=True, type_ab="bf16", type_c="f32",
                   seed=95)
    x = wl.make_inputs(p)
    dev = torch.device("cuda:0")
    A = torch.from_numpy(x.A.view(np.int16)).to(dev)
    B = torch.from_numpy(x.B.view(np.int16)).to(dev)
    C = torch.zeros(p.storage_elems()[2], dtype=torch.float32, device=dev)

    monkeypatch.setenv("DMT_BMM_PAIR", pair)
    monkeypatch.setenv("DMT_BMM_TEST_STALL_MMA", "1")
    monkeypatch.setenv("DMT_BMM_WAIT_TIMEOUT_MS", "50")
    with api.Plan(desc_for(p)) as plan:
        assert plan.info().cta_pair == int(pair)
        t0 = time.perf_counter()
        plan.run(A, B, C, 1.0, 0.0, torch.cuda.current_stream())
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        st, word = plan.device_error()
    assert st == api.BMM_ERR_DEVICE_TIMEOUT
    assert word >> 28 == 0xB and ((word >> 8) & 0xFF) in (1, 2, 3, 4, 5)
    assert elapsed < 5.0, f"kernel took {elapsed:.2f} s to give up"

    # the word was cleared by the read, and the context still works
    monkeypatch.delenv("DMT_BMM_TEST_STALL_MMA")
    monkeypatch.delenv("DMT_BMM_WAIT_TIMEOUT_MS")
    c, info = run_gpu(p, x)
    check_full(p, x, c)

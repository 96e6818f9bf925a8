"""The host-buffer entry point (bmm_host_*): operands copied in from host
memory and C copied back, in chunks of batch items or 256-row blocks whose
transfers overlap the computation.  Its C must equal bmm_run's bit for bit
(the chunks split independent rows or batch items) and the oracle within the
stated tolerance."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

from bmm_harness import check_full, desc_for

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _host(x: np.ndarray, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16 if x.dtype == np.uint16 else x.dtype))
    return t.pin_memory() if pin else t


def _c_host(p: wl.Problem, x: wl.Inputs, pin=True):
    nc = p.storage_elems()[2]
    if x.C_in is not None:
        c = x.C_in.copy()
    else:
        c = np.full(nc, 7.0, np.float32) if p.type_c == "f32" else np.full(nc, 0x40E0, np.uint16)
    return _host(c, pin)


def run_host(p, x, chunks=0, pin=True):
    hA, hB, hC = _host(x.A, pin), _host(x.B, pin), _c_host(p, x, pin)
    with api.HostPlan(desc_for(p), chunks) as plan:
        plan.run(hA, hB, hC, p.alpha, p.beta, torch.cuda.current_stream())
        torch.cuda.synchronize()
        st, word = plan.device_error()
        info = plan.chunks()
    assert st == api.BMM_OK, hex(word)
    out = hC.numpy()
    return (out.view(np.uint16) if p.type_c == "bf16" else out), info


def run_device(p, x):
    dev = torch.device("cuda:0")
    A = _host(x.A, False).to(dev)
    B = _host(x.B, False).to(dev)
    C = _c_host(p, x, False).to(dev)
    with api.Plan(desc_for(p)) as plan:
        plan.run(A, B, C, p.alpha, p.beta, torch.cuda.current_stream())
        torch.cuda.synchronize()
    out = C.cpu().numpy()
    return out.view(np.uint16) if p.type_c == "bf16" else out


CASES = {
    # batch items in 4 chunks, C_in read (beta != 0), fp32 out
    "batch_chunks": dict(p=wl.Problem(batch=6, M=300, N=200, K=136, transB=True, type_ab="bf16",
                                      type_c="f32", alpha=0.75, beta=0.5, seed=120), chunks=4,
                         expect=(4, False)),
    # batch 1, A row-major: 256-row blocks (the last one 232 rows), bf16 out
    "row_chunks": dict(p=wl.Problem(batch=1, M=1000, N=520, K=256, transB=True, type_ab="bf16",
                                    type_c="bf16", seed=121), chunks=0, expect=(4, True)),
    # batch 1, A stored transposed: one chunk
    "transposed_a": dict(p=wl.Problem(batch=1, M=384, N=256, K=200, transA=True, type_ab="f16",
                                      type_c="f32", seed=122), chunks=0, expect=(1, False)),
    # A shared by every batch item (stride 0): copied once
    "broadcast_a": dict(p=wl.Problem(batch=5, M=128, N=192, K=64, type_ab="bf16", type_c="f32",
                                     sA=0, seed=123), chunks=3, expect=(3, False)),
    # more chunks asked than batch items
    "few_items": dict(p=wl.Problem(batch=2, M=64, N=64, K=64, type_ab="bf16", type_c="f32",
                                   seed=124), chunks=8, expect=(2, False)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_host_run_equals_device_run_and_oracle(name):
    _need_gpu()
    case = CASES[name]
    p = case["p"]
    x = wl.make_inputs(p)
    got, info = run_host(p, x, case["chunks"])
    assert info == case["expect"]
    ref = run_device(p, x)
    assert np.array_equal(got, ref), "host-buffer result differs from bmm_run"
    check_full(p, x, got)


def test_pageable_host_memory_gives_the_same_result():
    _need_gpu()
    p = CASES["row_chunks"]["p"]
    x = wl.make_inputs(p)
    a, _ = run_host(p, x, pin=True)
    b, _ = run_host(p, x, pin=False)
    assert np.array_equal(a, b)


def test_alpha_zero_reads_no_operands():
    _need_gpu()
    p = wl.Problem(batch=3, M=96, N=80, K=64, type_ab="bf16", type_c="f32", alpha=0.0, beta=2.0,
                   seed=125)
    x = wl.make_inputs(p)
    hC = _c_host(p, x)
    with api.HostPlan(desc_for(p), 3) as plan:
        plan.run(None, None, hC, 0.0, 2.0, torch.cuda.current_stream())
        torch.cuda.synchronize()
    assert np.array_equal(hC.numpy(), (2.0 * x.C_in).astype(np.float32))


def test_square_gemm_through_host_buffers():
    """The 4096^3 TN bf16 product: row chunks, bit for bit the device result."""
    _need_gpu()
    p = wl.GEMM_4096
    x = wl.make_inputs(p)
    got, info = run_host(p, x)
    assert info == (4, True)
    assert np.array_equal(got, run_device(p, x))

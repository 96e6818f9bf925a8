"""bmm_run_noalloc: the entry point for callers that cannot call cudaMalloc
(an allocator owns the device's memory, or the call path cannot afford
cudaMalloc's cost and implicit device synchronisation).  It keeps its scratch
in a device array built into the library instead of allocating.

Its output must agree with the plan-based bmm_run on the same inputs, within
the parity tolerance the other GPU tests use, on two calls in a row (the
second call reuses the scratch the first one left behind).  The problem has
unaligned leading dimensions so the operand staging area is really used.
This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

from bmm_harness import decode_c, desc_for

pytestmark = pytest.mark.gpu


def _run_both(p, x, stream):
    dev = torch.device("cuda:0")
    A = torch.from_numpy(x.A.view(np.int16)).to(dev)
    B = torch.from_numpy(x.B.view(np.int16)).to(dev)
    cdt = torch.float32 if p.type_c == "f32" else torch.int16
    cin = torch.from_numpy(x.C_in if p.type_c == "f32" else x.C_in.view(np.int16))
    C_plan = cin.to(dev, dtype=cdt)
    C_na = cin.to(dev, dtype=cdt)
    err = torch.full((1,), -1, dtype=torch.int32, device=dev)
    desc = desc_for(p)
    with api.Plan(desc) as plan:
        plan.run(A, B, C_plan, p.alpha, p.beta, stream)
        api.bmm_run_noalloc(desc, A, B, C_na, p.alpha, p.beta, stream, device_error=err)
        torch.cuda.synchronize()
        assert plan.device_error()[0] == api.BMM_OK
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x}"
    as_np = (lambda t: t.cpu().numpy()) if p.type_c == "f32" else \
        (lambda t: t.cpu().numpy().view(np.uint16))
    return as_np(C_plan), as_np(C_na)


def test_noalloc_matches_bmm_run_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    stream = torch.cuda.Stream()
    for call, seed in enumerate((201, 202)):
        p = wl.Problem(batch=3, M=200, N=150, K=300, transA=bool(call), transB=True,
                       type_ab="f16", type_c="f32", alpha=0.5, beta=1.0,
                       lda=(203 if call else 301), ldb=305, ldc=151, seed=seed)
        info = api.bmm_plan_query(desc_for(p))
        assert info.pack_a == 1 and info.pack_b == 1 and info.workspace_bytes > 0
        x = wl.make_inputs(p)
        c_plan, c_na = _run_both(p, x, stream)
        ref, bnd = oracle.bmm(x.A, x.B, x.C_in, **p.oracle_kwargs())
        cin = decode_c(x.C_in, p)
        tol = oracle.tolerance(ref, bnd, cin, alpha=p.alpha, beta=p.beta, out_bf16=False)
        got_plan, got_na = decode_c(c_plan, p), decode_c(c_na, p)
        assert np.all(np.isfinite(got_na))
        assert np.all(np.abs(got_na - got_plan) <= tol), f"call {call}: differs from bmm_run"
        assert np.all(np.abs(got_na - ref) <= tol), f"call {call}: differs from the oracle"
        # the padding between C rows (ldc > N) is left as it was
        s = p.strides()
        pad = np.concatenate([np.arange(b * s["sC"] + i * s["ldc"] + p.N, b * s["sC"] + (i + 1) * s["ldc"])
                              for b in range(p.batch) for i in range(p.M - 1)])
        assert np.array_equal(c_na[pad], x.C_in[pad])


def test_noalloc_beyond_its_staging_area_reads_the_operand_in_place():
    """A needs 84 MB of staging (lda 1027 is not a multiple of 8 elements),
    more than the built-in 32 MiB: the call reads A in place through the
    kernels' row loader instead.  Its output equals bmm_run's (staged) bit
    for bit and meets the oracle's bound; the first call passes no
    device_error pointer, the second one does."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p = wl.Problem(batch=40, M=1024, N=256, K=1024, lda=1027, type_ab="f16", type_c="f32", seed=203)
    desc = desc_for(p)
    info = api.bmm_plan_query(desc)
    assert info.pack_a == 1 and info.workspace_bytes > (32 << 20)
    x = wl.make_inputs(p)
    dev = torch.device("cuda:0")
    A = torch.from_numpy(x.A.view(np.int16)).to(dev)
    B = torch.from_numpy(x.B.view(np.int16)).to(dev)
    nc = p.storage_elems()[2]
    C_plan = torch.full((nc,), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    with api.Plan(desc) as plan:
        plan.run(A, B, C_plan, p.alpha, p.beta, stream)
        torch.cuda.synchronize()
        assert plan.device_error()[0] == api.BMM_OK
    staged = C_plan.cpu().numpy()
    err = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for call in range(2):
        C_na = torch.full((nc,), float("nan"), dtype=torch.float32, device=dev)
        api.bmm_run_noalloc(desc, A, B, C_na, p.alpha, p.beta, stream,
                            device_error=(err if call else None))
        torch.cuda.synchronize()
        got = C_na.cpu().numpy()
        assert np.array_equal(got.view(np.uint8), staged.view(np.uint8)), f"call {call}"
    assert int(err.item()) == 0
    ref, bnd = oracle.bmm(x.A, x.B, None, **p.oracle_kwargs())
    tol = oracle.tolerance(ref, bnd, None, alpha=p.alpha, beta=p.beta, out_bf16=False)
    assert np.all(np.abs(decode_c(got, p) - ref) <= tol)

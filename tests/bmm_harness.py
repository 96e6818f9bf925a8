"""Test harness: run one ``workloads.Problem`` through the C ABI on the GPU
and compare the result with the fp64 oracle.

Every operand lives inside a larger device buffer whose guard elements hold
NaN (A, B) or a sentinel pattern (C): a read outside an operand shows up as
NaN in C, and a write outside C changes the sentinel.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

NAN_BITS = {"bf16": 0x7FC0, "f16": 0x7E00}
C_SENTINEL_F32 = np.float32(-12345.678)
C_SENTINEL_BF16 = np.uint16(0xC0DE)


def desc_for(p: wl.Problem) -> api.bmm_desc_t:
    s = p.strides()
    return api.make_desc(batch=p.batch, M=p.M, N=p.N, K=p.K, lda=s["lda"], ldb=s["ldb"],
                         ldc=s["ldc"], strideA=s["sA"], strideB=s["sB"], strideC=s["sC"],
                         transA=p.transA, transB=p.transB, typeA=p.type_ab, typeC=p.type_c)


def _as_i16(v) -> int:
    return int(np.array([v], dtype=np.uint16).view(np.int16)[0])


def _dev16(bits: np.ndarray, guard: int, fill: int, dev, offset_elems=0):
    n = bits.size
    buf = torch.full((guard + n + guard + 8,), _as_i16(fill), dtype=torch.int16, device=dev)
    start = guard + offset_elems
    if n:
        buf[start:start + n].copy_(torch.from_numpy(bits.view(np.int16)).to(dev))
    return buf, start


def decode_c(host: np.ndarray, p: wl.Problem) -> np.ndarray:
    """Dense float64 [batch, M, N] view of the C storage (host copy)."""
    s = p.strides()
    if p.type_c == "f32":
        vals = host.astype(np.float64)
    else:
        vals = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).double().numpy()
    out = np.empty((p.batch, p.M, p.N), dtype=np.float64)
    for b in range(p.batch):
        for i in range(p.M):
            o = b * s["sC"] + i * s["ldc"]
            out[b, i] = vals[o:o + p.N]
    return out


def c_storage(p: wl.Problem, x: wl.Inputs, c_fill: str):
    """Host C storage before the call: C_in where beta != 0, else NaN/garbage."""
    nc = p.storage_elems()[2]
    if x.C_in is not None:
        return x.C_in.copy()
    if p.type_c == "f32":
        return np.full(nc, np.nan if c_fill == "nan" else 7.0, dtype=np.float32)
    return np.full(nc, NAN_BITS["bf16"] if c_fill == "nan" else 0x40E0, dtype=np.uint16)


def run_gpu(p: wl.Problem, x: wl.Inputs, *, guard=4096, c_fill="nan", stream=None,
            a_offset=0, expect_status=api.BMM_OK):
    """Run ``p`` on inputs ``x`` through bmm_create/bmm_run.  Returns
    (C storage as a host numpy array, plan info)."""
    dev = torch.device("cuda:0")
    A, a0 = _dev16(x.A, guard, NAN_BITS[p.type_ab], dev, a_offset)
    B, b0 = _dev16(x.B, guard, NAN_BITS[p.type_ab], dev)
    chost = c_storage(p, x, c_fill)
    if p.type_c == "f32":
        C = torch.full((guard + chost.size + guard,), float(C_SENTINEL_F32), dtype=torch.float32,
                       device=dev)
        C[guard:guard + chost.size].copy_(torch.from_numpy(chost).to(dev))
    else:
        C = torch.full((guard + chost.size + guard,), _as_i16(C_SENTINEL_BF16), dtype=torch.int16,
                       device=dev)
        C[guard:guard + chost.size].copy_(torch.from_numpy(chost.view(np.int16)).to(dev))
    esz = 2
    cesz = 4 if p.type_c == "f32" else 2
    plan = api.Plan(desc_for(p))
    try:
        info = plan.info()
        st = api.load_library().bmm_run(
            plan.handle, api._ptr(A.data_ptr() + a0 * esz), api._ptr(B.data_ptr() + b0 * esz),
            api._ptr(C.data_ptr() + guard * cesz), float(p.alpha), float(p.beta),
            api._stream(stream if stream is not None else torch.cuda.current_stream()))
        assert st == expect_status, api.bmm_status_string(st)
        torch.cuda.synchronize()
        derr, word = plan.device_error()
        assert derr == api.BMM_OK, f"device error word {word:#x}"
    finally:
        plan.close()
    out = C.cpu().numpy()
    if p.type_c == "f32":
        assert np.all(out[:guard] == C_SENTINEL_F32) and np.all(out[guard + chost.size:] == C_SENTINEL_F32), \
            "write outside C"
        return out[guard:guard + chost.size], info
    out = out.view(np.uint16)
    assert np.all(out[:guard] == C_SENTINEL_BF16) and np.all(out[guard + chost.size:] == C_SENTINEL_BF16), \
        "write outside C"
    return out[guard:guard + chost.size].copy(), info


def check_full(p: wl.Problem, x: wl.Inputs, c_host: np.ndarray, *, exact=False):
    """Element-by-element comparison with the full oracle."""
    c_ref, bnd = oracle.bmm(x.A, x.B, x.C_in, **p.oracle_kwargs())
    got = decode_c(c_host, p)
    assert np.all(np.isfinite(got)), "non-finite values in C"
    if exact:
        bad = got != c_ref
        assert not bad.any(), f"{bad.sum()} elements differ from the exact result"
        return 0.0
    cin = None if x.C_in is None else decode_c(x.C_in if p.type_c == "f32" else x.C_in, p)
    tol = oracle.tolerance(c_ref, bnd, cin, alpha=p.alpha, beta=p.beta, out_bf16=p.type_c == "bf16")
    err = np.abs(got - c_ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{bad.sum()} of {bad.size} elements outside tolerance; first "
                             f"{[(tuple(i), got[tuple(i)], c_ref[tuple(i)], tol[tuple(i)]) for i in idx]}")
    return float(np.max(err / np.maximum(tol, 1e-300))) if err.size else 0.0


def sample_indices(p: wl.Problem, n: int, seed: int, tile_n: int = 256) -> np.ndarray:
    """Random samples plus the corners and tile edges of every kind."""
    rng = np.random.default_rng(seed)
    idx = [np.stack([rng.integers(0, p.batch, n), rng.integers(0, p.M, n),
                     rng.integers(0, p.N, n)], axis=1)]
    edges_m = sorted({0, p.M - 1, *[m for m in (127, 128, 129, 255, 256) if m < p.M]})
    edges_n = sorted({0, p.N - 1, *[v for v in (15, 16, 63, 64, 127, 128, 255, 256) if v < p.N]})
    for b in {0, p.batch - 1}:
        for i in edges_m:
            for j in edges_n:
                idx.append(np.array([[b, i, j]]))
    return np.concatenate(idx, axis=0).astype(np.int64)


def check_sampled(p: wl.Problem, x: wl.Inputs, c_host: np.ndarray, samples: np.ndarray):
    c_ref, bnd = oracle.bmm_sampled(x.A, x.B, x.C_in, samples, **p.oracle_kwargs())
    s = p.strides()
    off = samples[:, 0] * s["sC"] + samples[:, 1] * s["ldc"] + samples[:, 2]
    if p.type_c == "f32":
        got = c_host[off].astype(np.float64)
    else:
        got = torch.from_numpy(c_host[off].view(np.int16)).view(torch.bfloat16).double().numpy()
    cin = None
    if x.C_in is not None:
        cin = x.C_in[off].astype(np.float64) if p.type_c == "f32" else \
            torch.from_numpy(x.C_in[off].view(np.int16)).view(torch.bfloat16).double().numpy()
    tol = oracle.tolerance(c_ref, bnd, cin, alpha=p.alpha, beta=p.beta, out_bf16=p.type_c == "bf16")
    assert np.all(np.isfinite(got))
    err = np.abs(got - c_ref)
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} sampled elements outside tolerance: " \
        f"{[(tuple(samples[i]), got[i], c_ref[i], tol[i]) for i in np.argwhere(bad)[:5, 0]]}"
    return float(np.max(err / np.maximum(tol, 1e-300)))

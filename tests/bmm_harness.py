"""Test harness: run one ``workloads.Problem`` through the C ABI on the GPU
and compare the result with the fp64 oracle.

Every operand lives inside a larger device buffer whose guard elements hold
NaN (A, B) or a sentinel pattern (C): a read outside an operand shows up as
NaN in C, and a write outside C changes the sentinel.
"""
from __future__ import annotations

import dataclasses

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
        vals = np.ascontiguousarray(host, dtype=np.float32)
    else:
        vals = torch.from_numpy(np.ascontiguousarray(host).view(np.int16)).view(torch.bfloat16).float().numpy()
    if p.batch == 0 or p.M == 0 or p.N == 0:
        return np.empty((p.batch, p.M, p.N), dtype=np.float64)
    it = vals.itemsize
    view = np.lib.stride_tricks.as_strided(vals, shape=(p.batch, p.M, p.N),
                                           strides=(s["sC"] * it, s["ldc"] * it, it), writeable=False)
    return view.astype(np.float64)


def c_storage(p: wl.Problem, x: wl.Inputs, c_fill: str):
    """Host C storage before the call: C_in where beta != 0, else NaN/garbage."""
    nc = p.storage_elems()[2]
    if x.C_in is not None:
        return x.C_in.copy()
    if p.type_c == "f32":
        return np.full(nc, np.nan if c_fill == "nan" else 7.0, dtype=np.float32)
    return np.full(nc, NAN_BITS["bf16"] if c_fill == "nan" else 0x40E0, dtype=np.uint16)


def run_gpu(p: wl.Problem, x: wl.Inputs, *, guard=4096, c_fill="nan", stream=None,
            a_offset=0, c_offset=0, expect_status=api.BMM_OK):
    """Run ``p`` on inputs ``x`` through bmm_create/bmm_run.  Returns
    (C storage as a host numpy array, plan info).  ``c_offset`` moves C's
    base that many elements past its 16-byte-aligned place."""
    dev = torch.device("cuda:0")
    A, a0 = _dev16(x.A, guard, NAN_BITS[p.type_ab], dev, a_offset)
    B, b0 = _dev16(x.B, guard, NAN_BITS[p.type_ab], dev)
    chost = c_storage(p, x, c_fill)
    c0 = guard + c_offset
    if p.type_c == "f32":
        C = torch.full((c0 + chost.size + guard,), float(C_SENTINEL_F32), dtype=torch.float32,
                       device=dev)
        C[c0:c0 + chost.size].copy_(torch.from_numpy(chost).to(dev))
    else:
        C = torch.full((c0 + chost.size + guard,), _as_i16(C_SENTINEL_BF16), dtype=torch.int16,
                       device=dev)
        C[c0:c0 + chost.size].copy_(torch.from_numpy(chost.view(np.int16)).to(dev))
    esz = 2
    cesz = 4 if p.type_c == "f32" else 2
    plan = api.Plan(desc_for(p))
    try:
        info = plan.info()
        st = api.load_library().bmm_run(
            plan.handle, api._ptr(A.data_ptr() + a0 * esz), api._ptr(B.data_ptr() + b0 * esz),
            api._ptr(C.data_ptr() + c0 * cesz), float(p.alpha), float(p.beta),
            api._stream(stream if stream is not None else torch.cuda.current_stream()))
        assert st == expect_status, api.bmm_status_string(st)
        torch.cuda.synchronize()
        derr, word = plan.device_error()
        assert derr == api.BMM_OK, f"device error word {word:#x}"
    finally:
        plan.close()
    out = C.cpu().numpy()
    if p.type_c == "f32":
        assert np.all(out[:c0] == C_SENTINEL_F32) and np.all(out[c0 + chost.size:] == C_SENTINEL_F32), \
            "write outside C"
        return out[c0:c0 + chost.size], info
    out = out.view(np.uint16)
    assert np.all(out[:c0] == C_SENTINEL_BF16) and np.all(out[c0 + chost.size:] == C_SENTINEL_BF16), \
        "write outside C"
    return out[c0:c0 + chost.size].copy(), info


def _batch_slice(p: wl.Problem, x: wl.Inputs, c_host: np.ndarray, b0: int, b1: int):
    """Problem, inputs and C storage of batch items [b0, b1) of ``p``: the
    same strides, the buffers cut at item b0 (a broadcast operand, batch
    stride 0, is passed whole)."""
    s = p.strides()
    sub = dataclasses.replace(p, batch=b1 - b0, **s)
    na, nb, nc = sub.storage_elems()
    a0 = 0 if s["sA"] == 0 else b0 * s["sA"]
    bb0 = 0 if s["sB"] == 0 else b0 * s["sB"]
    c0 = b0 * s["sC"]
    xs = wl.Inputs(x.A[a0:a0 + na], x.B[bb0:bb0 + nb],
                   None if x.C_in is None else x.C_in[c0:c0 + nc])
    return sub, xs, c_host[c0:c0 + nc]


def check_full(p: wl.Problem, x: wl.Inputs, c_host: np.ndarray, *, exact=False,
               max_elems=1 << 26):
    """Element-by-element comparison of every element of C with the full
    oracle, and no NaN or Inf anywhere in C.  Large problems are compared in
    slices of whole batch items (at most ``max_elems`` outputs each, one
    item at least) so the fp64 reference never has to fit in memory at once.
    Returns the largest err/tol over all elements (0 for exact checks)."""
    per_item = max(1, p.M * p.N)
    step = max(1, max_elems // per_item)
    worst = 0.0
    for b0 in range(0, max(p.batch, 1), step):
        b1 = min(p.batch, b0 + step)
        if b1 <= b0:
            break
        sub, xs, cs = (p, x, c_host) if (b0 == 0 and b1 == p.batch) else _batch_slice(p, x, c_host, b0, b1)
        worst = max(worst, _check_full_once(sub, xs, cs, exact=exact, item0=b0))
    return worst


def _check_full_once(p: wl.Problem, x: wl.Inputs, c_host: np.ndarray, *, exact, item0):
    c_ref, bnd = oracle.bmm(x.A, x.B, x.C_in, want_bound=not exact, **p.oracle_kwargs())
    got = decode_c(c_host, p)
    assert np.all(np.isfinite(got)), "non-finite values in C"
    if exact:
        bad = got != c_ref
        if bad.any():
            idx = np.argwhere(bad)[:5]
            raise AssertionError(f"{bad.sum()} elements differ from the exact result; first (b,i,j) "
                                 f"{[(int(i[0]) + item0, int(i[1]), int(i[2])) for i in idx]}")
        return 0.0
    cin = None if x.C_in is None else decode_c(x.C_in, p)
    tol = oracle.tolerance(c_ref, bnd, cin, alpha=p.alpha, beta=p.beta, out_bf16=p.type_c == "bf16")
    del bnd, cin
    err = np.abs(got - c_ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{bad.sum()} of {bad.size} elements outside tolerance; first "
                             f"{[((int(i[0]) + item0, int(i[1]), int(i[2])), got[tuple(i)], c_ref[tuple(i)], tol[tuple(i)]) for i in idx]}")
    if not err.size:
        return 0.0
    np.divide(err, np.maximum(tol, 1e-300), out=err)
    return float(err.max())


def _seams(extent: int, tile: int) -> set:
    """Indices on both sides of every tile boundary below ``extent``, plus
    the first and last index and the first index of the last (possibly
    partial) tile."""
    out = {0, extent - 1}
    if tile > 0:
        for t in range(tile, extent, tile):
            out.update((t - 1, t))
        out.add(((extent - 1) // tile) * tile)
    return {v for v in out if 0 <= v < extent}


def sample_indices(p: wl.Problem, n: int, seed: int, *, tile_m: int = 128,
                   tile_n: int = 256, max_seams: int = 64) -> np.ndarray:
    """Random samples plus the corners and the seams of the tiles the plan
    actually uses (``tile_m`` rows, ``tile_n`` columns of C; for the swapped
    form pass the tile extents of C's transpose swapped back), on the first
    and last batch item.  At most ``max_seams`` seam indices per dimension
    (evenly spread) keep the set small on large outputs."""
    rng = np.random.default_rng(seed)
    idx = [np.stack([rng.integers(0, p.batch, n), rng.integers(0, p.M, n),
                     rng.integers(0, p.N, n)], axis=1)]

    def thin(v):
        v = sorted(v)
        if len(v) <= max_seams:
            return v
        keep = np.unique(np.linspace(0, len(v) - 1, max_seams).round().astype(int))
        return [v[k] for k in keep] + v[-2:]

    edges_m = thin(_seams(p.M, tile_m))
    edges_n = thin(_seams(p.N, tile_n))
    for b in {0, p.batch - 1}:
        grid = np.array([[b, i, j] for i in edges_m for j in edges_n], dtype=np.int64)
        idx.append(grid)
    return np.concatenate(idx, axis=0).astype(np.int64)


def plan_tiles(info):
    """(tile_m, tile_n) of C from a plan's info (the plan reports the MMA
    view, which for the swapped form tiles C's transpose)."""
    tm, tn = int(info.tile_m), int(info.tile_n)
    return (tn, tm) if info.swap_ab else (tm, tn)


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

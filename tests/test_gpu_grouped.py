"""Grouped launches: many independent problems of different sizes in one
persistent launch, each checked element by element against the fp64 oracle.
The problems mix ragged M, N, K tails, padded row strides, alpha/beta, and
problems with M or N of zero (skipped)."""
import itertools

import numpy as np
import pytest
import torch

import oracle
from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

from bmm_harness import decode_c

pytestmark = pytest.mark.gpu

NAN16 = {"bf16": 0x7FC0, "f16": 0x7E00}


def _problems(n, seed, transA, transB, type_ab, type_c, dims=(1, 17, 64, 100, 129, 200, 333),
              with_beta=True):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M, N, K = (int(rng.choice(dims)) for _ in range(3))
        if i == 3:
            M = 0                                    # skipped
        pad = int(rng.choice([0, 8]))
        ldc_align = 4 if type_c == "f32" else 8
        lda = ((M if transA else K) + 7) // 8 * 8 + pad
        ldb = ((K if transB else N) + 7) // 8 * 8 + pad
        ldc = (N + ldc_align - 1) // ldc_align * ldc_align + pad
        beta = float(rng.choice([0.0, 0.5])) if with_beta else 0.0
        p = wl.Problem(batch=1, M=M, N=N, K=K, transA=transA, transB=transB, type_ab=type_ab,
                       type_c=type_c, alpha=float(rng.choice([1.0, -0.75])), beta=beta,
                       lda=max(lda, 1), ldb=max(ldb, 1), ldc=max(ldc, 1), dist_ab="normal",
                       seed=seed * 100 + i)
        out.append(p)
    return out


def _run_group(problems, transA, transB, type_ab, type_c, stream=None):
    dev = torch.device("cuda:0")
    keep, items, xs = [], [], []
    for p in problems:
        x = wl.make_inputs(p)
        xs.append(x)
        s = p.strides()
        A = torch.from_numpy(np.concatenate([x.A, np.full(64, NAN16[type_ab], np.uint16)]).view(np.int16)).to(dev)
        B = torch.from_numpy(np.concatenate([x.B, np.full(64, NAN16[type_ab], np.uint16)]).view(np.int16)).to(dev)
        nc = max(p.storage_elems()[2], 1)
        if x.C_in is not None:
            c0 = x.C_in if type_c == "f32" else x.C_in
        else:
            c0 = np.full(nc, np.nan, np.float32) if type_c == "f32" else np.full(nc, 0x7FC0, np.uint16)
        C = torch.from_numpy(c0.copy() if type_c == "f32" else c0.view(np.int16).copy()).to(dev)
        keep += [A, B, C]
        items.append(dict(M=p.M, N=p.N, K=p.K, lda=s["lda"], ldb=s["ldb"], ldc=s["ldc"], A=A, B=B, C=C,
                          alpha=p.alpha, beta=p.beta))
    arr, n = api.make_problems(items)
    plan = api.bmm_grouped_create(arr, n, transA, transB, type_ab, type_c)
    try:
        info = api.bmm_grouped_get_info(plan)
        api.bmm_grouped_run(plan, arr, stream or torch.cuda.current_stream())
        torch.cuda.synchronize()
        st, word = api.bmm_grouped_get_device_error(plan)
        assert st == api.BMM_OK, f"device error {word:#x}"
    finally:
        api.bmm_grouped_destroy(plan)
    outs = []
    for p, it in zip(problems, items):
        c = it["C"].cpu().numpy()
        outs.append(c if type_c == "f32" else c.view(np.uint16))
    return outs, xs, info


def _check(p, x, c):
    if p.M == 0 or p.N == 0:
        return
    ref, bnd = oracle.bmm(x.A, x.B, x.C_in, **p.oracle_kwargs())
    got = decode_c(c, p)
    cin = None if x.C_in is None else decode_c(x.C_in, p)
    tol = oracle.tolerance(ref, bnd, cin, alpha=p.alpha, beta=p.beta, out_bf16=p.type_c == "bf16")
    assert np.all(np.isfinite(got))
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} elements outside tolerance"


@pytest.mark.parametrize("transA,transB", list(itertools.product([False, True], repeat=2)))
@pytest.mark.parametrize("type_ab,type_c", [("bf16", "f32"), ("f16", "bf16")])
def test_grouped_mixed_problems(transA, transB, type_ab, type_c):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    probs = _problems(12, 7 + 2 * transA + transB, transA, transB, type_ab, type_c)
    outs, xs, info = _run_group(probs, transA, transB, type_ab, type_c)
    assert info["tile_n"] in (64, 128, 256)
    for p, x, c in zip(probs, xs, outs):
        _check(p, x, c)


@pytest.mark.parametrize("width", ["256", "128"])
def test_grouped_pinned_widths(monkeypatch, width):
    """The default launch runs two CTAs per SM with 128-wide tiles; pinning
    256 runs one CTA per SM with 256-wide ones.  Problems up to 256 wide, so
    128-wide tiles split the wider ones in two N tiles."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("DMT_BMM_TILE_N", width)
    probs = _problems(20, 31, False, True, "bf16", "f32")
    outs, xs, info = _run_group(probs, False, True, "bf16", "f32")
    assert info["tile_n"] == int(width)
    for p, x, c in zip(probs, xs, outs):
        _check(p, x, c)


def test_grouped_many_small_problems():
    """A thousand small problems in one launch (the launch-bound case the
    grouping exists for); a sample of them is checked against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    probs = _problems(1000, 99, False, True, "bf16", "f32", dims=(16, 32, 48, 64), with_beta=False)
    outs, xs, info = _run_group(probs, False, True, "bf16", "f32")
    assert info["tile_n"] == 64
    rng = np.random.default_rng(5)
    for i in rng.choice(len(probs), 40, replace=False):
        _check(probs[i], xs[i], outs[i])


def test_grouped_rejections():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    A = torch.zeros(64 * 72, dtype=torch.bfloat16, device=dev)
    B = torch.zeros(64 * 72, dtype=torch.bfloat16, device=dev)
    C = torch.zeros(64 * 64, dtype=torch.float32, device=dev)
    base = dict(M=64, N=64, K=64, lda=64, ldb=64, ldc=64, A=A, B=B, C=C)
    for bad, code in [(dict(K=0), api.BMM_ERR_UNSUPPORTED), (dict(lda=65), api.BMM_ERR_UNSUPPORTED),
                      (dict(M=-1), api.BMM_ERR_INVALID_ARG), (dict(ldb=10), api.BMM_ERR_INVALID_ARG)]:
        arr, n = api.make_problems([dict(base, **bad)])
        with pytest.raises(api.BmmError) as e:
            api.bmm_grouped_create(arr, n, 0, 0, "bf16", "f32")
        assert e.value.status == code, bad
    arr, n = api.make_problems([base])
    plan = api.bmm_grouped_create(arr, n, 0, 0, "bf16", "f32")
    try:
        moved, _ = api.make_problems([dict(base, A=A.data_ptr() + 2)])      # not 16-byte aligned
        with pytest.raises(api.BmmError) as e:
            api.bmm_grouped_run(plan, moved, torch.cuda.current_stream())
        assert e.value.status == api.BMM_ERR_MISALIGNED
        resized, _ = api.make_problems([dict(base, N=32)])                  # sizes fixed at create
        with pytest.raises(api.BmmError) as e:
            api.bmm_grouped_run(plan, resized, torch.cuda.current_stream())
        assert e.value.status == api.BMM_ERR_INVALID_ARG
    finally:
        api.bmm_grouped_destroy(plan)


def test_reused_plan_follows_moved_outputs_and_new_scalars():
    """A grouped plan caches each problem's tensor maps and table entry by its
    pointers and scalars: run it, then with some problems writing to new C
    buffers and a new alpha, then with the original arguments again; every
    run must match the oracle (and the launch is dynamic: one CTA per tile,
    cluster launch control handing tiles out)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    problems = _problems(24, 77, False, True, "bf16", "f32", with_beta=False)
    xs = [wl.make_inputs(p) for p in problems]
    keep, items = [], []
    for p, x in zip(problems, xs):
        s = p.strides()
        A = torch.from_numpy(x.A.view(np.int16)).to(dev)
        B = torch.from_numpy(x.B.view(np.int16)).to(dev)
        C = torch.full((max(p.storage_elems()[2], 1),), float("nan"), device=dev)
        keep += [A, B, C]
        items.append(dict(M=p.M, N=p.N, K=p.K, lda=s["lda"], ldb=s["ldb"], ldc=s["ldc"], A=A, B=B, C=C,
                          alpha=p.alpha, beta=0.0))
    arr, n = api.make_problems(items)
    plan = api.bmm_grouped_create(arr, n, 0, 1, "bf16", "f32")
    try:
        def run_and_check(its, alphas):
            arr2, _ = api.make_problems(its)
            api.bmm_grouped_run(plan, arr2, torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert api.bmm_grouped_get_device_error(plan)[0] == api.BMM_OK
            for p, x, it, a in zip(problems, xs, its, alphas):
                q = wl.Problem(**{**p.__dict__, "alpha": a})
                _check(q, x, it["C"].cpu().numpy())

        run_and_check(items, [p.alpha for p in problems])
        moved = [dict(it) for it in items]
        for j in range(0, len(moved), 3):             # every third problem: new C, new alpha
            moved[j]["C"] = torch.full_like(items[j]["C"], float("nan"))
            moved[j]["alpha"] = 2.0
        run_and_check(moved, [2.0 if j % 3 == 0 else p.alpha for j, p in enumerate(problems)])
        for it in items:
            it["C"].fill_(float("nan"))
        run_and_check(items, [p.alpha for p in problems])
    finally:
        api.bmm_grouped_destroy(plan)

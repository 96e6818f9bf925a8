"""Products whose element offsets pass 2^31, through the C ABI on the GPU.

Each case is sized so that some offset into C (and, where noted, into A or
B) exceeds 2^31 elements, which int32 index arithmetic anywhere on the path
would wrap: the TMA box-store epilogue, the direct-store epilogue with an
unaligned ldc and beta != 0, the swapped (C^T) epilogue of skinny M, a K of
over a million (16385 k-blocks through a 6-stage ring), and eight million
small batch items; and the fused attention with 16 million keys and with
batch offsets past 2^31 in Q, K, V and O.  The inputs are drawn on the device (seeded); C starts as a
NaN pattern (beta = 0) or as seeded values with NaN padding (beta != 0).

Checks, all on the device except the last:
  - every element of C's logical region is finite (every element written,
    and no read outside A or B, whose guard elements hold NaN);
  - C's guards and its row padding still hold the NaN pattern bit for bit;
  - sampled elements (corners, the rows on both sides of the 2^31 offset,
    random ones) match the fp64 oracle within its bound: each sample's
    operand row and column are gathered from the device and the oracle takes
    them as a batch of 1 x 1 x K products.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_matmul_tensor_gb300 import bmm as api

pytestmark = pytest.mark.gpu

GUARD = 4096
NAN16 = 0x7FC0
NAN32 = 0x7FC00000
LIMIT = 1 << 31


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _span(items, stride, rows, ld, cols):
    if items <= 0 or rows <= 0 or cols <= 0:
        return 0
    return (items - 1) * stride + (rows - 1) * ld + cols


class Case:
    def __init__(self, *, batch, M, N, K, transA=False, transB=False, type_ab="bf16", type_c="f32",
                 alpha=1.0, beta=0.0, lda=None, ldb=None, ldc=None, seed=0):
        self.batch, self.M, self.N, self.K = batch, M, N, K
        self.transA, self.transB = transA, transB
        self.type_ab, self.type_c = type_ab, type_c
        self.alpha, self.beta, self.seed = alpha, beta, seed
        self.a_rows, self.a_cols = (K, M) if transA else (M, K)
        self.b_rows, self.b_cols = (N, K) if transB else (K, N)
        self.lda = lda or self.a_cols
        self.ldb = ldb or self.b_cols
        self.ldc = ldc or N
        self.sA = self.a_rows * self.lda
        self.sB = self.b_rows * self.ldb
        self.sC = M * self.ldc
        self.na = _span(batch, self.sA, self.a_rows, self.lda, self.a_cols)
        self.nb = _span(batch, self.sB, self.b_rows, self.ldb, self.b_cols)
        self.nc = _span(batch, self.sC, M, self.ldc, N)

    def desc(self):
        return api.make_desc(batch=self.batch, M=self.M, N=self.N, K=self.K, lda=self.lda, ldb=self.ldb,
                             ldc=self.ldc, strideA=self.sA, strideB=self.sB, strideC=self.sC,
                             transA=self.transA, transB=self.transB, typeA=self.type_ab,
                             typeC=self.type_c)


def _operand(n, dt, gen, dev):
    """Guard + n seeded uniform(-1, 1) values + guard, guards NaN (int16 view)."""
    buf = torch.full((GUARD + n + GUARD,), NAN16, dtype=torch.int16, device=dev)
    step = 1 << 28
    for s in range(0, n, step):
        e = min(n, s + step)
        x = torch.rand(e - s, generator=gen, device=dev, dtype=torch.float32) * 2 - 1
        buf[GUARD + s:GUARD + e] = x.to(dt).view(torch.int16)
        del x
    return buf


def _c_logical(c, case):
    """[batch, M, N] strided view of C's logical elements (int view)."""
    return torch.as_strided(c, (case.batch, case.M, case.N), (case.sC, case.ldc, 1), GUARD)


def _run_and_check(case, samples):
    _need_gpu()
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + case.seed)
    dt = torch.bfloat16 if case.type_ab == "bf16" else torch.float16
    A = _operand(case.na, dt, gen, dev)
    B = _operand(case.nb, dt, gen, dev)
    f32 = case.type_c == "f32"
    cint = torch.int32 if f32 else torch.int16
    C = torch.full((GUARD + case.nc + GUARD,), NAN32 if f32 else NAN16, dtype=cint, device=dev)
    if case.beta != 0.0:
        view = _c_logical(C, case)
        for b in range(case.batch):
            x = torch.rand(case.M, case.N, generator=gen, device=dev) * 2 - 1
            view[b] = (x if f32 else x.to(torch.bfloat16)).view(cint)
            del x
    s = np.asarray(samples, dtype=np.int64)
    c_off = torch.from_numpy(GUARD + s[:, 0] * case.sC + s[:, 1] * case.ldc + s[:, 2]).to(dev)
    c_in = C[c_off].cpu().numpy()

    with api.Plan(case.desc()) as plan:
        es = 2
        plan.run(A.data_ptr() + GUARD * es, B.data_ptr() + GUARD * es,
                 C.data_ptr() + GUARD * (4 if f32 else 2), case.alpha, case.beta,
                 torch.cuda.current_stream())
        torch.cuda.synchronize()
        st, word = plan.device_error()
    assert st == api.BMM_OK, f"device error word {word:#x}"

    # every logical element written and finite; guards and padding untouched
    logical = _c_logical(C, case)
    vals = logical.view(torch.float32) if f32 else logical.view(torch.bfloat16)
    assert bool(torch.isfinite(vals).all()), "C holds non-finite values (unwritten, or a read outside A/B)"
    nanbits = NAN32 if f32 else NAN16
    assert bool((C[:GUARD] == nanbits).all()) and bool((C[GUARD + case.nc:] == nanbits).all()), \
        "write outside C"
    if case.ldc > case.N and case.M > 1:
        pad = torch.as_strided(C, (case.batch, case.M - 1, case.ldc - case.N), (case.sC, case.ldc, 1),
                               GUARD + case.N)
        assert bool((pad == nanbits).all()), "write into C's row padding"
    del logical, vals

    # the samples against the oracle, one 1 x 1 x K product per sample
    k = torch.arange(case.K, device=dev, dtype=torch.int64)
    sb, si, sj = (torch.from_numpy(s[:, c].copy()).to(dev)[:, None] for c in range(3))
    a_idx = sb * case.sA + ((k[None, :] * case.lda + si) if case.transA else (si * case.lda + k[None, :]))
    b_idx = sb * case.sB + ((sj * case.ldb + k[None, :]) if case.transB else (k[None, :] * case.ldb + sj))
    a_bits = A[GUARD + a_idx].cpu().numpy().view(np.uint16).reshape(-1)
    b_bits = B[GUARD + b_idx].cpu().numpy().view(np.uint16).reshape(-1)
    got_raw = C[c_off].cpu().numpy()
    n = s.shape[0]
    if f32:
        cin = c_in.view(np.float32)
        got = got_raw.view(np.float32).astype(np.float64)
        cin64 = cin.astype(np.float64)
    else:
        cin = c_in.view(np.uint16)
        got = torch.from_numpy(got_raw).view(torch.bfloat16).double().numpy()
        cin64 = torch.from_numpy(c_in).view(torch.bfloat16).double().numpy()
    ref, bnd = oracle.bmm(a_bits, b_bits, cin if case.beta != 0.0 else None, batch=n, M=1, N=1, K=case.K,
                          lda=case.K, ldb=case.K, ldc=1, sA=case.K, sB=case.K, sC=1, transA=False,
                          transB=True, type_ab=case.type_ab, type_c=case.type_c, alpha=case.alpha,
                          beta=case.beta)
    ref, bnd = ref.reshape(-1), bnd.reshape(-1)
    tol = oracle.tolerance(ref, bnd, cin64 if case.beta != 0.0 else None, alpha=case.alpha,
                           beta=case.beta, out_bf16=not f32)
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), [(tuple(s[i]), got[i], ref[i], tol[i]) for i in np.nonzero(bad)[0][:5]]
    del A, B, C
    torch.cuda.empty_cache()


def _samples(case, n_random, seed, extra_rows=()):
    """Corners, the rows either side of the first row whose offset passes
    2^31, extra rows, and random elements: (b, i, j) triples."""
    rng = np.random.default_rng(seed)
    out = []
    bs = sorted({0, case.batch - 1})
    cross = LIMIT // case.ldc if case.batch == 1 else None
    rows = {0, case.M - 1, *[r for r in extra_rows if 0 <= r < case.M]}
    if cross is not None:
        rows |= {r for r in (cross - 1, cross, cross + 1) if 0 <= r < case.M}
    cols = sorted({0, 1, case.N - 1, case.N // 2})
    for b in bs:
        for i in sorted(rows):
            for j in cols:
                out.append((b, i, j))
    out += [(int(rng.integers(0, case.batch)), int(rng.integers(0, case.M)), int(rng.integers(0, case.N)))
            for _ in range(n_random)]
    return np.array(out, dtype=np.int64)


def test_bf16_tma_store_epilogue_past_2_31_elements():
    # 46403 x 46408 bf16 C (2.15e9 elements), row-major TN, ragged last row tile
    case = Case(batch=1, M=46403, N=46408, K=64, transB=True, type_ab="bf16", type_c="bf16", seed=1)
    assert case.nc > LIMIT
    _run_and_check(case, _samples(case, 96, 1))


def test_f32_direct_store_unaligned_ldc_with_beta_past_2_31():
    # ldc = N + 2 (odd: no TMA store), beta != 0 reads C_in there; A MN-major;
    # B's row stride (46341 halves) is not 16-byte aligned, so B is staged
    case = Case(batch=1, M=46400, N=46341, K=40, transA=True, type_ab="f16", type_c="f32",
                alpha=0.5, beta=-1.25, ldc=46343, seed=2)
    assert case.nc > LIMIT
    _run_and_check(case, _samples(case, 96, 2))


def test_skinny_swapped_epilogue_past_2_31():
    # M = 16: the product runs as C^T = B^T A^T, whose epilogue writes C
    # column-wise: C offsets reach 15 * ldc + N - 1 > 2^31
    case = Case(batch=1, M=16, N=134_217_800, K=16, transB=True, type_ab="bf16", type_c="bf16", seed=3)
    assert case.nc > LIMIT
    _run_and_check(case, _samples(case, 64, 3, extra_rows=range(16)))


def test_k_of_a_million_wraps_the_ring_many_times():
    # 256 x 256 (one CTA-pair tile), K = 2^20 + 40: 16385 k-blocks, a 40-wide tail
    case = Case(batch=1, M=256, N=256, K=(1 << 20) + 40, transB=True, type_ab="bf16", type_c="f32", seed=4)
    _run_and_check(case, _samples(case, 8, 4, extra_rows=(127, 128)))


def test_eight_million_batch_items_past_2_31():
    # 2^23 + 5 items of 16 x 16 x 16: batch offsets of A, B (bf16) and C (fp32)
    # all pass 2^31 elements
    case = Case(batch=(1 << 23) + 5, M=16, N=16, K=16, type_ab="bf16", type_c="f32", seed=5)
    assert case.na > LIMIT and case.nc > LIMIT
    samples = _samples(case, 64, 5)
    tail = np.array([(case.batch - 1 - d, i, j) for d in range(3) for i in (0, 15) for j in (0, 15)])
    mid = LIMIT // case.sC
    across = np.array([(b, i, j) for b in (mid - 1, mid, mid + 1) for i in (0, 15) for j in (0, 15)])
    _run_and_check(case, np.concatenate([samples, tail, across]))


# ---------------------------------------------------------------- fused attention

ATTN_D = 128
ATTN_ALPHA = float(np.float32(1.0 / np.sqrt(ATTN_D)))


def _attn_run_and_check(batch, Lq, Lk, sample_items, rows, seed):
    """Fused attention with dense [batch, L, 128] bf16 operands drawn on the
    device (normal), guards NaN; every output finite, guards untouched, and
    the sampled query rows of the sampled batch items against the oracle."""
    _need_gpu()
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev)
    gen.manual_seed(4321 + seed)

    def draw(n):
        buf = torch.full((GUARD + n + GUARD,), NAN16, dtype=torch.int16, device=dev)
        step = 1 << 28
        for s in range(0, n, step):
            e = min(n, s + step)
            buf[GUARD + s:GUARD + e] = torch.randn(e - s, generator=gen, device=dev).to(
                torch.bfloat16).view(torch.int16)
        return buf

    D = ATTN_D
    q, k, v = draw(batch * Lq * D), draw(batch * Lk * D), draw(batch * Lk * D)
    o = torch.full((GUARD + batch * Lq * D + GUARD,), NAN16, dtype=torch.int16, device=dev)
    es = 2
    with api.AttnPlan(api.make_attn_desc(batch=batch, Lq=Lq, Lk=Lk, alpha=ATTN_ALPHA)) as plan:
        plan.run(q.data_ptr() + GUARD * es, k.data_ptr() + GUARD * es, v.data_ptr() + GUARD * es,
                 o.data_ptr() + GUARD * es, torch.cuda.current_stream())
        torch.cuda.synchronize()
        st, word = plan.device_error()
    assert st == api.BMM_OK, f"device error word {word:#x}"
    body = o[GUARD:GUARD + batch * Lq * D]
    assert bool(torch.isfinite(body.view(torch.bfloat16)).all()), "non-finite O"
    assert bool((o[:GUARD] == NAN16).all()) and bool((o[GUARD + batch * Lq * D:] == NAN16).all()), \
        "write outside O"
    rows = np.array(sorted(set(rows)), dtype=np.int64)
    for b in sample_items:
        qb = q[GUARD + b * Lq * D:GUARD + (b + 1) * Lq * D].view(Lq, D)[torch.from_numpy(rows).to(dev)]
        kb = k[GUARD + b * Lk * D:GUARD + (b + 1) * Lk * D]
        vb = v[GUARD + b * Lk * D:GUARD + (b + 1) * Lk * D]
        ref, bnd = oracle.attention(qb.cpu().numpy().view(np.uint16)[None], kb.cpu().numpy().view(np.uint16),
                                    vb.cpu().numpy().view(np.uint16), batch=1, Lq=len(rows), Lk=Lk, D=D,
                                    alpha=ATTN_ALPHA)
        ob = o[GUARD + b * Lq * D:GUARD + (b + 1) * Lq * D].view(Lq, D)[torch.from_numpy(rows).to(dev)]
        got = ob.view(torch.bfloat16).double().cpu().numpy()
        err = np.abs(got - ref[0])
        tol = oracle.attention_tolerance(ref, bnd, qb.cpu().numpy().view(np.uint16)[None],
                                         kb.cpu().numpy().view(np.uint16), vb.cpu().numpy().view(np.uint16),
                                         alpha=ATTN_ALPHA)[0]
        assert np.all(err <= tol), (b, float((err / tol).max()))
    del q, k, v, o
    torch.cuda.empty_cache()


def test_attention_sixteen_million_keys():
    # one item of 128 queries over 2^24 + 100 keys: K and V offsets pass 2^31
    # elements and one CTA walks 131073 key blocks through its two K/V slots
    Lk = (1 << 24) + 100
    assert Lk * ATTN_D > LIMIT
    _attn_run_and_check(1, 128, Lk, [0], [0, 1, 63, 64, 126, 127], 11)


def test_attention_batch_offsets_past_2_31():
    # 2^17 + 3 items of 200 queries x 130 keys: Q, K, V and O batch offsets
    # pass 2^31 elements (Q and O at item 83886, K and V at item 129055)
    batch, Lq, Lk = (1 << 17) + 3, 200, 130
    assert batch * Lk * ATTN_D > LIMIT and batch * Lq * ATTN_D > LIMIT
    q_cross, k_cross = LIMIT // (Lq * ATTN_D), LIMIT // (Lk * ATTN_D)
    _attn_run_and_check(batch, Lq, Lk, [0, q_cross, q_cross + 1, k_cross, k_cross + 1, batch - 1],
                        [0, 127, 128, 199], 12)

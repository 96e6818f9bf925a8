"""Pins for the fp64 CPU oracle: each check ties it to something other than
itself — closed forms, exact small-integer arithmetic, brute force in
Python integers, float64 library routines, format definitions — so that a
dropped term, a wrong sign or index, or a transposed operand fails a test.

The storage convention under test ("Triton Optimization Reference (cuTile ->
Triton)", section 2: transposition lives in the strides used to address A and
B) is row-major with element strides; see ``workloads.Problem``.
"""
import itertools
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from dense_matmul_tensor_gb300 import workloads as wl

NAN16 = {"bf16": 0x7FC0, "f16": 0x7E00}


def encode(x, dtype):
    """Exactly representable float64 values -> 16-bit patterns (torch cast)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float64))
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def store(op, trans, ld=None, stride=None, dtype="bf16", pad=None):
    """Lay out the logical operands op[b] (R x C) in row-major storage.
    trans=True stores op[b]^T.  Padding elements get ``pad`` bits (NaN by
    default, so any read of padding poisons the result)."""
    op = np.asarray(op, dtype=np.float64)
    batch = op.shape[0]
    mats = np.transpose(op, (0, 2, 1)) if trans else op
    rows, cols = mats.shape[1], mats.shape[2]
    ld = cols if ld is None else ld
    stride = rows * ld if stride is None else stride
    n = 0 if batch == 0 else (batch - 1) * stride + (rows - 1) * ld + cols
    buf = np.full(max(n, 1), NAN16[dtype] if pad is None else pad, dtype=np.uint16)
    for b in range(batch if stride else min(batch, 1)):
        for r in range(rows):
            o = b * stride + r * ld
            buf[o:o + cols] = encode(mats[b, r], dtype)
    return buf, ld, stride


def run(opA, opB, *, transA=False, transB=False, dtype="bf16", alpha=1.0, beta=0.0,
        Cin=None, pads=(0, 0, 0), type_c="f32", threads=None, bcastA=False, bcastB=False):
    opA = np.asarray(opA, np.float64)
    opB = np.asarray(opB, np.float64)
    batch, M, K = opA.shape
    N = opB.shape[2]
    A, lda, sA = store(opA[:1] if bcastA else opA, transA,
                       ld=(K if not transA else M) + pads[0], dtype=dtype)
    B, ldb, sB = store(opB[:1] if bcastB else opB, transB,
                       ld=(N if not transB else K) + pads[1], dtype=dtype)
    if bcastA:
        sA = 0
    if bcastB:
        sB = 0
    ldc = N + pads[2]
    sC = M * ldc
    if Cin is None:
        cbuf = np.full(max(batch * sC, 1), np.nan, dtype=np.float32)
    else:
        cbuf = np.full(max(batch * sC, 1), np.nan, dtype=np.float32)
        for b in range(batch):
            for i in range(M):
                cbuf[b * sC + i * ldc: b * sC + i * ldc + N] = Cin[b, i]
    if type_c == "bf16":
        cbuf = encode(np.nan_to_num(cbuf.astype(np.float64), nan=np.nan), "bf16")
    return oracle.bmm(A, B, cbuf, batch=batch, M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc,
                      sA=sA, sB=sB, sC=sC, transA=transA, transB=transB, type_ab=dtype,
                      type_c=type_c, alpha=alpha, beta=beta, threads=threads)


def brute(opA, opB, alpha=1.0, beta=0.0, Cin=None):
    """Python-integer / exact-float reference: the definition, term by term."""
    batch, M, K = len(opA), len(opA[0]), len(opA[0][0])
    N = len(opB[0][0])
    out = np.zeros((batch, M, N))
    for b in range(batch):
        for i in range(M):
            for j in range(N):
                s = 0
                for k in range(K):
                    s += int(opA[b][i][k]) * int(opB[b][k][j])
                v = alpha * s
                if beta != 0.0:
                    v += beta * Cin[b][i][j]
                out[b, i, j] = v
    return out


# ------------------------------------------------------------ format pins

def test_decode_known_patterns():
    # IEEE binary16 and bfloat16 definitions
    cases_f16 = {0x3C00: 1.0, 0xC400: -4.0, 0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24,
                 0x0400: 2.0 ** -14, 0x7BFF: 65504.0, 0x3555: 1365 * 2.0 ** -12, 0x8000: -0.0}
    cases_bf16 = {0x3F80: 1.0, 0xC000: -2.0, 0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126,
                  0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x3E00: 0.125, 0xBF40: -0.75}
    for bits, v in cases_f16.items():
        assert oracle.decode(np.uint16(bits), "f16") == v
    for bits, v in cases_bf16.items():
        assert oracle.decode(np.uint16(bits), "bf16") == v
    assert math.copysign(1.0, float(oracle.decode(np.uint16(0x8000), "f16"))) == -1.0


def test_decode_all_patterns_match_library():
    allbits = np.arange(65536, dtype=np.uint16)
    ours16 = oracle.decode(allbits, "f16")
    lib16 = allbits.view(np.float16).astype(np.float64)
    fin = np.isfinite(lib16)
    assert np.array_equal(ours16[fin], lib16[fin])
    assert np.all(np.isnan(ours16[np.isnan(lib16)]))
    oursb = oracle.decode(allbits, "bf16")
    libb = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).double().numpy()
    fin = np.isfinite(libb)
    assert np.array_equal(oursb[fin], libb[fin])
    assert np.array_equal(np.isinf(oursb), np.isinf(libb))


def test_round_bf16_ties_and_no_double_rounding():
    one = 1.0
    # halfway between 1 and 1+2^-7 -> even (1.0); between 1+2^-7 and 1+2^-6 -> 1+2^-6
    assert oracle.round_bf16(one + 2.0 ** -8) == 0x3F80
    assert oracle.round_bf16(one + 3 * 2.0 ** -8) == encode(one + 2.0 ** -6, "bf16")[()]
    # just above a tie: direct rounding goes up; rounding through fp32 first would not
    assert oracle.round_bf16(one + 2.0 ** -8 + 2.0 ** -40) == encode(one + 2.0 ** -7, "bf16")[()]
    assert oracle.round_bf16(-(one + 2.0 ** -8 + 2.0 ** -40)) == encode(-(one + 2.0 ** -7), "bf16")[()]
    assert oracle.round_bf16(2.0 ** -133) == 0x0001
    assert oracle.round_bf16(3.0 * 2.0 ** -134) == 0x0002          # tie between 1 and 2 quanta -> 2
    assert oracle.round_bf16(2.0 ** 200) == 0x7F80


def test_round_bf16_matches_library_on_float32_values():
    x = (wl.draw(20000, 77, "normal") * np.float32(1e3)).astype(np.float64)   # exact fp32 values
    ours = oracle.round_bf16(x)
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)


# --------------------------------------------------------- product pins

@pytest.mark.parametrize("transA,transB", list(itertools.product([False, True], repeat=2)))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_permutation_matrices_exact(transA, transB, dtype):
    rng = np.random.default_rng(5)
    M = K = 7
    N = 5
    perm = rng.permutation(M)
    P = np.zeros((1, M, K))
    P[0, np.arange(M), perm] = 1.0
    Bv = rng.integers(-8, 9, size=(1, K, N)).astype(np.float64)
    c, bnd = run(P, Bv, transA=transA, transB=transB, dtype=dtype, pads=(3, 1, 2))
    assert np.array_equal(c[0], Bv[0][perm])            # row i of C = row perm[i] of B
    assert np.array_equal(bnd[0], np.abs(Bv[0][perm]))
    # permutation on the right: C = A Q^T gives column permutation
    Av = rng.integers(-8, 9, size=(1, M, K)).astype(np.float64)
    Q = np.zeros((1, K, K))
    Q[0, perm, np.arange(K)] = 1.0                      # (A Q)[:, j] = A[:, perm[j]]
    c2, _ = run(Av, Q, transA=transA, transB=transB, dtype=dtype)
    assert np.array_equal(c2[0], Av[0][:, perm])


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rank1_closed_form(dtype):
    rng = np.random.default_rng(11)
    batch, M, N, K = 3, 9, 13, 37
    u = rng.integers(-7, 8, size=(batch, M)).astype(np.float64)
    v = rng.integers(-7, 8, size=(batch, N)).astype(np.float64)
    A = np.repeat(u[:, :, None], K, axis=2)               # A = u 1^T
    B = np.repeat(v[:, None, :], K, axis=1)               # B = 1 v^T
    c, bnd = run(A, B, dtype=dtype, transB=True)
    expect = K * u[:, :, None] * v[:, None, :]
    assert np.array_equal(c, expect)
    assert np.array_equal(bnd, np.abs(expect))


@pytest.mark.parametrize("transA,transB", list(itertools.product([False, True], repeat=2)))
def test_small_integers_vs_python_brute_force(transA, transB):
    rng = np.random.default_rng(3 + 2 * transA + transB)
    batch, M, N, K = 2, 5, 6, 11
    A = rng.integers(-4, 5, size=(batch, M, K))
    B = rng.integers(-4, 5, size=(batch, K, N))
    Cin = rng.integers(-4, 5, size=(batch, M, N)).astype(np.float64)
    c, _ = run(A, B, transA=transA, transB=transB, alpha=0.5, beta=-2.0, Cin=Cin,
               pads=(2, 3, 1), threads=3)
    ref = brute(A.tolist(), B.tolist(), alpha=0.5, beta=-2.0, Cin=Cin.tolist())
    assert np.array_equal(c, ref)


def test_batch_broadcast_and_bf16_cin():
    rng = np.random.default_rng(8)
    batch, M, N, K = 3, 4, 5, 6
    A = np.repeat(rng.integers(-3, 4, size=(1, M, K)), batch, axis=0)
    B = rng.integers(-3, 4, size=(batch, K, N))
    Cin = rng.integers(-3, 4, size=(batch, M, N)).astype(np.float64)
    c, _ = run(A, B, bcastA=True, beta=1.0, Cin=Cin, type_c="bf16")
    ref = brute(A.tolist(), B.tolist(), beta=1.0, Cin=Cin.tolist())
    assert np.array_equal(c, ref)
    A2 = rng.integers(-3, 4, size=(batch, M, K))
    B2 = np.repeat(rng.integers(-3, 4, size=(1, K, N)), batch, axis=0)
    c2, _ = run(A2, B2, bcastB=True, transB=True)
    assert np.array_equal(c2, brute(A2.tolist(), B2.tolist()))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_random_vs_float64_library_matmul(dtype):
    p = wl.Problem(batch=3, M=37, N=29, K=83, transA=True, type_ab=dtype, seed=21)
    x = wl.make_inputs(p)
    s = p.strides()
    c, bnd = oracle.bmm(x.A, x.B, None, **p.oracle_kwargs())
    tA = wl.as_torch16(x.A, dtype).double()
    tB = wl.as_torch16(x.B, dtype).double()
    for b in range(p.batch):
        Ab = tA[b * s["sA"]: b * s["sA"] + p.a_rows * s["lda"]].view(p.a_rows, s["lda"])[:, :p.a_cols]
        Bb = tB[b * s["sB"]: b * s["sB"] + p.b_rows * s["ldb"]].view(p.b_rows, s["ldb"])[:, :p.b_cols]
        opA = Ab.T if p.transA else Ab
        opB = Bb.T if p.transB else Bb
        ref = (opA @ opB).numpy()
        absref = (opA.abs() @ opB.abs()).numpy()
        assert np.all(np.abs(c[b] - ref) <= 1e-12 * absref + 1e-300)
        assert np.allclose(bnd[b], absref, rtol=1e-12, atol=0)


def test_transpose_equivalence_bitwise():
    """op(A) stored transposed must give the very same bits as the same
    operand stored plainly (all four transpose pairs)."""
    rng = np.random.default_rng(99)
    batch, M, N, K = 2, 6, 7, 9
    A = wl.round16(rng.standard_normal(batch * M * K).astype(np.float32), "bf16")
    B = wl.round16(rng.standard_normal(batch * K * N).astype(np.float32), "bf16")
    Av = oracle.decode(A, "bf16").reshape(batch, M, K)
    Bv = oracle.decode(B, "bf16").reshape(batch, K, N)
    base, _ = run(Av, Bv)
    for tA, tB in itertools.product([False, True], repeat=2):
        c, _ = run(Av, Bv, transA=tA, transB=tB, pads=(1, 2, 0))
        assert np.array_equal(c, base), (tA, tB)


def test_alpha_beta_special_cases():
    rng = np.random.default_rng(4)
    batch, M, N, K = 2, 5, 4, 6
    A = rng.integers(-3, 4, size=(batch, M, K)).astype(np.float64)
    B = rng.integers(-3, 4, size=(batch, K, N)).astype(np.float64)
    Cin = rng.standard_normal((batch, M, N)).astype(np.float32).astype(np.float64)
    c0, _ = run(A, B, alpha=0.0, beta=0.75, Cin=Cin)
    assert np.array_equal(c0, 0.75 * Cin)                 # alpha = 0: beta*C exactly
    cn, _ = run(A, B, alpha=1.0, beta=0.0)                # C buffer is NaN: never read
    assert np.all(np.isfinite(cn))
    assert np.array_equal(cn, brute(A.astype(int).tolist(), B.astype(int).tolist()))
    ck, bk = run(A[:, :, :0], B[:, :0, :], beta=-1.5, Cin=Cin)   # K = 0
    assert np.array_equal(ck, -1.5 * Cin)
    assert np.all(bk == 0)


def test_empty_problems():
    c, b = run(np.zeros((0, 3, 4)), np.zeros((0, 4, 2)))
    assert c.shape == (0, 3, 2)
    c, b = run(np.zeros((2, 0, 4)), np.zeros((2, 4, 2)))
    assert c.shape == (2, 0, 2)


def test_sampled_equals_full_bitwise():
    p = wl.Problem(batch=3, M=33, N=47, K=129, transB=True, type_ab="f16", type_c="bf16",
                   alpha=-1.25, beta=0.5, seed=31, lda=140, ldc=50)
    x = wl.make_inputs(p)
    c, bnd = oracle.bmm(x.A, x.B, x.C_in, **p.oracle_kwargs())
    rng = np.random.default_rng(1)
    idx = np.stack([rng.integers(0, p.batch, 200), rng.integers(0, p.M, 200),
                    rng.integers(0, p.N, 200)], axis=1)
    cs, bs = oracle.bmm_sampled(x.A, x.B, x.C_in, idx, **p.oracle_kwargs())
    assert np.array_equal(cs, c[idx[:, 0], idx[:, 1], idx[:, 2]])
    assert np.array_equal(bs, bnd[idx[:, 0], idx[:, 1], idx[:, 2]])


def test_bound_dominates_and_is_tight_for_nonnegative():
    p = wl.Problem(batch=2, M=20, N=30, K=40, seed=41)
    x = wl.make_inputs(p)
    c, bnd = oracle.bmm(x.A, x.B, None, **p.oracle_kwargs())
    assert np.all(np.abs(c) <= bnd * (1 + 1e-15))
    absA = x.A & np.uint16(0x7FFF)
    absB = x.B & np.uint16(0x7FFF)
    c2, bnd2 = oracle.bmm(absA, absB, None, **p.oracle_kwargs())
    assert np.array_equal(c2, bnd2)
    assert np.array_equal(bnd2, bnd)


def test_threads_do_not_change_bits():
    p = wl.Problem(batch=2, M=41, N=23, K=57, transA=True, seed=51)
    x = wl.make_inputs(p)
    c1, b1 = oracle.bmm(x.A, x.B, None, threads=1, **p.oracle_kwargs())
    c7, b7 = oracle.bmm(x.A, x.B, None, threads=7, **p.oracle_kwargs())
    assert np.array_equal(c1, c7) and np.array_equal(b1, b7)


# ------------------------------------------------ attention-pair recipe

def test_attention_probs_rows_and_library_softmax():
    batch, L, D = 2, 40, 16
    base = 9000
    Q = wl.bits16(batch * L * D, base + 1, "normal", "bf16").reshape(batch, L, D)
    Kt = wl.bits16(batch * L * D, base + 2, "normal", "bf16").reshape(batch, L, D)
    alpha = float(np.float32(1 / math.sqrt(D)))
    P = oracle.attention_probs_bf16(Q, Kt, batch=batch, L=L, D=D, alpha=alpha)
    Pv = oracle.decode(P, "bf16")
    # every row of a softmax sums to 1; one bf16 rounding (unit roundoff 2^-8)
    # per entry moves the row sum by at most 2^-8
    assert np.all(np.abs(Pv.sum(axis=2) - 1.0) <= 2.0 ** -8 + 1e-12)
    q = torch.from_numpy(Q.view(np.int16)).view(torch.bfloat16).double()
    k = torch.from_numpy(Kt.view(np.int16)).view(torch.bfloat16).double()
    S = alpha * (q @ k.transpose(1, 2))
    ref = torch.softmax(S, dim=2).numpy()
    assert np.all(np.abs(Pv - ref) <= 2.0 ** -8 * ref + 1e-15)
    assert np.array_equal(P, oracle.round_bf16(ref)) or \
        np.mean(P == oracle.round_bf16(ref)) > 0.999   # ties in last ulp only


# ------------------------------------------ planted mistakes (mutations)

MUTATIONS = {
    # a dropped term: the last k never enters the sum
    "drop_last_k": ("for (int64_t k = 0; k < K; ++k) {\n      const double a = arow[k];",
                    "for (int64_t k = 0; k < K - 1; ++k) {\n      const double a = arow[k];"),
    # a transposed operand: B read as if transB had the other value
    "transpose_B": ("int64_t off = d->transB ? n * d->ldb + k : k * d->ldb + n;",
                    "int64_t off = d->transB ? k * d->ldb + n : n * d->ldb + k;"),
    # a wrong sign on the beta term
    "beta_sign": ("if (d->beta != 0.0) c += d->beta *", "if (d->beta != 0.0) c -= d->beta *"),
    # a wrong index: rows of C written transposed within the batch
    "index_swap": ("const int64_t o = (b * d->M + i) * N + n;",
                   "const int64_t o = b * d->M * N + n * d->M + i;"),
    # fp16 exponent bias off by one
    "f16_bias": ("ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
}


def _pin_suite(lib_module):
    """A compact subset of the pins above, run against ``lib_module``."""
    failures = []
    rng = np.random.default_rng(123)
    for tA, tB in itertools.product([False, True], repeat=2):
        batch, M, N, K = 2, 5, 3, 7
        A = rng.integers(-4, 5, size=(batch, M, K))
        B = rng.integers(-4, 5, size=(batch, K, N))
        Cin = rng.integers(-4, 5, size=(batch, M, N)).astype(np.float64)
        for dtype in ("bf16", "f16"):
            Ab, lda, sA = store(A, tA, dtype=dtype)
            Bb, ldb, sB = store(B, tB, dtype=dtype)
            cf = Cin.astype(np.float32).ravel()
            c, _ = lib_module.bmm(Ab, Bb, cf, batch=batch, M=M, N=N, K=K, lda=lda, ldb=ldb,
                                  ldc=N, sA=sA, sB=sB, sC=M * N, transA=tA, transB=tB,
                                  type_ab=dtype, alpha=1.0, beta=1.0)
            ref = brute(A.tolist(), B.tolist(), beta=1.0, Cin=Cin.tolist())
            if not np.array_equal(c, ref):
                failures.append((tA, tB, dtype))
    return failures


def test_pins_pass_on_the_oracle():
    assert _pin_suite(oracle) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    """Plant one plausible mistake in a copy of the oracle source, build it
    on the CPU, and check that the pins reject the mutant."""
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "bmm_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(mutant_src),
                    "-lm", "-lpthread"], check=True)
    import ctypes
    import types
    mut = types.SimpleNamespace()
    lib = ctypes.CDLL(str(so))
    i64, i32, f64, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    lib.oracle_bmm_f64.argtypes = [i64] * 10 + [i32] * 4 + [f64, f64] + [vp] * 5 + [i32]
    lib.oracle_bmm_f64.restype = i32

    def bmm(A, B, C_in, *, batch, M, N, K, lda, ldb, ldc, sA, sB, sC, transA, transB,
            type_ab, alpha, beta):
        cref = np.empty((batch, M, N))
        bnd = np.empty((batch, M, N))
        t = oracle._TYPE_CODES[type_ab]
        rc = lib.oracle_bmm_f64(batch, M, N, K, lda, ldb, ldc, sA, sB, sC, int(transA),
                                int(transB), t, oracle.F32, alpha, beta, oracle._ptr(A),
                                oracle._ptr(B), oracle._ptr(np.ascontiguousarray(C_in)),
                                oracle._ptr(cref), oracle._ptr(bnd), 2)
        assert rc == 0
        return cref, bnd

    mut.bmm = bmm
    if name == "f16_bias":
        # values near 1 in fp16 decode to twice their size: caught by the fp16 runs
        pass
    assert _pin_suite(mut) != [], f"pins did not catch mutation {name}"


# ------------------------------------------------- fused attention oracle

def _att_inputs(batch, Lq, Lk, D, seed):
    Q = wl.bits16(batch * Lq * D, seed + 1, "normal", "bf16").reshape(batch, Lq, D)
    Kt = wl.bits16(batch * Lk * D, seed + 2, "normal", "bf16").reshape(batch, Lk, D)
    V = wl.bits16(batch * Lk * D, seed + 3, "normal", "bf16").reshape(batch, Lk, D)
    return Q, Kt, V


def test_attention_oracle_vs_library_softmax():
    batch, Lq, Lk, D = 2, 33, 70, 16
    Q, Kt, V = _att_inputs(batch, Lq, Lk, D, 500)
    alpha = float(np.float32(1 / math.sqrt(D)))
    O, bnd = oracle.attention(Q, Kt, V, batch=batch, Lq=Lq, Lk=Lk, D=D, alpha=alpha)
    q, k, v = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double() for x in (Q, Kt, V))
    P = torch.softmax(alpha * (q @ k.transpose(1, 2)), dim=2)
    ref = (P @ v).numpy()
    absref = (P @ v.abs()).numpy()
    assert np.all(np.abs(O - ref) <= 1e-12 * absref + 1e-300)
    assert np.allclose(bnd, absref, rtol=1e-12, atol=0)


def test_attention_oracle_closed_forms():
    batch, Lq, Lk, D = 1, 5, 9, 8
    _, Kt, V = _att_inputs(batch, Lq, Lk, D, 600)
    # Q = 0: every score is 0, the softmax is uniform, O is the mean of V's rows
    Q0 = np.zeros((batch, Lq, D), np.uint16)
    O, _ = oracle.attention(Q0, Kt, V, batch=batch, Lq=Lq, Lk=Lk, D=D, alpha=1.0)
    mean = oracle.decode(V, "bf16").mean(axis=1)
    assert np.allclose(O, mean[:, None, :], rtol=0, atol=1e-15)
    # one key aligned with the query and a huge scale: O is that key's value row
    Qv = np.tile(encode(np.eye(D)[0] * 4.0, "bf16"), (batch, Lq, 1))
    Kv = np.tile(encode(np.zeros(D), "bf16"), (batch, Lk, 1))
    Kv[0, 6] = encode(np.eye(D)[0] * 4.0, "bf16")
    O1, _ = oracle.attention(Qv, Kv, V, batch=batch, Lq=Lq, Lk=Lk, D=D, alpha=100.0)
    assert np.allclose(O1[0], oracle.decode(V, "bf16")[0, 6][None, :], rtol=0, atol=1e-12)


def test_attention_oracle_key_permutation_invariance():
    batch, Lq, Lk, D = 1, 7, 12, 8
    Q, Kt, V = _att_inputs(batch, Lq, Lk, D, 700)
    perm = np.random.default_rng(3).permutation(Lk)
    O, _ = oracle.attention(Q, Kt, V, batch=batch, Lq=Lq, Lk=Lk, D=D, alpha=0.3)
    Op, _ = oracle.attention(Q, Kt[:, perm], V[:, perm], batch=batch, Lq=Lq, Lk=Lk, D=D, alpha=0.3)
    assert np.allclose(O, Op, rtol=1e-13, atol=1e-15)


def test_attention_oracle_matches_probs_then_product():
    """The fused definition equals the two-step path of the pair workload
    (probabilities from attention_probs, then their product with V) before
    any rounding of P: compare with fp64 P from the library softmax."""
    batch, L, D = 1, 40, 16
    Q, Kt, V = _att_inputs(batch, L, L, D, 800)
    alpha = 0.25
    O, _ = oracle.attention(Q, Kt, V, batch=batch, Lq=L, Lk=L, D=D, alpha=alpha)
    P = oracle.attention_probs_bf16(Q, Kt, batch=batch, L=L, D=D, alpha=alpha)
    Pv = oracle.decode(P, "bf16")
    Vv = oracle.decode(V, "bf16")
    two_step = Pv @ Vv
    bnd = np.abs(Pv) @ np.abs(Vv)
    assert np.all(np.abs(O - two_step) <= 2.0 ** -8 * bnd + 1e-12)   # P rounded to bf16 once


def test_bf16_values_match_the_oracle_decode_on_all_patterns():
    allbits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bf16_values(allbits).astype(np.float64)
    ref = oracle.decode(allbits, "bf16")
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(ref)) and np.array_equal(np.isinf(ours), np.isinf(ref))


def test_attention_tolerance_terms_and_what_it_admits():
    """The fused-attention bound at alpha = 0 reduces to its fixed terms; it
    admits the result of rounding every normalised probability and then O to
    bf16 (the two roundings it is derived from), and it rejects an O that
    drops one key of the softmax (a plausible kernel mistake)."""
    batch, Lq, Lk, D = 2, 24, 96, 16
    Q, Kt, V = _att_inputs(batch, Lq, Lk, D, 810)
    O, bnd = oracle.attention(Q, Kt, V, batch=batch, Lq=Lq, Lk=Lk, D=D, alpha=0.0)
    vmax = np.abs(oracle.decode(V, "bf16")).max(axis=1)
    tol0 = oracle.attention_tolerance(O, bnd, Q, Kt, V, alpha=0.0)
    want = (2.0 ** -8 + 2.0 ** -14) * (bnd + np.abs(O)) + Lk * 2.0 ** -126 * vmax[:, None, :]
    assert np.array_equal(tol0, want)
    alpha = 0.4
    O, bnd = oracle.attention(Q, Kt, V, batch=batch, Lq=Lq, Lk=Lk, D=D, alpha=alpha)
    tol = oracle.attention_tolerance(O, bnd, Q, Kt, V, alpha=alpha)
    q, k, v = (oracle.decode(x, "bf16") for x in (Q, Kt, V))
    s = alpha * np.einsum("bid,bcd->bic", q, k)
    p = np.exp(s - s.max(axis=2, keepdims=True))
    l = p.sum(axis=2, keepdims=True)
    p_bf = oracle.decode(oracle.round_bf16(p), "bf16")
    two_round = oracle.decode(oracle.round_bf16(np.einsum("bic,bcd->bid", p_bf, v) / l), "bf16")
    assert np.all(np.abs(two_round - O) <= tol)
    # the eta term grows with |alpha| and the norms of q and k
    assert np.all(tol >= (2.0 ** -8 + 2.0 ** -14) * (bnd + np.abs(O)))
    drop = np.einsum("bic,bcd->bid", p[:, :, 1:], v[:, 1:]) / p[:, :, 1:].sum(axis=2, keepdims=True)
    assert np.any(np.abs(drop - O) > tol)

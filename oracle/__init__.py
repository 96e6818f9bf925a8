"""TEST INFRASTRUCTURE — fp64 CPU oracle for the batched dense product.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The GPU library never does, and
this package imports nothing from the GPU library: the two share no code.

The arithmetic lives in ``bmm_oracle.c`` (plain C, fp64, k-ascending sums);
this module only compiles it with gcc and marshals numpy arrays through
ctypes.  What it computes is the plain definition

    C_ref[b,i,j] = alpha * sum_k opA[b,i,k] * opB[b,k,j] + beta * C_in[b,i,j]
    Bnd[b,i,j]   = sum_k |opA[b,i,k]| * |opB[b,k,j]|

which the tiled kernels of "Triton Optimization Reference (cuTile -> Triton)"
sections 1-2 (EVEN_K fast path, transpose in the addressing) reorganise but do
not change.  Inputs are raw 16-bit patterns (``numpy.uint16``) as produced by
the seeded input generator; C_in is ``float32`` values or bf16 bit patterns.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, brute force, exact small-integer cases and a float64 library matmul.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bmm_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle_bmm.so")

BF16, F16, F32 = 0, 1, 2
_TYPE_CODES = {"bf16": BF16, "f16": F16, "f32": F32}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags only) and return the path."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def build_command() -> list:
    """The gcc command line ``build()`` runs (for parallel builds)."""
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", _LIB, _SRC, "-lm", "-lpthread"]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    vp = ctypes.c_void_p
    lib.oracle_bmm_f64.argtypes = [i64] * 10 + [i32] * 4 + [f64, f64] + [vp] * 5 + [i32]
    lib.oracle_bmm_f64.restype = i32
    lib.oracle_bmm_sampled.argtypes = [i64] * 10 + [i32] * 4 + [f64, f64] + [vp] * 3 + [i64] + [vp] * 5
    lib.oracle_bmm_sampled.restype = i32
    lib.oracle_attention_probs_bf16.argtypes = [i64, i64, i64, f64, vp, vp, vp, i32]
    lib.oracle_attention_probs_bf16.restype = i32
    lib.oracle_attention_f64.argtypes = [i64, i64, i64, i64, f64, vp, vp, vp, vp, vp, i32]
    lib.oracle_attention_f64.restype = i32
    lib.oracle_round_bf16.argtypes = [f64]
    lib.oracle_round_bf16.restype = ctypes.c_uint16
    lib.oracle_decode16.argtypes = [ctypes.c_uint16, i32]
    lib.oracle_decode16.restype = f64
    _lib = lib
    return lib


def host_threads() -> int:
    """Threads the oracle uses by default: every core in this process's mask."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a, name):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name} must hold raw 16-bit patterns (numpy.uint16), got {a.dtype}")
    return a


def _cin(c, typeC):
    if c is None:
        return None
    c = np.ascontiguousarray(c)
    want = np.float32 if typeC == F32 else np.uint16
    if c.dtype != want:
        raise TypeError(f"C_in must be {np.dtype(want).name} for this output type, got {c.dtype}")
    return c


def bmm(A, B, C_in, *, batch, M, N, K, lda, ldb, ldc, sA, sB, sC,
        transA=False, transB=False, type_ab="bf16", type_c="f32",
        alpha=1.0, beta=0.0, threads=None, want_bound=True):
    """Full oracle.  Returns ``(C_ref, Bnd)`` as dense float64 [batch, M, N]
    arrays (``Bnd`` is None when ``want_bound`` is false)."""
    lib = _load()
    ta, tc = _TYPE_CODES[type_ab], _TYPE_CODES[type_c]
    A, B = _bits(A, "A"), _bits(B, "B")
    C_in = _cin(C_in, tc) if beta != 0.0 else None
    cref = np.empty((batch, M, N), dtype=np.float64)
    bnd = np.empty((batch, M, N), dtype=np.float64) if want_bound else None
    rc = lib.oracle_bmm_f64(batch, M, N, K, lda, ldb, ldc, sA, sB, sC,
                            int(bool(transA)), int(bool(transB)), ta, tc,
                            float(alpha), float(beta), _ptr(A), _ptr(B), _ptr(C_in),
                            _ptr(cref), _ptr(bnd), int(threads or host_threads()))
    if rc != 0:
        raise ValueError(f"oracle_bmm_f64 rejected the problem (code {rc})")
    return cref, bnd


def bmm_sampled(A, B, C_in, samples, *, batch, M, N, K, lda, ldb, ldc, sA, sB, sC,
                transA=False, transB=False, type_ab="bf16", type_c="f32",
                alpha=1.0, beta=0.0):
    """Oracle for chosen output elements.  ``samples`` is an int64 array of
    shape [n, 3] holding (b, i, j).  Returns ``(c_ref, bnd)`` float64 [n]."""
    lib = _load()
    ta, tc = _TYPE_CODES[type_ab], _TYPE_CODES[type_c]
    A, B = _bits(A, "A"), _bits(B, "B")
    C_in = _cin(C_in, tc) if beta != 0.0 else None
    s = np.ascontiguousarray(np.asarray(samples, dtype=np.int64).reshape(-1, 3))
    ib, ii, ij = (np.ascontiguousarray(s[:, c]) for c in range(3))
    n = s.shape[0]
    cref = np.empty(n, dtype=np.float64)
    bnd = np.empty(n, dtype=np.float64)
    rc = lib.oracle_bmm_sampled(batch, M, N, K, lda, ldb, ldc, sA, sB, sC,
                                int(bool(transA)), int(bool(transB)), ta, tc,
                                float(alpha), float(beta), _ptr(A), _ptr(B), _ptr(C_in),
                                n, _ptr(ib), _ptr(ii), _ptr(ij), _ptr(cref), _ptr(bnd))
    if rc != 0:
        raise ValueError(f"oracle_bmm_sampled rejected the problem (code {rc})")
    return cref, bnd


def attention_probs_bf16(Q, Kmat, *, batch, L, D, alpha, threads=None):
    """P = bf16(row-softmax(alpha * Q K^T)) from dense [batch, L, D] bf16 bit
    arrays, computed in fp64 and rounded once.  Returns uint16 [batch, L, L]."""
    lib = _load()
    Q, Kmat = _bits(Q, "Q"), _bits(Kmat, "K")
    P = np.empty((batch, L, L), dtype=np.uint16)
    rc = lib.oracle_attention_probs_bf16(batch, L, D, float(alpha), _ptr(Q), _ptr(Kmat),
                                         _ptr(P), int(threads or host_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention_probs_bf16 failed (code {rc})")
    return P


def attention(Q, Kmat, V, *, batch, Lq, Lk, D, alpha, threads=None, want_bound=True):
    """O = softmax(alpha * Q K^T) V in fp64 from dense bf16 bit arrays
    (Q: [batch, Lq, D]; K, V: [batch, Lk, D]).  Returns (O, Bnd) float64
    [batch, Lq, D] with Bnd = sum_c p_ic |V_cd| (None if not wanted)."""
    lib = _load()
    Q, Kmat, V = _bits(Q, "Q"), _bits(Kmat, "K"), _bits(V, "V")
    O = np.empty((batch, Lq, D), dtype=np.float64)
    bnd = np.empty((batch, Lq, D), dtype=np.float64) if want_bound else None
    rc = lib.oracle_attention_f64(batch, Lq, Lk, D, float(alpha), _ptr(Q), _ptr(Kmat), _ptr(V),
                                  _ptr(O), _ptr(bnd), int(threads or host_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention_f64 failed (code {rc})")
    return O, bnd


def bf16_values(bits):
    """bf16 bit patterns to float32 values: a bf16 pattern is the upper half
    of the binary32 pattern of the same value, so widening is exact."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rows_max(bits, D, fn, chunk_rows=1 << 20):
    """max over rows of fn(row values) for a [rows, D] bf16 bit array, in
    chunks of rows (the key count may run to millions)."""
    rows = bits.reshape(-1, D)
    out = None
    for r0 in range(0, rows.shape[0], chunk_rows):
        v = fn(bf16_values(rows[r0:r0 + chunk_rows]).astype(np.float64))
        m = v.max(axis=0)
        out = m if out is None else np.maximum(out, m)
    return out


ATTN_ROUND = 2.0 ** -8   # one RNE rounding to bf16 (8-bit significand), relative
ATTN_FP32 = 2.0 ** -14   # every fp32 step of the softmax and its sums, relative (see below)
STATED_FP32 = 1e-5       # the stated fp32 accumulation allowance, relative to sum |a||b|


def attention_tolerance(o_ref, bnd, Q, K, V, *, alpha):
    """Acceptance bound per element of the fused attention form
    O = softmax(alpha Q K^T) V, derived from the arithmetic it is held to
    (scores accumulated in fp32, probabilities p rounded to bf16 before the
    product with V, that product and the normaliser l = sum_c p_c summed in
    fp32 from the unrounded p, O rounded to bf16 once):

        tol = (2^-8 + eps + eta_i) * (B_id + |O_id|) + Lk * 2^-126 * max_c |V_cd|

    with B_id = sum_c p_ic |V_cd| (the oracle's bound; p normalised).

    * 2^-8 * B: each p_c moves by at most 2^-8 relative when rounded to bf16;
      only the numerator sum_c p_c V_c sees that rounding (l sums the
      unrounded p), so O moves by at most 2^-8 * B.
    * 2^-8 * |O|: the one rounding of O to bf16.
    * eta_i = |alpha| * 1e-5 * ||q_i||_2 * max_c ||k_c||_2: the stated fp32
      product allowance (1e-5 * sum_k |q_k||k_ck|, bounded by Cauchy-Schwarz)
      applied to each score; a score error ds scales p_c by exp(alpha ds),
      and weights w_c perturbed by relative errors eta_c move
      sum_c w_c V_c / sum_c w_c by at most max eta * (B + |O|).
    * eps = 2^-14 covers the remaining fp32 steps, all far smaller: the same
      1e-5 allowance for the P.V accumulation (relative to B) and for the sum
      l (relative to |O|), the rounding of the exponent argument and of the
      exponentials, the rescale products and the reciprocal of l (each a few
      units of 2^-24 for the weights that matter), and the second-order term
      2^-8 * 2^-8 * B of rounding an O that already carries the p error.
    * Lk * 2^-126 * max|V|: probabilities below 2^-126 may be flushed to zero
      (relative to a largest p of at least 1, so l >= 1).

    Q is [batch, Lq, D] (the query rows of o_ref), K and V [batch, Lk, D]
    (or flat), all bf16 bit patterns."""
    o_ref = np.asarray(o_ref)
    batch, Lq, D = o_ref.shape
    Qb = np.asarray(Q).reshape(batch, Lq, D)
    Kb = np.asarray(K).reshape(batch, -1, D)
    Vb = np.asarray(V).reshape(batch, -1, D)
    Lk = Kb.shape[1]
    qn = np.sqrt(np.square(bf16_values(Qb).astype(np.float64)).sum(axis=2))      # [batch, Lq]
    kn = np.array([_rows_max(Kb[b], D, lambda v: np.sqrt(np.square(v).sum(axis=1)))
                   for b in range(batch)]).reshape(batch)                         # [batch]
    vmax = np.array([_rows_max(Vb[b], D, np.abs) for b in range(batch)]).reshape(batch, D)
    eta = abs(float(alpha)) * STATED_FP32 * qn * kn[:, None]
    rel = ATTN_ROUND + ATTN_FP32 + eta[:, :, None]
    return rel * (np.asarray(bnd) + np.abs(o_ref)) + Lk * 2.0 ** -126 * vmax[:, None, :]


def round_bf16(x):
    """Round float64 values to bf16 (ties to even); returns uint16 bits."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    out = np.fromiter((lib.oracle_round_bf16(float(v)) for v in x.ravel()),
                      dtype=np.uint16, count=x.size)
    return out.reshape(x.shape)


def decode(bits, type_ab):
    """Decode 16-bit patterns to float64 the way the oracle does."""
    lib = _load()
    t = _TYPE_CODES[type_ab]
    b = np.asarray(bits, dtype=np.uint16)
    out = np.fromiter((lib.oracle_decode16(int(v), t) for v in b.ravel()),
                      dtype=np.float64, count=b.size)
    return out.reshape(b.shape)


def tolerance(c_ref, bnd, c_in, *, alpha, beta, out_bf16):
    """Acceptance bound per element: 1e-5*|alpha|*Bnd + 1e-5*|beta*C_in|,
    plus 2^-8*|C_ref| (one bf16 rounding, 8-bit significand) for bf16 output.
    With alpha=1, beta=0 and fp32 output this is the stated 1e-5*sum|a||b|."""
    tol = 1e-5 * abs(alpha) * bnd
    if beta != 0.0 and c_in is not None:
        tol = tol + 1e-5 * abs(beta) * np.abs(c_in)
    if out_bf16:
        tol = tol + 2.0 ** -8 * np.abs(c_ref)
    return tol

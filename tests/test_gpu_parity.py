"""GPU parity: the tcgen05 path through the C ABI against the fp64 oracle,
element by element, on seeded inputs.

Tolerance per element: 1e-5*|alpha|*sum_k|a_ik||b_kj| + 1e-5*|beta*C_in|,
plus 2^-8*|C_ref| when C is bf16 (one rounding of an 8-bit significand).
Small-integer inputs are exact in fp32 and must match bit for bit.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

from bmm_harness import check_full, check_sampled, decode_c, plan_tiles, run_gpu, sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load_library()


# ------------------------------------------------------------ small exact

@pytest.mark.parametrize("transA,transB", list(itertools.product([False, True], repeat=2)))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_small_integers_bitwise(transA, transB, dtype):
    """|x| <= 4 and K <= 4096 keep every partial sum an integer below 2^24:
    the fp32 result must equal the oracle exactly."""
    p = wl.Problem(batch=2, M=200, N=136, K=448, transA=transA, transB=transB, type_ab=dtype,
                   type_c="f32", seed=61)
    na, nb, _ = p.storage_elems()
    x = wl.Inputs(wl.small_ints16(na, 611, -4, 4, dtype), wl.small_ints16(nb, 612, -4, 4, dtype), None)
    c, info = run_gpu(p, x)
    check_full(p, x, c, exact=True)


def test_small_workload_full():
    p = wl.SMALL
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x)
    assert info.tile_n == 64 and info.swap_ab == 0 and info.even_k == 1
    check_full(p, x, c)


# ------------------------------------------------- sweep of shapes and flags

SWEEP_DIMS = [1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 257]
ALPHA_BETA = [(1.0, 0.0), (0.5, 1.0), (0.0, 1.0), (-2.0, 0.25)]


def _sweep_cases(n=48, seed=7):
    rng = np.random.default_rng(seed)
    cases = []
    for t in range(n):
        M, N, K = (int(rng.choice(SWEEP_DIMS)) for _ in range(3))
        batch = int(rng.choice([1, 3]))
        tA, tB = bool(rng.integers(2)), bool(rng.integers(2))
        dtype = ["bf16", "f16"][int(rng.integers(2))]
        tc = ["f32", "bf16"][int(rng.integers(2))]
        ab = ALPHA_BETA[int(rng.integers(4))]
        cases.append((batch, M, N, K, tA, tB, dtype, tc, ab))
    return cases


@pytest.mark.parametrize("case", _sweep_cases(), ids=lambda c: "b{}_{}x{}x{}_t{}{}_{}_{}_{}".format(
    c[0], c[1], c[2], c[3], int(c[4]), int(c[5]), c[6], c[7], c[8]))
def test_sweep(case):
    batch, M, N, K, tA, tB, dtype, tc, (alpha, beta) = case
    p = wl.Problem(batch=batch, M=M, N=N, K=K, transA=tA, transB=tB, type_ab=dtype, type_c=tc,
                   alpha=alpha, beta=beta, seed=100 + M + N + K)
    x = wl.make_inputs(p)
    c, _ = run_gpu(p, x)
    check_full(p, x, c)


@pytest.mark.parametrize("transA,transB", list(itertools.product([False, True], repeat=2)))
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (129, 257, 48), (17, 300, 1000), (640, 24, 130)])
def test_multi_tile_ragged(M, N, K, transA, transB):
    """Several tiles in M and N and a ragged K tail (K % 64 != 0)."""
    p = wl.Problem(batch=3, M=M, N=N, K=K, transA=transA, transB=transB, type_ab="bf16",
                   type_c="f32", alpha=1.0, beta=0.0, dist_ab="normal", seed=71)
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x)
    check_full(p, x, c)


def test_padded_and_unaligned_leading_dimensions():
    """lda/ldb not multiples of 8 elements go through the staging copy; ldc
    padding must stay untouched."""
    p = wl.Problem(batch=2, M=150, N=99, K=77, transA=True, transB=False, type_ab="f16",
                   type_c="f32", alpha=0.5, beta=1.0, lda=153, ldb=101, ldc=103, seed=81)
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x)
    assert info.pack_a == 1 and info.pack_b == 1
    check_full(p, x, c)


@pytest.mark.parametrize("N,tc", [(260, "bf16"), (264, "bf16"), (258, "f32"), (260, "f32")])
def test_box_store_edges(N, tc):
    """Row-major C with padded ldc: rows whose byte length is a multiple of
    16 go out through TMA box stores, the others through direct stores; the
    padding between rows and the guard after C must stay untouched."""
    p = wl.Problem(batch=2, M=130, N=N, K=72, transB=True, type_ab="bf16", type_c=tc,
                   ldc=N + 12, seed=83 + N)
    x = wl.make_inputs(p)
    c, _ = run_gpu(p, x, c_fill="garbage")
    check_full(p, x, c)
    s = p.strides()
    pad = np.concatenate([np.arange(b * s["sC"] + i * s["ldc"] + p.N, b * s["sC"] + (i + 1) * s["ldc"])
                          for b in range(p.batch) for i in range(p.M - 1)])
    fill = np.float32(7.0) if tc == "f32" else np.uint16(0x40E0)
    assert np.all(c[pad] == fill)


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("N,tc", [(4064, "bf16"), (4096, "f32"), (480, "f32")])
def test_skipped_boxes_never_recycle_a_buffer_in_flight(N, tc, pair, monkeypatch):
    """Tiles whose last columns lie past N: the epilogue skips the boxes wholly
    outside C.  A skipped box must not take a turn of the two box buffers, or
    the next box is written into the buffer the last real store is still
    reading (that store then sends the skipped box's zeros).  Widths are
    chosen so the last tile column has one or two real boxes followed by
    skipped ones; K is short so the epilogue runs back to back, and the run is
    repeated."""
    monkeypatch.setenv("DMT_BMM_PAIR", pair)
    p = wl.Problem(batch=2, M=512, N=N, K=64, transB=True, type_ab="bf16", type_c=tc,
                   seed=84 + N)
    x = wl.make_inputs(p)
    for _ in range(3):
        c, info = run_gpu(p, x)
        assert info.tile_n in (192, 224, 256) and info.cta_pair == int(pair)
        check_full(p, x, c)


def test_padded_aligned_leading_dimensions():
    p = wl.Problem(batch=2, M=130, N=260, K=100, transB=True, type_ab="bf16", type_c="bf16",
                   lda=136, ldb=112, ldc=272, sA=136 * 130 + 8, seed=82)
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x)
    assert info.pack_a == 0 and info.pack_b == 0
    check_full(p, x, c)


@pytest.mark.parametrize("which", ["A", "B"])
def test_batch_broadcast(which):
    p = wl.Problem(batch=4, M=96, N=80, K=72, type_ab="bf16", type_c="f32",
                   sA=0 if which == "A" else None, sB=0 if which == "B" else None, seed=83)
    x = wl.make_inputs(p)
    c, _ = run_gpu(p, x)
    check_full(p, x, c)


def test_beta_zero_does_not_read_nan_c():
    p = wl.Problem(batch=2, M=100, N=100, K=100, seed=84)
    x = wl.make_inputs(p)
    c, _ = run_gpu(p, x, c_fill="nan")
    assert np.all(np.isfinite(decode_c(c, p)))
    check_full(p, x, c)


@pytest.mark.parametrize("tc", ["f32", "bf16"])
def test_alpha_zero_and_k_zero(tc):
    p = wl.Problem(batch=2, M=33, N=65, K=40, type_c=tc, alpha=0.0, beta=-0.5, seed=85)
    x = wl.make_inputs(p)
    c, _ = run_gpu(p, x)
    check_full(p, x, c)
    # K = 0: A is M x 0 and needs lda >= 1 (BLAS convention); C = beta * C
    p0 = wl.Problem(batch=2, M=33, N=65, K=0, type_c=tc, alpha=1.0, beta=2.0, lda=8, seed=86)
    x0 = wl.make_inputs(p0)
    c0, _ = run_gpu(p0, x0)
    check_full(p0, x0, c0)
    pz = wl.Problem(batch=2, M=33, N=65, K=0, type_c=tc, alpha=1.0, beta=0.0, lda=8, seed=87)
    cz, _ = run_gpu(pz, wl.make_inputs(pz), c_fill="nan")
    assert np.all(decode_c(cz, pz) == 0.0)


def test_empty_problem_is_a_no_op():
    p = wl.Problem(batch=3, M=0, N=16, K=16, seed=88)
    c, _ = run_gpu(p, wl.make_inputs(p))
    assert c.size == 0


def test_misaligned_base_is_rejected():
    p = wl.Problem(batch=1, M=64, N=64, K=64, seed=89)
    x = wl.make_inputs(p)
    c, _ = run_gpu(p, x, a_offset=1, expect_status=api.BMM_ERR_MISALIGNED)


def test_repeated_runs_and_streams():
    """Same plan, several runs on a side stream: identical bits each time."""
    p = wl.Problem(batch=2, M=256, N=384, K=320, transB=True, type_c="f32", seed=90)
    x = wl.make_inputs(p)
    s = torch.cuda.Stream()
    first, _ = run_gpu(p, x, stream=s)
    for _ in range(2):
        again, _ = run_gpu(p, x, stream=s)
        assert np.array_equal(first, again)
    check_full(p, x, first)


# ------------------------------------------------- 1-CTA and CTA-pair tiles

@pytest.mark.parametrize("pair", ["1", "0"])
@pytest.mark.parametrize("transA,transB", list(itertools.product([False, True], repeat=2)))
def test_large_tile_class_both_kernels(pair, transA, transB, monkeypatch):
    """The 256-wide tile class runs on CTA pairs (2-SM MMA) by default and on
    single CTAs with DMT_BMM_PAIR=0; both must meet the tolerance, with
    ragged M, N and K tails and several tiles per CTA."""
    monkeypatch.setenv("DMT_BMM_PAIR", pair)
    p = wl.Problem(batch=2, M=1100, N=600, K=333, transA=transA, transB=transB, type_ab="bf16",
                   type_c="f32", alpha=1.5, beta=-0.5, dist_ab="normal", seed=91)
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x)
    assert info.cta_pair == int(pair) and info.tile_n >= 192
    check_full(p, x, c)


@pytest.mark.parametrize("type_c", ["f32", "bf16"])
def test_tile_configuration_does_not_change_exact_results(monkeypatch, type_c):
    """Changing the tile configuration must never change the output
    ("Optimize Triton Block Parameters", Correctness requirements).  With
    small integers every fp32 sum is exact, so every tile width on both
    kernels must match the oracle and each other bit for bit (for bf16 output
    the single rounding of those exact sums must agree too).  M, N, K are
    ragged against every tile."""
    p = wl.Problem(batch=2, M=520, N=1000, K=1000, transB=True, type_ab="bf16", type_c=type_c,
                   seed=92)
    na, nb, _ = p.storage_elems()
    x = wl.Inputs(wl.small_ints16(na, 921, -2, 2, "bf16"), wl.small_ints16(nb, 922, -2, 2, "bf16"), None)
    out = {}
    for pair in ("1", "0"):
        for tn in ("192", "224", "256"):
            monkeypatch.setenv("DMT_BMM_PAIR", pair)
            monkeypatch.setenv("DMT_BMM_TILE_N", tn)
            out[pair, tn], info = run_gpu(p, x)
            assert info.cta_pair == int(pair) and info.tile_n == int(tn)
            if type_c == "f32":
                check_full(p, x, out[pair, tn], exact=True)
    first = out["1", "256"]
    for k, v in out.items():
        assert np.array_equal(v, first), k


# ------------------------------------------------------- full-size workloads
#
# Every element of C at the full sizes is compared with the fp64 oracle (the
# oracle runs on the host cores, in slices of whole batch items), and no
# element may be NaN or Inf.  The tile corners and seams of the plan the
# library chose are checked once more on their own, so a failure there names
# the seam.


def _full_and_seams(p, x, c, info, seed, n=2000):
    worst = check_full(p, x, c)
    tm, tn = plan_tiles(info)
    check_sampled(p, x, c, sample_indices(p, n, seed, tile_m=tm, tile_n=tn))
    print(f"{p.name}: max err/tol over all {p.batch * p.M * p.N} elements = {worst:.4f}")
    return worst


def test_workload_gemm_4096():
    p = wl.GEMM_4096
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x, guard=8192)
    assert info.tile_n == 224 and info.cta_pair == 1 and info.even_k == 1 and info.swap_ab == 0
    _full_and_seams(p, x, c, info, 1)


def test_gemm_with_a_leftover_round():
    """4000 x 4500 x 4096: 288 pair tiles, no multiple of the 76 pairs (the
    bench's uneven GEMM), every element against the oracle."""
    p = wl.UNEVEN_GEMM
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x, guard=8192)
    assert info.cta_pair == 1 and info.tiles % 76 != 0
    _full_and_seams(p, x, c, info, 6)


def test_workload_ragged():
    p = wl.RAGGED
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x)
    assert info.even_k == 0 and info.pack_b == 1 and info.pack_a == 0
    _full_and_seams(p, x, c, info, 2)


def test_workload_skinny():
    p = wl.SKINNY
    x = wl.make_inputs(p)
    c, info = run_gpu(p, x)
    assert info.swap_ab == 1 and info.tile_n == 16
    _full_and_seams(p, x, c, info, 3)


def test_workload_attention_pair():
    """S = alpha Q K^T (fp32 out), then O = P V with P = bf16(softmax(S)) made
    by the oracle from its own S (never from the GPU's).  Both products are
    compared with the oracle on every element."""
    qk, pv = wl.ATTN_QK, wl.ATTN_PV
    Q, Kt, V = wl.attention_qkv()
    xs = wl.Inputs(Q.ravel(), Kt.ravel(), None)
    s_host, info = run_gpu(qk, xs)
    assert info.tile_n == 256
    _full_and_seams(qk, xs, s_host, info, 4)
    del s_host
    P = oracle.attention_probs_bf16(Q, Kt, batch=128, L=2048, D=128, alpha=qk.alpha)
    xo = wl.Inputs(P.ravel(), V.ravel(), None)
    o_host, info = run_gpu(pv, xo)
    assert info.tile_n == 128
    _full_and_seams(pv, xo, o_host, info, 5)

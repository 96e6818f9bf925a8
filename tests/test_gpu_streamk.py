"""Stream-K tail of the CTA-pair kernel against the fp64 oracle.

Plans with CTA pairs and K >= 2048 may split the tiles left over after the
last whole round along K over all pairs ("Triton Optimization Reference",
section 7: the last wave of a persistent grid): pieces without a tile's first
k-block leave fp32 partials in the plan's workspace, the piece with it adds
them and writes C.  Small-integer inputs keep every fp32 sum exact, so any
lost, doubled or misplaced partial shows as a bitwise difference from the
oracle; random inputs are held to the usual tolerance.
"""
import numpy as np
import pytest
import torch

from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

from bmm_harness import check_full, desc_for, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load_library()


@pytest.fixture(autouse=True)
def _split_whenever_allowed(monkeypatch):
    # the planner's estimate may prefer whole rounds of a narrower tile; these
    # tests want the split on every shape that allows it
    monkeypatch.setenv("DMT_BMM_STREAMK", "1")


# (batch, M, N, K, transA, transB): whole rounds plus a tail; only a tail (8
# tiles on 76 pairs); a ragged K tail inside split pieces; ragged M and N
# edges; MN-major operands; several batch items.  A leftover of at most half
# the pairs' tiles is split two ways (sk_piece2), a larger one in equal
# ranges (sk_piece): 72 tiles on 76 pairs and 74 leftover tiles after a round.
SHAPES = [
    (1, 4096, 4096, 4096, False, True),
    (1, 512, 1024, 4096, False, True),
    (1, 1000, 1000, 2100, True, False),
    (2, 1100, 700, 3000, False, False),
    (3, 800, 1300, 2048, True, True),
    (1, 2560, 3840, 2048, False, True),
]


def _ints(p, seed):
    na, nb, _ = p.storage_elems()
    return wl.Inputs(wl.small_ints16(na, seed, -2, 2, p.type_ab), wl.small_ints16(nb, seed + 1, -2, 2, p.type_ab),
                     None)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}_{}x{}x{}_t{}{}".format(*s[:4], int(s[4]), int(s[5])))
def test_split_tail_is_exact_on_small_integers(shape):
    batch, M, N, K, tA, tB = shape
    p = wl.Problem(batch=batch, M=M, N=N, K=K, transA=tA, transB=tB, type_ab="bf16", type_c="f32", seed=95)
    info = api.bmm_plan_query(desc_for(p))
    assert info.stream_k == 1 and info.tile_n == 256 and info.cta_pair == 1
    x = _ints(p, 951)
    c, _ = run_gpu(p, x)
    check_full(p, x, c, exact=True)


@pytest.mark.parametrize("type_c,beta", [("bf16", 0.0), ("f32", 0.75)])
def test_split_tail_meets_the_tolerance(type_c, beta):
    p = wl.Problem(batch=2, M=1500, N=1800, K=2500, transB=True, type_ab="f16", type_c=type_c,
                   alpha=-1.25, beta=beta, dist_ab="normal", seed=96)
    assert api.bmm_plan_query(desc_for(p)).stream_k == 1
    x = wl.make_inputs(p)
    c, _ = run_gpu(p, x)
    check_full(p, x, c)


def test_repeated_runs_are_bitwise_identical():
    """The flags a run raises are cleared by the run that reads them: the next
    runs of the same plan must see fresh partials (same bits every time)."""
    p = wl.Problem(batch=1, M=2048, N=3584, K=2048, transB=True, type_ab="bf16", type_c="f32", seed=97)
    x = _ints(p, 971)
    dev = torch.device("cuda:0")
    A = torch.from_numpy(x.A.view(np.int16)).to(dev)
    B = torch.from_numpy(x.B.view(np.int16)).to(dev)
    C = torch.empty(p.M * p.N, dtype=torch.float32, device=dev)
    outs = []
    with api.Plan(desc_for(p)) as plan:
        assert plan.info().stream_k == 1
        for _ in range(3):
            C.fill_(float("nan"))
            plan.run(A, B, C, 1.0, 0.0, torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert plan.device_error()[0] == api.BMM_OK
            outs.append(C.cpu().numpy().copy())
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    check_full(p, x, outs[0], exact=True)


def test_switched_off_gives_the_same_exact_result(monkeypatch):
    p = wl.Problem(batch=1, M=1024, N=2048, K=2048, transB=True, type_ab="bf16", type_c="f32", seed=98)
    x = _ints(p, 981)
    on, info_on = run_gpu(p, x)
    assert info_on.stream_k == 1
    monkeypatch.setenv("DMT_BMM_STREAMK", "0")
    off, info_off = run_gpu(p, x)
    assert info_off.stream_k == 0
    assert np.array_equal(on.view(np.uint32), off.view(np.uint32))
    check_full(p, x, on, exact=True)


@pytest.mark.parametrize("publish_kb", ["0", "100"])
def test_two_way_split_points(monkeypatch, publish_kb):
    """The owner's range: half the k-blocks (0: no transfer allowance) or all
    but one (an allowance longer than K)."""
    monkeypatch.setenv("DMT_BMM_SK_PUBLISH_KB", publish_kb)
    p = wl.Problem(batch=1, M=1024, N=1536, K=2100, transB=True, type_ab="bf16", type_c="f32", seed=99)
    x = _ints(p, 991)
    c, info = run_gpu(p, x)
    assert info.stream_k == 1 and info.sk_tiles == 24
    check_full(p, x, c, exact=True)


@pytest.mark.parametrize("M,N,K,two_way", [(8192, 8192, 4096, True), (6144, 6144, 4096, False)])
def test_planner_split_at_full_size(monkeypatch, M, N, K, two_way):
    """The planner's own choice (no forcing) on shapes where it splits: 8192^2
    x 4096 (36 leftover tiles, two ways) and 6144^2 x 4096 (44, equal ranges);
    random bf16 operands, every element against the oracle."""
    monkeypatch.delenv("DMT_BMM_STREAMK", raising=False)
    p = wl.Problem(batch=1, M=M, N=N, K=K, transB=True, type_ab="bf16", type_c="bf16", dist_ab="normal", seed=100)
    info = api.bmm_plan_query(desc_for(p))
    pairs = 76
    rem = info.tiles % pairs
    assert info.stream_k == 1 and info.sk_tiles == rem and (2 * rem <= pairs) == two_way
    x = wl.make_inputs(p)
    c, _ = run_gpu(p, x)
    worst = check_full(p, x, c)
    print(f"{M}x{N}x{K}: max err/tol over all {M * N} elements = {worst:.4f}")

"""Ring depth per launch of the CTA-pair kernel.

A plan with 256 x 224 (or 256 x 192) pair tiles and bf16 C keeps two shared-
memory layouts: launches whose C goes out through TMA box stores (beta = 0,
16-byte-aligned C) use half the epilogue region (2 KB boxes) and one more
ring stage; every other launch of the same plan (beta != 0, so direct stores
that read C first) uses the general region and the shorter ring.  Both must
give the oracle's result, one after the other on the same plan.
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


def _ints(p, seed):
    na, nb, nc = p.storage_elems()
    c_in = None
    if p.beta != 0.0:
        c_in = wl.small_ints16(nc, seed + 2, -2, 2, "bf16")
    return wl.Inputs(wl.small_ints16(na, seed, -2, 2, p.type_ab), wl.small_ints16(nb, seed + 1, -2, 2, p.type_ab),
                     c_in)


@pytest.mark.parametrize("N,width", [(4096, 224), (3648, 192)])
def test_both_layouts_of_one_plan_match_the_oracle(N, width):
    # K = 256 keeps every fp32 sum of small integers exact, and within bf16's
    # exact range after the alpha and beta terms (|sum| <= 4 * 256)
    p = wl.Problem(batch=1, M=4096, N=N, K=256, transB=True, type_ab="bf16", type_c="bf16", seed=61)
    info = api.bmm_plan_query(desc_for(p))
    assert info.cta_pair == 1 and info.tile_n == width
    assert info.stages_bf16_box == info.stages + 1
    assert info.smem_bytes == 232448
    x = _ints(p, 611)
    c, _ = run_gpu(p, x)  # beta = 0: box stores, the deeper ring
    check_full(p, x, c, exact=True)
    q = wl.Problem(batch=1, M=4096, N=N, K=256, transB=True, type_ab="bf16", type_c="bf16", beta=1.0,
                   alpha=1.0, seed=61)
    y = _ints(q, 611)
    c2, _ = run_gpu(q, y)  # beta != 0: direct stores, the general region
    check_full(q, y, c2, exact=True)


def test_fp32_output_keeps_one_layout():
    p = wl.Problem(batch=1, M=4096, N=4096, K=256, transB=True, type_ab="bf16", type_c="f32", seed=62)
    info = api.bmm_plan_query(desc_for(p))
    assert info.stages_bf16_box == info.stages

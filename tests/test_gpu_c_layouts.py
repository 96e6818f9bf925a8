"""C with beta != 0 in the layouts the direct-store epilogue serves.

Row strides whose byte length leaves every 4th, 2nd or no row on a 16-byte
boundary, C's base 4, 8 or 12 bytes past one, fp32 and bf16 C, batch strides
on and off 16-byte multiples, and 96 pair tiles on 76 pairs.  Small-integer
inputs keep every value exact, so a row or column read or written one off
shows as a bitwise difference from the oracle; the guard cells around C must
keep their sentinels.
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
    if p.type_c == "f32":
        c_in = np.random.Generator(np.random.PCG64(seed + 2)).integers(-3, 4, size=nc).astype(np.float32)
    else:
        c_in = wl.small_ints16(nc, seed + 2, -3, 3, "bf16")
    return wl.Inputs(wl.small_ints16(na, seed, -2, 2, p.type_ab), wl.small_ints16(nb, seed + 1, -2, 2, p.type_ab),
                     c_in)


def _run(p, x, c_offset=0):
    c, info = run_gpu(p, x, c_offset=c_offset)
    assert info.cta_pair == 1 and info.tile_n == 256
    check_full(p, x, c, exact=True)


# (B stored K x N, N contiguous: pair plans take 256-wide tiles for it.)
@pytest.mark.parametrize("ldc", [999, 1001, 1002, 1000])
@pytest.mark.parametrize("c_offset", [0, 1, 3])
def test_fp32_row_strides_and_base_offsets(ldc, c_offset):
    p = wl.Problem(batch=1, M=700, N=999, K=256, type_ab="bf16", type_c="f32", alpha=0.5, beta=-0.75,
                   ldc=ldc, seed=71)
    _run(p, _ints(p, 711 + ldc), c_offset)


@pytest.mark.parametrize("transA", [True, False])
def test_fp32_more_tiles_than_pairs(transA):
    p = wl.Problem(batch=8, M=700, N=999, K=200, transA=transA, type_ab="f16", type_c="f32",
                   alpha=1.0, beta=1.0, seed=72)
    _run(p, _ints(p, 721))


def test_batch_stride_off_sixteen_bytes():
    p = wl.Problem(batch=3, M=300, N=999, K=128, type_ab="bf16", type_c="f32", alpha=0.5, beta=1.0,
                   sC=300 * 999 + 1, seed=73)
    _run(p, _ints(p, 731))


@pytest.mark.parametrize("ldc", [1002, 1004, 1000, 999])
def test_bf16_row_strides(ldc):
    p = wl.Problem(batch=2, M=500, N=999, K=128, type_ab="bf16", type_c="bf16", alpha=1.0, beta=2.0,
                   ldc=ldc, seed=74)
    _run(p, _ints(p, 741 + ldc), c_offset=1)

"""The kernels' row loader: operands TMA cannot address (row or batch stride
off a 16-byte boundary) read in place by plain loads (DMT_BMM_LDG=1 at plan
time, or bmm_run_noalloc beyond its staging area) instead of the staging copy.

The row loader writes each stage in the layout the TMA box would give, so the
tensor core sees the same operands: its C must equal the staged path's bit for
bit, and the fp64 oracle within its bound.  The cases cover K-major and
MN-major A and B, one or both operands through the loader, CTA pairs and single
CTAs, ragged K tails and M/N edges, batch broadcast and the swapped (C^T)
skinny form.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

from bmm_harness import check_full, run_gpu

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


CASES = {
    # CTA pairs; A K-major with ld 201 (row loader), B K-major aligned (TMA)
    "pair_a_kmajor": dict(p=wl.Problem(batch=2, M=300, N=260, K=200, transB=True, lda=201,
                                       type_ab="bf16", type_c="f32", seed=301), pack=(2, 0)),
    # single CTA; A K-major (ld 79) and B MN-major (ld 93) both through the loader
    "single_both": dict(p=wl.Problem(batch=3, M=100, N=90, K=77, lda=79, ldb=93, type_ab="f16",
                                     type_c="f32", alpha=0.5, beta=0.25, seed=302), pack=(2, 2)),
    # CTA pairs; A MN-major (ld 515), B K-major (ld 131), ragged K
    "pair_mn_k": dict(p=wl.Problem(batch=1, M=513, N=300, K=130, transA=True, transB=True, lda=515,
                                   ldb=131, type_ab="bf16", type_c="bf16", seed=303), pack=(2, 2)),
    # broadcast A with odd ld, batched B with an odd batch stride
    "broadcast": dict(p=wl.Problem(batch=3, M=200, N=128, K=96, lda=97, sA=0, sB=96 * 128 + 3,
                                   type_ab="bf16", type_c="f32", seed=304), pack=(2, 2)),
    # M = 16 <= 64 < N: swapped to C^T; B (the MMA's A) MN-major with ld 301
    "swap": dict(p=wl.Problem(batch=2, M=16, N=300, K=104, ldb=301, type_ab="bf16", type_c="bf16",
                              seed=305), pack=(0, 2)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_row_loader_matches_staged_path_bit_for_bit(name, monkeypatch):
    _need_gpu()
    case = CASES[name]
    p = case["p"]
    x = wl.make_inputs(p)
    staged, info_s = run_gpu(p, x)
    assert info_s.pack_a in (0, 1) and info_s.pack_b in (0, 1)
    monkeypatch.setenv("DMT_BMM_LDG", "1")
    loaded, info_l = run_gpu(p, x)
    # pack_a / pack_b name the caller's A and B
    assert (info_l.pack_a, info_l.pack_b) == case["pack"], (info_l.pack_a, info_l.pack_b)
    assert info_l.workspace_bytes == 0
    assert np.array_equal(staged.view(np.uint8), loaded.view(np.uint8)), "differs from the staged path"
    check_full(p, x, loaded)


def test_row_loader_on_single_cta_256_wide_mn_major_tiles(monkeypatch):
    # DMT_BMM_PAIR=0: a 128 x 256 single-CTA tile whose MN-major B tile is four
    # 64-column atoms, written by the loader
    _need_gpu()
    monkeypatch.setenv("DMT_BMM_PAIR", "0")
    p = wl.Problem(batch=1, M=260, N=600, K=150, ldb=603, type_ab="bf16", type_c="f32", seed=306)
    x = wl.make_inputs(p)
    staged, _ = run_gpu(p, x)
    monkeypatch.setenv("DMT_BMM_LDG", "1")
    loaded, info = run_gpu(p, x)
    assert info.cta_pair == 0 and info.pack_b == 2
    assert np.array_equal(staged.view(np.uint8), loaded.view(np.uint8))
    check_full(p, x, loaded)


def test_row_loader_on_the_ragged_workload(monkeypatch):
    # 16 x 1000 x 999 x 1000, A MN-major (TMA), B with ld 999 through the loader
    _need_gpu()
    p = wl.RAGGED
    x = wl.make_inputs(p)
    staged, _ = run_gpu(p, x, guard=8192)
    monkeypatch.setenv("DMT_BMM_LDG", "1")
    loaded, info = run_gpu(p, x, guard=8192)
    assert info.pack_b == 2 and info.pack_a == 0
    assert np.array_equal(staged.view(np.uint8), loaded.view(np.uint8))
    check_full(p, x, loaded)


def test_noalloc_reads_operands_past_its_staging_area_in_place():
    # B stored K x N with ldb 4097 would need 64 MiB of staging (> 32 MiB): the
    # row loader reads it in place; the result equals bmm_run's (staged) bit for bit
    _need_gpu()
    p = wl.Problem(batch=2, M=64, N=4097, K=4096, ldb=4097, type_ab="bf16", type_c="f32", seed=307)
    x = wl.make_inputs(p)
    staged, info = run_gpu(p, x)
    assert info.pack_b == 1 and info.workspace_bytes > (32 << 20)
    s = p.strides()
    desc = api.make_desc(batch=p.batch, M=p.M, N=p.N, K=p.K, lda=s["lda"], ldb=s["ldb"], ldc=s["ldc"],
                         strideA=s["sA"], strideB=s["sB"], strideC=s["sC"], typeA="bf16", typeC="f32")
    dev = torch.device("cuda:0")
    A = torch.from_numpy(x.A.view(np.int16)).to(dev)
    B = torch.from_numpy(x.B.view(np.int16)).to(dev)
    C = torch.full((p.storage_elems()[2],), float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.bmm_run_noalloc(desc, A, B, C, 1.0, 0.0, torch.cuda.current_stream(), device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = C.cpu().numpy()
    assert np.array_equal(got.view(np.uint8), staged.view(np.uint8))
    check_full(p, x, got)

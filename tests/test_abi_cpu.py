"""The C ABI on the host, with no GPU: the library loads, exports every
symbol ``include/bmm.h`` declares, validates arguments before touching the
device, and plans each workload as intended.  No compute call is made."""
import os
import re

import pytest

from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import build
from dense_matmul_tensor_gb300 import workloads as wl

from bmm_harness import desc_for

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def declared_symbols():
    syms = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            syms |= set(re.findall(r"BMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))
    return syms


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert {"bmm_create", "bmm_run", "bmm_destroy"} <= syms
    for s in syms:
        assert hasattr(lib, s), f"{s} declared in include/ but not exported"
    assert set(api.EXPORTED) <= syms


def test_status_strings_and_version(lib):
    for code, name in [(0, "BMM_OK"), (1, "BMM_ERR_INVALID_ARG"), (3, "BMM_ERR_MISALIGNED"),
                       (5, "BMM_ERR_DEVICE_TIMEOUT")]:
        assert api.bmm_status_string(code) == name
    assert api.bmm_version() >= 1


def _desc(**kw):
    base = dict(batch=2, M=64, N=64, K=64, lda=64, ldb=64, ldc=64, strideA=4096, strideB=4096,
                strideC=4096, transA=0, transB=0, typeA="bf16", typeC="f32")
    base.update(kw)
    return api.make_desc(**base)


@pytest.mark.parametrize("bad", [
    dict(M=-1), dict(K=-5), dict(lda=63), dict(ldb=10), dict(ldc=63),
    dict(transA=2), dict(typeA="f32"), dict(typeC="f16"), dict(strideA=-8),
    dict(strideC=100),                        # C batch items would overlap
    dict(typeB=1),                            # A bf16, B fp16
])
def test_invalid_arguments_rejected_before_any_device_call(lib, bad):
    d = _desc(**bad)
    with pytest.raises(api.BmmError) as e:
        api.bmm_create(d)
    assert e.value.status == api.BMM_ERR_INVALID_ARG
    with pytest.raises(api.BmmError) as e:
        api.bmm_plan_query(d)
    assert e.value.status == api.BMM_ERR_INVALID_ARG


def test_null_arguments(lib):
    import ctypes
    assert lib.bmm_create(None, None) == api.BMM_ERR_INVALID_ARG
    assert lib.bmm_run(None, None, None, None, 1.0, 0.0, None) == api.BMM_ERR_INVALID_ARG
    assert lib.bmm_get_plan_info(None, None) == api.BMM_ERR_INVALID_ARG
    assert lib.bmm_destroy(None) == api.BMM_OK
    assert lib.bmm_get_device_error(None, None) == api.BMM_ERR_INVALID_ARG
    p = ctypes.c_void_p(1)
    assert lib.bmm_create(ctypes.byref(_desc(M=-3)), ctypes.byref(p)) == api.BMM_ERR_INVALID_ARG
    assert p.value is None  # set to NULL on error


def test_dimensions_beyond_int32_unsupported(lib):
    d = _desc(K=2 ** 31, lda=2 ** 31, strideA=2 ** 37)
    with pytest.raises(api.BmmError) as e:
        api.bmm_plan_query(d)
    assert e.value.status == api.BMM_ERR_UNSUPPORTED


def test_create_without_a_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(api.BmmError) as e:
        api.bmm_create(_desc())
    assert e.value.status == api.BMM_ERR_NO_DEVICE


SMEM_LIMIT = 227 * 1024


def _stage_bytes_formula(bm, bn, bk, esz=2):
    # stages x (A tile + B tile): "Optimize Triton Block Parameters", Step 2
    return (bm * bk + bk * bn) * esz


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_planner_on_workloads(lib, name):
    p = wl.WORKLOADS[name]
    info = api.bmm_plan_query(desc_for(p))
    assert info.tile_m == (256 if info.cta_pair else 128) and info.tile_k == 64
    assert info.smem_bytes <= SMEM_LIMIT
    # one CTA's share of the tile: all of a 128-row A tile, half of B on a pair
    raw = _stage_bytes_formula(128, info.tile_n // (2 if info.cta_pair else 1), info.tile_k)
    assert info.stage_bytes == -(-raw // 1024) * 1024
    assert info.stages * info.stage_bytes <= SMEM_LIMIT
    assert info.stages >= 4
    assert info.tmem_cols >= 2 * info.tile_n and info.tmem_cols <= 512
    assert info.even_k == (p.K % 64 == 0)
    assert info.stages <= 8
    if p is wl.SKINNY:
        assert info.swap_ab == 1 and info.tile_n == 16
        assert info.tiles == p.batch * 2          # N=256 over two 128-row MMA tiles
        # 18 KB stages would fit ten deep; eight measured faster on this
        # HBM-bound shape, and the planner builds at most eight
        assert info.stages == 8
    if p is wl.GEMM_4096:
        # CTA pairs with 256 x 224 tiles: 16 x 19 = 304 tiles = exactly 4 rounds
        # on 76 pairs (256-wide tiles would leave a 0.37 wave); 30 KB per CTA
        # per stage, six stages, and seven for the bf16 box-store launches
        # (7 x 30 KB + 16 KB of boxes + 512 B of barriers = 227 KB - 512 B)
        assert info.cta_pair == 1 and info.tile_n == 224 and info.tiles == 16 * 19
        assert info.stages == 6 and info.tmem_cols == 512
        assert info.stages_bf16_box == 7 and info.smem_bytes == 232448
        assert info.workspace_bytes == 0
    if p is wl.ATTN_QK:
        # 8192 pair tiles of 256 x 256 fill 108 rounds almost exactly
        assert info.cta_pair == 1 and info.tile_n == 256 and info.tiles == 128 * 8 * 8
    if p is wl.RAGGED:
        # B stored K x N with ld 999 (not a multiple of 8): staged; A (ld 1000) read in place
        assert info.pack_b == 1 and info.pack_a == 0
        assert info.workspace_bytes >= p.batch * p.K * 1000 * 2
    if p is wl.ATTN_PV:
        assert info.tile_n == 128


def test_planner_boundary_shapes(lib):
    # the pages' boundary shapes and the K = 48 tail against a 64-wide K tile
    for M in (17, 63, 129):
        info = api.bmm_plan_query(_desc(M=M, N=96, K=48, lda=48, ldb=96, ldc=96,
                                        strideA=M * 48, strideB=48 * 96, strideC=M * 96))
        assert info.even_k == 0
        assert info.tiles >= 1


def test_stage_cap_from_the_environment(lib, monkeypatch):
    monkeypatch.setenv("DMT_BMM_STAGES", "4")
    info = api.bmm_plan_query(desc_for(wl.GEMM_4096))
    assert info.stages == 4 and info.smem_bytes <= SMEM_LIMIT
    monkeypatch.setenv("DMT_BMM_STAGES", "1")     # below 2: ignored
    assert api.bmm_plan_query(desc_for(wl.GEMM_4096)).stages == 6
    monkeypatch.setenv("DMT_BMM_STAGES", "12")    # above what the planner builds: ignored
    assert api.bmm_plan_query(desc_for(wl.SKINNY)).stages == 8


def test_pair_mode_can_be_switched_off(lib, monkeypatch):
    monkeypatch.setenv("DMT_BMM_PAIR", "0")
    info = api.bmm_plan_query(desc_for(wl.GEMM_4096))
    # single CTAs: 128 x 224 tiles, 32 x 19 = 608 = 4 rounds on 152 SMs
    assert info.cta_pair == 0 and info.tile_m == 128 and info.tile_n == 224
    assert info.tiles == 32 * 19 and info.stages == 4
    monkeypatch.setenv("DMT_BMM_PAIR", "1")
    assert api.bmm_plan_query(desc_for(wl.GEMM_4096)).cta_pair == 1


def test_wave_balanced_tile_width(lib, monkeypatch):
    # the estimate rounds x tile_n picks the width with the least idle tail
    info = api.bmm_plan_query(desc_for(wl.RAGGED))
    assert info.cta_pair == 1 and info.tile_n == 256      # 256 tiles -> 4 rounds of 256
    monkeypatch.setenv("DMT_BMM_TILE_N", "192")
    assert api.bmm_plan_query(desc_for(wl.GEMM_4096)).tile_n == 192
    monkeypatch.setenv("DMT_BMM_TILE_N", "224")
    # MN-major B on a pair is loaded in 64-column boxes per CTA: 224 is not allowed
    assert api.bmm_plan_query(desc_for(wl.RAGGED)).tile_n == 256


def test_stream_k_tail_choice(lib, monkeypatch):
    # 8192^3 on 76 pairs: 1024 tiles of 256 x 256 = 13 whole rounds + 36 tiles;
    # splitting those along K beats the best whole-round width (256: 14 rounds)
    d = _desc(batch=1, M=8192, N=8192, K=8192, lda=8192, ldb=8192, ldc=8192, strideA=8192 * 8192,
              strideB=8192 * 8192, strideC=8192 * 8192, transB=1, typeC="bf16")
    info = api.bmm_plan_query(d)
    assert info.stream_k == 1 and info.tile_n == 256 and info.cta_pair == 1
    assert info.tiles == 1024 and info.sk_tiles == 1024 - 13 * 76
    assert info.sk_workspace_bytes >= 76 * 2 * 128 * 256 * 4
    # 4096^3: four whole rounds of 256 x 224 tiles (0.93 of a 256-wide round
    # each) cost less than three 256-wide rounds plus the two-way split's
    # owner range (40 of 64 k-blocks) and fixup, so no split
    g = api.bmm_plan_query(desc_for(wl.GEMM_4096))
    assert g.stream_k == 0 and g.sk_tiles == 0 and g.sk_workspace_bytes == 0 and g.tile_n == 224
    # 8192^2 x 4096: 36 leftover tiles after 13 rounds, split two ways
    h = api.bmm_plan_query(_desc(batch=1, M=8192, N=8192, K=4096, lda=4096, ldb=4096, ldc=8192,
                                 strideA=8192 * 4096, strideB=8192 * 4096, strideC=8192 * 8192, transB=1,
                                 typeC="bf16"))
    assert h.stream_k == 1 and h.sk_tiles == 36
    # 4000 x 4500 x 4096: 288 tiles, 60 leftover after 3 rounds (more than half
    # the pairs: equal ranges), whose estimate loses to a fourth 256-wide round
    u = api.bmm_plan_query(desc_for(wl.UNEVEN_GEMM))
    assert u.stream_k == 0 and u.tile_n == 256 and u.tiles == 288
    # forced on where allowed, off everywhere
    monkeypatch.setenv("DMT_BMM_STREAMK", "1")
    f = api.bmm_plan_query(desc_for(wl.GEMM_4096))
    assert f.stream_k == 1 and f.tile_n == 256 and f.sk_tiles == 256 - 3 * 76
    # short K (fewer than 32 k-blocks) and single-CTA tiles never split
    assert api.bmm_plan_query(desc_for(wl.RAGGED)).stream_k == 0
    assert api.bmm_plan_query(desc_for(wl.ATTN_QK)).stream_k == 0
    assert api.bmm_plan_query(desc_for(wl.SKINNY)).stream_k == 0
    monkeypatch.setenv("DMT_BMM_STREAMK", "0")
    assert api.bmm_plan_query(d).stream_k == 0


def test_grouped_create_validates_before_any_device_call(lib):
    ok = dict(M=64, N=64, K=64, lda=64, ldb=64, ldc=64)
    for bad, code in [(dict(M=-1), api.BMM_ERR_INVALID_ARG), (dict(lda=10), api.BMM_ERR_INVALID_ARG),
                      (dict(K=0), api.BMM_ERR_UNSUPPORTED), (dict(ldb=66), api.BMM_ERR_UNSUPPORTED)]:
        arr, n = api.make_problems([dict(ok, **bad)])
        with pytest.raises(api.BmmError) as e:
            api.bmm_grouped_create(arr, n, 0, 0, "bf16", "f32")
        assert e.value.status == code, bad
    arr, n = api.make_problems([ok])
    with pytest.raises(api.BmmError) as e:
        api.bmm_grouped_create(arr, n, 2, 0, "bf16", "f32")
    assert e.value.status == api.BMM_ERR_INVALID_ARG
    assert lib.bmm_grouped_destroy(None) == api.BMM_OK


def _attn(**kw):
    base = dict(batch=2, Lq=100, Lk=70, alpha=0.125)
    base.update(kw)
    return api.make_attn_desc(**base)


@pytest.mark.parametrize("bad,code", [
    (dict(Lq=-1), api.BMM_ERR_INVALID_ARG),
    (dict(ldk=64), api.BMM_ERR_INVALID_ARG),            # row stride below D
    (dict(alpha=float("nan")), api.BMM_ERR_INVALID_ARG),
    (dict(strideO=99 * 128), api.BMM_ERR_INVALID_ARG),   # O batch items would overlap
    (dict(D=64, ldq=64, ldk=64, ldv=64, ldo=64), api.BMM_ERR_UNSUPPORTED),
    (dict(ldv=130), api.BMM_ERR_UNSUPPORTED),           # not a multiple of 16 bytes
    (dict(Lk=0), api.BMM_ERR_UNSUPPORTED),              # softmax over no keys
    (dict(Lq=2 ** 30 + 1), api.BMM_ERR_UNSUPPORTED),
])
def test_attention_create_validates_before_any_device_call(lib, bad, code):
    with pytest.raises(api.BmmError) as e:
        api.bmm_attn_create(_attn(**bad))
    assert e.value.status == code, bad
    assert lib.bmm_attn_destroy(None) == api.BMM_OK
    assert lib.bmm_attn_run(None, None, None, None, None, None) == api.BMM_ERR_INVALID_ARG


def test_attention_create_without_a_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(api.BmmError) as e:
        api.bmm_attn_create(_attn())
    assert e.value.status == api.BMM_ERR_NO_DEVICE


def test_host_plan_validates_before_any_device_call(lib):
    import ctypes
    lib = api._host_lib()  # argument types set
    plan = ctypes.c_void_p(1)
    assert lib.bmm_host_create(ctypes.byref(_desc(M=-1)), 0, ctypes.byref(plan)) == api.BMM_ERR_INVALID_ARG
    assert plan.value is None
    assert lib.bmm_host_create(ctypes.byref(_desc()), 17, ctypes.byref(plan)) == api.BMM_ERR_INVALID_ARG
    assert lib.bmm_host_create(None, 0, ctypes.byref(plan)) == api.BMM_ERR_INVALID_ARG
    assert lib.bmm_host_destroy(None) == api.BMM_OK
    assert lib.bmm_host_run(None, None, None, None, 1.0, 0.0, None) == api.BMM_ERR_INVALID_ARG


def test_host_plan_without_a_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(api.BmmError) as e:
        api.HostPlan(_desc())
    assert e.value.status == api.BMM_ERR_NO_DEVICE


@pytest.mark.parametrize("typeC", ["bf16", "f32"])
@pytest.mark.parametrize("transB", [0, 1])
def test_every_ring_layout_fits_the_shared_memory_it_plans(lib, typeC, transB):
    """For a sweep of shapes: the general layout (1024 bytes of alignment
    slack, 32 KB of epilogue buffers, 512 bytes of barriers, the ring) fits
    the plan's shared memory, and a deeper ring for bf16 box-store runs fits
    the 227 KB limit with 2 KB boxes and no slack (the kernel checks the
    alignment it counts on at run time)."""
    stage_limit = 232448
    for M in (96, 1000, 4096):
        for N in (16, 100, 333, 999, 4096):
            for K in (64, 4096):
                lda, ldb = K, (K if transB else N)
                d = _desc(batch=1, M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=N, strideA=M * lda,
                          strideB=(N * K), strideC=M * N, transB=transB, typeC=typeC)
                i = api.bmm_plan_query(d)
                assert 2 <= i.stages <= 8
                assert 1024 + 32768 + 512 + i.stages * i.stage_bytes <= i.smem_bytes <= stage_limit
                assert i.stages_bf16_box >= i.stages
                if i.stages_bf16_box > i.stages:
                    assert i.cta_pair == 1 and typeC == "bf16" and i.swap_ab == 0
                    assert i.stages_bf16_box * i.stage_bytes + 16384 + 512 <= i.smem_bytes == stage_limit

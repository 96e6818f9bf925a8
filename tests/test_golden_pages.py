"""The pages' printed figures (tests/golden/pages_figures.json) pin the
host-side measurement arithmetic: arithmetic intensity, ridge point and the
shared-memory budget formula."""
import json
import os

from dense_matmul_tensor_gb300 import workloads as wl

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def test_ridge_point_a100():
    g = GOLDEN["ridge_a100"]
    assert g["peak_tflops_fp16"] * 1e12 / (g["hbm_tb_per_s"] * 1e12) == g["ridge_flop_per_byte"]


def test_intensity_of_square_gemm_matches_page_formula():
    # 2MNK / 2(MK+KN+MN) for M=N=K=4096 is 4096/3; the workload's own
    # flop and byte counts (bf16 in, bf16 out, beta=0) must agree
    p = wl.GEMM_4096
    M, N, K = p.M, p.N, p.K
    page_ai = (2 * M * N * K) / (2 * (M * K + K * N + M * N))
    assert abs(page_ai - 4096 / 3) < 1e-9
    assert abs(p.flops() / p.algorithmic_bytes() - page_ai) < 1e-9


def test_smem_stage_formula_matches_printed_example():
    g = GOLDEN["smem_overflow_example"]
    stage = (g["BLOCK_M"] * g["BLOCK_K"] + g["BLOCK_K"] * g["BLOCK_N"]) * g["elem_bytes"]
    assert round(stage / 1000) == g["stage_bytes_as_printed_kb"]            # 49,152 B printed as "49KB"
    # the page multiplies its rounded stage size by the stage count: 5 x 49 = 245
    assert g["num_stages"] * round(stage / 1000) == g["total_as_printed_kb"]
    assert g["num_stages"] * stage > g["limit_kb_a100"] * 1024


def test_workload_intensities_against_measured_ridge():
    # skinny and attention shapes sit under any ridge above ~120 FLOP/B;
    # the square GEMM sits far above it
    assert wl.SKINNY.flops() / wl.SKINNY.algorithmic_bytes() < 16
    assert wl.ATTN_QK.flops() / wl.ATTN_QK.algorithmic_bytes() < 61
    assert wl.GEMM_4096.flops() / wl.GEMM_4096.algorithmic_bytes() > 1000

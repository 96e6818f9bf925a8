"""The DRAM traffic bench.py reports (``roofline.traffic``) comes from an ncu
capture of a given kernel source; the table keys each figure by a hash of
those sources, and the bench reports null for a kernel whose sources no
longer match.  The committed figures must belong to the committed sources."""
import bench


def test_every_reported_kernel_has_a_current_traffic_figure():
    current = {
        "gemm_4096x4096x4096_tn_bf16": bench.kernel_source_hash(bench.GEMM_SOURCES),
        "attn_fused_b128_2048x2048x128_bf16": bench.kernel_source_hash(bench.ATTN_SOURCES),
    }
    for workload, h in current.items():
        assert (h, workload) in bench.NCU_TRAFFIC, f"no capture for the current sources of {workload}"
    for (h, workload), traffic in bench.NCU_TRAFFIC.items():
        assert current.get(workload) == h, f"stale traffic key {h} for {workload}"
        assert traffic > 0


def test_tensor_pipe_figures_belong_to_the_current_sources():
    current = {
        "gemm_4096x4096x4096_tn_bf16": bench.kernel_source_hash(bench.GEMM_SOURCES),
        "attn_fused_b128_2048x2048x128_bf16": bench.kernel_source_hash(bench.ATTN_SOURCES),
    }
    for (h, workload), pct in bench.NCU_TENSOR_ACTIVE_PCT.items():
        assert current.get(workload) == h, f"stale tensor-pipe key {h} for {workload}"
        assert 0.0 < pct <= 100.0

// C ABI of the fused attention-shaped contraction (declared in include/bmm.h):
// validation, tensor maps and the launch of attn_fwd_kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/bmm.h"
#include "attn_kernel.cuh"

struct bmm_attn_plan_s {
  bmm_attn_desc_t d;
  int sms;
  uint32_t* err;
  uint64_t timeout_ns;
  int test_stall;
  const void* map_ptr[3];
  CUtensorMap map[3];  // Q, K, V
};

namespace {

constexpr int64_t kMax31 = 0x7fffffffLL;
constexpr int64_t kMaxLen = int64_t(1) << 30;

PFN_cuTensorMapEncodeTiled_v12000 g_encode_attn = nullptr;
std::once_flag g_encode_attn_once;

bool encoder() {
  std::call_once(g_encode_attn_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_attn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode_attn != nullptr;
}

// [batch][rows][128] bf16 with row stride ld and batch stride sb (elements),
// read in (64 x 128) boxes with the 128-byte swizzle.
bool encode_rows(const void* base, int64_t batch, int64_t rows, int64_t ld, int64_t sb,
                 CUtensorMap* out) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dmt::kAttnD), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2),
                           static_cast<cuuint64_t>(batch > 1 ? sb * 2 : ((rows * ld * 2 + 15) / 16) * 16)};
  cuuint32_t box[3] = {64u, 128u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return g_encode_attn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

uint64_t attn_timeout_ns() {
  const char* e = std::getenv("DMT_BMM_WAIT_TIMEOUT_MS");
  if (e && *e) {
    const long long ms = std::atoll(e);
    if (ms > 0) return static_cast<uint64_t>(ms) * 1000000ull;
  }
  return 2000000000ull;
}

bmm_status_t attn_validate(const bmm_attn_desc_t* d) {
  if (!d) return BMM_ERR_INVALID_ARG;
  if (d->batch < 0 || d->Lq < 0 || d->Lk < 0 || d->D <= 0) return BMM_ERR_INVALID_ARG;
  if (d->D != dmt::kAttnD) return BMM_ERR_UNSUPPORTED;
  if (d->ldq < d->D || d->ldk < d->D || d->ldv < d->D || d->ldo < d->D) return BMM_ERR_INVALID_ARG;
  if (d->strideQ < 0 || d->strideK < 0 || d->strideV < 0 || d->strideO < 0) return BMM_ERR_INVALID_ARG;
  if (d->batch > 1 && d->Lq > 0 && d->strideO < (d->Lq - 1) * d->ldo + d->D) return BMM_ERR_INVALID_ARG;
  if (!std::isfinite(d->alpha)) return BMM_ERR_INVALID_ARG;
  // key and query indices (and TMA coordinates) stay in int32 with a block's slack
  if (d->batch > kMax31 || d->Lq > kMaxLen || d->Lk > kMaxLen) return BMM_ERR_UNSUPPORTED;
  if (d->batch > 0 && d->Lq > 0 && d->Lk == 0) return BMM_ERR_UNSUPPORTED;  // softmax over nothing
  // TMA row strides and the 16-byte output rows
  if (d->ldq % 8 || d->ldk % 8 || d->ldv % 8 || d->ldo % 8) return BMM_ERR_UNSUPPORTED;
  if (d->batch > 1 && (d->strideQ % 8 || d->strideK % 8 || d->strideV % 8 || d->strideO % 8))
    return BMM_ERR_UNSUPPORTED;
  return BMM_OK;
}

}  // namespace

extern "C" {

bmm_status_t bmm_attn_create(const bmm_attn_desc_t* desc, bmm_attn_plan_t* out) {
  if (!out) return BMM_ERR_INVALID_ARG;
  *out = nullptr;
  const bmm_status_t st = attn_validate(desc);
  if (st != BMM_OK) return st;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BMM_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BMM_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return BMM_ERR_NO_DEVICE;
  if (!encoder()) return BMM_ERR_CUDA;
  bmm_attn_plan_s* pl = new (std::nothrow) bmm_attn_plan_s();
  if (!pl) return BMM_ERR_CUDA;
  pl->d = *desc;
  pl->sms = sms;
  pl->timeout_ns = attn_timeout_ns();
  const char* ts = std::getenv("DMT_BMM_TEST_STALL_MMA");
  pl->test_stall = (ts && ts[0] == '1') ? 1 : 0;
  if (cudaMalloc(reinterpret_cast<void**>(&pl->err), 256) != cudaSuccess ||
      cudaMemset(pl->err, 0, 256) != cudaSuccess) {
    cudaFree(pl->err);
    delete pl;
    return BMM_ERR_CUDA;
  }
  *out = pl;
  return BMM_OK;
}

bmm_status_t bmm_attn_run(bmm_attn_plan_t pl, const void* Q, const void* K, const void* V, void* O,
                          void* stream_v) {
  if (!pl) return BMM_ERR_INVALID_ARG;
  const bmm_attn_desc_t& d = pl->d;
  if (d.batch == 0 || d.Lq == 0) return BMM_OK;
  if (!Q || !K || !V || !O) return BMM_ERR_INVALID_ARG;
  for (const void* ptr : {Q, K, V, static_cast<const void*>(O)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return BMM_ERR_MISALIGNED;
  const void* bases[3] = {Q, K, V};
  const int64_t rows[3] = {d.Lq, d.Lk, d.Lk};
  const int64_t lds[3] = {d.ldq, d.ldk, d.ldv};
  const int64_t sbs[3] = {d.strideQ, d.strideK, d.strideV};
  for (int i = 0; i < 3; ++i) {
    if (pl->map_ptr[i] != bases[i]) {
      if (!encode_rows(bases[i], d.batch, rows[i], lds[i], sbs[i], &pl->map[i])) return BMM_ERR_CUDA;
      pl->map_ptr[i] = bases[i];
    }
  }
  static std::once_flag once;
  static bool attr_ok = false;
  std::call_once(once, [] {
    attr_ok = cudaFuncSetAttribute(dmt::attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(dmt::kAttnSmem)) == cudaSuccess;
  });
  if (!attr_ok) return BMM_ERR_CUDA;
  const int rows_per_item = dmt::kAttnItemRows;
  dmt::AttnParams ap;
  std::memset(&ap, 0, sizeof(ap));
  ap.Lq = static_cast<int32_t>(d.Lq);
  ap.Lk = static_cast<int32_t>(d.Lk);
  ap.q_tiles = static_cast<int32_t>((d.Lq + rows_per_item - 1) / rows_per_item);
  ap.k_blocks = static_cast<int32_t>((d.Lk + dmt::kAttnN - 1) / dmt::kAttnN);
  ap.items = d.batch * ap.q_tiles;
  ap.scale_log2 = static_cast<float>(static_cast<double>(d.alpha) * 1.4426950408889634);
  // 128 x 128 x 16 MMAs, bf16 in, fp32 accumulate; B of O = P V is MN-major
  const uint32_t base = (1u << 4) | (1u << 7) | (1u << 10) | (16u << 17) |
                        (static_cast<uint32_t>(dmt::kAttnM >> 4) << 24);
  ap.idesc_s = base;
  ap.idesc_o = base | (1u << 16);
  ap.O = static_cast<__nv_bfloat16*>(O);
  ap.ldo = d.ldo;
  ap.so = d.strideO;
  ap.err = pl->err;
  ap.timeout_ns = pl->timeout_ns;
  ap.test_stall = pl->test_stall;
  const int64_t grid = ap.items < pl->sms ? ap.items : pl->sms;
  dmt::attn_fwd_kernel<<<static_cast<unsigned>(grid), dmt::kAttnThreads, dmt::kAttnSmem,
                         static_cast<cudaStream_t>(stream_v)>>>(ap, pl->map[0], pl->map[1], pl->map[2]);
  return cudaGetLastError() == cudaSuccess ? BMM_OK : BMM_ERR_CUDA;
}

bmm_status_t bmm_attn_get_device_error(bmm_attn_plan_t pl, uint32_t* detail) {
  if (!pl) return BMM_ERR_INVALID_ARG;
  uint32_t w = 0;
  if (cudaMemcpy(&w, pl->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return BMM_ERR_CUDA;
  if (w != 0 && cudaMemset(pl->err, 0, sizeof(w)) != cudaSuccess) return BMM_ERR_CUDA;
  if (detail) *detail = w;
  return w == 0 ? BMM_OK : BMM_ERR_DEVICE_TIMEOUT;
}

bmm_status_t bmm_attn_destroy(bmm_attn_plan_t pl) {
  if (!pl) return BMM_OK;
  bmm_status_t st = BMM_OK;
  if (pl->err && cudaFree(pl->err) != cudaSuccess) st = BMM_ERR_CUDA;
  delete pl;
  return st;
}

}  // extern "C"

// Host-buffer entry point of the batched product (declared in include/bmm.h):
// copies the operands in from host memory, runs the product and copies C
// back, overlapping the transfers with the computation in chunks.
//
// The work is cut into chunks of whole batch items (batch >= 2) or of rows of
// A and C (batch 1 with A row-major).  Chunk c's inputs go in on a copy
// stream, its product runs on the caller's stream once they have landed, and
// its C goes out on a second copy stream once the product is done, so chunk
// c+1 is copied in while chunk c computes and chunk c-1 is copied out.  Each
// chunk is an ordinary plan of the product (its own tensor maps, cached for
// the plan's fixed device buffers), so the result is the one bmm_run gives:
// the chunks only split independent rows or batch items.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>
#include <vector>

#include "../../include/bmm.h"

namespace {

constexpr int kMaxChunks = 16;
constexpr int64_t kRowQuantum = 256;  // row chunks in whole 256-row (CTA-pair) tiles

struct Extent {
  int64_t off;    // first element of the chunk's region
  int64_t elems;  // elements from there to the region's last element
};

// Elements an operand of `items` batch items spans: (items-1)*stride + one
// item's rows*ld reach (the last row only up to its last column).
int64_t span(int64_t items, int64_t stride, int64_t rows, int64_t ld, int64_t cols) {
  if (items <= 0 || rows <= 0 || cols <= 0) return 0;
  return (items - 1) * stride + (rows - 1) * ld + cols;
}

int64_t elem_bytes(int32_t t) { return t == BMM_F32 ? 4 : 2; }

}  // namespace

struct bmm_host_plan_s {
  bmm_desc_t d;
  int chunks;
  bool by_rows;                  // chunks of rows of A and C (batch 1), else of batch items
  int64_t first[kMaxChunks + 1]; // chunk c covers items / rows [first[c], first[c+1])
  bmm_plan_t sub[kMaxChunks];
  void* dA = nullptr;
  void* dB = nullptr;
  void* dC = nullptr;
  int64_t a_rows, a_cols, b_rows, b_cols;  // stored shapes of one batch item
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr, ev_end = nullptr;
  cudaEvent_t ev_in[kMaxChunks], ev_done[kMaxChunks];
};

namespace {

void release(bmm_host_plan_s* hp) {
  for (int c = 0; c < hp->chunks; ++c) {
    if (hp->sub[c]) bmm_destroy(hp->sub[c]);
    if (hp->ev_in[c]) cudaEventDestroy(hp->ev_in[c]);
    if (hp->ev_done[c]) cudaEventDestroy(hp->ev_done[c]);
  }
  if (hp->ev_start) cudaEventDestroy(hp->ev_start);
  if (hp->ev_end) cudaEventDestroy(hp->ev_end);
  if (hp->h2d) cudaStreamDestroy(hp->h2d);
  if (hp->d2h) cudaStreamDestroy(hp->d2h);
  cudaFree(hp->dA);
  cudaFree(hp->dB);
  cudaFree(hp->dC);
  delete hp;
}

// The region of operand X (A = 0, B = 1, C = 2) that chunk c reads or writes.
Extent region(const bmm_host_plan_s* hp, int x, int c) {
  const bmm_desc_t& d = hp->d;
  const int64_t lo = hp->first[c], hi = hp->first[c + 1];
  int64_t rows, cols, ld, stride;
  if (x == 0) {
    rows = hp->a_rows; cols = hp->a_cols; ld = d.lda; stride = d.strideA;
  } else if (x == 1) {
    rows = hp->b_rows; cols = hp->b_cols; ld = d.ldb; stride = d.strideB;
  } else {
    rows = d.M; cols = d.N; ld = d.ldc; stride = d.strideC;
  }
  if (hp->by_rows) {
    if (x == 1) return {0, span(1, 0, rows, ld, cols)};  // B: whole, with the first chunk
    return {lo * ld, span(1, 0, hi - lo, ld, cols)};
  }
  if (x != 2 && stride == 0) return {0, span(1, 0, rows, ld, cols)};  // broadcast: once
  return {lo * stride, span(hi - lo, stride, rows, ld, cols)};
}

}  // namespace

extern "C" {

bmm_status_t bmm_host_create(const bmm_desc_t* desc, int32_t chunks, bmm_host_plan_t* out) {
  if (!out) return BMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!desc || chunks < 0 || chunks > kMaxChunks) return BMM_ERR_INVALID_ARG;
  // validate the whole problem first (no device needed)
  bmm_plan_info_t info;
  const bmm_status_t vst = bmm_plan_query(desc, &info);
  if (vst != BMM_OK) return vst;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BMM_ERR_NO_DEVICE;

  bmm_host_plan_s* hp = new (std::nothrow) bmm_host_plan_s();
  if (!hp) return BMM_ERR_CUDA;
  hp->d = *desc;
  const bmm_desc_t& d = hp->d;
  hp->a_rows = d.transA ? d.K : d.M;
  hp->a_cols = d.transA ? d.M : d.K;
  hp->b_rows = d.transB ? d.N : d.K;
  hp->b_cols = d.transB ? d.K : d.N;
  int want = chunks == 0 ? 4 : chunks;
  hp->by_rows = d.batch == 1 && !d.transA;
  const int64_t units = hp->by_rows ? (d.M + kRowQuantum - 1) / kRowQuantum : d.batch;
  if (units < want) want = static_cast<int>(units > 0 ? units : 1);
  if (d.batch == 1 && d.transA) want = 1;  // A's rows are its K index: no row split
  hp->chunks = want;
  for (int c = 0; c <= want; ++c) {
    const int64_t u = units * c / want;
    hp->first[c] = hp->by_rows ? (u * kRowQuantum < d.M ? u * kRowQuantum : d.M) : u;
  }
  hp->first[want] = hp->by_rows ? d.M : d.batch;

  bmm_status_t st = BMM_OK;
  const int64_t ea = elem_bytes(d.typeA), ec = elem_bytes(d.typeC);
  const int64_t na = span(d.batch, d.strideA, hp->a_rows, d.lda, hp->a_cols);
  const int64_t nbe = span(d.batch, d.strideB, hp->b_rows, d.ldb, hp->b_cols);
  const int64_t nc = span(d.batch, d.strideC, d.M, d.ldc, d.N);
  if ((na && cudaMalloc(&hp->dA, na * ea) != cudaSuccess) ||
      (nbe && cudaMalloc(&hp->dB, nbe * ea) != cudaSuccess) ||
      (nc && cudaMalloc(&hp->dC, nc * ec) != cudaSuccess) ||
      cudaStreamCreateWithFlags(&hp->h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hp->d2h, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp->ev_start, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp->ev_end, cudaEventDisableTiming) != cudaSuccess)
    st = BMM_ERR_CUDA;
  for (int c = 0; c < hp->chunks && st == BMM_OK; ++c) {
    if (cudaEventCreateWithFlags(&hp->ev_in[c], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp->ev_done[c], cudaEventDisableTiming) != cudaSuccess) {
      st = BMM_ERR_CUDA;
      break;
    }
    bmm_desc_t sd = d;
    const int64_t n = hp->first[c + 1] - hp->first[c];
    if (hp->by_rows) sd.M = n; else sd.batch = n;
    st = bmm_create(&sd, &hp->sub[c]);
  }
  if (st != BMM_OK) {
    release(hp);
    return st;
  }
  *out = hp;
  return BMM_OK;
}

bmm_status_t bmm_host_run(bmm_host_plan_t hp, const void* hA, const void* hB, void* hC, float alpha,
                          float beta, void* stream_v) {
  if (!hp) return BMM_ERR_INVALID_ARG;
  const bmm_desc_t& d = hp->d;
  if (d.batch == 0 || d.M == 0 || d.N == 0) return BMM_OK;
  if (!hC) return BMM_ERR_INVALID_ARG;
  const bool reads_ab = alpha != 0.0f && d.K > 0;
  if (reads_ab && (!hA || !hB)) return BMM_ERR_INVALID_ARG;
  const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const int64_t ea = elem_bytes(d.typeA), ec = elem_bytes(d.typeC);
  auto in = [&](void* dst, const void* src, int x, int c, int64_t es) -> bool {
    const Extent e = region(hp, x, c);
    if (e.elems == 0) return true;
    return cudaMemcpyAsync(static_cast<char*>(dst) + e.off * es,
                           static_cast<const char*>(src) + e.off * es, e.elems * es,
                           cudaMemcpyHostToDevice, hp->h2d) == cudaSuccess;
  };
  // the copies start once the caller's earlier work on `stream` is done
  if (cudaEventRecord(hp->ev_start, stream) != cudaSuccess ||
      cudaStreamWaitEvent(hp->h2d, hp->ev_start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->d2h, hp->ev_start, 0) != cudaSuccess)
    return BMM_ERR_CUDA;
  const bool b_once = hp->by_rows || d.strideB == 0;
  const bool a_once = !hp->by_rows && d.strideA == 0;
  for (int c = 0; c < hp->chunks; ++c) {
    bool ok = true;
    if (reads_ab) {
      if (!a_once || c == 0) ok = ok && in(hp->dA, hA, 0, c, ea);
      if (!b_once || c == 0) ok = ok && in(hp->dB, hB, 1, c, ea);
    }
    if (beta != 0.0f) ok = ok && in(hp->dC, hC, 2, c, ec);
    if (!ok || cudaEventRecord(hp->ev_in[c], hp->h2d) != cudaSuccess) return BMM_ERR_CUDA;
  }
  for (int c = 0; c < hp->chunks; ++c) {
    if (cudaStreamWaitEvent(stream, hp->ev_in[c], 0) != cudaSuccess) return BMM_ERR_CUDA;
    const Extent ra = region(hp, 0, c), rb = region(hp, 1, c), rc = region(hp, 2, c);
    const bmm_status_t st =
        bmm_run(hp->sub[c], static_cast<const char*>(hp->dA) + ra.off * ea,
                static_cast<const char*>(hp->dB) + (hp->by_rows ? 0 : rb.off) * ea,
                static_cast<char*>(hp->dC) + rc.off * ec, alpha, beta, stream_v);
    if (st != BMM_OK) return st;
    if (cudaEventRecord(hp->ev_done[c], stream) != cudaSuccess ||
        cudaStreamWaitEvent(hp->d2h, hp->ev_done[c], 0) != cudaSuccess)
      return BMM_ERR_CUDA;
    if (rc.elems && cudaMemcpyAsync(static_cast<char*>(hC) + rc.off * ec,
                                    static_cast<const char*>(hp->dC) + rc.off * ec, rc.elems * ec,
                                    cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess)
      return BMM_ERR_CUDA;
  }
  // the caller's stream completes only when C is back in host memory
  if (cudaEventRecord(hp->ev_end, hp->d2h) != cudaSuccess ||
      cudaStreamWaitEvent(stream, hp->ev_end, 0) != cudaSuccess)
    return BMM_ERR_CUDA;
  return BMM_OK;
}

bmm_status_t bmm_host_get_device_error(bmm_host_plan_t hp, uint32_t* detail) {
  if (!hp) return BMM_ERR_INVALID_ARG;
  bmm_status_t result = BMM_OK;
  uint32_t first = 0;
  for (int c = 0; c < hp->chunks; ++c) {
    uint32_t w = 0;
    const bmm_status_t st = bmm_get_device_error(hp->sub[c], &w);
    if (st != BMM_OK && result == BMM_OK) {
      result = st;
      first = w;
    }
  }
  if (detail) *detail = first;
  return result;
}

bmm_status_t bmm_host_get_chunks(bmm_host_plan_t hp, int32_t* chunks, int32_t* by_rows) {
  if (!hp) return BMM_ERR_INVALID_ARG;
  if (chunks) *chunks = hp->chunks;
  if (by_rows) *by_rows = hp->by_rows ? 1 : 0;
  return BMM_OK;
}

bmm_status_t bmm_host_destroy(bmm_host_plan_t hp) {
  if (!hp) return BMM_OK;
  release(hp);
  return BMM_OK;
}

}  // extern "C"

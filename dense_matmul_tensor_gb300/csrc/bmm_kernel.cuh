// The batched-product kernels for sm_103a.
//
// bmm_tc_kernel: a persistent, warp-specialised tcgen05 GEMM over the whole
// batch x tile grid.  Per CTA (192 threads, one CTA per SM):
//   warp 0      TMA producer: fills a multi-stage shared-memory ring with the
//               A tile (128 x 64) and the B tile (BN x 64) of each k-block.
//   warp 1      allocates Tensor Memory and, from one lane, issues
//               tcgen05.mma (128 x BN x 16 per instruction) into a
//               double-buffered fp32 accumulator; tcgen05.commit releases
//               ring slots and hands finished accumulators to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld of their 32 accumulator lanes, scale by
//               alpha (+ beta * C), convert, and store with coalesced
//               global writes (row-major C goes through a padded shared
//               staging tile so that each warp store covers one C row).
//
// Design sources on the pages (prior art, restated for sm_103a):
//  - "Triton Optimization Reference (cuTile -> Triton)", section 1: EVEN_K.
//    Every full k-block runs with no bounds logic; when K % 64 != 0 the last
//    k-block is a separate tail whose out-of-range columns TMA fills with
//    zeros, and the MMA issues only ceil((K % 64) / 16) k-steps for it.
//  - same page, section 2: transposition lives in the addressing.  Here it
//    is the TMA box orientation plus the MN-major bit and byte offsets of the
//    tcgen05 shared-memory descriptor; no data is moved.
//  - same page, sections 3 and 7: the batch x tile grid is walked by a static
//    persistent loop over tile ids, decoded with GROUP_M grouping for L2
//    reuse.
//  - "FLA Triton -> Gluon porting", sections 3-5: ring of stages with one
//    "full" and one "empty" mbarrier per slot, separate barriers for TMA and
//    tcgen05 completion, accumulator in Tensor Memory zero-initialised by the
//    first MMA (enable-input-D off), load / MMA / epilogue partitions.
//
// Every mbarrier wait is bounded (%globaltimer).  On expiry the kernel
// records an error word, raises a CTA-wide abort flag, waits (bounded) for
// its own TMA loads and MMAs in flight, frees Tensor Memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace dmt {

constexpr int kTileM = 128;   // MMA M (TMEM lanes)
constexpr int kTileK = 64;    // k-block: 64 x 16-bit = one 128-byte swizzle row
constexpr int kUmmaK = 16;    // K of one tcgen05.mma kind::f16
constexpr int kThreads = 192; // producer, MMA, 4 epilogue warps
constexpr int kGroupM = 8;
constexpr int kEpiPitch = 33; // floats per staged row (bank-conflict-free)
constexpr uint32_t kEpiBytes = 4u * 32u * kEpiPitch * 4u;
constexpr uint32_t kBarBytes = 512;   // barriers, TMEM slot, abort flag
constexpr uint32_t kSmemLimit = 232448;  // 227 KB dynamic shared memory per CTA

// Device error word: kErrTag | (site << 8) | role-specific detail.
constexpr uint32_t kErrTag = 0xB0000000u;
enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaAccEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpiAccFull = 4,
};

struct KParams {
  int32_t Mv, Nv, K;       // MMA view: D (Mv x Nv) = opA (Mv x K) * opB (K x Nv)
  int32_t num_m, num_n;    // tiles per batch item
  int64_t tiles;           // batch * num_m * num_n
  int32_t k_blocks;        // ceil(K / 64)
  int32_t tail_steps;      // MMA k-steps in the last k-block (4 when K % 64 == 0)
  int32_t a_mn, b_mn;      // 1: operand is MN-major in memory (and in smem)
  int32_t a_bcast, b_bcast;// 1: batch stride 0 (tensor map has one batch item)
  int32_t stages;
  uint32_t stage_bytes;    // A tile + B tile, 1024-aligned
  uint32_t a_bytes;        // offset of the B tile inside a stage
  uint32_t tx_bytes;       // TMA bytes per stage
  uint32_t idesc;          // tcgen05 instruction descriptor
  uint32_t tmem_cols;
  void* C;
  int64_t ldc, sC;         // C strides (elements), user layout
  int32_t c_bf16;          // C element type: 1 = bf16, 0 = fp32
  int32_t c_trans;         // 1: D = C^T (operands swapped): D(i, j) -> C[j*ldc + i]
  float alpha, beta;
  uint32_t* err;           // device error word
  uint64_t timeout_ns;     // bound on any single wait
};

struct Abort {
  volatile uint32_t* flag;
  uint32_t* err;
  uint64_t timeout_ns;
};

// Slow path of a bounded wait: poll until the phase completes, another role
// raises the abort flag, or the time limit passes (then raise it).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, Abort ab, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*ab.flag) return false;
      if (global_timer_ns() - t0 > ab.timeout_ns) break;
    }
  }
  *ab.flag = 1u;
  atomicCAS(ab.err, 0u, kErrTag | (site << 8) | (blockIdx.x & 0xFFu));
  return false;
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, Abort ab, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, ab, site);
}

// Wait with a short fixed limit and no error report: used only on the abort
// path to let this CTA's own asynchronous copies and MMAs land before exit.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 15u) == 0 && global_timer_ns() - t0 > 100000000ull) return;
  }
}

__device__ __forceinline__ void decode_tile(int64_t t, const KParams& p, int& b, int& mb, int& nb) {
  const int64_t per = static_cast<int64_t>(p.num_m) * p.num_n;
  b = static_cast<int>(t / per);
  const int r = static_cast<int>(t - static_cast<int64_t>(b) * per);
  const int group = kGroupM * p.num_n;
  const int gid = r / group;
  const int first_m = gid * kGroupM;
  const int gsz = min(p.num_m - first_m, kGroupM);
  const int rin = r - gid * group;
  mb = first_m + rin % gsz;
  nb = rin / gsz;
}

__device__ __forceinline__ float load_c(const KParams& p, int64_t off) {
  if (p.c_bf16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p.C)[off]);
  return static_cast<const float*>(p.C)[off];
}

__device__ __forceinline__ void store_c(const KParams& p, int64_t off, float v) {
  if (p.c_bf16)
    static_cast<__nv_bfloat16*>(p.C)[off] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(p.C)[off] = v;
}

// One chunk of CW accumulator columns held by this thread (row `lane` of the
// warp's 32-lane quarter) -> C.
template <int CW>
__device__ __forceinline__ void store_chunk(const KParams& p, float (&v)[CW], float* stg, int lane,
                                            int row0, int col0, int64_t cbase) {
  const float alpha = p.alpha, beta = p.beta;
  if (p.c_trans) {
    // D row i = C column, D column j = C row: lanes write consecutive C columns.
    const int i = row0 + lane;
    if (i < p.Mv) {
#pragma unroll
      for (int r = 0; r < CW; ++r) {
        const int j = col0 + r;
        if (j < p.Nv) {
          const int64_t off = cbase + static_cast<int64_t>(j) * p.ldc + i;
          float out = alpha * v[r];
          if (beta != 0.0f) out = fmaf(beta, load_c(p, off), out);
          store_c(p, off, out);
        }
      }
    }
    return;
  }
  // Row-major C: stage the 32 x CW block (thread = row) and write it back
  // row by row (lane = column), so each warp store covers one C row.
#pragma unroll
  for (int r = 0; r < CW; ++r) stg[lane * kEpiPitch + r] = v[r];
  __syncwarp();
  const int j = col0 + lane;
  if (lane < CW && j < p.Nv) {
    const int rows = min(32, p.Mv - row0);
    for (int rr = 0; rr < rows; ++rr) {
      const int64_t off = cbase + static_cast<int64_t>(row0 + rr) * p.ldc + j;
      float out = alpha * stg[rr * kEpiPitch + lane];
      if (beta != 0.0f) out = fmaf(beta, load_c(p, off), out);
      store_c(p, off, out);
    }
  }
  __syncwarp();
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    bmm_tc_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmA,
                  const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  const int S = p.stages;
  const uint32_t ring_bytes = static_cast<uint32_t>(S) * p.stage_bytes;
  float* epi = reinterpret_cast<float*>(smem + ring_bytes);
  const uint32_t bar0 = sbase + ring_bytes + kEpiBytes;
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], drain; then the
  // Tensor Memory base address and the CTA-wide abort flag
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + ring_bytes + kEpiBytes + 8u * (2u * S + 5u));
  volatile uint32_t* abort_flag = tmem_slot + 1;

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 4);  // one arrive per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const Abort ab{abort_flag, p.err, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
        int b, mb, nb;
        decode_tile(t, p, b, mb, nb);
        const int m0 = mb * kTileM, n0 = nb * BN;
        const int za = p.a_bcast ? 0 : b, zb = p.b_bcast ? 0 : b;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1u;
          if (!wait_bounded(empty_bar(s), ph ^ 1u, ab, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + s * p.stage_bytes;
          const uint32_t b_dst = a_dst + p.a_bytes;
          mbar_arrive_expect_tx(full_bar(s), p.tx_bytes);
          const int k0 = kb * kTileK;
          if (!p.a_mn) {
            tma_load_3d(a_dst, &tmA, full_bar(s), k0, m0, za);
          } else {
            tma_load_3d(a_dst, &tmA, full_bar(s), m0, k0, za);
            tma_load_3d(a_dst + 8192u, &tmA, full_bar(s), m0 + 64, k0, za);
          }
          if (!p.b_mn) {
            tma_load_3d(b_dst, &tmB, full_bar(s), k0, n0, zb);
          } else {
#pragma unroll
            for (int h = 0; h < BN / 64; ++h)
              tma_load_3d(b_dst + 8192u * h, &tmB, full_bar(s), n0 + 64 * h, k0, zb);
          }
        }
      }
      // Let the loads issued for the last S k-blocks land before the CTA can
      // exit (after a normal run they have all landed and this returns at once).
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0u;
      for (uint32_t j = first; j < it; ++j) drain_wait(full_bar(j % S), (j / S) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, b_lbo = p.b_mn ? 8192u : 16u;
      const uint32_t a_step = p.a_mn ? 2048u : 32u, b_step = p.b_mn ? 2048u : 32u;
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++tl) {
        const uint32_t acc = tl & 1u, aph = (tl >> 1) & 1u;
        if (!wait_bounded(acce_bar(acc), aph ^ 1u, ab, kSiteMmaAccEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1u;
          if (!wait_bounded(full_bar(s), ph, ab, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = sbase + s * p.stage_bytes;
          const uint32_t b_addr = a_addr + p.a_bytes;
          const int nsteps = (kb == p.k_blocks - 1) ? p.tail_steps : kTileK / kUmmaK;
          for (int ks = 0; ks < nsteps; ++ks) {
            const uint64_t ad = smem_desc_sw128(a_addr + ks * a_step, a_lbo, 1024u);
            const uint64_t bd = smem_desc_sw128(b_addr + ks * b_step, b_lbo, 1024u);
            tc_mma_f16(d_tmem, ad, bd, p.idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(empty_bar(s));  // slot is free once these MMAs have read it
        }
        if (!ok) break;
        tc_commit(accf_bar(acc));  // accumulator complete
      }
      // Every MMA this thread issued must finish before Tensor Memory is freed
      // (on an aborted run nobody else waits for them).
      tc_commit(drain_bar);
      drain_wait(drain_bar, 0u);
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    float* stg = epi + (warp - 2) * 32 * kEpiPitch;
    uint32_t tl = 0;
    for (int64_t t = blockIdx.x; t < p.tiles; t += gridDim.x, ++tl) {
      const uint32_t acc = tl & 1u, aph = (tl >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(accf_bar(acc), aph, ab, kSiteEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after_sync();
      int b, mb, nb;
      decode_tile(t, p, b, mb, nb);
      const int row0 = mb * kTileM + q * 32;
      const int64_t cbase = static_cast<int64_t>(b) * p.sC;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if constexpr (BN == 16) {
        float v[16];
        tmem_ld_16cols(taddr, v);
        tmem_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(acc));
        store_chunk<16>(p, v, stg, lane, row0, nb * BN, cbase);
      } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld_32cols(taddr + 32u * c, v);
          tmem_wait_ld();
          if (c == BN / 32 - 1) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));  // accumulator may be reused
          }
          store_chunk<32>(p, v, stg, lane, row0, nb * BN + 32 * c, cbase);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// Copy a strided 16-bit operand into the workspace with ld rounded up to a
// multiple of 8 elements (16 bytes), which TMA needs for its row strides.
__global__ void pack16_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                              int64_t nb, int64_t rows, int64_t cols, int64_t ld_src,
                              int64_t s_src, int64_t ld_dst, int64_t s_dst) {
  const int64_t total_rows = nb * rows;
  for (int64_t r = blockIdx.y; r < total_rows; r += gridDim.y) {
    const int64_t b = r / rows, i = r - b * rows;
    const uint16_t* s = src + b * s_src + i * ld_src;
    uint16_t* d = dst + b * s_dst + i * ld_dst;
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < cols;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x)
      d[c] = s[c];
  }
}

// C = beta * C (beta == 0 writes zeros without reading C): the alpha == 0 or
// K == 0 case, where A and B are not read.
__global__ void scale_c_kernel(void* C, int c_bf16, int64_t batch, int64_t M, int64_t N,
                               int64_t ldc, int64_t sC, float beta) {
  const int64_t total_rows = batch * M;
  for (int64_t r = blockIdx.y; r < total_rows; r += gridDim.y) {
    const int64_t b = r / M, i = r - b * M;
    const int64_t base = b * sC + i * ldc;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < N;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      if (c_bf16) {
        __nv_bfloat16* c = static_cast<__nv_bfloat16*>(C) + base + j;
        *c = __float2bfloat16_rn(beta == 0.0f ? 0.0f : beta * __bfloat162float(*c));
      } else {
        float* c = static_cast<float*>(C) + base + j;
        *c = beta == 0.0f ? 0.0f : beta * *c;
      }
    }
  }
}

}  // namespace dmt

// Fused attention-shaped contraction for sm_103a:
//
//     O[b] = softmax(alpha * Q[b] K[b]^T) V[b]      (softmax over keys)
//
// Q: [batch][Lq][128], K, V: [batch][Lk][128], bf16, row-major; O bf16.  The
// score matrix S never leaves the chip: per 128-query tile, S blocks of 128
// keys live in Tensor Memory, the probabilities P in shared memory, and the
// output accumulates in registers with the running-maximum rescale of the
// online softmax.  This is the fused form of the attention pair the pages
// build from two batched products ("Triton Optimization Reference (cuTile ->
// Triton)": attention-style contractions; "FLA Triton -> Gluon porting",
// section 4: tcgen05 with Tensor Memory accumulators, section 5: warp
// specialisation).
//
// Per CTA (persistent, one 128-query tile at a time, 192 threads):
//   warp 0      TMA: Q (two 64-column halves) once per tile, then K_j and V_j
//               (128 keys each) into a two-stage ring.
//   warp 1      one lane issues tcgen05.mma: S_j = Q K_j^T (128 x 128 x 128,
//               both operands K-major) into S[j%2], one block ahead of
//               O_j = P_j V_j (V read MN-major: its rows are keys, the
//               contiguous index is the head dimension) into O[j%2].
//   warps 2..5  softmax and accumulation, one query row per thread: row
//               maximum, p = exp2(s*alpha*log2e - m) written to shared memory
//               as bf16 in the swizzled K-major layout the MMA reads (two P
//               buffers, so block j's softmax overlaps block j-1's product),
//               O = O * exp2(m_old - m_new) + O_j in registers, then O / l.
#pragma once

#include "bmm_kernel.cuh"

namespace dmt {

constexpr int kAttnD = 128;   // head dimension (two 64-wide swizzle atoms)
constexpr int kAttnM = 128;   // query rows per tile
constexpr int kAttnN = 128;   // keys per block
constexpr int kAttnStages = 2;
constexpr uint32_t kAttnHalf = 128u * 128u;             // one 64-column half: 16 KB
constexpr uint32_t kAttnQBytes = 2u * kAttnHalf;         // 32 KB
constexpr uint32_t kAttnPBytes = 2u * kAttnHalf;         // 32 KB per P buffer (two buffers)
constexpr uint32_t kAttnKVBytes = 4u * kAttnHalf;        // K and V halves: 64 KB
constexpr uint32_t kAttnBarBytes = 256;
constexpr uint32_t kAttnSmem =
    1024 + kAttnQBytes + 2 * kAttnPBytes + kAttnStages * kAttnKVBytes + kAttnBarBytes;
static_assert(kAttnSmem <= 232448, "shared memory per CTA");

struct AttnParams {
  int32_t Lq, Lk;
  int32_t q_tiles;        // ceil(Lq / 128)
  int32_t k_blocks;       // ceil(Lk / 128)
  int64_t items;          // batch * q_tiles
  float scale_log2;       // alpha * log2(e)
  uint32_t idesc_s;       // 128 x 128, bf16, A and B K-major
  uint32_t idesc_o;       // 128 x 128, bf16, A K-major, B MN-major
  __nv_bfloat16* O;
  int64_t ldo, so;        // O row and batch strides (elements)
  uint32_t* err;
  uint64_t timeout_ns;
  int32_t test_stall;     // 1: the MMA thread first waits on a barrier nothing completes
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float y;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}
// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1) as one paired fp32 instruction
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1) {
  asm("{\n\t.reg .b64 a, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 d, {%0, %1};\n\t"
      "add.rn.f32x2 d, d, a;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

// Largest (kMin: smallest) raw score of this thread's row in one S block over
// the first `valid` keys (all 128 when the block is full).
template <bool kMin>
__device__ __forceinline__ float row_extreme(uint32_t taddr, int valid) {
  const float init = kMin ? INFINITY : -INFINITY;
  float a = init, b = init;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float v[32];
    tmem_ld_32cols(taddr + 32u * c, v);
    tmem_wait_ld();
    if (valid < 128) {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (32 * c + e >= valid) v[e] = init;
    }
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      a = kMin ? min3(a, v[e], v[e + 1]) : max3(a, v[e], v[e + 1]);
      b = kMin ? min3(b, v[e + 2], v[e + 3]) : max3(b, v[e + 2], v[e + 3]);
    }
  }
  return kMin ? fminf(a, b) : fmaxf(a, b);
}

// Softmax of one S block for this thread's query row (warp-uniform control):
// the block's largest alpha * log2(e) * s over the valid keys, the new running
// maximum m and its rescale factor r = exp2(m_old - m_new), the probabilities
// p = exp2(alpha log2(e) s - m_new) written as bf16 into the P buffer (two
// 64-key halves, 128-byte rows, 16-byte chunks XOR-swizzled by row % 8 as
// TMA's 128-byte swizzle would place them), and l = l * r + sum(p).  Releases
// the S buffer and marks P ready.  P buffer g % 2 is reused once the product
// of block g - 2 has read it.
__device__ __forceinline__ bool softmax_block(const AttnParams& p, const Abort& ab, uint32_t s_full,
                                              uint32_t s_empty, uint32_t p_ready, uint32_t p_free,
                                              uint32_t g, uint32_t ph, uint32_t taddr,
                                              uint8_t* p_buf, int row, int lane, int key0,
                                              float& m, float& l, float& r) {
  int w = 1;
  if (lane == 0) w = wait_bounded<true>(s_full, ph, ab, kSiteEpiAccFull) ? 1 : 0;
  if (!__shfl_sync(0xffffffffu, w, 0)) return false;
  __syncwarp();
  tc_fence_after_sync();
  const int valid = p.Lk - key0 < 128 ? p.Lk - key0 : 128;
  const float sc = p.scale_log2;
  // at least one key is valid, so the block's extreme is finite
  const float m_blk = sc >= 0.0f ? row_extreme<false>(taddr, valid) * sc
                                 : row_extreme<true>(taddr, valid) * sc;
  const float m_new = fmaxf(m, m_blk);
  r = fast_exp2(m - m_new);  // exp2(-inf) = 0 for the first block
  if (g >= 2) {  // the product of block g - 2 must have read this P buffer
    if (lane == 0) w = wait_bounded<true>(p_free, ((g >> 1) & 1u) ^ 1u, ab, kSiteEpiAccFull) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, w, 0)) return false;
  }
  const float nm = -m_new;
  float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float v[32];
    tmem_ld_32cols(taddr + 32u * c, v);
    tmem_wait_ld();
    uint8_t* prow = p_buf + (c >> 1) * kAttnHalf + row * 128;
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      fma2(v[e], v[e + 1], v[e], v[e + 1], sc, sc, nm, nm);
      v[e] = fast_exp2(v[e]);
      v[e + 1] = fast_exp2(v[e + 1]);
    }
    if (valid < 128) {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (32 * c + e >= valid) v[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      add2(s0, s1, v[e], v[e + 1]);
      add2(s2, s3, v[e + 2], v[e + 3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // one 16-byte chunk: 8 keys
      uint32_t wds[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * k + 2 * e2], v[8 * k + 2 * e2 + 1]);
        wds[e2] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      const int chunk = (c & 1) * 4 + k;
      *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) =
          make_uint4(wds[0], wds[1], wds[2], wds[3]);
    }
  }
  tc_fence_before_sync();
  fence_proxy_async_shared();  // P is read by the tensor core (async proxy)
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(s_empty);
    mbar_arrive(p_ready);
  }
  // l sums the unrounded p: the bf16 rounding then perturbs only the
  // numerator of O = (P V) / l, by at most 2^-8 sum_c p_c |V_c| / l
  l = l * r + ((s0 + s1) + (s2 + s3));
  m = m_new;
  return true;
}

// Fold one finished P V block into the register accumulator:
// o = o * r + O_block, then release the block's Tensor Memory.
__device__ __forceinline__ bool fold_block(const Abort& ab, uint32_t o_full, uint32_t o_empty,
                                           uint32_t ph, uint32_t taddr, int lane, float r,
                                           float (&o)[kAttnD]) {
  int w = 1;
  if (lane == 0) w = wait_bounded<true>(o_full, ph, ab, kSiteEpiAccFull) ? 1 : 0;
  if (!__shfl_sync(0xffffffffu, w, 0)) return false;
  __syncwarp();
  tc_fence_after_sync();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float v[32];
    tmem_ld_32cols(taddr + 32u * c, v);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; e += 2)
      fma2(o[32 * c + e], o[32 * c + e + 1], o[32 * c + e], o[32 * c + e + 1], r, r, v[e], v[e + 1]);
  }
  tc_fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(o_empty);
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const uint32_t q_addr = sbase;
  uint8_t* p_tile = smem + kAttnQBytes;
  const uint32_t p_addr = sbase + kAttnQBytes;
  const uint32_t kv_addr0 = p_addr + 2 * kAttnPBytes;
  const uint32_t bar0 = kv_addr0 + kAttnStages * kAttnKVBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bar0 - sbase) + 8u * 20u);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  // barriers
  const uint32_t q_full = bar0, q_empty = bar0 + 8;
  auto kv_full = [&](uint32_t s) { return bar0 + 16 + 8 * s; };
  auto kv_empty = [&](uint32_t s) { return bar0 + 32 + 8 * s; };
  auto s_full = [&](uint32_t s) { return bar0 + 48 + 8 * s; };
  auto s_empty = [&](uint32_t s) { return bar0 + 64 + 8 * s; };
  const uint32_t p_ready = bar0 + 80;
  auto p_free = [&](uint32_t s) { return bar0 + 88 + 8 * s; };
  auto o_full = [&](uint32_t s) { return bar0 + 104 + 8 * s; };
  auto o_empty = [&](uint32_t s) { return bar0 + 120 + 8 * s; };
  const uint32_t drain_bar = bar0 + 136;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (uint32_t s = 0; s < 2; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), 4);
      mbar_init(o_full(s), 1);
      mbar_init(o_empty(s), 4);
      mbar_init(p_free(s), 1);
    }
    mbar_init(p_ready, 4);
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);  // S[0], S[1], O[0], O[1]: 128 columns each
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const Abort ab{abort_flag, p.err, p.timeout_ns};
  const int nb = p.k_blocks;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA
    if (lane == 0) {
      uint32_t gk = 0, ti = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
        const int b = static_cast<int>(item / p.q_tiles);
        const int q0 = static_cast<int>(item % p.q_tiles) * kAttnM;
        if (!wait_bounded<true>(q_empty, (ti & 1u) ^ 1u, ab, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(q_full, kAttnQBytes);
        tma_load_3d(q_addr, &tmQ, q_full, 0, q0, b);
        tma_load_3d(q_addr + kAttnHalf, &tmQ, q_full, 64, q0, b);
        for (int j = 0; j < nb; ++j, ++gk) {
          const uint32_t s = gk & 1u, ph = (gk >> 1) & 1u;
          if (!wait_bounded<true>(kv_empty(s), ph ^ 1u, ab, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t kv = kv_addr0 + s * kAttnKVBytes;
          mbar_arrive_expect_tx(kv_full(s), kAttnKVBytes);
          tma_load_3d(kv, &tmK, kv_full(s), 0, j * kAttnN, b);
          tma_load_3d(kv + kAttnHalf, &tmK, kv_full(s), 64, j * kAttnN, b);
          tma_load_3d(kv + 2 * kAttnHalf, &tmV, kv_full(s), 0, j * kAttnN, b);
          tma_load_3d(kv + 3 * kAttnHalf, &tmV, kv_full(s), 64, j * kAttnN, b);
        }
      }
      // let this CTA's last loads land before it can exit
      const uint32_t first = gk > 2u ? gk - 2u : 0u;
      for (uint32_t j = first; j < gk; ++j) drain_wait(kv_full(j & 1u), (j >> 1) & 1u);
      if (ti > 0) drain_wait(q_full, (ti - 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t hi_sw = desc_hi_sw128(1024u);
      const uint32_t q_lo = desc_lo(q_addr, 16u);
      const uint32_t p_lo = desc_lo(p_addr, 16u);
      uint32_t gk = 0, gs = 0, ti = 0;  // PV blocks issued, S blocks issued, tiles
      bool ok = !p.test_stall || wait_bounded(drain_bar, 0u, ab, kSiteTestStall);
      // S_g = Q K_g^T: k-steps 0..3 in the first 64-column halves, 4..7 in the second.
      auto issue_s = [&](uint32_t g) -> bool {
        const uint32_t s = g & 1u, ph = (g >> 1) & 1u;
        if (!wait_bounded<true>(kv_full(s), ph, ab, kSiteMmaFull)) return false;
        if (!wait_bounded<true>(s_empty(s), ph ^ 1u, ab, kSiteMmaAccEmpty)) return false;
        tc_fence_after_sync();
        const uint32_t k_lo = desc_lo(kv_addr0 + s * kAttnKVBytes, 16u);
        const uint32_t d_tmem = tmem_base + s * 128u;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * (kAttnHalf >> 4) + (ks & 3) * 2;  // (bytes >> 4)
          tc_mma_f16(d_tmem, desc_join(q_lo + off, hi_sw), desc_join(k_lo + off, hi_sw), p.idesc_s,
                     ks > 0 ? 1u : 0u);
        }
        tc_commit(s_full(s));
        return true;
      };
      for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
        if (!wait_bounded<true>(q_full, ti & 1u, ab, kSiteMmaFull)) break;
        for (int j = 0; j < nb && ok; ++j, ++gk) {
          if (j == 0) ok = issue_s(gs++);
          if (ok && j + 1 < nb) ok = issue_s(gs++);
          if (!ok) break;
          if (j + 1 == nb) tc_commit(q_empty);  // Q is free once every S of this tile is done
          const uint32_t s = gk & 1u, ph = (gk >> 1) & 1u;
          if (!wait_bounded<true>(p_ready, gk & 1u, ab, kSiteMmaFull) ||
              !wait_bounded<true>(o_empty(s), ph ^ 1u, ab, kSiteMmaAccEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // O_g = P_g V_g: P K-major over keys (two 64-key halves); V MN-major
          // (64-column halves of the head dimension 16 KB apart, 8 key rows per
          // 1024-byte group, 16 keys = 2048 bytes per k-step).
          const uint32_t v_lo = desc_lo(kv_addr0 + s * kAttnKVBytes + 2 * kAttnHalf, kAttnHalf);
          const uint32_t d_tmem = tmem_base + 256u + s * 128u;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t poff = (ks >> 2) * (kAttnHalf >> 4) + (ks & 3) * 2;
            tc_mma_f16(d_tmem, desc_join(p_lo + s * (kAttnPBytes >> 4) + poff, hi_sw),
                       desc_join(v_lo + ks * 128u, hi_sw), p.idesc_o, ks > 0 ? 1u : 0u);
          }
          tc_commit(o_full(s));
          tc_commit(p_free(s));
          tc_commit(kv_empty(s));
        }
      }
      tc_commit(drain_bar);
      drain_wait(drain_bar, 0u);
    }
  } else {
    // ------------------------------------------- softmax and accumulation
    const int q = warp & 3;
    const int row = q * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    uint32_t gk = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x) {
      const int b = static_cast<int>(item / p.q_tiles);
      const int qi = static_cast<int>(item % p.q_tiles) * kAttnM + row;
      float o[kAttnD];
#pragma unroll
      for (int d = 0; d < kAttnD; ++d) o[d] = 0.0f;
      float m = -INFINITY, l = 0.0f;
      float r_pend = 0.0f;  // rescale factor of the newest block not yet folded into o
      for (int j = 0; j < nb && ok; ++j) {
        const uint32_t g = gk + j;
        const uint32_t s = g & 1u, ph = (g >> 1) & 1u;
        float r;
        ok = softmax_block(p, ab, s_full(s), s_empty(s), p_ready, p_free(s), g, ph,
                           tmem_base + lane_off + s * 128u, p_tile + s * kAttnPBytes, row, lane,
                           j * kAttnN, m, l, r);
        if (!ok) break;
        if (j > 0) ok = fold_block(ab, o_full((g - 1) & 1u), o_empty((g - 1) & 1u), ((g - 1) >> 1) & 1u,
                                   tmem_base + lane_off + 256u + ((g - 1) & 1u) * 128u, lane, r_pend, o);
        r_pend = r;
      }
      if (ok) {
        const uint32_t g = gk + nb - 1;
        ok = fold_block(ab, o_full(g & 1u), o_empty(g & 1u), (g >> 1) & 1u,
                        tmem_base + lane_off + 256u + (g & 1u) * 128u, lane, r_pend, o);
      }
      if (!ok) break;
      gk += nb;
      // normalise and store this thread's row of O
      if (qi < p.Lq) {
        const float inv = 1.0f / l;
        __nv_bfloat16* dst = p.O + static_cast<int64_t>(b) * p.so + static_cast<int64_t>(qi) * p.ldo;
#pragma unroll
        for (int d = 0; d < kAttnD; d += 8) {
          uint32_t wds[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const __nv_bfloat162 h2 =
                __floats2bfloat162_rn(o[d + 2 * e2] * inv, o[d + 2 * e2 + 1] * inv);
            wds[e2] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(dst + d) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

}  // namespace dmt

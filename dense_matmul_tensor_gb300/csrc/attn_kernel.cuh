// Fused attention-shaped contraction for sm_103a:
//
//     O[b] = softmax(alpha * Q[b] K[b]^T) V[b]      (softmax over keys)
//
// Q: [batch][Lq][128], K, V: [batch][Lk][128], bf16, row-major; O bf16.  The
// score matrix S never leaves the chip: per 128-query tile, S blocks of 128
// keys live in Tensor Memory, the probabilities P in shared memory, and the
// output accumulates in Tensor Memory with the running-maximum rescale of
// the online softmax.  This is the fused form of the attention pair the
// pages build from two batched products ("Triton Optimization Reference
// (cuTile -> Triton)": attention-style contractions; "FLA Triton -> Gluon
// porting", section 4: tcgen05 with Tensor Memory accumulators, section 5:
// warp specialisation).
//
// Per CTA (persistent, one 128-query tile at a time, 320 threads):
//   warp 0      TMA: Q (two 64-column halves) once per tile; K_j and V_j
//               (128 keys each) into two K slots and two V slots, V one block
//               behind K.  A K slot is refilled once its S MMAs are done, a V
//               slot once its P V MMAs are done.
//   warp 1      one lane issues tcgen05.mma: S_j = Q K_j^T (both operands
//               K-major) into S[j%2], one block ahead of O += P_j V_j (V read
//               MN-major: its rows are keys, the contiguous index is the head
//               dimension) into the tile's O buffer (O[t%2] for tile t).
//   warps 2..9  softmax: two warpgroups, one query row per thread in each;
//               warpgroup w owns keys [64w, 64w+64) of every block and head
//               columns [64w, 64w+64) of O.  Both read the whole S row for its
//               maximum (so they agree on it without exchanging), then each
//               writes p = exp2(s*alpha*log2e - m) for its 64 keys into P[j%2]
//               as bf16 in the swizzled K-major layout the MMA reads.
//
// Lazy rescale: m is the largest scaled score seen when O was last rescaled.
// A block whose maximum exceeds m by more than 8 (in log2 units) first waits
// for the previous P V product, multiplies the row's O (in Tensor Memory) and
// l by exp2(m_old - m_new) and moves m; otherwise p = exp2(s - m) <= 2^8 and
// nothing is rescaled.  The result is the same softmax: only the common
// factor exp2(-m) of numerator and denominator differs.
#pragma once

#include "bmm_kernel.cuh"

namespace dmt {

constexpr int kAttnD = 128;        // head dimension (two 64-wide swizzle atoms)
constexpr int kAttnM = 128;        // query rows per tile
constexpr int kAttnN = 128;        // keys per block
constexpr int kAttnThreads = 320;  // TMA warp, MMA warp, two softmax warpgroups
constexpr uint32_t kAttnHalf = 128u * 128u;       // one 64-column half of 128 rows: 16 KB
constexpr uint32_t kAttnTile = 2u * kAttnHalf;    // Q, P, K or V tile: 32 KB
constexpr uint32_t kAttnBarBytes = 256;
constexpr uint32_t kAttnXchBytes = 2u * 128u * 4u;  // per-row partial sums of both warpgroups
// Q, P[2], K[2], V[2]
constexpr uint32_t kAttnSmem = 1024 + 7 * kAttnTile + kAttnBarBytes + kAttnXchBytes;
static_assert(kAttnSmem <= 232448, "shared memory per CTA");
constexpr float kAttnRescaleLog2 = 8.0f;  // lazy-rescale threshold

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

// Warp-uniform bounded wait: lane 0 polls, the warp follows its verdict (and
// is ordered after lane 0's acquire by the closing __syncwarp).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Abort& ab,
                                          uint32_t site, int lane) {
  int w = 1;
  if (lane == 0) w = wait_bounded<true>(bar, parity, ab, site) ? 1 : 0;
  w = __shfl_sync(0xffffffffu, w, 0);
  __syncwarp();
  return w != 0;
}

// Extreme (kMin: smallest, else largest) of acc and 32 raw scores, of which
// only the first `valid` count (all of them when valid >= 32).
template <bool kMin>
__device__ __forceinline__ float extreme32(const float (&v)[32], int valid, float acc) {
  const float init = kMin ? INFINITY : -INFINITY;
  float a = acc, b = init;
  if (valid >= 32) {
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      a = kMin ? min3(a, v[e], v[e + 1]) : max3(a, v[e], v[e + 1]);
      b = kMin ? min3(b, v[e + 2], v[e + 3]) : max3(b, v[e + 2], v[e + 3]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (e < valid) a = kMin ? fminf(a, v[e]) : fmaxf(a, v[e]);
  }
  return kMin ? fminf(a, b) : fmaxf(a, b);
}

// Largest alpha * log2(e) * s over the valid keys of this thread's row of an
// S block (128 columns at taddr); the warpgroup's own 64 columns (at
// own_col) are kept in `mine`.  kMin: alpha < 0, so the smallest raw score
// gives the largest scaled one.
template <bool kMin>
__device__ __forceinline__ float row_max_scaled(uint32_t taddr, uint32_t own_col, int valid,
                                                float sc, float (&mine)[2][32]) {
  float acc = kMin ? INFINITY : -INFINITY;
#pragma unroll
  for (int h = 0; h < 2; ++h) tmem_ld_32cols(taddr + own_col + 32u * h, mine[h]);
  tmem_wait_ld();
#pragma unroll
  for (int h = 0; h < 2; ++h)
    acc = extreme32<kMin>(mine[h], valid - static_cast<int>(own_col) - 32 * h, acc);
  const uint32_t other = own_col ^ 64u;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    float v[32];
    tmem_ld_32cols(taddr + other + 32u * h, v);
    tmem_wait_ld();
    acc = extreme32<kMin>(v, valid - static_cast<int>(other) - 32 * h, acc);
  }
  return acc * sc;  // at least one key of the block is valid: finite
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const uint32_t q_addr = sbase;
  uint8_t* p_tile = smem + kAttnTile;
  const uint32_t p_addr = sbase + kAttnTile;            // P[0], P[1]
  const uint32_t k_addr = sbase + 3 * kAttnTile;        // K[0], K[1]
  const uint32_t v_addr = sbase + 5 * kAttnTile;        // V[0], V[1]
  const uint32_t bar0 = sbase + 7 * kAttnTile;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 7 * kAttnTile + 224u);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  float* xch = reinterpret_cast<float*>(smem + 7 * kAttnTile + kAttnBarBytes);  // [2][128]

  // barriers (8 bytes each)
  const uint32_t q_full = bar0, q_empty = bar0 + 8;
  auto k_full = [&](uint32_t s) { return bar0 + 16 + 8 * s; };
  auto k_empty = [&](uint32_t s) { return bar0 + 32 + 8 * s; };
  auto v_full = [&](uint32_t s) { return bar0 + 48 + 8 * s; };
  auto v_empty = [&](uint32_t s) { return bar0 + 64 + 8 * s; };
  auto s_full = [&](uint32_t s) { return bar0 + 80 + 8 * s; };
  auto s_empty = [&](uint32_t s) { return bar0 + 96 + 8 * s; };
  const uint32_t p_ready = bar0 + 112;
  auto p_free = [&](uint32_t s) { return bar0 + 120 + 8 * s; };  // the P V of a block is done
  auto o_full = [&](uint32_t s) { return bar0 + 136 + 8 * s; };
  auto o_empty = [&](uint32_t s) { return bar0 + 152 + 8 * s; };
  const uint32_t xch_bar = bar0 + 168;   // both warpgroups' partial sums are written
  const uint32_t xch_read = bar0 + 176;  // ... and read: the slots may take the next tile's
  const uint32_t drain_bar = bar0 + 184;
  constexpr uint32_t kSoftmaxWarps = 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (uint32_t s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), kSoftmaxWarps);
      mbar_init(p_free(s), 1);
      mbar_init(o_full(s), 1);
      mbar_init(o_empty(s), kSoftmaxWarps);
    }
    mbar_init(p_ready, kSoftmaxWarps);
    mbar_init(xch_bar, kSoftmaxWarps);
    mbar_init(xch_read, kSoftmaxWarps);
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
      uint32_t gk = 0, gv = 0, ti = 0;  // K blocks, V blocks, tiles loaded
      bool ok = true;
      auto load_v = [&](int b, int j) -> bool {
        const uint32_t s = gv & 1u;
        if (!wait_bounded<true>(v_empty(s), ((gv >> 1) & 1u) ^ 1u, ab, kSiteProducerEmpty)) return false;
        mbar_arrive_expect_tx(v_full(s), kAttnTile);
        tma_load_3d(v_addr + s * kAttnTile, &tmV, v_full(s), 0, j * kAttnN, b);
        tma_load_3d(v_addr + s * kAttnTile + kAttnHalf, &tmV, v_full(s), 64, j * kAttnN, b);
        ++gv;
        return true;
      };
      for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
        const int b = static_cast<int>(item / p.q_tiles);
        const int q0 = static_cast<int>(item % p.q_tiles) * kAttnM;
        if (!wait_bounded<true>(q_empty, (ti & 1u) ^ 1u, ab, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(q_full, kAttnTile);
        tma_load_3d(q_addr, &tmQ, q_full, 0, q0, b);
        tma_load_3d(q_addr + kAttnHalf, &tmQ, q_full, 64, q0, b);
        // K_j, then V_{j-1}: a K slot frees as soon as its S is computed
        for (int j = 0; j < nb && ok; ++j) {
          const uint32_t s = gk & 1u;
          if (!wait_bounded<true>(k_empty(s), ((gk >> 1) & 1u) ^ 1u, ab, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(k_full(s), kAttnTile);
          tma_load_3d(k_addr + s * kAttnTile, &tmK, k_full(s), 0, j * kAttnN, b);
          tma_load_3d(k_addr + s * kAttnTile + kAttnHalf, &tmK, k_full(s), 64, j * kAttnN, b);
          ++gk;
          if (j > 0) ok = load_v(b, j - 1);
        }
        if (ok) ok = load_v(b, nb - 1);
      }
      // let this CTA's last loads land before it can exit
      for (uint32_t j = gk > 2u ? gk - 2u : 0u; j < gk; ++j) drain_wait(k_full(j & 1u), (j >> 1) & 1u);
      for (uint32_t j = gv > 2u ? gv - 2u : 0u; j < gv; ++j) drain_wait(v_full(j & 1u), (j >> 1) & 1u);
      if (ti > 0) drain_wait(q_full, (ti - 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t hi_sw = desc_hi_sw128(1024u);
      const uint32_t q_lo = desc_lo(q_addr, 16u);
      const uint32_t p_lo = desc_lo(p_addr, 16u);
      uint32_t gk = 0, gs = 0, ti = 0;  // P V blocks issued, S blocks issued, tiles
      bool ok = !p.test_stall || wait_bounded(drain_bar, 0u, ab, kSiteTestStall);
      // S_g = Q K_g^T: k-steps 0..3 in the first 64-column halves, 4..7 in the second.
      auto issue_s = [&](uint32_t g) -> bool {
        const uint32_t s = g & 1u, ph = (g >> 1) & 1u;
        if (!wait_bounded<true>(k_full(s), ph, ab, kSiteMmaFull)) return false;
        if (!wait_bounded<true>(s_empty(s), ph ^ 1u, ab, kSiteMmaAccEmpty)) return false;
        tc_fence_after_sync();
        const uint32_t k_lo = desc_lo(k_addr + s * kAttnTile, 16u);
        const uint32_t d_tmem = tmem_base + s * 128u;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * (kAttnHalf >> 4) + (ks & 3) * 2;  // (bytes >> 4)
          tc_mma_f16(d_tmem, desc_join(q_lo + off, hi_sw), desc_join(k_lo + off, hi_sw), p.idesc_s,
                     ks > 0 ? 1u : 0u);
        }
        tc_commit(s_full(s));
        tc_commit(k_empty(s));
        return true;
      };
      for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
        const uint32_t ob = ti & 1u;
        if (!wait_bounded<true>(q_full, ti & 1u, ab, kSiteMmaFull)) break;
        for (int j = 0; j < nb && ok; ++j, ++gk) {
          if (j == 0) ok = issue_s(gs++);
          if (ok && j + 1 < nb) ok = issue_s(gs++);
          if (!ok) break;
          if (j + 1 == nb) tc_commit(q_empty);  // Q is free once every S of this tile is done
          const uint32_t s = gk & 1u, ph = (gk >> 1) & 1u;
          if (!wait_bounded<true>(p_ready, gk & 1u, ab, kSiteMmaFull) ||
              (j == 0 && !wait_bounded<true>(o_empty(ob), ((ti >> 1) & 1u) ^ 1u, ab, kSiteMmaAccEmpty)) ||
              !wait_bounded<true>(v_full(s), ph, ab, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // O += P_g V_g: P K-major over keys (two 64-key halves); V MN-major
          // (64-column halves of the head dimension 16 KB apart, 8 key rows per
          // 1024-byte group, 16 keys = 2048 bytes per k-step).
          const uint32_t v_lo = desc_lo(v_addr + s * kAttnTile, kAttnHalf);
          const uint32_t d_tmem = tmem_base + 256u + ob * 128u;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t poff = (ks >> 2) * (kAttnHalf >> 4) + (ks & 3) * 2;
            tc_mma_f16(d_tmem, desc_join(p_lo + s * (kAttnTile >> 4) + poff, hi_sw),
                       desc_join(v_lo + ks * 128u, hi_sw), p.idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(p_free(s));
          tc_commit(v_empty(s));
          if (j + 1 == nb) tc_commit(o_full(ob));
        }
      }
      tc_commit(drain_bar);
      drain_wait(drain_bar, 0u);
    }
  } else {
    // --------------------------------------------------------- softmax
    const int wg = (warp - 2) >> 2;               // key half / O column half owned
    const int quad = warp & 3;                    // TMEM lane quarter this warp may access
    const int row = quad * 32 + lane;             // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t own_col = static_cast<uint32_t>(wg) * 64u;
    const float sc = p.scale_log2;
    uint32_t g = 0, ti = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
      const uint32_t ob = ti & 1u;
      const uint32_t o_col = 256u + ob * 128u + own_col;
      const int b = static_cast<int>(item / p.q_tiles);
      const int qi = static_cast<int>(item % p.q_tiles) * kAttnM + row;
      float m = 0.0f, l = 0.0f;
      for (int j = 0; j < nb; ++j, ++g) {
        const uint32_t s = g & 1u, ph = (g >> 1) & 1u;
        const int valid = p.Lk - j * kAttnN < 128 ? p.Lk - j * kAttnN : 128;
        if (!(ok = warp_wait(s_full(s), ph, ab, kSiteEpiAccFull, lane))) break;
        tc_fence_after_sync();
        float mine[2][32];
        const uint32_t taddr = tmem_base + lane_off + s * 128u;
        const float m_blk = sc >= 0.0f ? row_max_scaled<false>(taddr, own_col, valid, sc, mine)
                                       : row_max_scaled<true>(taddr, own_col, valid, sc, mine);
        // this S buffer is no longer needed: the next-but-one S may overwrite it
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty(s));
        bool grow = false;
        if (j == 0) {
          m = m_blk;
        } else {
          grow = m_blk > m + kAttnRescaleLog2;
        }
        if (__any_sync(0xffffffffu, grow)) {
          // rescale O and l by exp2(m_old - m_new) in the rows that need it,
          // after the previous block's product has landed in O
          const uint32_t h = g - 1;
          if (!(ok = warp_wait(p_free(h & 1u), (h >> 1) & 1u, ab, kSiteEpiAccFull, lane))) break;
          tc_fence_after_sync();
          const float r = grow ? fast_exp2(m - m_blk) : 1.0f;
          if (grow) {
            l *= r;
            m = m_blk;
          }
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            float v[32];
            tmem_ld_32cols(tmem_base + lane_off + o_col + 32u * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e += 2) fma2(v[e], v[e + 1], v[e], v[e + 1], r, r, 0.0f, 0.0f);
            tmem_st_32cols(tmem_base + lane_off + o_col + 32u * c, v);
          }
          tmem_wait_st();
        }
        if (g >= 2) {  // the product of block g - 2 must have read this P buffer
          if (!(ok = warp_wait(p_free(s), ph ^ 1u, ab, kSiteEpiAccFull, lane))) break;
        }
        // p for this warpgroup's 64 keys, into its 16 KB half of P[s]
        const float nm = -m;
        const int my_valid = valid - static_cast<int>(own_col);
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
        uint8_t* prow = p_tile + s * kAttnTile + wg * kAttnHalf + row * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float (&v)[32] = mine[h];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            fma2(v[e], v[e + 1], v[e], v[e + 1], sc, sc, nm, nm);
            v[e] = fast_exp2(v[e]);
            v[e + 1] = fast_exp2(v[e + 1]);
          }
          if (my_valid < 64) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * h + e >= my_valid) v[e] = 0.0f;
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
            const int chunk = h * 4 + k;
            *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) =
                make_uint4(wds[0], wds[1], wds[2], wds[3]);
          }
        }
        // l sums the unrounded p: the bf16 rounding then perturbs only the
        // numerator of O = (P V) / l, by at most 2^-8 sum_c p_c |V_c| / l
        l += (s0 + s1) + (s2 + s3);
        fence_proxy_async_shared();  // P is read by the tensor core (async proxy)
        tc_fence_before_sync();      // and any rescale of O precedes the next product
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready);
      }
      if (!ok) break;
      // both warpgroups' partial sums of this row; then O / l for own columns
      if (ti > 0 && !(ok = warp_wait(xch_read, (ti - 1) & 1u, ab, kSiteEpiAccFull, lane))) break;
      xch[wg * 128 + row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(xch_bar);
      if (!(ok = warp_wait(xch_bar, ti & 1u, ab, kSiteEpiAccFull, lane))) break;
      const float l_all = l + xch[(wg ^ 1) * 128 + row];
      __syncwarp();
      if (lane == 0) mbar_arrive(xch_read);
      if (!(ok = warp_wait(o_full(ob), (ti >> 1) & 1u, ab, kSiteEpiAccFull, lane))) break;
      tc_fence_after_sync();
      const float inv = 1.0f / l_all;
      __nv_bfloat16* dst =
          p.O + static_cast<int64_t>(b) * p.so + static_cast<int64_t>(qi) * p.ldo + own_col;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float v[32];
        tmem_ld_32cols(tmem_base + lane_off + o_col + 32u * c, v);
        tmem_wait_ld();
        if (c == 1) {  // this O buffer may take the tile after next
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_empty(ob));
        }
        if (qi < p.Lq) {
#pragma unroll
          for (int d = 0; d < 32; d += 8) {
            uint32_t wds[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const __nv_bfloat162 h2 =
                  __floats2bfloat162_rn(v[d + 2 * e2] * inv, v[d + 2 * e2 + 1] * inv);
              wds[e2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(dst + 32 * c + d) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
          }
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

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
// Per CTA (persistent, 320 threads) one item = 256 query rows of one batch
// entry, as two 128-row tiles X = A, B that share every K/V block:
//   warp 0      TMA: Q_A and Q_B (two 64-column halves each) once per item;
//               K_j and V_j (128 keys each) into two K slots and two V slots,
//               V one block behind K.
//   warp 1      one lane issues tcgen05.mma in ping-pong order
//                 S_A(0), S_B(0), then per block j:
//                 O_A += P_A(j) V_j, S_A(j+1), O_B += P_B(j) V_j, S_B(j+1)
//               S_X = Q_X K_j^T (both operands K-major, from shared memory);
//               P_X V_j reads P_X from Tensor Memory and V MN-major from
//               shared memory.  While one warpgroup works on its scores the
//               tensor core works on the other tile.
//   warps 2..9  softmax: warpgroup X (warps 2..5: A, 6..9: B), one query row
//               per thread.  It reads its row of S_X, takes the row maximum,
//               writes p = exp2(s*alpha*log2e - m) as bf16 pairs over the
//               first 64 columns of S_X (P_X), and at the end of the item
//               stores its 128 rows of O_X / l.
// Tensor Memory: S_A, S_B, O_A, O_B, 128 columns each.  The commit that
// signals S_X(j) also covers P_X(j-1) V_{j-1} (a commit tracks every MMA
// issued before it), so when a warpgroup sees its scores, O_X is final for
// the previous block and the columns it overwrites with P are free.
//
// Lazy rescale: m is the largest scaled score seen when O_X was last
// rescaled.  A block whose maximum exceeds m by more than 8 (in log2 units)
// multiplies the row's O_X (in Tensor Memory) and l by exp2(m_old - m_new)
// and moves m; otherwise p = exp2(s - m) <= 2^8 and nothing is rescaled.
// Either way the result is the same softmax: only the common factor of
// numerator and denominator differs.
#pragma once

#include "bmm_kernel.cuh"

namespace dmt {

constexpr int kAttnD = 128;        // head dimension (two 64-wide swizzle atoms)
constexpr int kAttnM = 128;        // query rows per tile
constexpr int kAttnItemRows = 256; // query rows per item: two tiles
constexpr int kAttnN = 128;        // keys per block
constexpr int kAttnThreads = 320;  // TMA warp, MMA warp, two softmax warpgroups
constexpr uint32_t kAttnHalf = 128u * 128u;       // one 64-column half of 128 rows: 16 KB
constexpr uint32_t kAttnTile = 2u * kAttnHalf;    // Q, K or V tile: 32 KB
constexpr uint32_t kAttnBarBytes = 256;
// Q_A, Q_B, K[2], V[2]
constexpr uint32_t kAttnSmem = 1024 + 6 * kAttnTile + kAttnBarBytes;
static_assert(kAttnSmem <= 232448, "shared memory per CTA");
constexpr float kAttnRescaleLog2 = 8.0f;  // lazy-rescale threshold

struct AttnParams {
  int32_t Lq, Lk;
  int32_t q_tiles;        // items per batch entry: ceil(Lq / 256)
  int32_t k_blocks;       // ceil(Lk / 128)
  int64_t items;          // batch * q_tiles
  float scale_log2;       // alpha * log2(e)
  uint32_t idesc_s;       // 128 x 128, bf16, A and B K-major
  uint32_t idesc_o;       // 128 x 128, bf16, A (in Tensor Memory) K-major, B MN-major
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

// Loads this thread's row of an S block (128 columns at taddr) into `v` with
// one wait, and returns the largest alpha * log2(e) * s over its valid keys.
// kMin: alpha < 0, so the smallest raw score gives the largest scaled one.
template <bool kMin>
__device__ __forceinline__ float row_max_scaled(uint32_t taddr, int valid, float sc,
                                                float (&v)[4][32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld_32cols(taddr + 32u * c, v[c]);
  tmem_wait_ld();
  float acc = kMin ? INFINITY : -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c) acc = extreme32<kMin>(v[c], valid - 32 * c, acc);
  return acc * sc;  // at least one key of the block is valid: finite
}

// p = exp2(s * sc - m) for 32 keys of the row (key0 = their first index
// within the block; keys from `valid` on are zero), summed into (s0..s3) and
// packed as bf16 pairs (lower key in the low half) into 16 words.
__device__ __forceinline__ void exp_pack(float (&v)[32], int key0, int valid, float sc, float nm,
                                         float* w, float& s0, float& s1, float& s2, float& s3) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    fma2(v[e], v[e + 1], v[e], v[e + 1], sc, sc, nm, nm);
    v[e] = fast_exp2(v[e]);
    v[e + 1] = fast_exp2(v[e + 1]);
  }
  if (valid < key0 + 32) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (key0 + e >= valid) v[e] = 0.0f;
  }
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    add2(s0, s1, v[e], v[e + 1]);
    add2(s2, s3, v[e + 2], v[e + 3]);
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
    w[e] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h2));
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const uint32_t q_addr = sbase;                        // Q_A, Q_B
  const uint32_t k_addr = sbase + 2 * kAttnTile;        // K[0], K[1]
  const uint32_t v_addr = sbase + 4 * kAttnTile;        // V[0], V[1]
  const uint32_t bar0 = sbase + 6 * kAttnTile;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 6 * kAttnTile + 224u);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  // barriers (8 bytes each); X = tile A (0) or B (1)
  const uint32_t q_full = bar0, q_empty = bar0 + 8;
  auto k_full = [&](uint32_t s) { return bar0 + 16 + 8 * s; };
  auto k_empty = [&](uint32_t s) { return bar0 + 32 + 8 * s; };
  auto v_full = [&](uint32_t s) { return bar0 + 48 + 8 * s; };
  auto v_empty = [&](uint32_t s) { return bar0 + 64 + 8 * s; };
  auto s_full = [&](uint32_t x) { return bar0 + 80 + 8 * x; };   // S_X(j) and P_X(j-1) V done
  auto p_ready = [&](uint32_t x) { return bar0 + 96 + 8 * x; };  // P_X(j) written
  auto o_full = [&](uint32_t x) { return bar0 + 112 + 8 * x; };  // the item's last P_X V done
  auto o_empty = [&](uint32_t x) { return bar0 + 128 + 8 * x; }; // O_X read out
  const uint32_t drain_bar = bar0 + 144;
  constexpr uint32_t kGroupWarps = 4;

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
      mbar_init(p_ready(s), kGroupWarps);
      mbar_init(o_full(s), 1);
      mbar_init(o_empty(s), kGroupWarps);
    }
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
    tmem_alloc(smem_addr(tmem_slot), 512);  // S_A, S_B, O_A, O_B: 128 columns each
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
      uint32_t gk = 0, gv = 0, ti = 0;  // K blocks, V blocks, items loaded
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
        const int q0 = static_cast<int>(item % p.q_tiles) * kAttnItemRows;
        if (!wait_bounded<true>(q_empty, (ti & 1u) ^ 1u, ab, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(q_full, 2 * kAttnTile);
        tma_load_3d(q_addr, &tmQ, q_full, 0, q0, b);
        tma_load_3d(q_addr + kAttnHalf, &tmQ, q_full, 64, q0, b);
        tma_load_3d(q_addr + kAttnTile, &tmQ, q_full, 0, q0 + kAttnM, b);
        tma_load_3d(q_addr + kAttnTile + kAttnHalf, &tmQ, q_full, 64, q0 + kAttnM, b);
        // K_j, then V_{j-1}: a K slot frees as soon as both S of its block are done
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
      uint32_t gs = 0, gv = 0, ti = 0;  // K blocks used by S, V blocks used by P V, items
      bool ok = !p.test_stall || wait_bounded(drain_bar, 0u, ab, kSiteTestStall);
      // S_X = Q_X K^T into S_X: k-steps 0..3 in the first 64-column halves,
      // 4..7 in the second.
      auto issue_s = [&](uint32_t x, uint32_t ks_) {
        const uint32_t k_lo = desc_lo(k_addr + ks_ * kAttnTile, 16u);
        const uint32_t qx = q_lo + x * (kAttnTile >> 4);
        const uint32_t d_tmem = tmem_base + x * 128u;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * (kAttnHalf >> 4) + (ks & 3) * 2;  // (bytes >> 4)
          tc_mma_f16(d_tmem, desc_join(qx + off, hi_sw), desc_join(k_lo + off, hi_sw), p.idesc_s,
                     ks > 0 ? 1u : 0u);
        }
        tc_commit(s_full(x));
      };
      // both S of the next K block, once it has landed
      auto issue_s_pair_half = [&](uint32_t x) -> bool {
        const uint32_t ks_ = gs & 1u;
        if (x == 0 && !wait_bounded<true>(k_full(ks_), (gs >> 1) & 1u, ab, kSiteMmaFull)) return false;
        issue_s(x, ks_);
        if (x == 1) {
          tc_commit(k_empty(ks_));
          ++gs;
        }
        return true;
      };
      // O_X (+)= P_X V: P from the first 64 columns of S_X (8 per k-step), V
      // MN-major (64-column halves 16 KB apart, 16 keys = 2048 bytes per k-step)
      auto issue_pv = [&](uint32_t x, uint32_t vs, bool first) {
        const uint32_t v_lo = desc_lo(v_addr + vs * kAttnTile, kAttnHalf);
        const uint32_t d_tmem = tmem_base + 256u + x * 128u;
        const uint32_t a_tmem = tmem_base + x * 128u;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma_f16_ts(d_tmem, a_tmem + 8u * ks, desc_join(v_lo + ks * 128u, hi_sw), p.idesc_o,
                        (!first || ks > 0) ? 1u : 0u);
      };
      for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
        if (!wait_bounded<true>(q_full, ti & 1u, ab, kSiteMmaFull)) break;
        ok = issue_s_pair_half(0u) && issue_s_pair_half(1u);
        if (ok && nb == 1) tc_commit(q_empty);  // Q is free once every S of the item is done
        for (int j = 0; j < nb && ok; ++j) {
          const uint32_t vs = gv & 1u, vph = (gv >> 1) & 1u;
          // P_X(j) is warpgroup X's (ti * nb + j)-th block: every item has nb blocks
          const uint32_t pph = (ti * static_cast<uint32_t>(nb) + static_cast<uint32_t>(j)) & 1u;
          for (uint32_t x = 0; x < 2 && ok; ++x) {
            // V and O first, the softmax's release last: each wait costs the
            // MMA thread a barrier round trip, and only the last one sits
            // between the release and the next MMA.  The release is awaited
            // asleep (a suspend-time hint): the barrier's completion wakes the
            // thread sooner than its next poll would see it.
            if ((x == 0 && !wait_bounded<true>(v_full(vs), vph, ab, kSiteMmaFull)) ||
                (j == 0 && !wait_bounded<true>(o_empty(x), (ti & 1u) ^ 1u, ab, kSiteMmaAccEmpty)) ||
                !(mbar_try_wait_hint(p_ready(x), pph, 500u) ||
                  wait_bounded<true>(p_ready(x), pph, ab, kSiteMmaFull))) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_pv(x, vs, j == 0);
            if (j + 1 == nb) tc_commit(o_full(x));
            if (x == 1) tc_commit(v_empty(vs));
            if (j + 1 < nb) {
              if (!(ok = issue_s_pair_half(x))) break;
              if (x == 1 && j + 2 == nb) tc_commit(q_empty);
            }
          }
          ++gv;
        }
      }
      tc_commit(drain_bar);
      drain_wait(drain_bar, 0u);
    }
  } else {
    // --------------------------------------------------------- softmax
    const uint32_t x = static_cast<uint32_t>(warp - 2) >> 2;  // tile A (0) or B (1)
    const int quad = warp & 3;                    // TMEM lane quarter this warp may access
    const int row = quad * 32 + lane;             // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_col = tmem_base + lane_off + x * 128u;          // S_X, and P_X over it
    const uint32_t o_col = tmem_base + lane_off + 256u + x * 128u;   // O_X
    const float sc = p.scale_log2;
    uint32_t n = 0, ti = 0;  // blocks done, items
    bool ok = true;
    for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
      const int b = static_cast<int>(item / p.q_tiles);
      const int qi = static_cast<int>(item % p.q_tiles) * kAttnItemRows + static_cast<int>(x) * kAttnM + row;
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < nb; ++j, ++n) {
        const int valid = p.Lk - j * kAttnN < 128 ? p.Lk - j * kAttnN : 128;
        if (!(ok = warp_wait(s_full(x), n & 1u, ab, kSiteEpiAccFull, lane))) break;
        tc_fence_after_sync();
        // this thread's whole 128-column row of S: one Tensor Memory round trip
        float v[4][32];
        const float m_blk = sc >= 0.0f ? row_max_scaled<false>(s_col, valid, sc, v)
                                       : row_max_scaled<true>(s_col, valid, sc, v);
        const bool grow = j > 0 && m_blk > m + kAttnRescaleLog2;
        if (j == 0) m = m_blk;
        if (__any_sync(0xffffffffu, grow)) {
          // rescale O_X and l by exp2(m_old - m_new) in the rows that need it
          // (O_X is final for the previous block: see the header)
          const float r = grow ? fast_exp2(m - m_blk) : 1.0f;
          if (grow) {
            l *= r;
            m = m_blk;
          }
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float o[16];
            tmem_ld_16cols(o_col + 16u * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e += 2) fma2(o[e], o[e + 1], o[e], o[e + 1], r, r, 0.0f, 0.0f);
            tmem_st_16cols(o_col + 16u * c, o);
          }
          tmem_wait_st();
        }
        // P over the first 64 columns of S_X (keys 32c..32c+31 into columns
        // 16c..16c+15): every score is already in registers
        const float nm = -m;
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float w[16];
          exp_pack(v[c], 32 * c, valid, sc, nm, w, s0, s1, s2, s3);
          tmem_st_16cols(s_col + 16u * c, w);
        }
        // l sums the unrounded p: the bf16 rounding then perturbs only the
        // numerator of O = (P V) / l, by at most 2^-8 sum_c p_c |V_c| / l
        l += (s0 + s1) + (s2 + s3);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready(x));
      }
      if (!ok) break;
      // O_X / l for this row, once the item's last product has landed
      if (!(ok = warp_wait(o_full(x), ti & 1u, ab, kSiteEpiAccFull, lane))) break;
      tc_fence_after_sync();
      const float inv = 1.0f / l;
      __nv_bfloat16* dst = p.O + static_cast<int64_t>(b) * p.so + static_cast<int64_t>(qi) * p.ldo;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float o[16];
        tmem_ld_16cols(o_col + 16u * c, o);
        tmem_wait_ld();
        if (c == 7) {  // O_X may take the next item
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_empty(x));
        }
        if (qi < p.Lq) {
#pragma unroll
          for (int d = 0; d < 16; d += 8) {
            uint32_t wds[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const __nv_bfloat162 h2 =
                  __floats2bfloat162_rn(o[d + 2 * e2] * inv, o[d + 2 * e2 + 1] * inv);
              wds[e2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(dst + 16 * c + d) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
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

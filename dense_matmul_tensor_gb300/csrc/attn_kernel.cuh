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
//               K-major) into S[j%2], two blocks ahead of O[j%2] += P_j V_j
//               (V read MN-major: its rows are keys, the contiguous index is
//               the head dimension): S_{j+2} goes out as soon as block j's
//               softmax has read S_j, so a warpgroup finds its next S ready.
//   warps 2..9  softmax: two warpgroups, one query row per thread in each.
//               Warpgroup w takes the blocks j = w (mod 2) of every tile with
//               its own S[w], P[w] and output accumulator O[w], running
//               maximum m_w and sum l_w, so the two run staggered: one's
//               exponentials overlap the other's reads and waits.  Each reads
//               its S row, writes p = exp2(s*alpha*log2e - m_w) as bf16 into
//               P[w] in the swizzled K-major layout the MMA reads.  At the end
//               of a tile the two halves are merged,
//                 O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)),
//               m = max(m_0, m_1): warpgroup 1 hands (m_1, l_1) to warpgroup
//               0, which returns both coefficients, and each warpgroup stores
//               64 of the row's 128 columns.
//
// Lazy rescale: m_w is the largest scaled score seen when O[w] was last
// rescaled.  A block whose maximum exceeds m_w by more than 8 (in log2 units)
// multiplies the row's O[w] (in Tensor Memory) and l_w by exp2(m_old - m_new)
// and moves m_w; otherwise p = exp2(s - m_w) <= 2^8 and nothing is rescaled.
// Either way the result is the same softmax: only the common factor of
// numerator and denominator differs.
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
constexpr uint32_t kAttnXchBytes = 2u * 128u * 4u;  // per row: (m_1, l_1), then the coefficients
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
// S block (128 columns at taddr); the first 64 scores stay in `v`.  kMin:
// alpha < 0, so the smallest raw score gives the largest scaled one.
template <bool kMin>
__device__ __forceinline__ float row_max_scaled(uint32_t taddr, int valid, float sc,
                                                float (&v)[2][32]) {
  float acc = kMin ? INFINITY : -INFINITY;
  {  // the second half first: it is read again later
    float u[2][32];
    tmem_ld_32cols(taddr + 64u, u[0]);
    tmem_ld_32cols(taddr + 96u, u[1]);
    tmem_wait_ld();
    acc = extreme32<kMin>(u[0], valid - 64, acc);
    acc = extreme32<kMin>(u[1], valid - 96, acc);
  }
  tmem_ld_32cols(taddr, v[0]);
  tmem_ld_32cols(taddr + 32u, v[1]);
  tmem_wait_ld();
  acc = extreme32<kMin>(v[0], valid, acc);
  acc = extreme32<kMin>(v[1], valid - 32, acc);
  return acc * sc;  // at least one key of the block is valid: finite
}

// p = exp2(s * sc - m) for 32 keys of the row (key0 = their first index
// within the block; keys from `valid` on are zero), summed into (s0..s3) and
// written as bf16 into the row of P (128-byte rows, two 64-key halves 16 KB
// apart, 16-byte chunks XOR-swizzled by row % 8 as TMA's 128-byte swizzle
// places them).
__device__ __forceinline__ void exp_chunk(float (&v)[32], int key0, int valid, float sc, float nm,
                                          uint8_t* prow, int row, float& s0, float& s1, float& s2,
                                          float& s3) {
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
  const int c = key0 >> 5;
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // one 16-byte chunk: 8 keys
    uint32_t wds[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * k + 2 * e2], v[8 * k + 2 * e2 + 1]);
      wds[e2] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    const int chunk = (c & 1) * 4 + k;
    *reinterpret_cast<uint4*>(prow + (c >> 1) * kAttnHalf + ((chunk ^ (row & 7)) << 4)) =
        make_uint4(wds[0], wds[1], wds[2], wds[3]);
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
  // per warpgroup w: S[w], P[w] and O[w]
  auto s_full = [&](uint32_t w) { return bar0 + 80 + 8 * w; };
  auto s_empty = [&](uint32_t w) { return bar0 + 96 + 8 * w; };
  auto p_ready = [&](uint32_t w) { return bar0 + 112 + 8 * w; };
  auto p_free = [&](uint32_t w) { return bar0 + 128 + 8 * w; };  // its last P V is done
  const uint32_t o_full = bar0 + 144;    // the tile's last P V is done
  const uint32_t o_empty = bar0 + 152;   // both O buffers have been read
  const uint32_t xch_up = bar0 + 160;    // warpgroup 1's (m, l) are in the slot
  const uint32_t xch_down = bar0 + 168;  // warpgroup 0's merge coefficients are in the slot
  const uint32_t drain_bar = bar0 + 176;
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
      mbar_init(s_empty(s), kGroupWarps);
      mbar_init(p_ready(s), kGroupWarps);
      mbar_init(p_free(s), 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, 2 * kGroupWarps);
    mbar_init(xch_up, kGroupWarps);
    mbar_init(xch_down, kGroupWarps);
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
      uint32_t us0 = 0, us1 = 0, up0 = 0, up1 = 0;  // uses of S[w] and P[w]
      bool ok = !p.test_stall || wait_bounded(drain_bar, 0u, ab, kSiteTestStall);
      // S_j = Q K_j^T into S[j % 2]: k-steps 0..3 in the first 64-column
      // halves, 4..7 in the second.
      auto issue_s = [&](uint32_t w) -> bool {
        const uint32_t ks_ = gs & 1u;
        if (!wait_bounded<true>(k_full(ks_), (gs >> 1) & 1u, ab, kSiteMmaFull)) return false;
        const uint32_t u = w ? us1 : us0;
        if (!wait_bounded<true>(s_empty(w), (u & 1u) ^ 1u, ab, kSiteMmaAccEmpty)) return false;
        tc_fence_after_sync();
        const uint32_t k_lo = desc_lo(k_addr + ks_ * kAttnTile, 16u);
        const uint32_t d_tmem = tmem_base + w * 128u;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * (kAttnHalf >> 4) + (ks & 3) * 2;  // (bytes >> 4)
          tc_mma_f16(d_tmem, desc_join(q_lo + off, hi_sw), desc_join(k_lo + off, hi_sw), p.idesc_s,
                     ks > 0 ? 1u : 0u);
        }
        tc_commit(s_full(w));
        tc_commit(k_empty(ks_));
        if (w) ++us1; else ++us0;
        ++gs;
        return true;
      };
      for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
        if (!wait_bounded<true>(q_full, ti & 1u, ab, kSiteMmaFull)) break;
        // S_0 and S_1 first; then S_{j+2} before P_j V_j
        ok = issue_s(0u) && (nb < 2 || issue_s(1u));
        if (ok && nb <= 2) tc_commit(q_empty);  // Q is free once every S of this tile is done
        for (int j = 0; j < nb && ok; ++j, ++gk) {
          const uint32_t w = static_cast<uint32_t>(j) & 1u;
          if (j + 2 < nb) {
            if (!(ok = issue_s(w))) break;
            if (j + 3 == nb) tc_commit(q_empty);
          }
          const uint32_t vs = gk & 1u;
          if (!wait_bounded<true>(p_ready(w), (w ? up1 : up0) & 1u, ab, kSiteMmaFull) ||
              (j == 0 && !wait_bounded<true>(o_empty, (ti & 1u) ^ 1u, ab, kSiteMmaAccEmpty)) ||
              !wait_bounded<true>(v_full(vs), (gk >> 1) & 1u, ab, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // O[w] += P_j V_j: P K-major over keys (two 64-key halves); V MN-major
          // (64-column halves of the head dimension 16 KB apart, 8 key rows per
          // 1024-byte group, 16 keys = 2048 bytes per k-step).  The tile's
          // first block of each warpgroup starts its O[w] afresh.
          const uint32_t v_lo = desc_lo(v_addr + vs * kAttnTile, kAttnHalf);
          const uint32_t d_tmem = tmem_base + 256u + w * 128u;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t poff = (ks >> 2) * (kAttnHalf >> 4) + (ks & 3) * 2;
            tc_mma_f16(d_tmem, desc_join(p_lo + w * (kAttnTile >> 4) + poff, hi_sw),
                       desc_join(v_lo + ks * 128u, hi_sw), p.idesc_o, (j >= 2 || ks > 0) ? 1u : 0u);
          }
          tc_commit(p_free(w));
          tc_commit(v_empty(vs));
          if (j + 1 == nb) tc_commit(o_full);
          if (w) ++up1; else ++up0;
        }
      }
      tc_commit(drain_bar);
      drain_wait(drain_bar, 0u);
    }
  } else {
    // --------------------------------------------------------- softmax
    const uint32_t wg = static_cast<uint32_t>(warp - 2) >> 2;  // blocks j = wg (mod 2)
    const int quad = warp & 3;                    // TMEM lane quarter this warp may access
    const int row = quad * 32 + lane;             // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_col = lane_off + wg * 128u;           // S[wg]
    const uint32_t o_col = lane_off + 256u + wg * 128u;    // O[wg]
    uint8_t* prow = p_tile + wg * kAttnTile + row * 128;   // this row of P[wg]
    const float sc = p.scale_log2;
    uint32_t n = 0, ti = 0;  // blocks this warpgroup has done, tiles
    bool ok = true;
    for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
      const int b = static_cast<int>(item / p.q_tiles);
      const int qi = static_cast<int>(item % p.q_tiles) * kAttnM + row;
      float m = -INFINITY, l = 0.0f;
      for (int j = static_cast<int>(wg); j < nb; j += 2, ++n) {
        const int valid = p.Lk - j * kAttnN < 128 ? p.Lk - j * kAttnN : 128;
        if (!(ok = warp_wait(s_full(wg), n & 1u, ab, kSiteEpiAccFull, lane))) break;
        tc_fence_after_sync();
        float v[2][32];
        const float m_blk = sc >= 0.0f ? row_max_scaled<false>(tmem_base + s_col, valid, sc, v)
                                       : row_max_scaled<true>(tmem_base + s_col, valid, sc, v);
        // this warpgroup's previous product must be done: P[wg] is then free
        // and O[wg] final until the next product
        if (n > 0 && !(ok = warp_wait(p_free(wg), (n - 1) & 1u, ab, kSiteEpiAccFull, lane))) break;
        const bool first = j < 2;
        const bool grow = !first && m_blk > m + kAttnRescaleLog2;
        if (first) m = m_blk;
        if (__any_sync(0xffffffffu, grow)) {
          // rescale O[wg] and l by exp2(m_old - m_new) in the rows that need it
          tc_fence_after_sync();
          const float r = grow ? fast_exp2(m - m_blk) : 1.0f;
          if (grow) {
            l *= r;
            m = m_blk;
          }
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float o[16];
            tmem_ld_16cols(tmem_base + o_col + 16u * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e += 2) fma2(o[e], o[e + 1], o[e], o[e + 1], r, r, 0.0f, 0.0f);
            tmem_st_16cols(tmem_base + o_col + 16u * c, o);
          }
          tmem_wait_st();
        }
        // p for the block's 128 keys, into P[wg]: the first 64 from registers,
        // the rest read again from S[wg], which is then released
        const float nm = -m;
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
        exp_chunk(v[0], 0, valid, sc, nm, prow, row, s0, s1, s2, s3);
        exp_chunk(v[1], 32, valid, sc, nm, prow, row, s0, s1, s2, s3);
        tmem_ld_32cols(tmem_base + s_col + 64u, v[0]);
        tmem_ld_32cols(tmem_base + s_col + 96u, v[1]);
        tmem_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty(wg));  // the warpgroup's next S may overwrite it
        exp_chunk(v[0], 64, valid, sc, nm, prow, row, s0, s1, s2, s3);
        exp_chunk(v[1], 96, valid, sc, nm, prow, row, s0, s1, s2, s3);
        // l sums the unrounded p: the bf16 rounding then perturbs only the
        // numerator of O = (P V) / l, by at most 2^-8 sum_c p_c |V_c| / l
        l += (s0 + s1) + (s2 + s3);
        fence_proxy_async_shared();  // P is read by the tensor core (async proxy)
        tc_fence_before_sync();      // and any rescale of O precedes the next product
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready(wg));
      }
      if (!ok) break;
      // merge: warpgroup 1 hands over (m_1, l_1); warpgroup 0 returns the
      // coefficients c_w = 2^(m_w - m) / l of both halves
      float* xa = xch;        // per row: m_1, then c_0
      float* xb = xch + 128;  // per row: l_1, then c_1
      const bool two = nb >= 2;  // warpgroup 1 had a block in this tile
      float c0, c1;
      if (wg == 1) {
        xa[row] = m;
        xb[row] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive(xch_up);
        if (!(ok = warp_wait(xch_down, ti & 1u, ab, kSiteEpiAccFull, lane))) break;
        c0 = xa[row];
        c1 = xb[row];
      } else {
        if (!(ok = warp_wait(xch_up, ti & 1u, ab, kSiteEpiAccFull, lane))) break;
        const float m1 = xa[row], l1 = xb[row];
        const float mm = two ? fmaxf(m, m1) : m;
        const float a0 = fast_exp2(m - mm);
        const float a1 = two ? fast_exp2(m1 - mm) : 0.0f;
        const float inv = 1.0f / (l * a0 + l1 * a1);
        c0 = a0 * inv;
        c1 = a1 * inv;
        xa[row] = c0;
        xb[row] = c1;
        __syncwarp();
        if (lane == 0) mbar_arrive(xch_down);
      }
      if (!(ok = warp_wait(o_full, ti & 1u, ab, kSiteEpiAccFull, lane))) break;
      tc_fence_after_sync();
      // this warpgroup's 64 columns of the row: c_0 O_0 + c_1 O_1
      const uint32_t col0 = wg * 64u;
      __nv_bfloat16* dst =
          p.O + static_cast<int64_t>(b) * p.so + static_cast<int64_t>(qi) * p.ldo + col0;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float o0[16], o1[16];
        tmem_ld_16cols(tmem_base + lane_off + 256u + col0 + 16u * c, o0);
        if (two) tmem_ld_16cols(tmem_base + lane_off + 384u + col0 + 16u * c, o1);
        tmem_wait_ld();
        if (c == 3) {  // both O buffers may take the next tile
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_empty);
        }
        if (!two) {
#pragma unroll
          for (int e = 0; e < 16; ++e) o1[e] = 0.0f;
        }
        if (qi < p.Lq) {
#pragma unroll
          for (int d = 0; d < 16; d += 8) {
            uint32_t wds[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const int e = d + 2 * e2;
              float x0, x1;
              fma2(x0, x1, o0[e], o0[e + 1], c0, c0, 0.0f, 0.0f);
              fma2(x0, x1, o1[e], o1[e + 1], c1, c1, x0, x1);
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
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

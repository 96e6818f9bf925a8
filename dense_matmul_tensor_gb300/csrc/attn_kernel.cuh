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
//               shared memory.  While the softmax warps work on one tile's
//               scores the tensor core works on the other tile.
//   warps 2..9  softmax, all eight warps on tile A, then on tile B, per key
//               block.  Warps w and w+4 share a Tensor Memory lane quarter and
//               split each of its 32 rows: w takes keys 0..63 of the block,
//               w+4 keys 64..127.  Each thread reads its 64 scores of S_X,
//               trades its half-row maximum with its partner (a 64-thread
//               named barrier), writes p = exp2(s*alpha*log2e - m) as bf16
//               pairs into columns 32..95 of S_X (P_X; every thread writes
//               only columns it has read), and at the end of the item stores
//               its 64 columns of O_X / l.
// Tensor Memory: S_A, S_B, O_A, O_B, 128 columns each.  The commit that
// signals S_X(j) also covers P_X(j-1) V_{j-1} (a commit tracks every MMA
// issued before it), so when the softmax warps see S_X, O_X is final for
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
constexpr int kAttnThreads = 320;  // TMA warp, MMA warp, eight softmax warps
constexpr uint32_t kAttnHalf = 128u * 128u;       // one 64-column half of 128 rows: 16 KB
constexpr uint32_t kAttnTile = 2u * kAttnHalf;    // Q, K or V tile: 32 KB
constexpr uint32_t kAttnBarBytes = 256;
// Q_A, Q_B, K[2], V[2]
constexpr uint32_t kAttnXchBytes = 2 * 2 * 128 * 8;  // two buffers x two key halves x 128 rows x (value, verdict)
constexpr uint32_t kAttnSmem = 1024 + 6 * kAttnTile + kAttnBarBytes + kAttnXchBytes;
static_assert(kAttnSmem <= 232448, "shared memory per CTA");
constexpr float kAttnRescaleLog2 = 8.0f;  // lazy-rescale threshold
constexpr uint32_t kAttnPCol = 32;        // P_X's first column within S_X
constexpr float kAttnSpecLog2 = 64.0f;    // bound on log2 p before the row maximum is known

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

// Extreme (kMin: smallest, else largest) of 64 scores: eight independent
// chains of four steps, then two merge steps, so the longest dependent chain
// is six instructions (one running extreme over all 64 would be 32).
template <bool kMin>
__device__ __forceinline__ float extreme64(const float (&v)[2][32]) {
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = k >> 2, o = 2 * (k & 3);
    a[k] = kMin ? fminf(v[c][o], v[c][o + 1]) : fmaxf(v[c][o], v[c][o + 1]);
#pragma unroll
    for (int i = 8; i < 32; i += 8)
      a[k] = kMin ? min3(a[k], v[c][i + o], v[c][i + o + 1]) : max3(a[k], v[c][i + o], v[c][i + o + 1]);
  }
  const float x = kMin ? min3(a[0], a[1], a[2]) : max3(a[0], a[1], a[2]);
  const float y = kMin ? min3(a[3], a[4], a[5]) : max3(a[3], a[4], a[5]);
  const float z = kMin ? fminf(a[6], a[7]) : fmaxf(a[6], a[7]);
  return kMin ? min3(x, y, z) : max3(x, y, z);
}

// Loads this thread's half row of an S block (64 columns at taddr) into `v`
// with one wait, and returns the largest alpha * log2(e) * s over its valid
// keys (-inf when the half holds none).  kMin: alpha < 0, so the smallest raw
// score gives the largest scaled one.
template <bool kMin>
__device__ __forceinline__ float half_row_max_scaled(uint32_t taddr, int valid, float sc,
                                                     float (&v)[2][32]) {
  tmem_ld_32cols(taddr, v[0]);
  tmem_ld_32cols(taddr + 32u, v[1]);
  tmem_wait_ld();
  if (valid >= 64) return extreme64<kMin>(v) * sc;
  if (valid <= 0) return -INFINITY;
  float acc = kMin ? INFINITY : -INFINITY;
  acc = extreme32<kMin>(v[0], valid, acc);
  acc = extreme32<kMin>(v[1], valid - 32, acc);
  return acc * sc;
}

// Named barrier `id` over `count` threads (whole warps).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// p = exp2(s * sc - m) in place for the 64 keys of a half row (key0 = the
// first one's index within the block; keys from `valid` on are zero).  All
// 64 exponentials are independent: nothing waits on one before the next.
__device__ __forceinline__ void exp64(float (&v)[2][32], int key0, int valid, float sc, float nm) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      fma2(v[c][e], v[c][e + 1], v[c][e], v[c][e + 1], sc, sc, nm, nm);
      v[c][e] = fast_exp2(v[c][e]);
      v[c][e + 1] = fast_exp2(v[c][e + 1]);
    }
  }
  if (valid < key0 + 64) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (key0 + 32 * c + e >= valid) v[c][e] = 0.0f;
  }
}

__device__ __forceinline__ void scale64(float (&v)[2][32], float r) {
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int e = 0; e < 32; e += 2) fma2(v[c][e], v[c][e + 1], v[c][e], v[c][e + 1], r, r, 0.0f, 0.0f);
}

// Packs the 64 p of a half row as bf16 pairs (lower key in the low half) into
// w and returns their sum (eight partial sums: short dependent chains).
__device__ __forceinline__ float sum_pack64(const float (&v)[2][32], float (&w)[2][16]) {
  float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f, s4 = 0.0f, s5 = 0.0f, s6 = 0.0f, s7 = 0.0f;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
#pragma unroll
    for (int e = 0; e < 32; e += 8) {
      add2(s0, s1, v[c][e], v[c][e + 1]);
      add2(s2, s3, v[c][e + 2], v[c][e + 3]);
      add2(s4, s5, v[c][e + 4], v[c][e + 5]);
      add2(s6, s7, v[c][e + 6], v[c][e + 7]);
    }
  }
#pragma unroll
  for (int c = 0; c < 2; ++c) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[c][2 * e], v[c][2 * e + 1]);
      w[c][e] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h2));
    }
  }
  return ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
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
  // Q_X of the item landed / free again (one pair per tile, so Q_A of the next
  // item loads as soon as the item's last S_A is done)
  auto q_full = [&](uint32_t x) { return x ? bar0 + 152 : bar0; };
  auto q_empty = [&](uint32_t x) { return x ? bar0 + 160 : bar0 + 8; };
  auto k_full = [&](uint32_t s) { return bar0 + 16 + 8 * s; };
  auto k_empty = [&](uint32_t s) { return bar0 + 32 + 8 * s; };
  auto v_full = [&](uint32_t s) { return bar0 + 48 + 8 * s; };
  auto v_empty = [&](uint32_t s) { return bar0 + 64 + 8 * s; };
  auto s_full = [&](uint32_t x) { return bar0 + 80 + 8 * x; };   // S_X(j) and P_X(j-1) V done
  auto p_ready = [&](uint32_t x) { return bar0 + 96 + 8 * x; };  // P_X(j) written
  auto o_full = [&](uint32_t x) { return bar0 + 112 + 8 * x; };  // the item's last P_X V done
  auto o_empty = [&](uint32_t x) { return bar0 + 128 + 8 * x; }; // O_X read out
  const uint32_t drain_bar = bar0 + 144;
  constexpr uint32_t kSoftmaxWarps = 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (uint32_t x = 0; x < 2; ++x) {
      mbar_init(q_full(x), 1);
      mbar_init(q_empty(x), 1);
    }
    for (uint32_t s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(p_ready(s), kSoftmaxWarps);
      mbar_init(o_full(s), 1);
      mbar_init(o_empty(s), kSoftmaxWarps);
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
        for (uint32_t x = 0; x < 2 && ok; ++x) {
          if (!wait_bounded<true>(q_empty(x), (ti & 1u) ^ 1u, ab, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t qx = q_addr + x * kAttnTile;
          mbar_arrive_expect_tx(q_full(x), kAttnTile);
          tma_load_3d(qx, &tmQ, q_full(x), 0, q0 + static_cast<int>(x) * kAttnM, b);
          tma_load_3d(qx + kAttnHalf, &tmQ, q_full(x), 64, q0 + static_cast<int>(x) * kAttnM, b);
        }
        if (!ok) break;
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
      if (ti > 0) {
        drain_wait(q_full(0), (ti - 1) & 1u);
        drain_wait(q_full(1), (ti - 1) & 1u);
      }
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
      // O_X (+)= P_X V: P from columns 32..95 of S_X (8 per k-step), V
      // MN-major (64-column halves 16 KB apart, 16 keys = 2048 bytes per k-step)
      auto issue_pv = [&](uint32_t x, uint32_t vs, bool first) {
        const uint32_t v_lo = desc_lo(v_addr + vs * kAttnTile, kAttnHalf);
        const uint32_t d_tmem = tmem_base + 256u + x * 128u;
        const uint32_t a_tmem = tmem_base + x * 128u + kAttnPCol;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma_f16_ts(d_tmem, a_tmem + 8u * ks, desc_join(v_lo + ks * 128u, hi_sw), p.idesc_o,
                        (!first || ks > 0) ? 1u : 0u);
      };
      for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
        // Q_X is free once the item's last S_X is done
        for (uint32_t x = 0; x < 2 && ok; ++x) {
          ok = wait_bounded<true>(q_full(x), ti & 1u, ab, kSiteMmaFull) && issue_s_pair_half(x);
          if (ok && nb == 1) tc_commit(q_empty(x));
        }
        for (int j = 0; j < nb && ok; ++j) {
          const uint32_t vs = gv & 1u, vph = (gv >> 1) & 1u;
          // P_X(j) is tile X's (ti * nb + j)-th block: every item has nb blocks
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
              if (j + 2 == nb) tc_commit(q_empty(x));
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
    // Warps w and w + 4 may access the same Tensor Memory lane quarter: both
    // take its 32 query rows in both tiles (A, then B, per key block), w the
    // keys 0..63 of each block and w + 4 the keys 64..127.
    const int quad = warp & 3;
    const uint32_t h = static_cast<uint32_t>(warp - 2) >> 2;  // key half
    const int row = quad * 32 + lane;                         // query row within a tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sc = p.scale_log2;
    float2* xch = reinterpret_cast<float2*>(smem + 6 * kAttnTile + kAttnBarBytes);
    uint32_t nx = 0;
    // Trades a value and the wait verdict with the thread of the same row in
    // the partner warp.  Two buffers: a thread rewrites a buffer only after
    // the next barrier, which its partner passes only once it has read it.
    // Both warps take every exchange, so a failed wait in either ends both
    // loops at the same point.
    auto exchange = [&](float mine, bool& ok_io) -> float {
      float2* buf = xch + (nx++ & 1u) * 256u;
      buf[h * 128u + row] = make_float2(mine, ok_io ? 1.0f : 0.0f);
      named_bar_sync(1u + static_cast<uint32_t>(quad), 64u);
      const float2 o = buf[(h ^ 1u) * 128u + row];
      ok_io = ok_io && o.y != 0.0f;
      return o.x;
    };
    uint32_t n = 0, ti = 0;  // blocks done, items
    bool ok = true;
    for (int64_t item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ti) {
      const int b = static_cast<int>(item / p.q_tiles);
      // per tile: running maximum and this half's sum of p (kept in registers:
      // the tile loop below is not unrolled, so no arrays indexed by it)
      float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
      for (int j = 0; j < nb && ok; ++j, ++n) {
        const int valid = p.Lk - j * kAttnN < 128 ? p.Lk - j * kAttnN : 128;
        const int valid_h = valid - 64 * static_cast<int>(h);  // keys of this half in range
#pragma unroll 1
        for (uint32_t x = 0; x < 2; ++x) {
          const uint32_t s_col = tmem_base + lane_off + x * 128u;          // S_X
          const uint32_t o_col = tmem_base + lane_off + 256u + x * 128u;   // O_X
          ok = warp_wait(s_full(x), n & 1u, ab, kSiteEpiAccFull, lane);
          float mx = x ? m_b : m_a, lx = x ? l_b : l_a;
          // this thread's 64 columns of S: one Tensor Memory round trip
          float v[2][32];
          float mine = -INFINITY, m_use = 0.0f;
          if (ok) {
            tc_fence_after_sync();
            mine = sc >= 0.0f ? half_row_max_scaled<false>(s_col + 64u * h, valid_h, sc, v)
                              : half_row_max_scaled<true>(s_col + 64u * h, valid_h, sc, v);
            // The exponentials start before the partner's maximum arrives:
            // against the running maximum (raised if need be so that
            // p <= 2^64), or in a row's first block against this half's own
            // maximum.  Below, p moves to the row's common maximum where the
            // two differ (p * exp2(m_use - m_new) = exp2(s - m_new)).
            m_use = j == 0 ? mine : fmaxf(mx, mine - kAttnSpecLog2);
            exp64(v, 64 * static_cast<int>(h), valid, sc, -m_use);
          }
          const float other = exchange(mine, ok);
          if (!ok) break;
          const float m_blk = fmaxf(mine, other);  // key 0 is valid: finite
          // both threads of a row take the same decisions from the same values
          const bool grow = j > 0 && m_blk > mx + kAttnRescaleLog2;
          const float m_new = (j == 0 || grow) ? m_blk : mx;
          if (__any_sync(0xffffffffu, m_use != m_new))
            scale64(v, m_use == m_new ? 1.0f : fast_exp2(m_use - m_new));
          if (__any_sync(0xffffffffu, grow)) {
            // rescale this half of O_X and l by exp2(m_old - m_new) in the rows
            // that need it (O_X is final for the previous block: see the header)
            const float r = grow ? fast_exp2(mx - m_new) : 1.0f;
            if (grow) lx *= r;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              float o[16];
              const uint32_t oc = o_col + 64u * h + 16u * c;
              tmem_ld_16cols(oc, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; e += 2) fma2(o[e], o[e + 1], o[e], o[e + 1], r, r, 0.0f, 0.0f);
              tmem_st_16cols(oc, o);
            }
            tmem_wait_st();
          }
          mx = m_new;
          // P as bf16 pairs: key k of the block into column kAttnPCol + k / 2 of
          // S_X, so each thread writes only columns whose scores it has loaded
          float w[2][16];
          const float p_sum = sum_pack64(v, w);
          tmem_st_16cols(s_col + kAttnPCol + 32u * h, w[0]);
          tmem_st_16cols(s_col + kAttnPCol + 32u * h + 16u, w[1]);
          // l sums the unrounded p: the bf16 rounding then perturbs only the
          // numerator of O = (P V) / l, by at most 2^-8 sum_c p_c |V_c| / l
          lx += p_sum;
          if (x) {
            m_b = mx;
            l_b = lx;
          } else {
            m_a = mx;
            l_a = lx;
          }
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_ready(x));
        }
      }
      if (!ok) break;
      // O_X / l for this row (this thread's 64 of its 128 columns), once the
      // item's last product has landed
#pragma unroll 1
      for (uint32_t x = 0; x < 2; ++x) {
        ok = warp_wait(o_full(x), ti & 1u, ab, kSiteEpiAccFull, lane);
        const float lx = x ? l_b : l_a;
        const float l_row = lx + exchange(lx, ok);  // the same sum in both threads
        if (!ok) break;
        tc_fence_after_sync();
        const float inv = 1.0f / l_row;
        const uint32_t o_col = tmem_base + lane_off + 256u + x * 128u + 64u * h;
        const int qi = static_cast<int>(item % p.q_tiles) * kAttnItemRows + static_cast<int>(x) * kAttnM + row;
        __nv_bfloat16* dst =
            p.O + static_cast<int64_t>(b) * p.so + static_cast<int64_t>(qi) * p.ldo + 64 * static_cast<int>(h);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float o[16];
          tmem_ld_16cols(o_col + 16u * c, o);
          tmem_wait_ld();
          if (c == 3) {  // O_X may take the next item
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
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

}  // namespace dmt

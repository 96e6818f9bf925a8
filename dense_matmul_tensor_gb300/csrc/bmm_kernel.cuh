// The batched-product kernels for sm_103a.
//
// bmm_tc_kernel: a persistent, warp-specialised tcgen05 GEMM over the whole
// batch x tile grid.  Per CTA (256 threads, one CTA per SM):
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
//   warps 6..7  row loader, for an operand TMA cannot address (row or batch
//               stride, or base, off a 16-byte boundary): plain loads of its
//               elements, written into the stage in the layout the TMA box
//               would give (idle otherwise).
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
constexpr int kThreads = 256; // producer, MMA, 4 epilogue warps, 2 row-loader warps
constexpr int kLdgWarps = 2;
constexpr int kGroupM = 8;
constexpr int kEpiPitch = 33; // floats per staged row (bank-conflict-free)
// Epilogue staging, shared by the two store paths: four 32 x 33 fp32 tiles
// (coalesced direct stores) or two 4 KB TMA-store boxes per epilogue warp.
constexpr uint32_t kEpiBoxBytes = 4096u;
constexpr int kMaxStages = 8;      // deepest operand ring the planner builds
constexpr uint32_t kEpiBytes = 4u * 2u * kEpiBoxBytes;
static_assert(kEpiBytes >= 4u * 32u * kEpiPitch * 4u, "direct-store staging must fit");
constexpr uint32_t kBarBytes = 512;   // barriers, TMEM slot, abort flag
// full[S], empty[S], two acc_full, two acc_empty, drain, then the TMEM slot and
// the abort flag must end before byte 256 of the barrier block (the grouped
// launches' schedule state starts there)
static_assert(8u * (2u * kMaxStages + 5u) + 8u <= 256u, "barrier block layout");
constexpr uint32_t kSmemLimit = 232448;  // 227 KB dynamic shared memory per CTA

// Device error word: kErrTag | (site << 8) | role-specific detail.
constexpr uint32_t kErrTag = 0xB0000000u;
enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaAccEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpiAccFull = 4,
  kSiteTestStall = 5,
  kSiteSchedule = 6,
  kSiteStreamK = 7,
  kSiteSmemLayout = 8,  // the launch's shared memory does not hold the ring, epilogue and barriers
};

// Epilogue region of the CTA-pair kernel for launches whose C goes out as
// bf16 through TMA box stores: two 2 KB boxes (32 rows x 64 bytes) per
// epilogue warp, half the general region, which leaves room for one more
// ring stage of 256 x 224 or 256 x 192 tiles.
constexpr uint32_t kEpiBoxBytesBf16 = 2048u;
constexpr uint32_t kEpiBytesBf16 = 4u * 2u * kEpiBoxBytesBf16;

// Stream-K tail of the CTA-pair kernel: a piece of k-blocks [ka, kb) of one
// tile has at least this many k-blocks, and at least half the tile's (so a
// tile has at most three pieces and its owner adds at most two partials).
constexpr int kSkMinUnits = 8;

// One problem of a grouped launch: an entry of a device table built by the
// host (tensor maps first, so each is 128-byte aligned).  tile_begin is the
// launch-wide index of the problem's first tile.
struct alignas(128) GroupEntry {
  CUtensorMap map_a, map_b, map_c;
  void* C;
  int64_t tile_begin;
  int64_t ldc;
  int32_t Mv, Nv, k_blocks, tail_steps, num_m, num_n;
  float alpha, beta;
  int32_t c_tma;
};

// An operand read by the row loader: [batch][rows][cols] 16-bit elements with
// row stride ld and batch stride `stride` (0: one item for the whole batch).
struct LdgOperand {
  const uint16_t* ptr;
  int64_t ld, stride;
  int64_t rows, cols;
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
  int32_t c_tma;           // 1: row-major C written with TMA box stores (tensor map tmC)
  float alpha, beta;
  uint32_t* err;           // device error word
  uint64_t timeout_ns;     // bound on any single wait
  int32_t test_stall;      // 1: the MMA thread first waits on a barrier nothing completes
  const GroupEntry* groups;// grouped launches: the problem table (device memory)
  const int32_t* group_first;  // ... and each entry's first tile, compact
  int32_t ngroups;
  int32_t ldg_mask;        // bit 0: A, bit 1: B read by the row loader (tx_bytes excludes them)
  LdgOperand ldg[2];       // A, B
  // Stream-K tail (CTA-pair kernel; sk_tiles == 0: off).  The first
  // sk_first tiles run whole, round-robin over the pairs; the
  // k-blocks of the last sk_tiles tiles are cut into sk_pairs equal ranges,
  // one per pair.  A piece without k-block 0 leaves its fp32 partial in
  // sk_ws and raises its flags to sk_epoch; the piece with k-block 0 adds the
  // other pieces' partials and writes C.
  int32_t sk_tiles, sk_pairs;
  int64_t sk_first;        // first tile of the tail (whole rounds x pairs)
  uint32_t sk_epoch;       // this launch's flag value (never 0)
  int32_t sk_ko;           // two-way split: the owner's k-blocks [0, sk_ko), the contributor's the rest
  float4* sk_ws;           // [pair][rank][quarter][chunk][8][32 rows] float4
  uint32_t* sk_flags;      // [pair][rank][quarter]
  // CTA-pair kernel: bytes of the epilogue region after the ring and of one
  // box buffer in it (kEpiBytes and kEpiBoxBytes, or for bf16 box-store
  // launches kEpiBytesBf16 and kEpiBoxBytesBf16)
  uint32_t epi_bytes, box_bytes;
};

// A stream-K piece: k-blocks [ka, kb) of tile `tile`.  kind 0: the whole
// tile (a range that happens to cover it); kind 1: no k-block 0 (its partial
// goes to the workspace slot of its pair); kind 2: the piece with k-block 0
// of a split tile, which adds the partials of pairs [q_lo, q_hi) and writes C.
struct SkPiece {
  int64_t tile;
  int32_t ka, kb, kind, q_lo, q_hi;
};

// Piece si (0 or 1) of pair `pair`: the pair's range of the tail's
// sk_tiles * k_blocks k-blocks, cut at tile boundaries (a range is at most
// one tile long, so it has at most two pieces).  False: no such piece.
__device__ __forceinline__ bool sk_piece(const KParams& p, int64_t pair, int si, SkPiece& it) {
  if (!p.sk_tiles || pair >= p.sk_pairs) return false;
  const int64_t KB = p.k_blocks;
  const int64_t U = static_cast<int64_t>(p.sk_tiles) * KB;
  const int64_t G = p.sk_pairs;
  const int64_t u0 = pair * U / G, u1 = (pair + 1) * U / G;
  if (u1 <= u0) return false;
  const int64_t t0 = u0 / KB;  // tile of the first piece, within the tail
  int64_t tt, s, e;
  if (si == 0) {
    tt = t0;
    s = u0;
    e = (t0 + 1) * KB < u1 ? (t0 + 1) * KB : u1;
  } else if (u1 > (t0 + 1) * KB) {
    tt = t0 + 1;
    s = tt * KB;
    e = u1;
  } else {
    return false;
  }
  it.tile = p.sk_first + tt;
  it.ka = static_cast<int32_t>(s - tt * KB);
  it.kb = static_cast<int32_t>(e - tt * KB);
  it.q_lo = it.q_hi = 0;
  if (it.ka > 0) {
    it.kind = 1;
  } else if (it.kb == KB) {
    it.kind = 0;
  } else {
    // the rest of the tile belongs to the next pairs, each in its first piece
    it.kind = 2;
    it.q_lo = static_cast<int32_t>(pair + 1);
    int64_t q = pair + 1;
    while (q < G && q * U / G < (tt + 1) * KB) ++q;
    it.q_hi = static_cast<int32_t>(q);
  }
  return true;
}

// The two-way split: each of the last sk_tiles tiles runs on two pairs,
// k-blocks [0, sk_ko) on pair 2i (the owner, which adds the other's partial
// and writes C) and [sk_ko, k_blocks) on pair 2i+1.  The owner's range is the
// longer one, by about the time a partial takes to reach the workspace, so
// the contributor's partial is there when the owner's accumulator is done.
// At most one piece per pair; false: none.
__device__ __forceinline__ bool sk_piece2(const KParams& p, int64_t pair, SkPiece& it) {
  if (pair >= 2 * static_cast<int64_t>(p.sk_tiles)) return false;
  it.tile = p.sk_first + pair / 2;
  if ((pair & 1) == 0) {
    it.ka = 0;
    it.kb = p.sk_ko;
    it.kind = 2;
    it.q_lo = static_cast<int32_t>(pair + 1);
    it.q_hi = static_cast<int32_t>(pair + 2);
  } else {
    it.ka = p.sk_ko;
    it.kb = p.k_blocks;
    it.kind = 1;
    it.q_lo = it.q_hi = 0;
  }
  return true;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* ptr, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// What the epilogue needs about C, for the launch or for one grouped problem.
struct EpiArgs {
  void* C;
  int64_t ldc;
  int32_t Mv, Nv, c_bf16, c_trans, c_tma;
  float alpha, beta;
};

__device__ __forceinline__ EpiArgs epi_args(const KParams& p) {
  return EpiArgs{p.C, p.ldc, p.Mv, p.Nv, p.c_bf16, p.c_trans, p.c_tma, p.alpha, p.beta};
}

struct Abort {
  volatile uint32_t* flag;
  uint32_t* err;
  uint64_t timeout_ns;
};

template <bool kSpin>
__device__ __forceinline__ bool mbar_probe(uint32_t bar, uint32_t parity) {
  return kSpin ? mbar_try_wait_spin(bar, parity) : mbar_try_wait(bar, parity);
}

// Slow path of a bounded wait: poll until the phase completes, another role
// raises the abort flag, or the time limit passes (then raise it).  kSpin
// polls without parking the thread (producer and MMA threads, whose wake-up
// latency sits on the pipeline's critical path).
template <bool kSpin>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, Abort ab, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_probe<kSpin>(bar, parity)) return true;
    if ((it & (kSpin ? 63u : 15u)) == 0) {
      if (*ab.flag) return false;
      if (global_timer_ns() - t0 > ab.timeout_ns) break;
    }
  }
  *ab.flag = 1u;
  atomicCAS(ab.err, 0u, kErrTag | (site << 8) | (blockIdx.x & 0xFFu));
  return false;
}

template <bool kSpin = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, Abort ab, uint32_t site) {
  if (mbar_probe<kSpin>(bar, parity)) return true;
  return wait_slow<kSpin>(bar, parity, ab, site);
}

// Wait with a short fixed limit and no error report: before exit, lets this
// CTA's own asynchronous copies and MMAs land (at once after a normal run;
// bounded after an abort).
static __device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 15u) == 0 && global_timer_ns() - t0 > 100000000ull) return;
  }
}

template <bool B>
struct BoolC {
  static constexpr bool value = B;
};

// Bounded wait with cluster-scope acquire (see mbar_try_wait_spin_cluster).
static __device__ __noinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, Abort ab, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait_spin_cluster(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*ab.flag) return false;
      if (global_timer_ns() - t0 > ab.timeout_ns) break;
    }
  }
  *ab.flag = 1u;
  atomicCAS(ab.err, 0u, kErrTag | (site << 8) | (blockIdx.x & 0xFFu));
  return false;
}

// Warp-uniform bounded wait (lane 0 polls, the warp takes its verdict).
__device__ __forceinline__ bool warp_wait_bounded(uint32_t bar, uint32_t parity, Abort ab, uint32_t site,
                                                  int lane) {
  int w = 1;
  if (lane == 0) w = wait_bounded<true>(bar, parity, ab, site) ? 1 : 0;
  w = __shfl_sync(0xffffffffu, w, 0);
  __syncwarp();
  return w != 0;
}

// 16 bytes starting at even byte offset sh (0..14) of the 32 bytes lo:hi.
__device__ __forceinline__ uint4 extract16(const uint4& lo, const uint4& hi, uint32_t sh) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const uint32_t b = (sh & 3u) * 8u;  // bits: 0 or 16
  uint32_t o[4];
  switch (sh >> 2) {  // whole words: the same for every chunk of a row
    case 0:
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(w[i], w[i + 1], b);
      break;
    case 1:
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(w[i + 1], w[i + 2], b);
      break;
    case 2:
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(w[i + 2], w[i + 3], b);
      break;
    default:
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(w[i + 3], w[i + 4], b);
      break;
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One operand tile of a ring stage written by the row loader, in the layout
// a 128-byte-swizzled TMA box gives: rows of 64 contiguous elements (128
// bytes), 16-byte chunk j of row r at chunk position j ^ (r mod 8); an
// MN-major tile is `atoms` blocks of 64 such rows, 8 KB apart.  Storage row
// row0 + r, elements col0 + 64 * atom + 8 * j .. + 7; elements outside the
// operand are zero, as TMA fills them.  The chunks are spread over
// `nthreads` threads (a multiple of 8; this thread is `tid`: chunk j =
// tid mod 8 of every (nthreads / 8)-th row).  A chunk starts on any 2-byte
// boundary: the thread loads the one or two 16-byte-aligned chunks that hold
// it (a second one only if it holds bytes of the row) and shifts the 16 bytes
// out; eight chunks' loads are in flight before the first store.
__device__ __forceinline__ void ldg_fill(uint8_t* tile, const LdgOperand& o, int bz, int64_t row0,
                                         int64_t col0, int tile_rows, int atoms, int tid, int nthreads) {
  constexpr int U = 8;
  const int j = tid & 7, rstep = nthreads >> 3;
  const uint16_t* base = o.ptr + static_cast<int64_t>(bz) * o.stride;
  for (int a = 0; a < atoms; ++a) {
    const int64_t scol = col0 + 64 * a + 8 * j;
    const int64_t left = o.cols - scol;  // elements of this chunk inside the row
    uint8_t* atom = tile + a * 8192;
    for (int r0 = tid >> 3; r0 < tile_rows; r0 += U * rstep) {
      uint4 lo[U], hi[U];
      uint32_t sh[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = r0 + u * rstep;
        const int64_t srow = row0 + r;
        lo[u] = hi[u] = make_uint4(0u, 0u, 0u, 0u);
        sh[u] = 0u;
        if (r < tile_rows && srow < o.rows && left > 0) {
          const uintptr_t at = reinterpret_cast<uintptr_t>(base + srow * o.ld + scol);
          const uintptr_t q = at & ~static_cast<uintptr_t>(15);
          const uintptr_t end = at + 2u * static_cast<uintptr_t>(left < 8 ? left : 8);
          sh[u] = static_cast<uint32_t>(at - q);
          lo[u] = __ldg(reinterpret_cast<const uint4*>(q));
          if (q + 16u < end) hi[u] = __ldg(reinterpret_cast<const uint4*>(q) + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = r0 + u * rstep;
        if (r >= tile_rows) continue;
        uint4 v = extract16(lo[u], hi[u], sh[u]);
        if (left < 8) {  // zero the elements past the row end
          uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e >= left) w[e >> 1] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
          v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        *reinterpret_cast<uint4*>(atom + r * 128 + ((j ^ (r & 7)) << 4)) = v;
      }
    }
  }
}

// Shared-memory descriptor words: the low word carries the start address
// (>> 4) and the leading byte offset, the high word the stride byte offset,
// the version and the 128-byte swizzle.  Start addresses stay below 256 KB,
// so stepping the low word by (bytes >> 4) never carries into the LBO field.
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint32_t desc_hi_sw128(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint64_t desc_join(uint32_t lo, uint32_t hi) {
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// MMAs of one k-block (4 k-steps of 16, or `nsteps` on a ragged tail) with
// the descriptors stepped by (k-step bytes >> 4) in their low words.
template <bool kPair>
__device__ __forceinline__ void issue_kblock(uint32_t d_tmem, uint32_t alo, uint32_t blo,
                                             uint32_t ahi, uint32_t bhi, uint32_t astep,
                                             uint32_t bstep, uint32_t idesc, int nsteps,
                                             bool first) {
  if (nsteps == kTileK / kUmmaK) {
#pragma unroll
    for (int ks = 0; ks < kTileK / kUmmaK; ++ks) {
      const uint64_t ad = desc_join(alo + ks * astep, ahi), bd = desc_join(blo + ks * bstep, bhi);
      const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
      if (kPair) tc_mma_f16_pair(d_tmem, ad, bd, idesc, acc);
      else tc_mma_f16(d_tmem, ad, bd, idesc, acc);
    }
  } else {
    for (int ks = 0; ks < nsteps; ++ks) {
      const uint64_t ad = desc_join(alo + ks * astep, ahi), bd = desc_join(blo + ks * bstep, bhi);
      const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
      if (kPair) tc_mma_f16_pair(d_tmem, ad, bd, idesc, acc);
      else tc_mma_f16(d_tmem, ad, bd, idesc, acc);
    }
  }
}

// Tile r of one (num_m x num_n) grid, in GROUP_M-row groups for L2 reuse.
__device__ __forceinline__ void decode_mn(int r, int num_m, int num_n, int& mb, int& nb) {
  const int group = kGroupM * num_n;
  const int gid = r / group;
  const int first_m = gid * kGroupM;
  const int gsz = min(num_m - first_m, kGroupM);
  const int rin = r - gid * group;
  mb = first_m + rin % gsz;
  nb = rin / gsz;
}

__device__ __forceinline__ void decode_tile(int64_t t, const KParams& p, int& b, int& mb, int& nb) {
  const int64_t per = static_cast<int64_t>(p.num_m) * p.num_n;
  b = static_cast<int>(t / per);
  decode_mn(static_cast<int>(t - static_cast<int64_t>(b) * per), p.num_m, p.num_n, mb, nb);
}

// Everything a role needs about tile t: its place, its K extent and the
// tensor maps of its operands (the launch's, or its grouped problem's).
struct TileCtx {
  int b, mb, nb, k_blocks, tail_steps;
  const CUtensorMap* map_a;
  const CUtensorMap* map_b;
  const CUtensorMap* map_c;
  const GroupEntry* g;
};

// Grouped launches: the table entry that tile t belongs to (the last whose
// first tile is <= t), by binary search over the compact first-tile array.
__device__ __forceinline__ int group_of(int64_t t, const KParams& p) {
  int lo = 0, hi = p.ngroups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.group_first + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Tile context of tile t of table entry gi (grouped launches).
__device__ __forceinline__ TileCtx tile_ctx_group(int64_t t, int gi, const KParams& p) {
  TileCtx c;
  const GroupEntry* g = p.groups + gi;
  decode_mn(static_cast<int>(t - g->tile_begin), g->num_m, g->num_n, c.mb, c.nb);
  c.b = 0;
  c.k_blocks = g->k_blocks;
  c.tail_steps = g->tail_steps;
  c.map_a = &g->map_a;
  c.map_b = &g->map_b;
  c.map_c = &g->map_c;
  c.g = g;
  return c;
}

template <bool kGrouped>
__device__ __forceinline__ TileCtx tile_ctx(int64_t t, const KParams& p, const CUtensorMap* tmA,
                                            const CUtensorMap* tmB, const CUtensorMap* tmC) {
  TileCtx c;
  if constexpr (!kGrouped) {
    decode_tile(t, p, c.b, c.mb, c.nb);
    c.k_blocks = p.k_blocks;
    c.tail_steps = p.tail_steps;
    c.map_a = tmA;
    c.map_b = tmB;
    c.map_c = tmC;
    c.g = nullptr;
  } else {
    c = tile_ctx_group(t, group_of(t, p), p);
  }
  return c;
}

__device__ __forceinline__ float load_c(const EpiArgs& p, int64_t off) {
  if (p.c_bf16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p.C)[off]);
  return static_cast<const float*>(p.C)[off];
}

__device__ __forceinline__ void store_c(const EpiArgs& p, int64_t off, float v) {
  if (p.c_bf16)
    static_cast<__nv_bfloat16*>(p.C)[off] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(p.C)[off] = v;
}

// One chunk of CW accumulator columns held by this thread (row `lane` of the
// warp's 32-lane quarter) -> C with coalesced direct stores (any alignment,
// beta != 0, or the swapped C^T form).  Rows go in groups of eight: the
// group's loads are all issued before its first store (C may alias nothing
// the compiler can prove, so interleaving would serialise one memory latency
// per row), while the live registers stay bounded.
template <int CW>
__device__ __forceinline__ void store_chunk(const EpiArgs& p, float (&v)[CW], float* stg, int lane,
                                            int row0, int col0, int64_t cbase) {
  constexpr int G = 8;
  const float alpha = p.alpha, beta = p.beta;
#pragma unroll
  for (int r = 0; r < CW; ++r) v[r] *= alpha;
  if (p.c_trans) {
    // D row i = C column, D column j = C row: lanes write consecutive C columns.
    const int i = row0 + lane;
    if (i < p.Mv) {
      const int ncols = min(CW, p.Nv - col0);
      int64_t off = cbase + static_cast<int64_t>(col0) * p.ldc + i;
#pragma unroll
      for (int g = 0; g < CW; g += G) {
        if (beta != 0.0f) {
          float cin[G];
          int64_t o = off;
#pragma unroll
          for (int r = 0; r < G; ++r, o += p.ldc)
            if (g + r < ncols) cin[r] = load_c(p, o);
#pragma unroll
          for (int r = 0; r < G; ++r) v[g + r] = fmaf(beta, cin[r], v[g + r]);
        }
#pragma unroll
        for (int r = 0; r < G; ++r, off += p.ldc)
          if (g + r < ncols) store_c(p, off, v[g + r]);
      }
    }
    return;
  }
  // Row-major C: stage the 32 x CW block (thread = row) and read it back
  // transposed (lane = column), so each warp store covers one C row.
#pragma unroll
  for (int r = 0; r < CW; ++r) stg[lane * kEpiPitch + r] = v[r];
  __syncwarp();
  const int j = col0 + lane;
  const bool active = lane < CW && j < p.Nv;
  const int rows = min(32, p.Mv - row0);
  int64_t off = cbase + static_cast<int64_t>(row0) * p.ldc + j;
  if (beta != 0.0f) {
    // All 32 rows of C_in are requested before anything is stored: one
    // memory latency per chunk instead of one per group of rows.
    float cin[32];
    int64_t o = off;
#pragma unroll
    for (int r = 0; r < 32; ++r, o += p.ldc)
      if (active && r < rows) cin[r] = load_c(p, o);
#pragma unroll
    for (int g = 0; g < 32; g += G) {
      float w[G];
#pragma unroll
      for (int r = 0; r < G; ++r) w[r] = fmaf(beta, cin[g + r], stg[(g + r) * kEpiPitch + lane]);
#pragma unroll
      for (int r = 0; r < G; ++r, off += p.ldc)
        if (active && g + r < rows) store_c(p, off, w[r]);
    }
    __syncwarp();
    return;
  }
#pragma unroll
  for (int g = 0; g < 32; g += G) {
    float w[G];
#pragma unroll
    for (int r = 0; r < G; ++r) w[r] = stg[(g + r) * kEpiPitch + lane];
    if (active) {
#pragma unroll
      for (int r = 0; r < G; ++r, off += p.ldc)
        if (g + r < rows) store_c(p, off, w[r]);
    }
  }
  __syncwarp();  // staging tile free for the next chunk
}

// Request C_in for one 32-column chunk of a warp's 32 rows of row-major C
// (lane = column): the loads are in flight while the previous chunk is
// stored, and the first chunk of a tile while its mainloop still runs.
__device__ __forceinline__ void prefetch_cin(const EpiArgs& p, float (&cin)[32], int lane, int row0,
                                             int col0, int64_t cbase) {
  const int j = col0 + lane;
  const bool active = j < p.Nv;
  const int rows = min(32, p.Mv - row0);
  int64_t o = cbase + static_cast<int64_t>(row0) * p.ldc + j;
#pragma unroll
  for (int r = 0; r < 32; ++r, o += p.ldc)
    if (active && r < rows) cin[r] = load_c(p, o);
}

// store_chunk for row-major C with beta != 0 and C_in already requested.
__device__ __forceinline__ void store_chunk_cin(const EpiArgs& p, float (&v)[32], const float (&cin)[32],
                                                float* stg, int lane, int row0, int col0,
                                                int64_t cbase) {
  constexpr int G = 8;
  const float alpha = p.alpha, beta = p.beta;
#pragma unroll
  for (int r = 0; r < 32; ++r) stg[lane * kEpiPitch + r] = alpha * v[r];
  __syncwarp();
  const int j = col0 + lane;
  const bool active = j < p.Nv;
  const int rows = min(32, p.Mv - row0);
  int64_t off = cbase + static_cast<int64_t>(row0) * p.ldc + j;
#pragma unroll
  for (int g = 0; g < 32; g += G) {
    float w[G];
#pragma unroll
    for (int r = 0; r < G; ++r) w[r] = fmaf(beta, cin[g + r], stg[(g + r) * kEpiPitch + lane]);
#pragma unroll
    for (int r = 0; r < G; ++r, off += p.ldc)
      if (active && g + r < rows) store_c(p, off, w[r]);
  }
  __syncwarp();  // staging tile free for the next chunk
}

// One chunk of 32 accumulator columns -> C through a TMA box store.  The
// warp writes its 32 rows into a 4 KB box buffer laid out with the tensor
// map's swizzle (128-byte rows for fp32, 64-byte rows for bf16), then one
// lane stores the box; TMA clips rows and columns outside C.  Two buffers
// per warp alternate, so a box is written while the previous one drains.
__device__ __forceinline__ void store_chunk_tma(const EpiArgs& p, const CUtensorMap* tmC,
                                                float (&v)[32], uint8_t* box, uint32_t box_addr,
                                                int lane, int row0, int col0, int b) {
  const float alpha = p.alpha;
  if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous box has been read
  __syncwarp();
  if (!p.c_bf16) {
    uint8_t* row = box + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) =
          make_float4(alpha * v[4 * j], alpha * v[4 * j + 1], alpha * v[4 * j + 2],
                      alpha * v[4 * j + 3]);
  } else {
    uint8_t* row = box + lane * 64;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h =
            __floats2bfloat162_rn(alpha * v[8 * j + 2 * e], alpha * v[8 * j + 2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(row + ((j ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(tmC, box_addr, col0, row0, b);
    bulk_commit_group();
  }
}

// kGrouped: the launch covers a table of independent problems (p.groups):
// every role maps its tile to a problem and takes that problem's sizes,
// tensor maps and C from the table; otherwise one batched problem.
// Tiles of a grouped launch differ in cost (K, and so the k-block count,
// varies by problem), so they are handed out dynamically with cluster launch
// control: the launch has one CTA per tile, each running CTA starts with its
// own tile and then cancels CTAs that have not started yet and takes their
// tiles.  The producer thread asks for the next tile while it loads the
// current one and passes each tile index (or the end) to the MMA thread and
// the epilogue warps through a four-entry ring in shared memory.  A plain
// launch hands tiles out round-robin over a persistent grid.
// kPerSM = 2 (grouped launches of narrow tiles): two CTAs of 192 threads
// share an SM, so the compiler keeps each thread within 168 registers.
template <int BN, bool kGrouped = false, int kPerSM = 1>
__global__ void __launch_bounds__(kPerSM == 2 ? kThreads - 32 * kLdgWarps : kThreads, kPerSM)
    bmm_tc_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmA,
                  const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC) {
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
  // dynamic schedule (grouped launches): the cancel response, the tile ring
  // and its barriers, from byte 256 of the barrier block
  const uint32_t clc_resp = bar0 + 256;
  volatile int32_t* sched_tile = reinterpret_cast<volatile int32_t*>(smem + ring_bytes + kEpiBytes + 272u);
  volatile int32_t* sched_group = reinterpret_cast<volatile int32_t*>(smem + ring_bytes + kEpiBytes + 368u);
  auto sched_full = [&](uint32_t i) { return bar0 + 288u + 8u * i; };
  auto sched_empty = [&](uint32_t i) { return bar0 + 320u + 8u * i; };
  const uint32_t clc_bar = bar0 + 352u;
  constexpr uint32_t kSched = 4;
  constexpr bool kDyn = kGrouped;  // grouped launches are scheduled dynamically

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1 + (p.ldg_mask ? kLdgWarps : 0));  // + the row-loader warps
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 4);  // one arrive per epilogue warp
    }
    mbar_init(drain_bar, 1);
    if constexpr (kDyn) {
      for (uint32_t i = 0; i < kSched; ++i) {
        mbar_init(sched_full(i), 1);
        mbar_init(sched_empty(i), 5);  // the MMA thread and the four epilogue warps
      }
      mbar_init(clc_bar, 1);
    }
    *abort_flag = 0u;
    fence_barrier_init();
  }

  if (warp == 0 && lane == 0 && !kGrouped) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.c_tma) tma_prefetch_desc(&tmC);
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
  // Tile i of this CTA for the MMA thread and the epilogue warps: round-robin
  // over a persistent grid, or read from the schedule ring with its table
  // entry (lane 0 waits and releases the entry, the lanes in `mask` take its
  // values: all 32 for an epilogue warp, lane 0 alone for the MMA thread; a
  // full-warp shuffle also gathers the warp back after lane 0's wait).
  // >= p.tiles: no more.
  auto next_tile = [&](uint32_t i, int64_t& t, int& gi, uint32_t mask) -> bool {
    if constexpr (!kDyn) {
      t = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(i) * gridDim.x;
      gi = 0;
      return true;
    } else {
      int v = 0, gv = 0, w = 1;
      if (lane == 0) {
        w = wait_bounded(sched_full(i % kSched), (i / kSched) & 1u, ab, kSiteSchedule) ? 1 : 0;
        if (w) {
          v = sched_tile[i % kSched];
          gv = sched_group[i % kSched];
          mbar_arrive(sched_empty(i % kSched));
        }
      }
      w = __shfl_sync(mask, w, 0);
      v = __shfl_sync(mask, v, 0);
      gv = __shfl_sync(mask, gv, 0);
      t = v;
      gi = gv;
      return w != 0;
    }
  };
  // the tile context from a tile and (dynamic schedule) its table entry
  auto ctx_of = [&](int64_t t, int gi) -> TileCtx {
    if constexpr (kDyn) return tile_ctx_group(t, gi, p);
    else return tile_ctx<kGrouped>(t, p, &tmA, &tmB, &tmC);
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      int64_t t = blockIdx.x;
      uint32_t si = 0;              // schedule entries published (grouped)
      bool cancel_pending = false;  // a cancel request whose response has not been read
      int gi = 0;  // table entry of tile t (dynamic schedule)
      if constexpr (kDyn) {
        gi = group_of(t, p);
        sched_tile[0] = static_cast<int32_t>(t);
        sched_group[0] = gi;
        mbar_arrive(sched_full(0));
        si = 1;
      }
      // kLdg: some operand comes from the row loader (its TMA loads are
      // skipped, and there may be no bytes to expect).  A separate copy of the
      // loop keeps the TMA-only issue sequence as it is.
      auto produce = [&](auto has_ldg) {
        constexpr bool kLdg = decltype(has_ldg)::value;
        while (t < p.tiles && ok) {
          if constexpr (kDyn) {  // ask for the next tile while this one loads
            mbar_arrive_expect_tx(clc_bar, 16);
            clc_try_cancel(clc_resp, clc_bar);
            cancel_pending = true;
          }
          const TileCtx tc = ctx_of(t, gi);
          const int m0 = tc.mb * kTileM, n0 = tc.nb * BN;
          const int za = p.a_bcast ? 0 : tc.b, zb = p.b_bcast ? 0 : tc.b;
          for (int kb = 0; kb < tc.k_blocks; ++kb, ++it) {
            const uint32_t s = it % S, ph = (it / S) & 1u;
            if (!wait_bounded<true>(empty_bar(s), ph ^ 1u, ab, kSiteProducerEmpty)) {
              ok = false;
              break;
            }
            const uint32_t a_dst = sbase + s * p.stage_bytes;
            const uint32_t b_dst = a_dst + p.a_bytes;
            if constexpr (kLdg) {
              if (p.tx_bytes) mbar_arrive_expect_tx(full_bar(s), p.tx_bytes);
              else mbar_arrive(full_bar(s));  // both operands come from the row loader
            } else {
              mbar_arrive_expect_tx(full_bar(s), p.tx_bytes);
            }
            const int k0 = kb * kTileK;
            if (!kLdg || !(p.ldg_mask & 1)) {
              if (!p.a_mn) {
                tma_load_3d(a_dst, tc.map_a, full_bar(s), k0, m0, za);
              } else {
                tma_load_3d(a_dst, tc.map_a, full_bar(s), m0, k0, za);
                tma_load_3d(a_dst + 8192u, tc.map_a, full_bar(s), m0 + 64, k0, za);
              }
            }
            if (!kLdg || !(p.ldg_mask & 2)) {
              if (!p.b_mn) {
                tma_load_3d(b_dst, tc.map_b, full_bar(s), k0, n0, zb);
              } else {
#pragma unroll
                for (int h = 0; h < BN / 64; ++h)
                  tma_load_3d(b_dst + 8192u * h, tc.map_b, full_bar(s), n0 + 64 * h, k0, zb);
              }
            }
          }
          if constexpr (kDyn) {
            // publish the next tile (a cancelled CTA's) or the end
            int64_t nxt = p.tiles;
            if (!ok || !wait_bounded<true>(clc_bar, (si - 1) & 1u, ab, kSiteSchedule)) {
              ok = false;
              break;
            }
            cancel_pending = false;
            uint32_t x = 0;
            if (clc_decode(clc_resp, x) && static_cast<int64_t>(x) < p.tiles) nxt = x;
            const uint32_t slot = si % kSched;
            if (si >= kSched &&
                !wait_bounded<true>(sched_empty(slot), ((si / kSched) - 1u) & 1u, ab, kSiteSchedule)) {
              ok = false;
              break;
            }
            const int ngi = nxt < p.tiles ? group_of(nxt, p) : 0;
            sched_tile[slot] = static_cast<int32_t>(nxt);
            sched_group[slot] = ngi;
            mbar_arrive(sched_full(slot));
            ++si;
            t = nxt;
            gi = ngi;
          } else {
            t += gridDim.x;
          }
        }
      };
      if (!kDyn && p.ldg_mask) produce(BoolC<true>{});
      else produce(BoolC<false>{});
      if constexpr (kDyn) {  // a cancel response still on its way must land first
        if (cancel_pending) drain_wait(clc_bar, (si - 1) & 1u);
      }
      // Let the loads issued for the last S k-blocks land before the CTA can
      // exit (after a normal run they have all landed and this returns at once).
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0u;
      for (uint32_t j = first; j < it; ++j) drain_wait(full_bar(j % S), (j / S) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // Descriptor words for stage 0; stage s adds s * (stage_bytes >> 4).
      const uint32_t alo0 = desc_lo(sbase, p.a_mn ? 8192u : 16u);
      const uint32_t blo0 = desc_lo(sbase + p.a_bytes, p.b_mn ? 8192u : 16u);
      const uint32_t hi = desc_hi_sw128(1024u);
      const uint32_t astep = (p.a_mn ? 2048u : 32u) >> 4, bstep = (p.b_mn ? 2048u : 32u) >> 4;
      const uint32_t sstep = p.stage_bytes >> 4;
      uint32_t s = 0, ph = 0, tl = 0;
      // Failure-detection test: phase 0 of the drain barrier completes only
      // after this thread's final commit, so this wait must run out.
      bool ok = !p.test_stall || wait_bounded(drain_bar, 0u, ab, kSiteTestStall);
      for (uint32_t ti = 0; ok; ++ti, ++tl) {
        int64_t t;
        int gi;
        if (!next_tile(ti, t, gi, 1u)) {  // lane 0 only
          ok = false;
          break;
        }
        if (t >= p.tiles) break;
        const uint32_t acc = tl & 1u, aph = (tl >> 1) & 1u;
        if (!wait_bounded<true>(acce_bar(acc), aph ^ 1u, ab, kSiteMmaAccEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        int k_blocks = p.k_blocks, tail_steps = p.tail_steps;
        if constexpr (kGrouped) {
          const TileCtx tc = ctx_of(t, gi);
          k_blocks = tc.k_blocks;
          tail_steps = tc.tail_steps;
        }
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!wait_bounded<true>(full_bar(s), ph, ab, kSiteMmaFull)) {
            ok = false;
            break;
          }
          // No tcgen05 fence here: the TMA writes and the MMA reads of this
          // slot are both async-proxy operations ordered by the barrier's
          // transaction count, and a fence inside the accumulation chain
          // stalls the tensor pipe.
          const int nsteps = (kb == k_blocks - 1) ? tail_steps : kTileK / kUmmaK;
          issue_kblock<false>(d_tmem, alo0 + s * sstep, blo0 + s * sstep, hi, hi, astep, bstep,
                              p.idesc, nsteps, kb == 0);
          tc_commit(empty_bar(s));  // slot is free once these MMAs have read it
          if (++s == static_cast<uint32_t>(S)) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(accf_bar(acc));  // accumulator complete
      }
      // Every MMA this thread issued must finish before Tensor Memory is freed
      // (on an aborted run nobody else waits for them).
      tc_commit(drain_bar);
      drain_wait(drain_bar, 0u);
    }
  } else if (warp < 6) {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    float* stg = epi + (warp - 2) * 32 * kEpiPitch;
    uint8_t* boxes = reinterpret_cast<uint8_t*>(epi) + (warp - 2) * 2 * kEpiBoxBytes;
    const uint32_t boxes_addr = smem_addr(boxes);
    uint32_t nbox = 0;
    uint32_t tl = 0;
    for (uint32_t ti = 0;; ++ti, ++tl) {
      int64_t t;
      int gi;
      if (!next_tile(ti, t, gi, 0xffffffffu) || t >= p.tiles) break;
      const uint32_t acc = tl & 1u, aph = (tl >> 1) & 1u;
      const TileCtx tc = ctx_of(t, gi);
      const int b = tc.b, mb = tc.mb, nb = tc.nb;
      EpiArgs ea = epi_args(p);
      if constexpr (kGrouped) {
        ea = EpiArgs{tc.g->C, tc.g->ldc, tc.g->Mv, tc.g->Nv, p.c_bf16, 0, tc.g->c_tma,
                     tc.g->alpha, tc.g->beta};
      }
      const int row0 = mb * kTileM + q * 32;
      const int64_t cbase = static_cast<int64_t>(b) * p.sC;
      // row-major C with beta != 0 on the direct path: C_in two chunks deep,
      // the first chunk requested before the accumulator is ready
      const bool pre = BN >= 128 && ea.beta != 0.0f && !ea.c_tma && !ea.c_trans;
      float cin[32];
      if (pre) prefetch_cin(ea, cin, lane, row0, nb * BN, cbase);
      int ok = 1;
      if (lane == 0) ok = wait_bounded(accf_bar(acc), aph, ab, kSiteEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if constexpr (BN == 16) {
        float v[16];
        tmem_ld_16cols(taddr, v);
        tmem_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(acc));
        store_chunk<16>(ea, v, stg, lane, row0, nb * BN, cbase);
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
          if (ea.c_tma) {
            // A box wholly outside C is skipped outright: it neither writes a
            // box buffer nor takes a turn, so the buffer alternation matches
            // the committed store groups that the read-wait counts.
            if (row0 < ea.Mv && nb * BN + 32 * c < ea.Nv) {
              const uint32_t k = nbox++ & 1u;
              store_chunk_tma(ea, tc.map_c, v, boxes + k * kEpiBoxBytes,
                              boxes_addr + k * kEpiBoxBytes, lane, row0, nb * BN + 32 * c, b);
            }
          } else if (pre) {
            float nxt[32];
            if (c + 1 < BN / 32) prefetch_cin(ea, nxt, lane, row0, nb * BN + 32 * (c + 1), cbase);
            store_chunk_cin(ea, v, cin, stg, lane, row0, nb * BN + 32 * c, cbase);
#pragma unroll
            for (int r = 0; r < 32; ++r) cin[r] = nxt[r];
          } else {
            store_chunk<32>(ea, v, stg, lane, row0, nb * BN + 32 * c, cbase);
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();  // box stores done before shared memory is released
  } else {
    // ------------------------------------------------------- row loader
    if constexpr (!kDyn) {
      if (p.ldg_mask) {
        const int tid = (warp - 6) * 32 + lane;
        uint32_t it = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
          int b, mb, nb;
          decode_tile(t, p, b, mb, nb);
          const int m0 = mb * kTileM, n0 = nb * BN;
          for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
            const uint32_t s = it % S, ph = (it / S) & 1u;
            if (!(ok = warp_wait_bounded(empty_bar(s), ph ^ 1u, ab, kSiteProducerEmpty, lane))) break;
            uint8_t* a_tile = smem + s * p.stage_bytes;
            uint8_t* b_tile = a_tile + p.a_bytes;
            const int k0 = kb * kTileK;
            if (p.ldg_mask & 1)
              ldg_fill(a_tile, p.ldg[0], p.a_bcast ? 0 : b, p.a_mn ? k0 : m0, p.a_mn ? m0 : k0,
                       p.a_mn ? 64 : kTileM, p.a_mn ? 2 : 1, tid, kLdgWarps * 32);
            if (p.ldg_mask & 2)
              ldg_fill(b_tile, p.ldg[1], p.b_bcast ? 0 : b, p.b_mn ? k0 : n0, p.b_mn ? n0 : k0,
                       p.b_mn ? 64 : BN, p.b_mn ? BN / 64 : 1, tid, kLdgWarps * 32);
            fence_proxy_async_shared();  // the tensor core reads the stage through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(s));
          }
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

// Stream-K fixup of one epilogue warp's 32 accumulator rows (the piece with a
// split tile's first k-block): adds the partials that pairs [q_lo, q_hi)
// left in their workspace slots to the accumulator in Tensor Memory (columns
// taddr .. taddr + BN - 1), after which the epilogue reads it as a whole
// tile.  Chunk c of pair x's partial is 4 KB at p.sk_ws + (slot(x) + c) * 256
// float4.  The operand ring is idle when this runs (this piece is its pair's
// last item and all its MMAs are complete), so the partials come in by bulk
// copies into `region` (this warp's quarter of the ring: an mbarrier, then
// 4 KB buffers), as many chunks per batch as the buffers hold.
// Warp-wide bounded wait (acquire) for a contributor's flag to reach this
// launch's epoch.  False: the time limit passed (reported) or another role
// aborted.
__device__ __forceinline__ bool sk_wait_flag(const KParams& p, const uint32_t* f, int lane, Abort ab) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t spin = 0;; ++spin) {
    if (__all_sync(0xffffffffu, ld_acquire_gpu(f) == p.sk_epoch)) return true;
    if ((spin & 15u) == 15u) {
      int bad = 0;
      if (lane == 0) bad = *ab.flag ? 1 : (global_timer_ns() - t0 > ab.timeout_ns ? 2 : 0);
      bad = __shfl_sync(0xffffffffu, bad, 0);
      if (bad) {
        if (bad == 2 && lane == 0) {
          *ab.flag = 1u;
          atomicCAS(ab.err, 0u, kErrTag | (kSiteStreamK << 8) | (blockIdx.x & 0xFFu));
        }
        return false;
      }
    }
  }
}

template <int BN>
__device__ __forceinline__ bool sk_fixup(const KParams& p, uint8_t* region, uint32_t region_addr,
                                      uint32_t region_bytes, int64_t slot_base_stride, int64_t slot_off,
                                      int q_lo, int q_hi, uint32_t taddr, int lane, Abort ab) {
  const int n = q_hi - q_lo;
  // the contributors' flags: partial written (bounded wait, acquire)
  for (int x = q_lo; x < q_hi; ++x)
    if (!sk_wait_flag(p, p.sk_flags + (x * slot_base_stride + slot_off) / (BN / 32), lane, ab)) return false;
  const uint32_t bar = region_addr;
  const uint32_t nbuf = (region_bytes - 128u) / 4096u;
  const int per_batch = static_cast<int>(nbuf) / n;  // chunks per batch (n <= 2: at least 4)
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  uint32_t phase = 0;
  for (int c0 = 0; c0 < BN / 32; c0 += per_batch) {
    const int c1 = c0 + per_batch < BN / 32 ? c0 + per_batch : BN / 32;
    // contributor x's chunks c0 .. c1-1 are contiguous in its slot: one copy
    // each, into consecutive buffers
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>((c1 - c0) * n) * 4096u);
      for (int x = q_lo; x < q_hi; ++x)
        bulk_load(region_addr + 128u + static_cast<uint32_t>((x - q_lo) * (c1 - c0)) * 4096u,
                  p.sk_ws + (x * slot_base_stride + slot_off + c0) * 256, static_cast<uint32_t>(c1 - c0) * 4096u,
                  bar);
    }
    if (!warp_wait_bounded(bar, phase, ab, kSiteStreamK, lane)) return false;
    phase ^= 1u;
    for (int c = c0; c < c1; ++c) {
      float v[32];
      tmem_ld_32cols(taddr + 32u * c, v);
      tmem_wait_ld();
      for (int x = 0; x < n; ++x) {
        const float4* src = reinterpret_cast<const float4*>(region + 128u + (x * (c1 - c0) + (c - c0)) * 4096u) + lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 s4 = src[j * 32];
          v[4 * j] += s4.x;
          v[4 * j + 1] += s4.y;
          v[4 * j + 2] += s4.z;
          v[4 * j + 3] += s4.w;
        }
      }
      tmem_st_32cols(taddr + 32u * c, v);
    }
    tmem_wait_st();
    // the next batch's copies (async proxy) overwrite what was just read
    fence_proxy_async_shared();
    __syncwarp();
  }
  // consumed: clear the flags for the next launch
  if (lane == 0)
    for (int x = q_lo; x < q_hi; ++x) p.sk_flags[(x * slot_base_stride + slot_off) / (BN / 32)] = 0u;
  tc_fence_before_sync();
  return true;
}

// The owner's side of the two-way split: wait for contributor x's flag, bring
// its partial rows (BN / 32 chunks of 4 KB, contiguous in the slot) into
// this warp's quarter of the idle operand ring (`region`, past a 128-byte
// barrier) with one bulk copy, and clear the flag.  The epilogue then adds
// chunk c (float4 j of lane r at region + 128 + c * 4096 + (j * 32 + r) * 16)
// to the accumulator's columns as it stores them.
template <int BN>
__device__ __forceinline__ bool sk_fetch_partial(const KParams& p, uint32_t region_addr, int64_t slot_base_stride,
                                              int64_t slot_off, int x, int lane, Abort ab) {
  uint32_t* f = p.sk_flags + (x * slot_base_stride + slot_off) / (BN / 32);
  if (!sk_wait_flag(p, f, lane, ab)) return false;
  const uint32_t bar = region_addr;
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(BN / 32) * 4096u);
    bulk_load(region_addr + 128u, p.sk_ws + (x * slot_base_stride + slot_off) * 256,
              static_cast<uint32_t>(BN / 32) * 4096u, bar);
  }
  __syncwarp();
  if (!warp_wait_bounded(bar, 0u, ab, kSiteStreamK, lane)) return false;
  if (lane == 0) *f = 0u;  // consumed: cleared for the next launch
  return true;
}

// sk_keep_partial for a piece that is its pair's last item: the operand ring
// is idle once its accumulator is complete, so the warp lays out all its
// chunks in its quarter of the ring (`region`, past 128 bytes) and sends the
// whole partial (BN / 32 chunks of 4 KB, contiguous in the slot) by one bulk
// copy, then raises the flag.
template <int BN>
__device__ __forceinline__ void sk_keep_partial_ring(const KParams& p, float4* dst, uint32_t* flag,
                                                  uint32_t taddr, uint32_t acce, uint8_t* region,
                                                  uint32_t region_addr, int lane) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld_32cols(taddr + 32u * c, v);
    tmem_wait_ld();
    if (c == BN / 32 - 1) {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce);
    }
    float4* sb = reinterpret_cast<float4*>(region + 128u + c * 4096u) + lane;
#pragma unroll
    for (int j = 0; j < 8; ++j) sb[j * 32] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    bulk_store(dst, region_addr + 128u, static_cast<uint32_t>(BN / 32) * 4096u);
    bulk_commit_group();
    bulk_wait_group_all();       // the partial is written
    fence_proxy_async_global();  // ... and ordered before the flag
    __threadfence();
    st_release_gpu(flag, p.sk_epoch);
  }
  __syncwarp();
}

// Stream-K piece without its tile's first k-block (kind 1): this warp's 32
// accumulator rows go to its workspace slot `dst` instead of C, 4 KB per
// 32-column chunk (rows as lanes, 8 float4 per row: float4 j of lane r at
// j * 32 + r).  Each chunk is laid out in one of the warp's two box buffers
// and sent by one bulk copy (plain stores from the warp would queue in the
// SM's load/store path); the accumulator is released to the leader
// (`acce`), and once the copies have completed the flag is raised to this
// launch's epoch (release).  `nbox` is the warp's box count, shared with the
// C box stores so the buffer rotation and the read-waits stay in step.
template <int BN>
__device__ __forceinline__ void sk_keep_partial(const KParams& p, float4* dst, uint32_t* flag, uint32_t taddr,
                                             uint32_t acce, uint8_t* boxes, uint32_t boxes_addr,
                                             uint32_t& nbox, int lane) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld_32cols(taddr + 32u * c, v);
    tmem_wait_ld();
    if (c == BN / 32 - 1) {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce);
    }
    const uint32_t k = nbox++ & 1u;
    if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous copy has been read
    __syncwarp();
    float4* sb = reinterpret_cast<float4*>(boxes + k * kEpiBoxBytes) + lane;
#pragma unroll
    for (int j = 0; j < 8; ++j) sb[j * 32] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      bulk_store(dst + c * 256, boxes_addr + k * kEpiBoxBytes, kEpiBoxBytes);
      bulk_commit_group();
    }
  }
  if (lane == 0) {
    bulk_wait_group_all();       // the partial is written
    fence_proxy_async_global();  // ... and ordered before the flag
    __threadfence();
    st_release_gpu(flag, p.sk_epoch);
  }
  __syncwarp();
}

// bmm_tc2_kernel: the same pipeline over CTA pairs (a cluster of 2).  The
// pair computes a 256 x BN tile with tcgen05.mma.cta_group::2: CTA r holds
// rows [128r, 128r+128) of the A tile and rows [r*BN/2, (r+1)*BN/2) of the
// K x BN B tile in its own ring stage (32 KB at BN = 256), so each SM takes in
// a third less operand data per FLOP than a 1-CTA 128 x 256 tile and its
// tensor core reads half of B from the peer's shared memory.
//   - Both CTAs' TMA loads count on the leader's "full" barrier (the leader
//     expects the bytes of both halves); only the leader waits on it.
//   - The leader's single MMA thread issues 256 x BN x 16 MMAs and
//     multicasts each tcgen05.commit to the "empty" (slot) and "acc full"
//     barriers of both CTAs.
//   - Each CTA's epilogue drains its own 128 accumulator rows; the peer's
//     four warps release the accumulator by arriving on the leader's "acc
//     empty" barrier (8 arrivals per phase).
//   - A cluster barrier at the end keeps either CTA from exiting (or freeing
//     Tensor Memory) while the other can still signal it.
//   - kTail (stream-K tail, p.sk_tiles > 0): after its whole tiles each
//     pair runs at most two pieces, kSkEven: equal ranges (sk_piece; see
//     sk_keep_partial and sk_fixup), kSkTwoWay: one piece of a tile split in
//     two (sk_piece2; the owner adds the partial in its epilogue, see
//     sk_fetch_partial).  Separate instantiations, so launches without a
//     split run code with none of it.
constexpr int kSkEven = 1;
constexpr int kSkTwoWay = 2;

template <int BN, int kTail = 0>
__global__ void __launch_bounds__(kThreads, 1)
    bmm_tc2_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC) {
  constexpr bool kSK = kTail != 0;
  constexpr bool kTwo = kTail == kSkTwoWay;
  constexpr int BNH = BN / 2;  // B tile rows held by each CTA
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  const int S = p.stages;
  const uint32_t ring_bytes = static_cast<uint32_t>(S) * p.stage_bytes;
  float* epi = reinterpret_cast<float*>(smem + ring_bytes);
  const uint32_t bar0 = sbase + ring_bytes + p.epi_bytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + ring_bytes + p.epi_bytes + 8u * (2u * S + 5u));
  volatile uint32_t* abort_flag = tmem_slot + 1;

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);

  // The host sizes the ring to the launch's shared memory assuming the
  // dynamic region starts 1024-byte aligned (no pad); if it does not, every
  // CTA of the grid (all see the same base) leaves before touching shared
  // memory, with the error reported, instead of overrunning the region.
  if (pad + ring_bytes + p.epi_bytes + kBarBytes > dynamic_smem_size()) {
    if (threadIdx.x == 0) atomicCAS(p.err, 0u, kErrTag | (kSiteSmemLayout << 8) | (blockIdx.x & 0xFFu));
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  // whole tiles, round-robin over the pairs; then (stream-K) at most two pieces
  const int64_t dp_end = kSK ? p.sk_first : p.tiles;
  auto piece = [&](int si, SkPiece& pc) -> bool {
    if constexpr (kTwo) return si == 0 && sk_piece2(p, pair, pc);
    else return sk_piece(p, pair, si, pc);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1 + (p.ldg_mask ? 2 * kLdgWarps : 0));  // + both CTAs' row loaders
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 8);  // four epilogue warps in each CTA of the pair
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.c_tma) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), p.tmem_cols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const Abort ab{abort_flag, p.err, p.timeout_ns};

  if (warp == 0) {
    // --------------------------------------------- TMA producer (each CTA)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      // kLdg: some operand comes from the row loaders (its TMA loads are
      // skipped, and the leader may have no bytes to expect).  A separate copy
      // of the loop keeps the TMA-only issue sequence as it is.
      auto produce_dp = [&](auto has_ldg) {
        constexpr bool kLdg = decltype(has_ldg)::value;
        for (int64_t t = pair; t < p.tiles && ok; t += npairs) {
          int b, mb, nb;
          decode_tile(t, p, b, mb, nb);
          const int m_own = mb * (2 * kTileM) + static_cast<int>(rank) * kTileM;
          const int n_own = nb * BN + static_cast<int>(rank) * BNH;
          const int za = p.a_bcast ? 0 : b, zb = p.b_bcast ? 0 : b;
          for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
            const uint32_t s = it % S, ph = (it / S) & 1u;
            if (!wait_bounded<true>(empty_bar(s), ph ^ 1u, ab, kSiteProducerEmpty)) {
              ok = false;
              break;
            }
            const uint32_t a_dst = sbase + s * p.stage_bytes;
            const uint32_t b_dst = a_dst + p.a_bytes;
            if constexpr (kLdg) {
              if (leader) {
                if (p.tx_bytes) mbar_arrive_expect_tx(full_bar(s), 2u * p.tx_bytes);
                else mbar_arrive(full_bar(s));  // both operands come from the row loaders
              }
            } else {
              if (leader) mbar_arrive_expect_tx(full_bar(s), 2u * p.tx_bytes);
            }
            const uint32_t fb = mapa_shared(full_bar(s), 0);  // the leader's barrier
            const int k0 = kb * kTileK;
            if (!kLdg || !(p.ldg_mask & 1)) {
              if (!p.a_mn) {
                tma_load_3d_pair(a_dst, &tmA, fb, k0, m_own, za);
              } else {
                tma_load_3d_pair(a_dst, &tmA, fb, m_own, k0, za);
                tma_load_3d_pair(a_dst + 8192u, &tmA, fb, m_own + 64, k0, za);
              }
            }
            if (!kLdg || !(p.ldg_mask & 2)) {
              if (!p.b_mn) {
                tma_load_3d_pair(b_dst, &tmB, fb, k0, n_own, zb);
              } else {
#pragma unroll
                for (int h = 0; h < BNH / 64; ++h)
                  tma_load_3d_pair(b_dst + 8192u * h, &tmB, fb, n_own + 64 * h, k0, zb);
              }
            }
          }
        }
      };
      auto produce = [&](auto has_ldg) {
        constexpr bool kLdg = decltype(has_ldg)::value;
        // k-blocks [k_lo, k_hi) of tile t
        auto load_tile = [&](int64_t t, int k_lo, int k_hi) {
          int b, mb, nb;
          decode_tile(t, p, b, mb, nb);
          const int m_own = mb * (2 * kTileM) + static_cast<int>(rank) * kTileM;
          const int n_own = nb * BN + static_cast<int>(rank) * BNH;
          const int za = p.a_bcast ? 0 : b, zb = p.b_bcast ? 0 : b;
          for (int kb = k_lo; kb < k_hi; ++kb, ++it) {
            const uint32_t s = it % S, ph = (it / S) & 1u;
            if (!wait_bounded<true>(empty_bar(s), ph ^ 1u, ab, kSiteProducerEmpty)) {
              ok = false;
              break;
            }
            const uint32_t a_dst = sbase + s * p.stage_bytes;
            const uint32_t b_dst = a_dst + p.a_bytes;
            if constexpr (kLdg) {
              if (leader) {
                if (p.tx_bytes) mbar_arrive_expect_tx(full_bar(s), 2u * p.tx_bytes);
                else mbar_arrive(full_bar(s));  // both operands come from the row loaders
              }
            } else {
              if (leader) mbar_arrive_expect_tx(full_bar(s), 2u * p.tx_bytes);
            }
            const uint32_t fb = mapa_shared(full_bar(s), 0);  // the leader's barrier
            const int k0 = kb * kTileK;
            if (!kLdg || !(p.ldg_mask & 1)) {
              if (!p.a_mn) {
                tma_load_3d_pair(a_dst, &tmA, fb, k0, m_own, za);
              } else {
                tma_load_3d_pair(a_dst, &tmA, fb, m_own, k0, za);
                tma_load_3d_pair(a_dst + 8192u, &tmA, fb, m_own + 64, k0, za);
              }
            }
            if (!kLdg || !(p.ldg_mask & 2)) {
              if (!p.b_mn) {
                tma_load_3d_pair(b_dst, &tmB, fb, k0, n_own, zb);
              } else {
#pragma unroll
                for (int h = 0; h < BNH / 64; ++h)
                  tma_load_3d_pair(b_dst + 8192u * h, &tmB, fb, n_own + 64 * h, k0, zb);
              }
            }
          }
        };
        for (int64_t t = pair; t < dp_end && ok; t += npairs) load_tile(t, 0, p.k_blocks);
        if constexpr (kSK) {
          SkPiece pc;
          for (int si = 0; si < 2 && ok && piece(si, pc); ++si) load_tile(pc.tile, pc.ka, pc.kb);
        }
      };
      if constexpr (!kSK) {
        if (p.ldg_mask) produce_dp(BoolC<true>{});
        else produce_dp(BoolC<false>{});
      } else {
        if (p.ldg_mask) produce(BoolC<true>{});
        else produce(BoolC<false>{});
      }
      // The leader's full barriers count both CTAs' bytes: once the last S
      // have completed, no load of either CTA is still in flight.
      if (leader) {
        const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0u;
        for (uint32_t j = first; j < it; ++j) drain_wait(full_bar(j % S), (j / S) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer (leader only)
    if (lane == 0 && leader) {
      const uint32_t alo0 = desc_lo(sbase, p.a_mn ? 8192u : 16u);
      const uint32_t blo0 = desc_lo(sbase + p.a_bytes, p.b_mn ? 8192u : 16u);
      const uint32_t hi = desc_hi_sw128(1024u);
      const uint32_t astep = (p.a_mn ? 2048u : 32u) >> 4, bstep = (p.b_mn ? 2048u : 32u) >> 4;
      const uint32_t sstep = p.stage_bytes >> 4;
      uint32_t s = 0, ph = 0, tl = 0;
      bool ok = !p.test_stall || wait_bounded(drain_bar, 0u, ab, kSiteTestStall);
      // kClusterAcq: the peer's row loader writes its stage with plain stores,
      // so the full waits take its release at cluster scope (a separate copy
      // of the loop keeps the TMA-only path's issue loop as it is)
      auto mma_dp = [&](auto cluster_acq) {
        constexpr bool kClusterAcq = decltype(cluster_acq)::value;
        for (int64_t t = pair; t < p.tiles && ok; t += npairs, ++tl) {
          const uint32_t acc = tl & 1u, aph = (tl >> 1) & 1u;
          if (!wait_bounded<true>(acce_bar(acc), aph ^ 1u, ab, kSiteMmaAccEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + acc * BN;
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!(kClusterAcq ? wait_bounded_cluster(full_bar(s), ph, ab, kSiteMmaFull)
                              : wait_bounded<true>(full_bar(s), ph, ab, kSiteMmaFull))) {
              ok = false;
              break;
            }
            // No tcgen05 fence here (see the single-CTA kernel).
            const int nsteps = (kb == p.k_blocks - 1) ? p.tail_steps : kTileK / kUmmaK;
            issue_kblock<true>(d_tmem, alo0 + s * sstep, blo0 + s * sstep, hi, hi, astep, bstep,
                               p.idesc, nsteps, kb == 0);
            tc_commit_pair_multicast(empty_bar(s), 0x3);  // slot free in both CTAs
            if (++s == static_cast<uint32_t>(S)) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_pair_multicast(accf_bar(acc), 0x3);  // accumulator halves complete
        }
      };
      auto mma_tiles = [&](auto cluster_acq) {
        constexpr bool kClusterAcq = decltype(cluster_acq)::value;
        // k-blocks [k_lo, k_hi) of the next tile into accumulator tl & 1
        auto mma_tile = [&](int k_lo, int k_hi) {
          const uint32_t acc = tl & 1u, aph = (tl >> 1) & 1u;
          if (!wait_bounded<true>(acce_bar(acc), aph ^ 1u, ab, kSiteMmaAccEmpty)) {
            ok = false;
            return;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + acc * BN;
          for (int kb = k_lo; kb < k_hi; ++kb) {
            if (!(kClusterAcq ? wait_bounded_cluster(full_bar(s), ph, ab, kSiteMmaFull)
                              : wait_bounded<true>(full_bar(s), ph, ab, kSiteMmaFull))) {
              ok = false;
              break;
            }
            // No tcgen05 fence here (see the single-CTA kernel).
            const int nsteps = (kb == p.k_blocks - 1) ? p.tail_steps : kTileK / kUmmaK;
            issue_kblock<true>(d_tmem, alo0 + s * sstep, blo0 + s * sstep, hi, hi, astep, bstep,
                               p.idesc, nsteps, kb == k_lo);
            tc_commit_pair_multicast(empty_bar(s), 0x3);  // slot free in both CTAs
            if (++s == static_cast<uint32_t>(S)) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!ok) return;
          tc_commit_pair_multicast(accf_bar(acc), 0x3);  // accumulator halves complete
        };
        for (int64_t t = pair; t < dp_end && ok; t += npairs, ++tl) mma_tile(0, p.k_blocks);
        if constexpr (kSK) {
          SkPiece pc;
          for (int si = 0; si < 2 && ok && piece(si, pc); ++si, ++tl) mma_tile(pc.ka, pc.kb);
        }
      };
      if constexpr (!kSK) {
        if (p.ldg_mask) mma_dp(BoolC<true>{});
        else mma_dp(BoolC<false>{});
      } else {
        if (p.ldg_mask) mma_tiles(BoolC<true>{});
        else mma_tiles(BoolC<false>{});
      }
      tc_commit_pair(drain_bar);
      drain_wait(drain_bar, 0u);
    }
  } else if (warp < 6) {
    // ------------------------------------------------ epilogue (each CTA)
    const int q = warp & 3;
    const uint32_t box_bytes = p.box_bytes;
    uint8_t* boxes = reinterpret_cast<uint8_t*>(epi) + (warp - 2) * 2 * box_bytes;
    // the direct-store staging tile: packed after the other warps' tiles, or
    // (stream-K) inside this warp's own box space, which a piece that keeps
    // its partial also stages through, so no warp's tile overlaps another's
    // buffers
    float* stg = kSK ? reinterpret_cast<float*>(boxes) : epi + (warp - 2) * 32 * kEpiPitch;
    const uint32_t boxes_addr = smem_addr(boxes);
    uint32_t nbox = 0;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    const uint32_t acce_leader1 = mapa_shared(acce_bar(1), 0);
    uint32_t tl = 0;
    const EpiArgs ea = epi_args(p);
    // row-major C with beta != 0 on the direct path: C_in two chunks deep
    const bool pre = p.beta != 0.0f && !p.c_tma && !p.c_trans;
    // Whole tiles first (round-robin), then at most two stream-K pieces: a
    // piece without its tile's first k-block keeps its partial, the piece
    // with it adds the others' partials before storing the tile as usual.
    int64_t t_next = pair;
    int si = 0;
    for (;; ++tl) {
      int64_t t;
      int kind = 0;
      SkPiece pc;
      if (t_next < dp_end) {
        t = t_next;
        t_next += npairs;
      } else if (kSK && si < 2 && piece(si, pc)) {
        ++si;
        t = pc.tile;
        kind = pc.kind;
      } else {
        break;
      }
      const uint32_t acc = tl & 1u, aph = (tl >> 1) & 1u;
      int b, mb, nb;
      decode_tile(t, p, b, mb, nb);
      const int row0 = mb * (2 * kTileM) + static_cast<int>(rank) * kTileM + q * 32;
      const int n0 = nb * BN;  // the tile's first column
      const int64_t cbase = static_cast<int64_t>(b) * p.sC;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      float cin[32];
      if (pre && kind == 0) prefetch_cin(ea, cin, lane, row0, n0, cbase);
      // the epilogue waits a whole mainloop: lane 0 parks (no spinning that
      // would take issue slots from the producer and MMA threads)
      int okw = 1;
      if (lane == 0) okw = wait_bounded(accf_bar(acc), aph, ab, kSiteEpiAccFull) ? 1 : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      if (!okw) break;
      __syncwarp();
      tc_fence_after_sync();
      constexpr int64_t slot_stride = 2 * 4 * (BN / 32);  // float4 blocks of 4 KB per pair
      if (kSK && kind == 1) {
        const int64_t slot_off = (rank * 4 + q) * (BN / 32);
        float4* dst = p.sk_ws + (pair * slot_stride + slot_off) * 256;
        uint32_t* flag = p.sk_flags + (pair * 2 + rank) * 4 + q;
        const uint32_t acce = acc ? acce_leader1 : acce_leader0;
        SkPiece after;
        if (!piece(si, after)) {  // the pair's last item: the ring is idle
          const uint32_t quarter_bytes = ring_bytes / 4u;
          sk_keep_partial_ring<BN>(p, dst, flag, taddr, acce, smem + (warp - 2) * quarter_bytes,
                                   sbase + (warp - 2) * quarter_bytes, lane);
        } else {
          sk_keep_partial<BN>(p, dst, flag, taddr, acce, boxes, boxes_addr, nbox, lane);
        }
        continue;
      }
      // two-way split owner: the contributor's partial rows, added chunk by chunk below
      const float4* part = nullptr;
      if (kSK && kind == 2) {
        const int64_t slot_off = (rank * 4 + q) * (BN / 32);
        const uint32_t quarter_bytes = ring_bytes / 4u;
        if constexpr (kTwo) {
          if (!sk_fetch_partial<BN>(p, sbase + (warp - 2) * quarter_bytes, slot_stride, slot_off, pc.q_lo, lane,
                                    ab))
            break;
          part = reinterpret_cast<const float4*>(smem + (warp - 2) * quarter_bytes + 128u) + lane;
        } else {
          if (!sk_fixup<BN>(p, smem + (warp - 2) * quarter_bytes, sbase + (warp - 2) * quarter_bytes,
                            quarter_bytes, slot_stride, slot_off, pc.q_lo, pc.q_hi, taddr, lane, ab))
            break;
        }
        if (pre) prefetch_cin(ea, cin, lane, row0, n0, cbase);
      }
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld_32cols(taddr + 32u * c, v);
        tmem_wait_ld();
        if (c == BN / 32 - 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc ? acce_leader1 : acce_leader0);
        }
        if (kTwo && part) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 s4 = part[c * 256 + j * 32];
            v[4 * j] += s4.x;
            v[4 * j + 1] += s4.y;
            v[4 * j + 2] += s4.z;
            v[4 * j + 3] += s4.w;
          }
        }
        if (p.c_tma) {
          // skipped outright when wholly outside C (see the single-CTA kernel)
          if (row0 < p.Mv && n0 + 32 * c < p.Nv) {
            const uint32_t k = nbox++ & 1u;
            store_chunk_tma(ea, &tmC, v, boxes + k * box_bytes, boxes_addr + k * box_bytes, lane,
                            row0, n0 + 32 * c, b);
          }
        } else if (pre) {
          float nxt[32];
          if (c + 1 < BN / 32) prefetch_cin(ea, nxt, lane, row0, n0 + 32 * (c + 1), cbase);
          store_chunk_cin(ea, v, cin, stg, lane, row0, n0 + 32 * c, cbase);
#pragma unroll
          for (int r = 0; r < 32; ++r) cin[r] = nxt[r];
        } else {
          store_chunk<32>(ea, v, stg, lane, row0, n0 + 32 * c, cbase);
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();
  } else {
    // ---------------------------------------------- row loader (each CTA)
    if (p.ldg_mask) {
      const int tid = (warp - 6) * 32 + lane;
      uint32_t it = 0;
      bool ok = true;
      for (int64_t t = pair; t < p.tiles && ok; t += npairs) {
        int b, mb, nb;
        decode_tile(t, p, b, mb, nb);
        const int m_own = mb * (2 * kTileM) + static_cast<int>(rank) * kTileM;
        const int n_own = nb * BN + static_cast<int>(rank) * BNH;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1u;
          if (!(ok = warp_wait_bounded(empty_bar(s), ph ^ 1u, ab, kSiteProducerEmpty, lane))) break;
          uint8_t* a_tile = smem + s * p.stage_bytes;
          uint8_t* b_tile = a_tile + p.a_bytes;
          const int k0 = kb * kTileK;
          if (p.ldg_mask & 1)
            ldg_fill(a_tile, p.ldg[0], p.a_bcast ? 0 : b, p.a_mn ? k0 : m_own, p.a_mn ? m_own : k0,
                     p.a_mn ? 64 : kTileM, p.a_mn ? 2 : 1, tid, kLdgWarps * 32);
          if (p.ldg_mask & 2)
            ldg_fill(b_tile, p.ldg[1], p.b_bcast ? 0 : b, p.b_mn ? k0 : n_own, p.b_mn ? n_own : k0,
                     p.b_mn ? 64 : BNH, p.b_mn ? BNH / 64 : 1, tid, kLdgWarps * 32);
          fence_proxy_async_shared();  // the tensor core reads the stage through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(full_bar(s), 0));  // the leader's barrier
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // no CTA of the pair signals the other after this point
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem_base, p.tmem_cols);
}

// Copy a strided 16-bit operand into the workspace with ld rounded up to a
// multiple of 8 elements (16 bytes), which TMA needs for its row strides.
// Each thread moves one 8-element segment of a row: the one or two aligned
// 16-byte words that hold it are loaded (the second only when the segment
// reaches into it, so no load touches a 16-byte word without a byte of the
// operand: every load stays on a page the operand occupies) and the segment
// is shifted out of them in registers (source rows need only 2-byte
// alignment), then stored with one 16-byte store.  Columns past the row end
// are written as zero; TMA never reads them.
static __global__ void pack16_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                              int64_t nb, int64_t rows, int64_t cols, int64_t ld_src,
                              int64_t s_src, int64_t ld_dst, int64_t s_dst) {
  const int64_t segs = (cols + 7) / 8;
  const int64_t total = nb * rows * segs;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = t / segs, seg = t - row * segs;
    const int64_t b = row / rows, i = row - b * rows;
    const uint16_t* s = src + b * s_src + i * ld_src + seg * 8;
    const int64_t n = (cols - seg * 8) < 8 ? (cols - seg * 8) : 8;
    const uintptr_t a = reinterpret_cast<uintptr_t>(s);
    const uint4* w = reinterpret_cast<const uint4*>(a & ~static_cast<uintptr_t>(15));
    const uint32_t sh = static_cast<uint32_t>(a & 15u);
    const uint4 lo = __ldg(w);
    const uint4 hi = sh + 2u * static_cast<uint32_t>(n) > 16u ? __ldg(w + 1) : make_uint4(0u, 0u, 0u, 0u);
    uint4 q = extract16(lo, hi, sh);
    if (n < 8) {  // the row's last segment: zero the columns past its end
      uint32_t e[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (2 * j >= n) e[j] = 0u;
        else if (2 * j + 1 >= n) e[j] &= 0xFFFFu;
      }
      q = make_uint4(e[0], e[1], e[2], e[3]);
    }
    *reinterpret_cast<uint4*>(dst + b * s_dst + i * ld_dst + seg * 8) = q;
  }
}

// C = beta * C (beta == 0 writes zeros without reading C): the alpha == 0 or
// K == 0 case, where A and B are not read.
static __global__ void scale_c_kernel(void* C, int c_bf16, int64_t batch, int64_t M, int64_t N,
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

// C ABI of the batched product (declared in include/bmm.h): validation,
// planning, tensor-map encoding and kernel launches.  All compute runs in the
// kernels of bmm_kernel.cuh; this file only decides and enqueues.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/bmm.h"
#include "bmm_kernel.cuh"

namespace {

using dmt::KParams;

constexpr int32_t kVersion = (0 << 16) | 1;
constexpr int kGb300Sms = 152;
constexpr int64_t kMaxDim = 0x7fffffffLL;

// One MMA operand (A = rows of D, B = columns of D) as it sits in memory.
struct Operand {
  int user;          // 0: the caller's A, 1: the caller's B
  int mn_major;      // 1: the MMA's M (or N) index is the contiguous one
  int64_t rows, cols;// stored matrix per batch item (row-major, `ld`)
  int64_t ld, stride;
  int bcast;         // one batch item shared by all
  int pack;          // 0: TMA from the caller's memory; 1: staged into the workspace
                     // first; 2: read by the kernel's row loader (no staging)
  int64_t pld, pstride, ws_off;
  int box_rows;      // TMA box rows for a K-major operand (128 or BN)
};

struct Planned {
  int swap;
  int pair;          // 1: CTA pairs (2-SM MMA, 256-row tiles)
  int64_t batch, Mv, Nv, K;
  Operand a, b;
  int bn, stages;
  int stages_bf16_box;       // CTA pairs: ring depth of launches whose C goes out as bf16 box stores
  uint32_t stage_bytes, a_bytes, tx_bytes, idesc, tmem_cols;
  int64_t tiles, smem_bytes, workspace_bytes;
  int32_t num_m, num_n, k_blocks, tail_steps;
  int sk;                    // stream-K tail allowed (CTA pairs, K >= kSkMinKBlocks k-blocks)
  int64_t sk_bytes;          // its workspace: flags, then one partial slot per CTA pair
};

// Stream-K needs enough k-blocks per tile for a piece of the tail to be worth
// its partial's round trip through memory.
constexpr int kSkMinKBlocks = 32;
constexpr int64_t kSkFlagBytes = 64 * 1024;  // flags region: up to 2048 pairs x 2 CTAs x 4 warps

// Workspace of the stream-K tail for `pairs` CTA pairs and tile width bn:
// the flags, then per pair its two CTAs' 128 x bn fp32 partials.
int64_t sk_workspace_bytes(int64_t pairs, int bn) {
  return kSkFlagBytes + pairs * 2 * dmt::kTileM * bn * 4;
}

// DMT_BMM_STREAMK: "0" never splits, "1" splits whenever a plan allows it,
// unset lets the planner's estimate decide.
int stream_k_mode() {
  const char* e = std::getenv("DMT_BMM_STREAMK");
  if (e && e[0] == '0') return 0;
  if (e && e[0] == '1') return 2;
  return 1;
}

// Fewest k-blocks in a stream-K piece: kSkMinUnits, and at least half a
// tile's, so the owner of a split tile adds at most two partials.
int64_t sk_min_units(int64_t k_blocks) {
  const int64_t half = (k_blocks + 1) / 2;
  return half > dmt::kSkMinUnits ? half : dmt::kSkMinUnits;
}

// Two-way split: the contributor's k-blocks.  Its partial reaches the
// workspace about kSkPublishKBlocks k-block times after its accumulator (the
// owner's side then costs little more than the usual epilogue), so the
// owner takes that many more k-blocks than the contributor.
// DMT_BMM_SK_PUBLISH_KB overrides the constant (comparisons).
constexpr int64_t kSkPublishKBlocks = 16;

int64_t sk_publish_kblocks() {
  const char* e = std::getenv("DMT_BMM_SK_PUBLISH_KB");
  if (e && *e) {
    const long v = std::atol(e);
    if (v >= 0 && v < 4096) return v;
  }
  return kSkPublishKBlocks;
}

int64_t sk_contributor_kblocks(int64_t k_blocks) {
  const int64_t c = (k_blocks - sk_publish_kblocks()) / 2;
  return c < 1 ? 1 : (c > k_blocks / 2 ? k_blocks / 2 : c);
}

// Cost of the split tail's fixup (a piece's partial written and read back,
// and the owner's wait) in units of "one round of tile columns": measured
// as about a quarter of a round of 256-wide tiles.
constexpr int64_t kSkFixupCost = 64;

// ... and of the two-way split's: the owner's copy of the partial and its
// add in the epilogue, and 256-wide rounds against the balanced width's
// (measured on 4096^3: the split ends with 224-wide whole rounds, its three
// 256-wide rounds taking 3.6 us longer than three 224-wide ones).
constexpr int64_t kSkTwoWayCost = 40;

// Time of one round of CTA-pair tiles of width bn in the same units (a
// round of 256-wide tiles = 256): measured over four whole rounds, a
// 224-wide round takes 0.93 and a 192-wide one 0.90 of a 256-wide one (the
// k-block's cost hardly depends on the tile width).
int64_t round_cost(int bn) { return bn == 256 ? 256 : bn == 224 ? 238 : bn == 192 ? 232 : bn; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool is16(int32_t t) { return t == BMM_BF16 || t == BMM_F16; }

bmm_status_t validate(const bmm_desc_t* d) {
  if (!d) return BMM_ERR_INVALID_ARG;
  if (d->batch < 0 || d->M < 0 || d->N < 0 || d->K < 0) return BMM_ERR_INVALID_ARG;
  if (d->transA != 0 && d->transA != 1) return BMM_ERR_INVALID_ARG;
  if (d->transB != 0 && d->transB != 1) return BMM_ERR_INVALID_ARG;
  if (!is16(d->typeA) || d->typeB != d->typeA) return BMM_ERR_INVALID_ARG;
  if (d->typeC != BMM_F32 && d->typeC != BMM_BF16) return BMM_ERR_INVALID_ARG;
  if (d->strideA < 0 || d->strideB < 0 || d->strideC < 0) return BMM_ERR_INVALID_ARG;
  const int64_t a_cols = d->transA ? d->M : d->K;
  const int64_t b_cols = d->transB ? d->K : d->N;
  if (d->lda < (a_cols > 1 ? a_cols : 1)) return BMM_ERR_INVALID_ARG;
  if (d->ldb < (b_cols > 1 ? b_cols : 1)) return BMM_ERR_INVALID_ARG;
  if (d->ldc < (d->N > 1 ? d->N : 1)) return BMM_ERR_INVALID_ARG;
  if (d->batch > 1 && d->M > 0 && d->N > 0 && d->strideC < (d->M - 1) * d->ldc + d->N)
    return BMM_ERR_INVALID_ARG;  // batch items of C would overlap
  if (d->batch > kMaxDim || d->M > kMaxDim || d->N > kMaxDim || d->K > kMaxDim)
    return BMM_ERR_UNSUPPORTED;
  return BMM_OK;
}

// Tile N for the large class, chosen to balance waves: the persistent grid
// runs ceil(tiles / units) rounds of tiles whose cost grows with N, so the
// estimate rounds x N is minimised over the tile widths the operand layout
// allows (a 4096-wide problem on 76 CTA pairs: 256 -> 4 rounds of 256,
// 224 -> 4 rounds of 224, so 224).  Ties keep the wider tile.
int balanced_tile_n(int64_t batch, int64_t Mv, int64_t Nv, int tile_m, int64_t units,
                    const int* cands, int ncand) {
  int best = cands[0];
  int64_t best_cost = -1;
  for (int i = 0; i < ncand; ++i) {
    const int bn = cands[i];
    const int64_t tiles = batch * ((Mv + tile_m - 1) / tile_m) * ((Nv + bn - 1) / bn);
    const int64_t rounds = (tiles + units - 1) / units;
    const int64_t cost = rounds * bn;
    if (best_cost < 0 || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

// Shape classes and resources.  Pure host arithmetic (no CUDA calls); `sms`
// is the device's SM count (152 on GB300).
// row_loader: operands TMA cannot address go through the kernel's row loader
// instead of the staging copy (DMT_BMM_LDG=1, or no workspace to stage in).
bool row_loader_requested() {
  const char* e = std::getenv("DMT_BMM_LDG");
  return e && e[0] == '1';
}

void plan(const bmm_desc_t* d, Planned* P, int sms, bool row_loader, bool allow_sk = true) {
  std::memset(P, 0, sizeof(*P));
  // Skinny M: compute C^T = op(B)^T op(A)^T so that N fills the 128-row MMA.
  P->swap = (d->M <= 64 && d->N > d->M) ? 1 : 0;
  P->batch = d->batch;
  P->K = d->K;
  Operand ua{}, ub{};
  ua.user = 0;
  ua.rows = d->transA ? d->K : d->M;
  ua.cols = d->transA ? d->M : d->K;
  ua.ld = d->lda;
  ua.stride = d->strideA;
  ub.user = 1;
  ub.rows = d->transB ? d->N : d->K;
  ub.cols = d->transB ? d->K : d->N;
  ub.ld = d->ldb;
  ub.stride = d->strideB;
  if (!P->swap) {
    P->Mv = d->M;
    P->Nv = d->N;
    P->a = ua;
    P->b = ub;
    P->a.mn_major = d->transA ? 1 : 0;  // A stored K x M: M contiguous
    P->b.mn_major = d->transB ? 0 : 1;  // B stored K x N: N contiguous
  } else {
    P->Mv = d->N;
    P->Nv = d->M;
    P->a = ub;
    P->b = ua;
    P->a.mn_major = d->transB ? 0 : 1;
    P->b.mn_major = d->transA ? 1 : 0;
  }
  // Tile N: the smallest of 16..256 that covers Nv.  An MN-major B tile is
  // loaded in 64-wide boxes (one 128-byte swizzle row), so it needs BN >= 64.
  int bn = 256;
  if (P->Nv <= 16 && !P->b.mn_major) bn = 16;
  else if (P->Nv <= 32 && !P->b.mn_major) bn = 32;
  else if (P->Nv <= 64) bn = 64;
  else if (P->Nv <= 128) bn = 128;
  // Large tiles run on CTA pairs (tcgen05 cta_group::2, 256 rows per pair):
  // each SM then takes in a third less operand data per FLOP.  The
  // environment variable DMT_BMM_PAIR=0 keeps the 1-CTA kernel (comparisons).
  const char* pe = std::getenv("DMT_BMM_PAIR");
  const bool pair_off = pe && pe[0] == '0';
  P->pair = (bn == 256 && P->Mv > dmt::kTileM && !pair_off) ? 1 : 0;
  const int tile_m = P->pair ? 2 * dmt::kTileM : dmt::kTileM;
  const int64_t k_blocks = (P->K + dmt::kTileK - 1) / dmt::kTileK;
  // Stream-K tail: with the leftover tiles split along K, the widest tile is
  // the fastest per FLOP (a round of 256-wide pair tiles takes about as long
  // as one of 224-wide), so no width is traded for a whole number of rounds.
  const int sk_mode = stream_k_mode();
  const bool sk_ok = allow_sk && P->pair && k_blocks >= kSkMinKBlocks && !row_loader && sk_mode > 0;
  const bool large = bn == 256;
  if (large) {
    // K-major B tiles may be any multiple of 16 rows; MN-major B tiles are
    // loaded in 64-column boxes (per CTA of a pair: BN/2 columns).
    static const int kK[3] = {256, 224, 192};
    static const int kMnSingle[2] = {256, 192};
    const int units = P->pair ? sms / 2 : sms;
    const int64_t u = units > 0 ? units : 1;
    if (!P->b.mn_major)
      bn = balanced_tile_n(P->batch, P->Mv, P->Nv, tile_m, u, kK, 3);
    else if (!P->pair)
      bn = balanced_tile_n(P->batch, P->Mv, P->Nv, tile_m, u, kMnSingle, 2);
    if (sk_ok) {
      // Estimated cost in rounds of 256-wide tiles (x 256): whole rounds of
      // the balanced width, against 256-wide tiles whose leftover round is
      // split along K: two ways (the owner's share of a round plus its
      // fixup) when at most half the pairs hold a leftover tile, else in
      // equal ranges (the leftover's share of a round plus the fixup).  No
      // leftover: no split.
      const int64_t tiles_b = P->batch * ((P->Mv + tile_m - 1) / tile_m) * ((P->Nv + bn - 1) / bn);
      const int64_t cost_b = (tiles_b + u - 1) / u * round_cost(bn);
      const int64_t tiles_s = P->batch * ((P->Mv + tile_m - 1) / tile_m) * ((P->Nv + 255) / 256);
      const int64_t rem = tiles_s % u;
      const int64_t owner = k_blocks - sk_contributor_kblocks(k_blocks);
      const int64_t cost_s = rem == 0       ? tiles_s / u * 256
                             : 2 * rem <= u ? tiles_s / u * 256 + owner * 256 / k_blocks + kSkTwoWayCost
                                            : tiles_s * 256 / u + kSkFixupCost;
      if (sk_mode == 2 || cost_s < cost_b) {
        bn = 256;
        P->sk = rem != 0 ? 1 : 0;
      }
    }
  }
  if (large) {
    static const int kK[3] = {256, 224, 192};
    static const int kMnSingle[2] = {256, 192};
    // DMT_BMM_TILE_N pins one of the widths this layout allows (comparisons).
    const char* te = std::getenv("DMT_BMM_TILE_N");
    if (te && *te) {
      const int want = std::atoi(te);
      const int* c = !P->b.mn_major ? kK : (P->pair ? kK : kMnSingle);
      const int n = !P->b.mn_major ? 3 : (P->pair ? 1 : 2);
      for (int i = 0; i < n; ++i)
        if (c[i] == want) bn = want;
    }
  }
  P->bn = bn;
  P->sk_bytes = P->sk ? sk_workspace_bytes(sms / 2 > 0 ? sms / 2 : 1, bn) : 0;
  const int b_rows = P->pair ? bn / 2 : bn;  // B tile rows held by one CTA
  P->a.box_rows = dmt::kTileM;
  P->b.box_rows = b_rows;

  // TMA needs 16-byte row and batch strides; otherwise stage a copy with
  // ld rounded up to 8 elements.
  int64_t ws = 0;
  for (Operand* o : {&P->a, &P->b}) {
    o->bcast = (o->stride == 0 || d->batch <= 1) ? 1 : 0;
    const bool ld_ok = (o->ld * 2) % 16 == 0;
    const bool st_ok = o->bcast || (o->stride * 2) % 16 == 0;
    o->pack = (ld_ok && st_ok) ? 0 : (row_loader ? 2 : 1);
    if (o->pack == 1) {
      o->pld = round_up(o->cols, 8);
      o->pstride = o->rows * o->pld;
      o->ws_off = ws;
      const int64_t nb = o->bcast ? 1 : d->batch;
      ws = round_up(ws + nb * o->pstride * 2, 256);
    }
  }
  P->workspace_bytes = ws;

  P->a_bytes = static_cast<uint32_t>(dmt::kTileM * dmt::kTileK * 2);
  const uint32_t b_bytes = static_cast<uint32_t>(b_rows * dmt::kTileK * 2);
  P->stage_bytes = static_cast<uint32_t>(round_up(P->a_bytes + b_bytes, 1024));
  // TMA bytes per stage and CTA: the row loader's operands are not counted
  P->tx_bytes = (P->a.pack == 2 ? 0u : P->a_bytes) + (P->b.pack == 2 ? 0u : b_bytes);
  const int64_t fixed = 1024 + dmt::kEpiBytes + dmt::kBarBytes;
  int stages = static_cast<int>((dmt::kSmemLimit - fixed) / P->stage_bytes);
  // At most 8 stages: only the narrow tiles (BN 16 and 32) fit more, and on the
  // HBM-bound skinny product 8 in flight per SM measured 4% faster than 10
  // (more outstanding loads than HBM serves well); 6, 5 and 4 were slower.
  if (stages > dmt::kMaxStages) stages = dmt::kMaxStages;
  // DMT_BMM_STAGES caps the ring depth (comparisons; at least 2)
  const char* se = std::getenv("DMT_BMM_STAGES");
  if (se && *se) {
    const int cap = std::atoi(se);
    if (cap >= 2 && cap < stages) stages = cap;
  }
  P->stages = stages;
  P->smem_bytes = fixed + static_cast<int64_t>(stages) * P->stage_bytes;
  // CTA pairs whose C may go out as bf16 through TMA box stores: those
  // launches need only half the epilogue region, and the ring takes what it
  // frees (256 x 224 and 256 x 192 tiles: one more stage).  This layout
  // counts on the dynamic region starting 1024-byte aligned; the kernel
  // checks that and reports an error (no access) if it does not.
  P->stages_bf16_box = stages;
  if (P->pair && d->typeC == BMM_BF16 && !P->swap) {
    int deep = static_cast<int>((dmt::kSmemLimit - dmt::kEpiBytesBf16 - dmt::kBarBytes) / P->stage_bytes);
    if (deep > dmt::kMaxStages) deep = dmt::kMaxStages;
    if (se && *se) {
      const int cap = std::atoi(se);
      if (cap >= 2 && cap < deep) deep = cap;
    }
    if (deep > stages) {
      P->stages_bf16_box = deep;
      P->smem_bytes = dmt::kSmemLimit;
    }
  }

  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(2 * bn)) cols <<= 1;
  P->tmem_cols = cols;

  const uint32_t fmt = (d->typeA == BMM_BF16) ? 1u : 0u;  // 0 = fp16, 1 = bf16
  P->idesc = (1u << 4)                                   // D format: fp32
             | (fmt << 7) | (fmt << 10)                  // A and B formats
             | (static_cast<uint32_t>(P->a.mn_major) << 15) |
             (static_cast<uint32_t>(P->b.mn_major) << 16) |
             (static_cast<uint32_t>(bn >> 3) << 17)      // N / 8
             | (static_cast<uint32_t>(tile_m >> 4) << 24);  // M / 16

  P->num_m = static_cast<int32_t>((P->Mv + tile_m - 1) / tile_m);
  P->num_n = static_cast<int32_t>((P->Nv + bn - 1) / bn);
  P->tiles = P->batch * P->num_m * P->num_n;
  P->k_blocks = static_cast<int32_t>((P->K + dmt::kTileK - 1) / dmt::kTileK);
  const int64_t rem = P->K % dmt::kTileK;
  P->tail_steps = rem == 0 ? dmt::kTileK / dmt::kUmmaK
                           : static_cast<int32_t>((rem + dmt::kUmmaK - 1) / dmt::kUmmaK);
}

void fill_info(const Planned& P, const bmm_desc_t* d, bmm_plan_info_t* info) {
  std::memset(info, 0, sizeof(*info));
  info->tile_m = P.pair ? 2 * dmt::kTileM : dmt::kTileM;
  info->tile_n = P.bn;
  info->tile_k = dmt::kTileK;
  info->stages = P.stages;
  info->stages_bf16_box = P.stages_bf16_box;
  info->swap_ab = P.swap;
  info->pack_a = P.swap ? P.b.pack : P.a.pack;
  info->pack_b = P.swap ? P.a.pack : P.b.pack;
  info->even_k = (d->K % dmt::kTileK) == 0 ? 1 : 0;
  info->tmem_cols = static_cast<int32_t>(P.tmem_cols);
  info->cta_pair = P.pair;
  info->tiles = P.tiles;
  info->smem_bytes = P.smem_bytes;
  info->stage_bytes = P.stage_bytes;
  info->workspace_bytes = P.workspace_bytes;
  info->stream_k = P.sk;
  if (P.sk) {
    const int64_t pairs = kGb300Sms / 2;
    const int64_t rem = P.tiles % pairs;
    info->sk_tiles = static_cast<int32_t>(rem);
    info->sk_workspace_bytes = P.sk_bytes;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

template <int BN>
bool prepare_kernel(int64_t smem) {
  static std::once_flag once;
  static bool ok = false;
  std::call_once(once, [] {
    ok = cudaFuncSetAttribute(dmt::bmm_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(dmt::kSmemLimit)) == cudaSuccess;
  });
  (void)smem;
  return ok;
}

template <int BN, int kTail = 0>
bool prepare_pair_kernel() {
  static std::once_flag once;
  static bool ok = false;
  std::call_once(once, [] {
    ok = cudaFuncSetAttribute(dmt::bmm_tc2_kernel<BN, kTail>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(dmt::kSmemLimit)) == cudaSuccess;
  });
  return ok;
}

uint64_t wait_timeout_ns() {
  const char* e = std::getenv("DMT_BMM_WAIT_TIMEOUT_MS");
  if (e && *e) {
    const long long ms = std::atoll(e);
    if (ms > 0) return static_cast<uint64_t>(ms) * 1000000ull;
  }
  return 2000000000ull;  // 2 s
}

}  // namespace

struct bmm_plan_s {
  bmm_desc_t d;
  Planned P;
  int device;
  int sms;
  int max_pairs;  // co-resident CTA pairs for the pair kernel (0: not queried)
  void* ws;
  void* sk_ws;        // stream-K flags and partials (P.sk_bytes; flags start at zero)
  uint32_t sk_epoch;  // flag value of the last launch (never 0)
  uint32_t* err;
  uint64_t timeout_ns;
  int test_stall;
  const void* map_ptr[3];
  CUtensorMap map[3];  // A, B, and C (C only when written by TMA box stores)
};

namespace {

bool encode_map(const bmm_plan_s* pl, const Operand& o, const void* base, CUtensorMap* out) {
  const int64_t ld = o.pack ? o.pld : o.ld;
  const int64_t stride = o.pack ? o.pstride : o.stride;
  const int64_t nb = o.bcast ? 1 : pl->P.batch;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(o.cols), static_cast<cuuint64_t>(o.rows),
                        static_cast<cuuint64_t>(nb)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2),
                           static_cast<cuuint64_t>(nb > 1 ? stride * 2 : round_up(o.rows * ld * 2, 16))};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(dmt::kTileK),
                       static_cast<cuuint32_t>(o.mn_major ? 64 : o.box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapDataType dt = pl->d.typeA == BMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = g_encode(out, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Threads per CTA: the row-loader warps (6 and 7) only when an operand needs them.
unsigned block_threads(const KParams& kp) {
  return static_cast<unsigned>(kp.ldg_mask ? dmt::kThreads : dmt::kThreads - 32 * dmt::kLdgWarps);
}

cudaLaunchConfig_t pair_config(int64_t pairs, int64_t smem, cudaStream_t stream,
                               cudaLaunchAttribute* attr, unsigned threads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Persistent grid of CTA pairs: as many as can be co-resident (queried once
// per plan), at most one per pair tile.
template <int BN>
cudaError_t launch_gemm_pair(bmm_plan_s* pl, KParams kp, cudaStream_t stream) {
  if (!prepare_pair_kernel<BN>()) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  if (pl->max_pairs == 0) {
    cudaLaunchConfig_t q = pair_config(pl->sms / 2, pl->P.smem_bytes, stream, attr, dmt::kThreads);
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, dmt::bmm_tc2_kernel<BN>, &q);
    if (e != cudaSuccess) return e;
    pl->max_pairs = n > 0 ? n : 1;
  }
  int64_t pairs = pl->P.tiles < pl->max_pairs ? pl->P.tiles : pl->max_pairs;
  // Stream-K tail: whole rounds over all resident pairs, then the leftover
  // tiles' k-blocks.  At most half as many leftover tiles as pairs: each tile
  // on two pairs, the owner's range longer by the partial's transfer time
  // (sk_piece2).  More: equal ranges (at least kSkMinUnits each) over as many
  // pairs as that allows (sk_piece).
  const int64_t G = pl->max_pairs;
  bool two_way = false;
  // (the fixup and a last piece's partial use a quarter of the operand ring:
  // it must hold a tile row's partial, BN / 32 chunks of 4 KB, and a barrier)
  const bool ring_ok = static_cast<int64_t>(pl->P.stages) * pl->P.stage_bytes / 4 >= (BN / 32) * 4096 + 128;
  if (BN == 256 && pl->P.sk && pl->sk_ws && ring_ok && G <= kSkFlagBytes / 32 &&
      sk_workspace_bytes(G, BN) <= pl->P.sk_bytes) {
    const int64_t waves = pl->P.tiles / G, rem = pl->P.tiles % G;
    if (rem > 0) {
      const int64_t units = rem * pl->P.k_blocks;
      int64_t skp = units / sk_min_units(pl->P.k_blocks);
      skp = skp < 1 ? 1 : (skp > G ? G : skp);
      if (2 * rem <= G) {
        two_way = true;
        skp = 2 * rem;
        kp.sk_ko = pl->P.k_blocks - sk_contributor_kblocks(pl->P.k_blocks);
      }
      if (++pl->sk_epoch == 0) pl->sk_epoch = 1;
      kp.sk_tiles = static_cast<int32_t>(rem);
      kp.sk_pairs = static_cast<int32_t>(skp);
      kp.sk_first = waves * G;
      kp.sk_epoch = pl->sk_epoch;
      kp.sk_flags = static_cast<uint32_t*>(pl->sk_ws);
      kp.sk_ws = reinterpret_cast<float4*>(static_cast<char*>(pl->sk_ws) + kSkFlagBytes);
      pairs = waves > 0 ? G : skp;
    }
  }
  if constexpr (BN == 256) {
    if (kp.sk_tiles > 0 && two_way) {
      if (!prepare_pair_kernel<BN, dmt::kSkTwoWay>()) return cudaErrorInvalidValue;
      cudaLaunchConfig_t cfg = pair_config(pairs, pl->P.smem_bytes, stream, attr, block_threads(kp));
      return cudaLaunchKernelEx(&cfg, dmt::bmm_tc2_kernel<BN, dmt::kSkTwoWay>, kp, pl->map[0], pl->map[1],
                                pl->map[2]);
    }
    if (kp.sk_tiles > 0) {
      if (!prepare_pair_kernel<BN, dmt::kSkEven>()) return cudaErrorInvalidValue;
      cudaLaunchConfig_t cfg = pair_config(pairs, pl->P.smem_bytes, stream, attr, block_threads(kp));
      return cudaLaunchKernelEx(&cfg, dmt::bmm_tc2_kernel<BN, dmt::kSkEven>, kp, pl->map[0], pl->map[1],
                                pl->map[2]);
    }
  }
  cudaLaunchConfig_t cfg = pair_config(pairs, pl->P.smem_bytes, stream, attr, block_threads(kp));
  return cudaLaunchKernelEx(&cfg, dmt::bmm_tc2_kernel<BN>, kp, pl->map[0], pl->map[1], pl->map[2]);
}

// C as a 3-D tensor (N, M, batch) with 32 x 32 boxes: 128-byte box rows for
// fp32 (128-byte swizzle), 64-byte rows for bf16 (64-byte swizzle), matching
// the layout the epilogue writes into its box buffers.
bool encode_c_map(const bmm_plan_s* pl, void* C, CUtensorMap* out) {
  const bmm_desc_t& d = pl->d;
  const int64_t es = d.typeC == BMM_F32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d.N), static_cast<cuuint64_t>(d.M),
                        static_cast<cuuint64_t>(d.batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d.ldc * es),
                           static_cast<cuuint64_t>(d.batch > 1 ? d.strideC * es
                                                               : round_up(d.M * d.ldc * es, 16))};
  cuuint32_t box[3] = {32u, 32u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(out, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              3, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_gemm(const bmm_plan_s* pl, const KParams& kp, cudaStream_t stream) {
  if (!prepare_kernel<BN>(pl->P.smem_bytes)) return cudaErrorInvalidValue;
  int64_t grid = pl->P.tiles < pl->sms ? pl->P.tiles : pl->sms;
  dmt::bmm_tc_kernel<BN><<<static_cast<unsigned>(grid), block_threads(kp),
                           static_cast<size_t>(pl->P.smem_bytes), stream>>>(kp, pl->map[0],
                                                                           pl->map[1], pl->map[2]);
  return cudaGetLastError();
}

}  // namespace

extern "C" {

int32_t bmm_version(void) { return kVersion; }

const char* bmm_status_string(bmm_status_t s) {
  switch (s) {
    case BMM_OK: return "BMM_OK";
    case BMM_ERR_INVALID_ARG: return "BMM_ERR_INVALID_ARG";
    case BMM_ERR_UNSUPPORTED: return "BMM_ERR_UNSUPPORTED";
    case BMM_ERR_MISALIGNED: return "BMM_ERR_MISALIGNED";
    case BMM_ERR_CUDA: return "BMM_ERR_CUDA";
    case BMM_ERR_DEVICE_TIMEOUT: return "BMM_ERR_DEVICE_TIMEOUT";
    case BMM_ERR_NO_DEVICE: return "BMM_ERR_NO_DEVICE";
  }
  return "BMM_ERR_UNKNOWN";
}

bmm_status_t bmm_plan_query(const bmm_desc_t* desc, bmm_plan_info_t* info) {
  if (!info) return BMM_ERR_INVALID_ARG;
  const bmm_status_t st = validate(desc);
  if (st != BMM_OK) return st;
  Planned P;
  plan(desc, &P, kGb300Sms, row_loader_requested());
  fill_info(P, desc, info);
  (void)kGb300Sms;
  return BMM_OK;
}

bmm_status_t bmm_create(const bmm_desc_t* desc, bmm_plan_t* out) {
  if (!out) return BMM_ERR_INVALID_ARG;
  *out = nullptr;
  const bmm_status_t st = validate(desc);
  if (st != BMM_OK) return st;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BMM_ERR_NO_DEVICE;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BMM_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return BMM_ERR_NO_DEVICE;  // built for sm_103a only
  if (!get_encoder()) return BMM_ERR_CUDA;

  bmm_plan_s* pl = new (std::nothrow) bmm_plan_s();
  if (!pl) return BMM_ERR_CUDA;
  pl->d = *desc;
  plan(desc, &pl->P, sms, row_loader_requested());
  pl->device = dev;
  pl->sms = sms;
  pl->timeout_ns = wait_timeout_ns();
  // Test hook for failure detection: the MMA thread waits on a barrier that
  // nothing completes, so its bounded wait must expire (see bmm.h, errors).
  const char* ts = std::getenv("DMT_BMM_TEST_STALL_MMA");
  pl->test_stall = (ts && ts[0] == '1') ? 1 : 0;
  if (cudaMalloc(reinterpret_cast<void**>(&pl->err), 256) != cudaSuccess ||
      cudaMemset(pl->err, 0, 256) != cudaSuccess) {
    cudaFree(pl->err);
    delete pl;
    return BMM_ERR_CUDA;
  }
  if (pl->P.workspace_bytes > 0 &&
      cudaMalloc(&pl->ws, static_cast<size_t>(pl->P.workspace_bytes)) != cudaSuccess) {
    cudaFree(pl->err);
    delete pl;
    return BMM_ERR_CUDA;
  }
  if (pl->P.sk_bytes > 0 &&
      (cudaMalloc(&pl->sk_ws, static_cast<size_t>(pl->P.sk_bytes)) != cudaSuccess ||
       cudaMemset(pl->sk_ws, 0, static_cast<size_t>(kSkFlagBytes)) != cudaSuccess)) {
    cudaFree(pl->sk_ws);
    cudaFree(pl->ws);
    cudaFree(pl->err);
    delete pl;
    return BMM_ERR_CUDA;
  }
  *out = pl;
  return BMM_OK;
}

bmm_status_t bmm_get_plan_info(bmm_plan_t pl, bmm_plan_info_t* info) {
  if (!pl || !info) return BMM_ERR_INVALID_ARG;
  fill_info(pl->P, &pl->d, info);
  return BMM_OK;
}

bmm_status_t bmm_run(bmm_plan_t pl, const void* A, const void* B, void* C, float alpha,
                     float beta, void* stream_v) {
  if (!pl) return BMM_ERR_INVALID_ARG;
  const bmm_desc_t& d = pl->d;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  if (d.batch == 0 || d.M == 0 || d.N == 0) return BMM_OK;
  if (!C) return BMM_ERR_INVALID_ARG;

  if (alpha == 0.0f || d.K == 0) {
    // A and B are not read: C = beta * C.
    const int64_t rows = d.batch * d.M;
    dim3 grid(static_cast<unsigned>((d.N + 255) / 256 < 64 ? (d.N + 255) / 256 : 64),
              static_cast<unsigned>(rows < 65535 ? rows : 65535));
    dmt::scale_c_kernel<<<grid, 256, 0, stream>>>(C, d.typeC == BMM_BF16, d.batch, d.M, d.N, d.ldc,
                                                  d.strideC, beta);
    return cudaGetLastError() == cudaSuccess ? BMM_OK : BMM_ERR_CUDA;
  }
  if (!A || !B) return BMM_ERR_INVALID_ARG;

  const Planned& P = pl->P;
  const void* base[2];
  const Operand* ops[2] = {&P.a, &P.b};
  for (int i = 0; i < 2; ++i) {
    const Operand& o = *ops[i];
    const void* src = o.user == 0 ? A : B;
    if (o.pack == 2) {
      if ((reinterpret_cast<uintptr_t>(src) & 1u) != 0) return BMM_ERR_MISALIGNED;
      base[i] = src;  // read by the row loader: no tensor map
      continue;
    }
    if (o.pack) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(static_cast<char*>(pl->ws) + o.ws_off);
      const int64_t nb = o.bcast ? 1 : d.batch;
      const int64_t segs = nb * o.rows * ((o.cols + 7) / 8);
      const int64_t blocks = (segs + 255) / 256;
      const unsigned grid = static_cast<unsigned>(blocks < 8 * pl->sms ? blocks : 8 * pl->sms);
      dmt::pack16_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(src), dst, nb,
                                                   o.rows, o.cols, o.ld, o.bcast ? 0 : o.stride,
                                                   o.pld, o.pstride);
      if (cudaGetLastError() != cudaSuccess) return BMM_ERR_CUDA;
      base[i] = dst;
    } else {
      if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0) return BMM_ERR_MISALIGNED;
      base[i] = src;
    }
    if (pl->map_ptr[i] != base[i]) {
      if (!encode_map(pl, o, base[i], &pl->map[i])) return BMM_ERR_CUDA;
      pl->map_ptr[i] = base[i];
    }
  }

  KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.Mv = static_cast<int32_t>(P.Mv);
  kp.Nv = static_cast<int32_t>(P.Nv);
  kp.K = static_cast<int32_t>(P.K);
  kp.num_m = P.num_m;
  kp.num_n = P.num_n;
  kp.tiles = P.tiles;
  kp.k_blocks = P.k_blocks;
  kp.tail_steps = P.tail_steps;
  kp.a_mn = P.a.mn_major;
  kp.b_mn = P.b.mn_major;
  kp.a_bcast = P.a.bcast;
  kp.b_bcast = P.b.bcast;
  kp.stages = P.stages;
  kp.stage_bytes = P.stage_bytes;
  kp.a_bytes = P.a_bytes;
  kp.tx_bytes = P.tx_bytes;
  kp.idesc = P.idesc;
  kp.tmem_cols = P.tmem_cols;
  for (int i = 0; i < 2; ++i) {
    const Operand& o = *ops[i];
    if (o.pack != 2) continue;
    kp.ldg_mask |= 1 << i;
    kp.ldg[i] = dmt::LdgOperand{static_cast<const uint16_t*>(base[i]), o.ld, o.bcast ? 0 : o.stride,
                                o.rows, o.cols};
  }
  kp.C = C;
  kp.ldc = d.ldc;
  kp.sC = d.strideC;
  kp.c_bf16 = d.typeC == BMM_BF16 ? 1 : 0;
  kp.c_trans = P.swap;
  // Row-major C with beta == 0 goes out through TMA box stores when its base,
  // strides and row length are 16-byte multiples (a box store writes whole
  // 16-byte chunks at the row end, which would spill past a ragged row);
  // otherwise coalesced direct stores.
  {
    const int64_t es = d.typeC == BMM_F32 ? 4 : 2;
    const bool aligned = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && (d.ldc * es) % 16 == 0 &&
                         (d.N * es) % 16 == 0 && (d.batch <= 1 || (d.strideC * es) % 16 == 0);
    kp.c_tma = (!P.swap && beta == 0.0f && aligned && P.bn >= 32) ? 1 : 0;
    if (kp.c_tma && pl->map_ptr[2] != C) {
      if (!encode_c_map(pl, C, &pl->map[2])) return BMM_ERR_CUDA;
      pl->map_ptr[2] = C;
    }
  }
  // the pair kernel's epilogue region: half size (and a deeper ring) when C
  // goes out as bf16 box stores
  kp.epi_bytes = dmt::kEpiBytes;
  kp.box_bytes = dmt::kEpiBoxBytes;
  if (P.pair && kp.c_tma && kp.c_bf16 && P.stages_bf16_box > P.stages) {
    kp.stages = P.stages_bf16_box;
    kp.epi_bytes = dmt::kEpiBytesBf16;
    kp.box_bytes = dmt::kEpiBoxBytesBf16;
  }
  kp.alpha = alpha;
  kp.beta = beta;
  kp.err = pl->err;
  kp.timeout_ns = pl->timeout_ns;
  kp.test_stall = pl->test_stall;

  cudaError_t e;
  if (P.pair) {
    switch (P.bn) {
      case 192: e = launch_gemm_pair<192>(pl, kp, stream); break;
      case 224: e = launch_gemm_pair<224>(pl, kp, stream); break;
      default: e = launch_gemm_pair<256>(pl, kp, stream); break;
    }
    return e == cudaSuccess ? BMM_OK : BMM_ERR_CUDA;
  }
  switch (P.bn) {
    case 16: e = launch_gemm<16>(pl, kp, stream); break;
    case 32: e = launch_gemm<32>(pl, kp, stream); break;
    case 64: e = launch_gemm<64>(pl, kp, stream); break;
    case 128: e = launch_gemm<128>(pl, kp, stream); break;
    case 192: e = launch_gemm<192>(pl, kp, stream); break;
    case 224: e = launch_gemm<224>(pl, kp, stream); break;
    default: e = launch_gemm<256>(pl, kp, stream); break;
  }
  return e == cudaSuccess ? BMM_OK : BMM_ERR_CUDA;
}

bmm_status_t bmm_get_device_error(bmm_plan_t pl, uint32_t* detail) {
  if (!pl) return BMM_ERR_INVALID_ARG;
  uint32_t w = 0;
  if (cudaMemcpy(&w, pl->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return BMM_ERR_CUDA;
  if (w != 0 && cudaMemset(pl->err, 0, sizeof(w)) != cudaSuccess) return BMM_ERR_CUDA;
  if (detail) *detail = w;
  return w == 0 ? BMM_OK : BMM_ERR_DEVICE_TIMEOUT;
}

bmm_status_t bmm_destroy(bmm_plan_t pl) {
  if (!pl) return BMM_OK;
  bmm_status_t st = BMM_OK;
  if (pl->ws && cudaFree(pl->ws) != cudaSuccess) st = BMM_ERR_CUDA;
  if (pl->sk_ws && cudaFree(pl->sk_ws) != cudaSuccess) st = BMM_ERR_CUDA;
  if (pl->err && cudaFree(pl->err) != cudaSuccess) st = BMM_ERR_CUDA;
  delete pl;
  return st;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of bmm_run.
//
// Some callers cannot call cudaMalloc: code that runs under an allocator that
// owns the device's memory (a framework's caching pool, a fixed memory budget
// carved out up front), and latency-critical call paths where cudaMalloc's
// cost and its implicit device synchronisation are not acceptable.  For them,
// bmm_run_noalloc takes the problem description directly and keeps all of its
// scratch (the device error word and the staging area for operands whose
// strides TMA cannot read in place) in one file-scope device array.  That
// array is part of the library image: every GPU that loads the library holds
// it until the process exits.
namespace {

constexpr size_t kNoAllocWordBytes = 256;             // device error word region
constexpr size_t kNoAllocStagingMax = size_t(32) << 20;  // 32 MiB operand staging area
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocWordBytes + kNoAllocStagingMax];

std::mutex g_noalloc_mu;
unsigned char* g_noalloc_addr[kNoAllocMaxDevices];

// Co-resident CTA pairs per (device, tile width, shared memory), remembered
// from the first call that launched the pair kernel with them, so later calls
// skip the occupancy query (a plan keeps this number; these calls have none).
struct NoAllocPairs {
  int dev;
  int tile_n;
  int64_t smem;
  int pairs;
};
constexpr int kNoAllocPairSlots = 64;
NoAllocPairs g_noalloc_pairs[kNoAllocPairSlots];
int g_noalloc_pairs_used = 0;

int noalloc_cached_pairs(int dev, const Planned& P) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  for (int i = 0; i < g_noalloc_pairs_used; ++i)
    if (g_noalloc_pairs[i].dev == dev && g_noalloc_pairs[i].tile_n == P.bn &&
        g_noalloc_pairs[i].smem == P.smem_bytes)
      return g_noalloc_pairs[i].pairs;
  return 0;
}

void noalloc_remember_pairs(int dev, const Planned& P, int pairs) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  for (int i = 0; i < g_noalloc_pairs_used; ++i)
    if (g_noalloc_pairs[i].dev == dev && g_noalloc_pairs[i].tile_n == P.bn &&
        g_noalloc_pairs[i].smem == P.smem_bytes)
      return;
  if (g_noalloc_pairs_used < kNoAllocPairSlots)
    g_noalloc_pairs[g_noalloc_pairs_used++] = NoAllocPairs{dev, P.bn, P.smem_bytes, pairs};
}

// Device address of the scratch array on device `dev` (which must be
// current).  Looked up with cudaGetSymbolAddress on the first call per device.
bmm_status_t noalloc_scratch(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return BMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return BMM_ERR_CUDA;
    g_noalloc_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_noalloc_addr[dev];
  return BMM_OK;
}

}  // namespace

extern "C" bmm_status_t bmm_run_noalloc(const bmm_desc_t* desc, const void* A, const void* B,
                                        void* C, float alpha, float beta, void* stream,
                                        uint32_t* device_error) {
  const bmm_status_t st = validate(desc);
  if (st != BMM_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BMM_ERR_NO_DEVICE;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BMM_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return BMM_ERR_NO_DEVICE;
  if (!get_encoder()) return BMM_ERR_CUDA;

  bmm_plan_s pl;  // on the stack: nothing is allocated for the call
  std::memset(static_cast<void*>(&pl), 0, sizeof(pl));
  pl.d = *desc;
  // no stream-K tail here: its partials would need more scratch than the array holds
  plan(desc, &pl.P, sms, row_loader_requested(), false);
  // staging larger than the built-in scratch: the row loader reads those operands
  if (pl.P.workspace_bytes > static_cast<int64_t>(kNoAllocStagingMax)) plan(desc, &pl.P, sms, true, false);
  unsigned char* scratch = nullptr;
  const bmm_status_t sst = noalloc_scratch(dev, &scratch);
  if (sst != BMM_OK) return sst;
  pl.device = dev;
  pl.sms = sms;
  pl.timeout_ns = wait_timeout_ns();
  pl.err = reinterpret_cast<uint32_t*>(scratch);
  pl.ws = scratch + kNoAllocWordBytes;

  if (pl.P.pair) pl.max_pairs = noalloc_cached_pairs(dev, pl.P);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the error word must start at zero.
  if (cudaMemsetAsync(pl.err, 0, sizeof(uint32_t), s) != cudaSuccess) return BMM_ERR_CUDA;
  const bmm_status_t rst = bmm_run(&pl, A, B, C, alpha, beta, stream);
  if (rst != BMM_OK) return rst;
  if (pl.P.pair && pl.max_pairs > 0) noalloc_remember_pairs(dev, pl.P, pl.max_pairs);
  if (device_error &&
      cudaMemcpyAsync(device_error, pl.err, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess)
    return BMM_ERR_CUDA;
  return BMM_OK;
}

// ---------------------------------------------------------------------------
// Grouped launches: one persistent launch over a table of independent
// problems (see bmm.h).  The single-CTA kernel runs in its grouped mode: each
// role looks its tile up in the device table (binary search over each
// problem's first tile) and takes that problem's sizes, tensor maps and C.

struct bmm_grouped_plan_s {
  int32_t count;                       // problems given by the caller
  std::vector<int32_t> live;           // indices of the problems with tiles
  std::vector<bmm_group_problem_t> shape;
  int32_t transA, transB, typeAB, typeC;
  int bn, stages;
  int per_sm;                          // CTAs sharing an SM (2: narrow tiles, half the shared memory each)
  uint32_t stage_bytes, a_bytes, tx_bytes, idesc, tmem_cols;
  int64_t smem_bytes, tiles;
  int sms;
  std::vector<dmt::GroupEntry> host;   // staging copy of the device table
  std::vector<bmm_group_problem_t> last;  // pointers and scalars the device table holds
  bool table_valid = false;               // the device table matches `host`
  dmt::GroupEntry* table;
  int32_t* first_tile;                    // device: each table entry's first tile (for the search)
  uint32_t* err;
  uint64_t timeout_ns;
};

namespace {

constexpr int32_t kMaxGroups = 65536;

// One operand of a grouped problem as a (cols, rows, 1) tensor map: K-major
// with a (64 x box_rows) box, MN-major with (64 x 64) boxes.
bool encode_group_operand(int32_t type, int64_t rows, int64_t cols, int64_t ld, int box_rows,
                          int mn_major, const void* base, CUtensorMap* out) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2),
                           static_cast<cuuint64_t>(round_up(rows * ld * 2, 16))};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(dmt::kTileK),
                       static_cast<cuuint32_t>(mn_major ? 64 : box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return g_encode(out, type == BMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_group_c(int32_t typeC, int64_t M, int64_t N, int64_t ldc, void* C, CUtensorMap* out) {
  const int64_t es = typeC == BMM_F32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), 1};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldc * es),
                           static_cast<cuuint64_t>(round_up(M * ldc * es, 16))};
  cuuint32_t box[3] = {32u, 32u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return g_encode(out, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, C,
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int kPerSM>
bool prepare_grouped_kernel() {
  static std::once_flag once;
  static bool ok = false;
  std::call_once(once, [] {
    ok = cudaFuncSetAttribute(dmt::bmm_tc_kernel<BN, true, kPerSM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(dmt::kSmemLimit)) == cudaSuccess;
    // two CTAs per SM need the largest shared-memory share of the SM
    if (ok && kPerSM == 2)
      ok = cudaFuncSetAttribute(dmt::bmm_tc_kernel<BN, true, kPerSM>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                100) == cudaSuccess;
  });
  return ok;
}

template <int BN, int kPerSM>
cudaError_t launch_grouped(const bmm_grouped_plan_s* pl, const KParams& kp, cudaStream_t stream) {
  if (!prepare_grouped_kernel<BN, kPerSM>()) return cudaErrorInvalidValue;
  // one CTA per tile: running CTAs take the tiles of CTAs that have not
  // started (cluster launch control), so the load balances itself
  const int64_t grid = pl->tiles;
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  dmt::bmm_tc_kernel<BN, true, kPerSM><<<static_cast<unsigned>(grid), block_threads(kp),
                                         static_cast<size_t>(pl->smem_bytes), stream>>>(kp, unused, unused, unused);
  return cudaGetLastError();
}

}  // namespace

extern "C" {

bmm_status_t bmm_grouped_create(int32_t count, const bmm_group_problem_t* problems, int32_t transA,
                                int32_t transB, int32_t typeAB, int32_t typeC,
                                bmm_grouped_plan_t* out) {
  if (!out) return BMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (count < 0 || (count > 0 && !problems)) return BMM_ERR_INVALID_ARG;
  if (count > kMaxGroups) return BMM_ERR_UNSUPPORTED;
  if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return BMM_ERR_INVALID_ARG;
  if (!is16(typeAB) || (typeC != BMM_F32 && typeC != BMM_BF16)) return BMM_ERR_INVALID_ARG;
  const int64_t ces = typeC == BMM_F32 ? 4 : 2;
  int64_t max_n = 0;
  for (int32_t i = 0; i < count; ++i) {
    const bmm_group_problem_t& q = problems[i];
    if (q.M < 0 || q.N < 0 || q.K < 0) return BMM_ERR_INVALID_ARG;
    const int64_t a_cols = transA ? q.M : q.K, b_cols = transB ? q.K : q.N;
    if (q.lda < (a_cols > 1 ? a_cols : 1) || q.ldb < (b_cols > 1 ? b_cols : 1) ||
        q.ldc < (q.N > 1 ? q.N : 1))
      return BMM_ERR_INVALID_ARG;
    if (q.M > kMaxDim || q.N > kMaxDim || q.K > kMaxDim) return BMM_ERR_UNSUPPORTED;
    if (q.M == 0 || q.N == 0) continue;
    if (q.K == 0) return BMM_ERR_UNSUPPORTED;
    if ((q.lda * 2) % 16 || (q.ldb * 2) % 16 || (q.ldc * ces) % 16) return BMM_ERR_UNSUPPORTED;
    if (q.N > max_n) max_n = q.N;
  }
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BMM_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BMM_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return BMM_ERR_NO_DEVICE;
  if (!get_encoder()) return BMM_ERR_CUDA;

  bmm_grouped_plan_s* pl = new (std::nothrow) bmm_grouped_plan_s();
  if (!pl) return BMM_ERR_CUDA;
  pl->count = count;
  pl->shape.assign(problems, problems + count);
  pl->transA = transA;
  pl->transB = transB;
  pl->typeAB = typeAB;
  pl->typeC = typeC;
  pl->sms = sms;
  pl->timeout_ns = wait_timeout_ns();
  // One tile shape for the launch: 64 wide if it covers the widest N, else
  // 128 (a wider problem takes several N tiles), with two CTAs per SM: the
  // tiles are short (K <= a few k-blocks), and a second CTA's loads, MMAs
  // and stores run while the first waits on its own (1000 problems of
  // 64..256: 50.4 us against 54.0 for 256-wide tiles, one CTA per SM).
  pl->bn = max_n <= 64 ? 64 : 128;
  pl->per_sm = 2;
  // DMT_BMM_TILE_N=64|128|256 pins the launch's tile width (comparisons;
  // 256 runs one CTA per SM)
  const char* te = std::getenv("DMT_BMM_TILE_N");
  if (te && *te) {
    const int w = std::atoi(te);
    if (w == 64 || w == 128 || w == 256) pl->bn = w;
  }
  if (pl->bn == 256) pl->per_sm = 1;
  const int a_mn = transA ? 1 : 0, b_mn = transB ? 0 : 1;
  pl->a_bytes = static_cast<uint32_t>(dmt::kTileM * dmt::kTileK * 2);
  const uint32_t b_bytes = static_cast<uint32_t>(pl->bn * dmt::kTileK * 2);
  pl->stage_bytes = static_cast<uint32_t>(round_up(pl->a_bytes + b_bytes, 1024));
  pl->tx_bytes = pl->a_bytes + b_bytes;
  const int64_t fixed = 1024 + dmt::kEpiBytes + dmt::kBarBytes;
  // per CTA: all of the SM's shared memory, or half of it (1 KB of each
  // half is the system's) for two CTAs per SM
  const int64_t budget = pl->per_sm == 2 ? (dmt::kSmemLimit + 1024) / 2 - 1024 : dmt::kSmemLimit;
  pl->stages = static_cast<int>((budget - fixed) / pl->stage_bytes);
  if (pl->stages > dmt::kMaxStages) pl->stages = dmt::kMaxStages;
  pl->smem_bytes = fixed + static_cast<int64_t>(pl->stages) * pl->stage_bytes;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(2 * pl->bn)) cols <<= 1;
  pl->tmem_cols = cols;
  const uint32_t fmt = typeAB == BMM_BF16 ? 1u : 0u;
  pl->idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(a_mn) << 15) |
              (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(pl->bn >> 3) << 17) |
              (static_cast<uint32_t>(dmt::kTileM >> 4) << 24);
  pl->tiles = 0;
  for (int32_t i = 0; i < count; ++i) {
    const bmm_group_problem_t& q = problems[i];
    if (q.M == 0 || q.N == 0) continue;
    dmt::GroupEntry e;
    std::memset(static_cast<void*>(&e), 0, sizeof(e));
    e.Mv = static_cast<int32_t>(q.M);
    e.Nv = static_cast<int32_t>(q.N);
    e.num_m = static_cast<int32_t>((q.M + dmt::kTileM - 1) / dmt::kTileM);
    e.num_n = static_cast<int32_t>((q.N + pl->bn - 1) / pl->bn);
    e.k_blocks = static_cast<int32_t>((q.K + dmt::kTileK - 1) / dmt::kTileK);
    const int64_t rem = q.K % dmt::kTileK;
    e.tail_steps = rem == 0 ? dmt::kTileK / dmt::kUmmaK
                            : static_cast<int32_t>((rem + dmt::kUmmaK - 1) / dmt::kUmmaK);
    e.tile_begin = pl->tiles;
    e.ldc = q.ldc;
    pl->tiles += static_cast<int64_t>(e.num_m) * e.num_n;
    pl->live.push_back(i);
    pl->host.push_back(e);
  }
  // one CTA per tile, and tile indices travel as int32 in the kernel's schedule
  if (pl->tiles > 0x7fffffffLL) {
    delete pl;
    return BMM_ERR_UNSUPPORTED;
  }
  const size_t table_bytes = sizeof(dmt::GroupEntry) * (pl->host.empty() ? 1 : pl->host.size());
  if (cudaMalloc(reinterpret_cast<void**>(&pl->table), table_bytes) != cudaSuccess) {
    delete pl;
    return BMM_ERR_CUDA;
  }
  // the entries' first tiles as a compact int32 array: the kernel's
  // tile -> problem search reads 4 bytes per entry (cache resident) instead
  // of one 512-byte table record per step.  Fixed at create: sizes are.
  std::vector<int32_t> first(pl->host.empty() ? 1 : pl->host.size(), 0);
  for (size_t j = 0; j < pl->host.size(); ++j) first[j] = static_cast<int32_t>(pl->host[j].tile_begin);
  pl->first_tile = nullptr;
  if (cudaMalloc(reinterpret_cast<void**>(&pl->first_tile), first.size() * sizeof(int32_t)) != cudaSuccess ||
      cudaMemcpy(pl->first_tile, first.data(), first.size() * sizeof(int32_t), cudaMemcpyHostToDevice) !=
          cudaSuccess) {
    cudaFree(pl->table);
    cudaFree(pl->first_tile);
    delete pl;
    return BMM_ERR_CUDA;
  }
  if (cudaMalloc(reinterpret_cast<void**>(&pl->err), 256) != cudaSuccess ||
      cudaMemset(pl->err, 0, 256) != cudaSuccess) {
    cudaFree(pl->table);
    cudaFree(pl->first_tile);
    cudaFree(pl->err);
    delete pl;
    return BMM_ERR_CUDA;
  }
  *out = pl;
  return BMM_OK;
}

bmm_status_t bmm_grouped_run(bmm_grouped_plan_t pl, const bmm_group_problem_t* problems,
                             void* stream_v) {
  if (!pl || (pl->count > 0 && !problems)) return BMM_ERR_INVALID_ARG;
  if (pl->tiles == 0) return BMM_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const int64_t ces = pl->typeC == BMM_F32 ? 4 : 2;
  const int b_box = pl->bn;
  if (pl->last.size() != pl->live.size()) pl->last.assign(pl->live.size(), bmm_group_problem_t{});
  bool changed = !pl->table_valid;
  for (size_t j = 0; j < pl->live.size(); ++j) {
    const int32_t i = pl->live[j];
    const bmm_group_problem_t& q = problems[i];
    const bmm_group_problem_t& s = pl->shape[i];
    if (q.M != s.M || q.N != s.N || q.K != s.K || q.lda != s.lda || q.ldb != s.ldb || q.ldc != s.ldc)
      return BMM_ERR_INVALID_ARG;  // sizes are fixed at create
    if (!q.A || !q.B || !q.C) return BMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q.A) & 15u) || (reinterpret_cast<uintptr_t>(q.B) & 15u))
      return BMM_ERR_MISALIGNED;
    // an entry is re-encoded only when its operands or scalars moved
    const bmm_group_problem_t& l = pl->last[j];
    if (pl->table_valid && q.A == l.A && q.B == l.B && q.C == l.C && q.alpha == l.alpha &&
        q.beta == l.beta)
      continue;
    // from here the device table no longer matches: an error return below
    // leaves it marked stale, so the next run encodes every entry again
    changed = true;
    pl->table_valid = false;
    pl->last[j] = q;
    dmt::GroupEntry& e = pl->host[j];
    const int64_t a_rows = pl->transA ? q.K : q.M, a_cols = pl->transA ? q.M : q.K;
    const int64_t b_rows = pl->transB ? q.N : q.K, b_cols = pl->transB ? q.K : q.N;
    if (!encode_group_operand(pl->typeAB, a_rows, a_cols, q.lda, dmt::kTileM, pl->transA ? 1 : 0, q.A,
                              &e.map_a) ||
        !encode_group_operand(pl->typeAB, b_rows, b_cols, q.ldb, b_box, pl->transB ? 0 : 1, q.B,
                              &e.map_b))
      return BMM_ERR_CUDA;
    const bool c_ok = (reinterpret_cast<uintptr_t>(q.C) & 15u) == 0 && (q.N * ces) % 16 == 0;
    e.c_tma = (q.beta == 0.0f && c_ok) ? 1 : 0;
    if (e.c_tma && !encode_group_c(pl->typeC, q.M, q.N, q.ldc, q.C, &e.map_c)) return BMM_ERR_CUDA;
    e.C = q.C;
    e.alpha = q.alpha;
    e.beta = q.beta;
  }
  // Pageable source: the copy is staged before this call returns, so the host
  // table may be rewritten by the next run.  Skipped when no entry changed.
  if (changed) {
    if (cudaMemcpyAsync(pl->table, pl->host.data(), sizeof(dmt::GroupEntry) * pl->host.size(),
                        cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return BMM_ERR_CUDA;
    pl->table_valid = true;
  }

  KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.tiles = pl->tiles;
  kp.a_mn = pl->transA ? 1 : 0;
  kp.b_mn = pl->transB ? 0 : 1;
  kp.stages = pl->stages;
  kp.stage_bytes = pl->stage_bytes;
  kp.a_bytes = pl->a_bytes;
  kp.tx_bytes = pl->tx_bytes;
  kp.idesc = pl->idesc;
  kp.tmem_cols = pl->tmem_cols;
  kp.c_bf16 = pl->typeC == BMM_BF16 ? 1 : 0;
  kp.err = pl->err;
  kp.timeout_ns = pl->timeout_ns;
  kp.groups = pl->table;
  kp.group_first = pl->first_tile;
  kp.ngroups = static_cast<int32_t>(pl->host.size());
  cudaError_t e;
  switch (pl->bn) {
    // 64 and 128 wide: two CTAs per SM; 256 wide (pinned): one
    case 64: e = launch_grouped<64, 2>(pl, kp, stream); break;
    case 128: e = launch_grouped<128, 2>(pl, kp, stream); break;
    default: e = launch_grouped<256, 1>(pl, kp, stream); break;
  }
  return e == cudaSuccess ? BMM_OK : BMM_ERR_CUDA;
}

bmm_status_t bmm_grouped_get_device_error(bmm_grouped_plan_t pl, uint32_t* detail) {
  if (!pl) return BMM_ERR_INVALID_ARG;
  uint32_t w = 0;
  if (cudaMemcpy(&w, pl->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return BMM_ERR_CUDA;
  if (w != 0 && cudaMemset(pl->err, 0, sizeof(w)) != cudaSuccess) return BMM_ERR_CUDA;
  if (detail) *detail = w;
  return w == 0 ? BMM_OK : BMM_ERR_DEVICE_TIMEOUT;
}

bmm_status_t bmm_grouped_get_info(bmm_grouped_plan_t pl, int32_t* tile_n, int64_t* tiles,
                                  int32_t* stages) {
  if (!pl) return BMM_ERR_INVALID_ARG;
  if (tile_n) *tile_n = pl->bn;
  if (tiles) *tiles = pl->tiles;
  if (stages) *stages = pl->stages;
  return BMM_OK;
}

bmm_status_t bmm_grouped_destroy(bmm_grouped_plan_t pl) {
  if (!pl) return BMM_OK;
  bmm_status_t st = BMM_OK;
  if (pl->table && cudaFree(pl->table) != cudaSuccess) st = BMM_ERR_CUDA;
  if (pl->first_tile && cudaFree(pl->first_tile) != cudaSuccess) st = BMM_ERR_CUDA;
  if (pl->err && cudaFree(pl->err) != cudaSuccess) st = BMM_ERR_CUDA;
  delete pl;
  return st;
}

}  // extern "C"

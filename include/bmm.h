/*
 * bmm.h — C ABI of the GB300 (sm_103a) batched dense matrix product
 *
 *     C[b] = alpha * op(A[b]) * op(B[b]) + beta * C[b],   b = 0 .. batch-1
 *
 * op() is the identity or the transpose; A and B hold bf16 or fp16 values
 * (both the same type); products accumulate in fp32 on the tensor cores
 * (tcgen05, accumulator in Tensor Memory); alpha and beta scale in fp32; C
 * is stored as fp32 or bf16 (round to nearest even).
 *
 * Where the operation is defined:
 *  - "Triton Optimization Reference (cuTile -> Triton)", section 1 (EVEN_K
 *    fast path): the K loop adds tl.dot of A and B tiles into an fp32
 *    accumulator; when K is not a multiple of the tile, the last tile's
 *    out-of-range elements are loaded as zero.
 *  - same page, section 2: a transposed A or B is expressed by the strides
 *    used to address the loaded tile, never by a transpose inside the loop.
 *  - same page, section 3: batch items are independent problems laid out
 *    with a stride between them (batch on its own grid axis).
 *  - "Optimize Triton Block Parameters", Correctness requirements: any tile
 *    configuration must give the same result for M, N, K that are not
 *    multiples of the tile (for example K = 48 with a 64-wide K tile).
 *
 * Storage convention (row-major, strides in ELEMENTS):
 *   transA = 0: A[b] is M x K;  element (i,k) at A + b*strideA + i*lda + k
 *   transA = 1: A[b] is K x M;  element (i,k) at A + b*strideA + k*lda + i
 *   transB = 0: B[b] is K x N;  element (k,j) at B + b*strideB + k*ldb + j
 *   transB = 1: B[b] is N x K;  element (k,j) at B + b*strideB + j*ldb + k
 *   C[b] is M x N;              element (i,j) at C + b*strideC + i*ldc + j
 * A batch stride of 0 broadcasts A (or B) over the batch.  C's batch stride
 * must keep distinct batch items apart (strideC >= (M-1)*ldc + N when M > 0).
 *
 * Semantics:
 *   beta == 0  -> C is not read (NaN or garbage in C does not propagate).
 *   alpha == 0 or K == 0 -> A and B are not read; C = beta * C.
 *   batch, M or N == 0 -> nothing is launched; BMM_OK.
 *   C must not overlap A or B.
 *
 * Threading and streams: every call is host-side thread-safe for distinct
 * plans.  One plan may have one bmm_run in flight at a time on the GPU (its
 * operand-staging workspace and device error word are per plan).  bmm_run
 * is asynchronous with respect to the host: it enqueues work on `stream`
 * and returns.
 *
 * Errors: return codes only; nothing crosses the ABI as an exception.
 * A device-side wait that runs past its time limit does not trap: the
 * kernel records BMM_ERR_DEVICE_TIMEOUT in the plan's device error word,
 * releases its resources and exits; read it with bmm_get_device_error()
 * after synchronising the stream.
 */
#ifndef DMT_BMM_H
#define DMT_BMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define BMM_API __attribute__((visibility("default")))
#else
#define BMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types (values of bmm_desc_t.typeA/typeB/typeC). */
typedef enum {
  BMM_BF16 = 0,
  BMM_F16 = 1,
  BMM_F32 = 2
} bmm_dtype_t;

typedef enum {
  BMM_OK = 0,
  BMM_ERR_INVALID_ARG = 1,    /* a size, stride, type or pointer argument is invalid */
  BMM_ERR_UNSUPPORTED = 2,    /* valid but outside what this build supports */
  BMM_ERR_MISALIGNED = 3,     /* a base pointer lacks the alignment the plan needs */
  BMM_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed */
  BMM_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait expired (see above) */
  BMM_ERR_NO_DEVICE = 6       /* no usable sm_103 device is current */
} bmm_status_t;

/* Problem description.  All sizes and strides are in elements. */
typedef struct {
  int64_t batch, M, N, K;
  int64_t lda, ldb, ldc;
  int64_t strideA, strideB, strideC;
  int32_t transA, transB;     /* 0 or 1 */
  int32_t typeA, typeB, typeC; /* bmm_dtype_t: A,B in {BF16,F16} and equal; C in {F32,BF16} */
} bmm_desc_t;

/* What the planner chose for a problem (for tests, benchmarks and logs). */
typedef struct {
  int32_t tile_m, tile_n, tile_k; /* MMA-view tile (after any operand swap) */
  int32_t stages;                 /* shared-memory ring depth */
  int32_t swap_ab;                /* 1: computes C^T = op(B)^T op(A)^T (skinny M) */
  int32_t pack_a, pack_b;         /* 0: read in place by TMA; 1: staged through the
                                     workspace first; 2: read in place by the
                                     kernel's row loader (plain loads, no staging) */
  int32_t even_k;                 /* 1: K is a multiple of tile_k (no tail tile) */
  int32_t tmem_cols;              /* Tensor Memory columns allocated per CTA */
  int32_t cta_pair;               /* 1: tiles run on CTA pairs (2-SM MMA, tile_m = 256) */
  int64_t tiles;                  /* output tiles over the whole batch */
  int64_t smem_bytes;             /* dynamic shared memory per CTA */
  int64_t stage_bytes;            /* bytes of one CTA's ring stage (its A and B tile parts) */
  int64_t workspace_bytes;        /* device workspace for staged operands */
  int32_t stream_k;               /* 1: the tiles left over after the last whole round
                                     are split along K over the CTA pairs (see bmm_run) */
  int32_t sk_tiles;               /* tiles split that way when all of the device's CTA
                                     pairs are resident (0: none) */
  int64_t sk_workspace_bytes;     /* device memory the plan keeps for the split's fp32
                                     partial sums and flags */
  int32_t stages_bf16_box;        /* ring depth of runs whose C goes out as bf16 through
                                     TMA box stores (beta = 0, 16-byte-aligned C): CTA-pair
                                     plans give those runs half the epilogue buffers and
                                     the ring the rest; otherwise equal to stages */
  int32_t reserved0;
} bmm_plan_info_t;

typedef struct bmm_plan_s* bmm_plan_t;

/*
 * Validate `desc` and plan the product: tile shape by shape class (including
 * the swap to C^T for skinny M), ring depth from the shared-memory budget
 * (stages x (A tile + B tile), "Optimize Triton Block Parameters", Step 2;
 * at most 8, fewer with DMT_BMM_STAGES),
 * and, per operand, whether TMA reads it in place or it is first copied into
 * an aligned workspace (TMA needs 16-byte strides and bases; "FLA Triton ->
 * Gluon porting", section 3, TMA).
 *
 * Needs a current CUDA device of compute capability 10.3: it queries the SM
 * count and allocates the plan's device error word and workspace
 * (cudaMalloc).  Arguments are validated before any CUDA call.
 * On success *plan owns those allocations until bmm_destroy.
 * Returns BMM_OK, BMM_ERR_INVALID_ARG (null pointer, negative size, ld less
 * than the stored row length, bad type combination, overlapping C batches),
 * BMM_ERR_UNSUPPORTED (dimension beyond 2^31-1), BMM_ERR_NO_DEVICE or
 * BMM_ERR_CUDA.  On error *plan is set to NULL.
 */
BMM_API bmm_status_t bmm_create(const bmm_desc_t* desc, bmm_plan_t* plan);

/*
 * Planning only, on the host, for a GB300 (152 SMs, 227 KB shared memory
 * per CTA): fills *info with what bmm_create would choose.  Makes no CUDA
 * call.  Returns BMM_OK or BMM_ERR_INVALID_ARG / BMM_ERR_UNSUPPORTED as
 * bmm_create would.
 */
BMM_API bmm_status_t bmm_plan_query(const bmm_desc_t* desc, bmm_plan_info_t* info);

/* Copy the plan's choices into *info.  BMM_ERR_INVALID_ARG on null. */
BMM_API bmm_status_t bmm_get_plan_info(bmm_plan_t plan, bmm_plan_info_t* info);

/*
 * Enqueue C = alpha*op(A)*op(B) + beta*C on `stream` (a cudaStream_t; NULL
 * is the legacy default stream).  A, B, C are device pointers owned by the
 * caller and laid out as `desc` said at bmm_create.  Operands that the plan
 * reads in place by TMA must have 16-byte-aligned base pointers; otherwise
 * BMM_ERR_MISALIGNED is returned and nothing is enqueued.  Operands whose row
 * or batch strides are not 16-byte multiples are staged through the plan's
 * workspace (or, with the environment variable DMT_BMM_LDG=1 at plan time,
 * read in place by the kernel's row loader) and need only element
 * alignment, as does C.  Returns BMM_OK once the work is enqueued,
 * BMM_ERR_INVALID_ARG (null plan or pointer), or BMM_ERR_CUDA (launch
 * failure).  Does not synchronise.
 *
 * Stream-K tail (plans with cta_pair = 1, K >= 2048 and no operand read by
 * the row loader; stream_k in bmm_plan_info_t): the CTA pairs first run
 * whole 256 x 256 tiles in rounds; the tiles left over after the last whole
 * round ("Triton Optimization Reference", section 7: the last wave of a
 * persistent grid) are cut along K.  At most half as many leftover tiles as
 * resident pairs: each tile runs on two pairs, the one with the first
 * k-block (the owner) taking a longer range than the other by about the time
 * the other's partial takes to reach the workspace.  More leftover tiles:
 * equal ranges of k-blocks, one per pair, a range covering the end of one
 * tile and the start of the next.  Either way the piece of a tile without its
 * first k-block leaves its fp32 partial sum in the plan's stream-K workspace
 * and raises a flag, and the piece with the first k-block waits for those
 * flags, adds the partials and writes C.  The sum is still accumulated in
 * fp32 (only its order changes).  Every pair of the launch must be resident
 * at once: with other kernels holding SMs concurrently, a wait for a flag can
 * run out, which is reported as BMM_ERR_DEVICE_TIMEOUT.  The environment
 * variable DMT_BMM_STREAMK=0 at plan time turns the split off.  A plan whose
 * launch was cut short by a device error should be destroyed: its flags may
 * be left raised.
 */
BMM_API bmm_status_t bmm_run(bmm_plan_t plan, const void* A, const void* B, void* C,
                     float alpha, float beta, void* stream);

/*
 * Read and clear the plan's device error word.  Call only after the stream
 * used by bmm_run has been synchronised (this call does a blocking copy).
 * Returns BMM_OK, BMM_ERR_DEVICE_TIMEOUT, or BMM_ERR_CUDA.  If `detail` is
 * not NULL it receives the raw word (role and wait site, 0 when clean).
 */
BMM_API bmm_status_t bmm_get_device_error(bmm_plan_t plan, uint32_t* detail);

/*
 * Free the plan's device allocations and host state.  Calls cudaFree, which
 * synchronises with the device; it does not otherwise wait on user streams.
 * NULL is accepted.  Returns BMM_OK or BMM_ERR_CUDA.
 */
BMM_API bmm_status_t bmm_destroy(bmm_plan_t plan);

/*
 * Grouped launch: many independent products C_i = alpha_i*op(A_i)*op(B_i) +
 * beta_i*C_i of different sizes in one persistent launch ("Triton
 * Optimization Reference (cuTile -> Triton)", section 8: grouping many small
 * tensors into one launch instead of one launch each, applied here to the
 * contraction).  Every problem shares transA/transB and the element types;
 * each has its own sizes, row strides, pointers and scalars.  Sizes and
 * strides follow bmm_desc_t with batch = 1.
 */
typedef struct {
  int64_t M, N, K;
  int64_t lda, ldb, ldc;  /* elements */
  const void* A;
  const void* B;
  void* C;
  float alpha, beta;
} bmm_group_problem_t;

typedef struct bmm_grouped_plan_s* bmm_grouped_plan_t;

/*
 * Plan a grouped launch over `count` problems (host array; the sizes and
 * strides are fixed here, pointers and scalars are read again at each run).
 * Requirements beyond bmm_create's: K >= 1, and lda, ldb, ldc multiples of
 * 16 bytes (no staging copies in a grouped launch).  Problems with M or N of
 * 0 are skipped.  Allocates the plan's device problem table and error word.
 * Returns BMM_OK, BMM_ERR_INVALID_ARG, BMM_ERR_UNSUPPORTED (K = 0, stride not
 * a 16-byte multiple, count beyond 65536), BMM_ERR_NO_DEVICE or BMM_ERR_CUDA.
 */
BMM_API bmm_status_t bmm_grouped_create(int32_t count, const bmm_group_problem_t* problems,
                                        int32_t transA, int32_t transB, int32_t typeAB,
                                        int32_t typeC, bmm_grouped_plan_t* plan);

/*
 * Enqueue the grouped launch on `stream`: `problems` (host array, same count
 * and sizes as at bmm_grouped_create) supplies this run's pointers and
 * alpha/beta.  The problem table is copied to the device on `stream` before
 * the kernel; one run of a plan may be in flight at a time.  A and B need
 * 16-byte-aligned base pointers (BMM_ERR_MISALIGNED otherwise).  Unlike
 * bmm_run, alpha == 0 still reads A and B.  Device-side wait timeouts are
 * read with bmm_grouped_get_device_error.
 */
BMM_API bmm_status_t bmm_grouped_run(bmm_grouped_plan_t plan, const bmm_group_problem_t* problems,
                                     void* stream);

/* As bmm_get_device_error, for a grouped plan. */
BMM_API bmm_status_t bmm_grouped_get_device_error(bmm_grouped_plan_t plan, uint32_t* detail);

/* Tile width, tiles and stages the grouped plan uses (NULL pointers allowed). */
BMM_API bmm_status_t bmm_grouped_get_info(bmm_grouped_plan_t plan, int32_t* tile_n,
                                          int64_t* tiles, int32_t* stages);

/* Free the grouped plan's device table and error word (cudaFree). */
BMM_API bmm_status_t bmm_grouped_destroy(bmm_grouped_plan_t plan);

/*
 * Fused attention-shaped contraction: O[b] = softmax(alpha * Q[b] K[b]^T) V[b]
 * with the softmax over keys, computed in one pass without writing the score
 * matrix (the attention pair of the pages is S = alpha Q K^T, P = softmax(S),
 * O = P V; "Triton Optimization Reference (cuTile -> Triton)", attention-style
 * contractions).  Q: [batch][Lq][D], K and V: [batch][Lk][D], O: [batch][Lq][D],
 * all bf16, row-major with row strides ld* and batch strides stride*
 * (elements).  The probabilities are rounded to bf16 before their product
 * with V (as in the two-step pair); accumulation is fp32; O is rounded to
 * bf16 once.  This build supports D = 128 only.
 */
typedef struct {
  int64_t batch, Lq, Lk, D;
  int64_t ldq, ldk, ldv, ldo;
  int64_t strideQ, strideK, strideV, strideO;
  float alpha;
} bmm_attn_desc_t;

typedef struct bmm_attn_plan_s* bmm_attn_plan_t;

/*
 * Validate and plan.  Requirements: D = 128; row strides >= D; every stride a
 * multiple of 8 elements (16 bytes); Lk >= 1 when there are queries; Lq and Lk
 * at most 2^30 and batch below 2^31 (else BMM_ERR_UNSUPPORTED).  Allocates
 * the plan's device error word.  Returns BMM_OK, BMM_ERR_INVALID_ARG,
 * BMM_ERR_UNSUPPORTED, BMM_ERR_NO_DEVICE or BMM_ERR_CUDA.
 */
BMM_API bmm_status_t bmm_attn_create(const bmm_attn_desc_t* desc, bmm_attn_plan_t* plan);

/* Enqueue O = softmax(alpha Q K^T) V on `stream`.  All four base pointers must
 * be 16-byte aligned (BMM_ERR_MISALIGNED).  Asynchronous; one run of a plan in
 * flight at a time. */
BMM_API bmm_status_t bmm_attn_run(bmm_attn_plan_t plan, const void* Q, const void* K, const void* V,
                                  void* O, void* stream);

/* As bmm_get_device_error, for an attention plan. */
BMM_API bmm_status_t bmm_attn_get_device_error(bmm_attn_plan_t plan, uint32_t* detail);

/* Free the plan (cudaFree of its error word). */
BMM_API bmm_status_t bmm_attn_destroy(bmm_attn_plan_t plan);

/*
 * Host-buffer form: A, B (and C_in when beta != 0) are read from host memory,
 * C is written back to host memory, in the layouts `desc` describes (the same
 * strides as on the device).  The plan owns device copies of the operands and
 * two copy streams; the work is cut into chunks of whole batch items (batch
 * >= 2) or of 256-row blocks of A and C (batch 1, A row-major), and chunk c's
 * inputs are copied in while chunk c-1 computes and chunk c-2's C is copied
 * out.  The result is bit for bit the one bmm_run gives (the chunks split
 * independent rows or batch items).  Host buffers should be page-locked
 * (cudaHostAlloc / cudaHostRegister) for the copies to overlap; pageable
 * memory works but serialises.  This is the call the end-to-end throughput
 * is measured through.
 */
typedef struct bmm_host_plan_s* bmm_host_plan_t;

/* Validate `desc` (as bmm_create), plan `chunks` pipeline chunks (0: four;
 * at most 16; fewer when the problem has fewer batch items or 256-row
 * blocks; one when batch is 1 and A is stored transposed), allocate the
 * device copies, streams and events.  BMM_ERR_INVALID_ARG, BMM_ERR_UNSUPPORTED,
 * BMM_ERR_NO_DEVICE or BMM_ERR_CUDA on failure (*plan set to NULL). */
BMM_API bmm_status_t bmm_host_create(const bmm_desc_t* desc, int32_t chunks, bmm_host_plan_t* plan);

/* C = alpha op(A) op(B) + beta C with host pointers A, B, C.  Asynchronous:
 * ordered after the work already queued on `stream`, and `stream` completes
 * once C is in host memory.  One run of a plan in flight at a time. */
BMM_API bmm_status_t bmm_host_run(bmm_host_plan_t plan, const void* A, const void* B, void* C,
                                  float alpha, float beta, void* stream);

/* The first device error word among the chunks' plans (as bmm_get_device_error). */
BMM_API bmm_status_t bmm_host_get_device_error(bmm_host_plan_t plan, uint32_t* detail);

/* The chunk count and whether chunks are row blocks (1) or batch items (0). */
BMM_API bmm_status_t bmm_host_get_chunks(bmm_host_plan_t plan, int32_t* chunks, int32_t* by_rows);

/* Free the plan: its device copies, streams, events and the chunks' plans. */
BMM_API bmm_status_t bmm_host_destroy(bmm_host_plan_t plan);

/*
 * bmm_run without any allocation, for callers that cannot call cudaMalloc:
 * code running under an allocator that owns the device's memory (a caching
 * pool, a fixed budget reserved up front) and latency-critical call paths
 * that cannot afford cudaMalloc's cost and implicit device synchronisation.
 * The pages have no counterpart to this entry point.
 *
 * It plans `desc` on the host for this call and enqueues the same kernels as
 * bmm_run on `stream`.  Its only scratch is one device array inside the
 * library (every GPU that loads the library holds it until exit): a 256-byte
 * error-word region plus a 32 MiB staging area for operands whose strides or
 * batch strides are not multiples of 16 bytes.  When such operands would need
 * more than 32 MiB of staging, the kernel's row loader reads them in place
 * instead (slower per byte than TMA, but with no staging copy).  It calls no
 * cudaMalloc, cudaFree or allocating library routine.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  The address is kept for the life of the
 * process: after a reset of the device (cudaDeviceReset, or any teardown of
 * its primary context) it is stale, so do not call this entry point again in
 * a process that has reset the device.  Every call shares the array and it keeps the
 * last call's contents, so calls whose work overlaps on the GPU (other
 * streams, other host threads) race on it: serialise them.  The error word
 * is cleared on `stream` at the start of each call.  If `device_error` is a
 * device pointer (not NULL), the call also copies the word there on
 * `stream`: 0, or the BMM_ERR_DEVICE_TIMEOUT detail described for
 * bmm_get_device_error, once the stream reaches it.
 *
 * Pointers, alignment and return codes are as for bmm_create + bmm_run.
 */
BMM_API bmm_status_t bmm_run_noalloc(const bmm_desc_t* desc, const void* A, const void* B,
                                     void* C, float alpha, float beta, void* stream,
                                     uint32_t* device_error);

/* Static, human-readable name of a status code. */
BMM_API const char* bmm_status_string(bmm_status_t status);

/* Library version as (major << 16) | minor. */
BMM_API int32_t bmm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DMT_BMM_H */

/*
 * TEST INFRASTRUCTURE — the fp64 CPU oracle for the batched dense product.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  It shares no code, header or table with the GPU
 * library: it decodes its own 16-bit inputs, keeps its own loops and never
 * includes anything from the product package.
 *
 * What it computes (the plain definition; the pages only reorganise it):
 *
 *   C_ref[b,i,j] = alpha * sum_{k=0}^{K-1} opA[b,i,k] * opB[b,k,j]
 *                  + beta * C_in[b,i,j]            (beta term only if beta != 0)
 *   Bnd[b,i,j]   = sum_{k=0}^{K-1} |opA[b,i,k]| * |opB[b,k,j]|
 *
 * "Triton Optimization Reference (cuTile -> Triton)", section 1 (EVEN_K fast
 * path): every tile step adds tl.dot(a, b) into an fp32 accumulator, and the
 * masked tail loads contribute zeros, so the tiled kernel reaches exactly this
 * sum up to rounding order.  Section 2 of the same page gives the storage
 * convention for transposed operands: transposition only swaps the strides
 * used to address the tile.
 *
 * Storage convention (row-major, element strides):
 *   transA = 0: A[b] is M x K, element (i,k) at A + b*sA + i*lda + k
 *   transA = 1: A[b] is K x M, element (i,k) at A + b*sA + k*lda + i
 *   transB = 0: B[b] is K x N, element (k,j) at B + b*sB + k*ldb + j
 *   transB = 1: B[b] is N x K, element (k,j) at B + b*sB + j*ldb + k
 *   C[b] is M x N, element (i,j) at C + b*sC + i*ldc + j
 *
 * Inputs A and B are raw bf16 or fp16 bit patterns (already rounded by the
 * input generator); C_in is fp32 values or bf16 bit patterns.  All sums run
 * in fp64 with k ascending.  The product of two 16-bit floats is exact in
 * fp64, so the only rounding is the fp64 addition.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BF16 0
#define ORC_F16 1
#define ORC_F32 2

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)

/* bf16 is the top half of an IEEE binary32: widen and convert exactly. */
static double orc_bf16_to_f64(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double orc_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1.m) * 2^(e-15) */
  }
  return sign ? -v : v;
}

static double orc_decode16(uint16_t h, int type) {
  return type == ORC_BF16 ? orc_bf16_to_f64(h) : orc_f16_to_f64(h);
}

static double orc_decode_c(const void* C, int64_t off, int typeC) {
  if (typeC == ORC_F32) return (double)((const float*)C)[off];
  return orc_bf16_to_f64(((const uint16_t*)C)[off]);
}

/* Exposed for the tests: decode a bit pattern the way the oracle does. */
double oracle_decode16(uint16_t h, int type) { return orc_decode16(h, type); }

/*
 * Round an fp64 value to the nearest bf16 (ties to even) and return its bits.
 * bf16 keeps 8 significant bits and binary32's exponent range, so the quantum
 * at |x| in [2^(E-1), 2^E) is 2^(E-8), floored at the subnormal quantum
 * 2^-133.  x / q is exact (q is a power of two) and rint() rounds it to the
 * nearest integer with ties to even in the default rounding mode.
 */
uint16_t oracle_round_bf16(double x) {
  if (isnan(x)) return 0x7fc0;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  if (isinf(x)) return signbit(x) ? 0xff80 : 0x7f80;
  int E;
  (void)frexp(x, &E); /* |x| = m * 2^E, m in [0.5, 1) */
  int qe = E - 8;
  if (qe < -133) qe = -133;
  double r = ldexp(rint(ldexp(x, -qe)), qe);
  if (fabs(r) >= ldexp(1.0, 128)) return signbit(x) ? 0xff80 : 0x7f80;
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

typedef struct {
  int64_t batch, M, N, K;
  int64_t lda, ldb, ldc;
  int64_t sA, sB, sC;
  int transA, transB, typeAB, typeC;
  double alpha, beta;
} orc_desc;

static int orc_check(const orc_desc* d) {
  if (d->batch < 0 || d->M < 0 || d->N < 0 || d->K < 0) return ORC_EINVAL;
  if (d->typeAB != ORC_BF16 && d->typeAB != ORC_F16) return ORC_EINVAL;
  if (d->typeC != ORC_F32 && d->typeC != ORC_BF16) return ORC_EINVAL;
  if (d->sA < 0 || d->sB < 0 || d->sC < 0) return ORC_EINVAL;
  return ORC_OK;
}

/* ---------------------------------------------------------------- full */

typedef struct {
  const orc_desc* d;
  const uint16_t* A;
  const uint16_t* B;
  const void* Cin;
  double* Cref;
  double* Bnd;
  const double* Bdec; /* op(B[b]) decoded, K x N row-major, shared */
  int64_t b;
  int64_t lo, hi; /* rows [lo, hi) for the row phase, k rows for decode */
  int phase;      /* 0 = decode op(B[b]), 1 = rows of C[b] */
  int rc;
} orc_job;

static void* orc_worker(void* p) {
  orc_job* j = (orc_job*)p;
  const orc_desc* d = j->d;
  const int64_t N = d->N, K = d->K;
  const int64_t b = j->b;
  if (j->phase == 0) {
    double* Bd = (double*)j->Bdec;
    const uint16_t* Bb = j->B + b * d->sB;
    for (int64_t k = j->lo; k < j->hi; ++k)
      for (int64_t n = 0; n < N; ++n) {
        int64_t off = d->transB ? n * d->ldb + k : k * d->ldb + n;
        Bd[k * N + n] = orc_decode16(Bb[off], d->typeAB);
      }
    return NULL;
  }
  double* arow = (double*)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
  double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
  double* bnd = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
  if (!arow || !acc || !bnd) {
    free(arow); free(acc); free(bnd);
    j->rc = ORC_ENOMEM;
    return NULL;
  }
  const uint16_t* Ab = j->A + b * d->sA;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    for (int64_t k = 0; k < K; ++k) {
      int64_t off = d->transA ? k * d->lda + i : i * d->lda + k;
      arow[k] = orc_decode16(Ab[off], d->typeAB);
    }
    for (int64_t n = 0; n < N; ++n) { acc[n] = 0.0; bnd[n] = 0.0; }
    /* k ascending for every (i, n): the plain definition of the sum. */
    for (int64_t k = 0; k < K; ++k) {
      const double a = arow[k];
      const double* brow = j->Bdec + k * N;
      for (int64_t n = 0; n < N; ++n) {
        const double p = a * brow[n];
        acc[n] += p;
        bnd[n] += fabs(p);
      }
    }
    for (int64_t n = 0; n < N; ++n) {
      const int64_t o = (b * d->M + i) * N + n; /* dense output */
      double c = d->alpha * acc[n];
      if (d->beta != 0.0) c += d->beta * orc_decode_c(j->Cin, b * d->sC + i * d->ldc + n, d->typeC);
      j->Cref[o] = c;
      if (j->Bnd) j->Bnd[o] = bnd[n];
    }
  }
  free(arow); free(acc); free(bnd);
  return NULL;
}

static int orc_run_phase(orc_job* jobs, int nthreads, int64_t total) {
  pthread_t th[256];
  int started[256];
  int64_t per = (total + nthreads - 1) / nthreads;
  /* Spawn workers 1..n-1, run share 0 on the calling thread, then join. */
  for (int t = nthreads - 1; t >= 0; --t) {
    jobs[t].lo = t * per < total ? t * per : total;
    jobs[t].hi = (t + 1) * per < total ? (t + 1) * per : total;
    jobs[t].rc = ORC_OK;
    started[t] = 0;
    if (jobs[t].lo >= jobs[t].hi) continue;
    if (t == 0 || pthread_create(&th[t], NULL, orc_worker, &jobs[t]) != 0)
      orc_worker(&jobs[t]); /* inline: share 0, or if spawning fails */
    else
      started[t] = 1;
  }
  int rc = ORC_OK;
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) pthread_join(th[t], NULL);
    if (jobs[t].rc != ORC_OK) rc = jobs[t].rc;
  }
  return rc;
}

/*
 * Full oracle: writes Cref (and Bnd unless it is NULL) densely as
 * [batch][M][N] fp64.  Returns 0, or a negative code for bad arguments.
 */
int oracle_bmm_f64(int64_t batch, int64_t M, int64_t N, int64_t K,
                   int64_t lda, int64_t ldb, int64_t ldc,
                   int64_t sA, int64_t sB, int64_t sC,
                   int transA, int transB, int typeAB, int typeC,
                   double alpha, double beta,
                   const uint16_t* A, const uint16_t* B, const void* Cin,
                   double* Cref, double* Bnd, int nthreads) {
  orc_desc d = {batch, M, N, K, lda, ldb, ldc, sA, sB, sC,
                transA, transB, typeAB, typeC, alpha, beta};
  if (orc_check(&d) != ORC_OK || !Cref) return ORC_EINVAL;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (batch == 0 || M == 0 || N == 0) return ORC_OK;
  double* Bdec = (double*)malloc((size_t)(K > 0 ? K : 1) * (size_t)N * sizeof(double));
  orc_job* jobs = (orc_job*)calloc((size_t)nthreads, sizeof(orc_job));
  if (!Bdec || !jobs) { free(Bdec); free(jobs); return ORC_ENOMEM; }
  int rc = ORC_OK;
  for (int64_t b = 0; b < batch && rc == ORC_OK; ++b) {
    for (int t = 0; t < nthreads; ++t) {
      jobs[t].d = &d; jobs[t].A = A; jobs[t].B = B; jobs[t].Cin = Cin;
      jobs[t].Cref = Cref; jobs[t].Bnd = Bnd; jobs[t].Bdec = Bdec; jobs[t].b = b;
      jobs[t].phase = 0;
    }
    rc = orc_run_phase(jobs, nthreads, K);
    if (rc != ORC_OK) break;
    for (int t = 0; t < nthreads; ++t) jobs[t].phase = 1;
    rc = orc_run_phase(jobs, nthreads, M);
  }
  free(Bdec);
  free(jobs);
  return rc;
}

/* ------------------------------------------------------------- sampled */

/*
 * One output element at a time, straight from the definition: for each of
 * the n samples (ib[s], ii[s], ij[s]) it sums opA[b,i,k]*opB[b,k,j] over k
 * ascending.  Used for the full-size problems where the whole product would
 * take the host too long.
 */
int oracle_bmm_sampled(int64_t batch, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc,
                       int64_t sA, int64_t sB, int64_t sC,
                       int transA, int transB, int typeAB, int typeC,
                       double alpha, double beta,
                       const uint16_t* A, const uint16_t* B, const void* Cin,
                       int64_t n, const int64_t* ib, const int64_t* ii, const int64_t* ij,
                       double* cref, double* bnd) {
  orc_desc d = {batch, M, N, K, lda, ldb, ldc, sA, sB, sC,
                transA, transB, typeAB, typeC, alpha, beta};
  if (orc_check(&d) != ORC_OK) return ORC_EINVAL;
  for (int64_t s = 0; s < n; ++s) {
    const int64_t b = ib[s], i = ii[s], j = ij[s];
    if (b < 0 || b >= batch || i < 0 || i >= M || j < 0 || j >= N) return ORC_EINVAL;
    double acc = 0.0, bd = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      int64_t oa = b * sA + (transA ? k * lda + i : i * lda + k);
      int64_t ob = b * sB + (transB ? j * ldb + k : k * ldb + j);
      double p = orc_decode16(A[oa], typeAB) * orc_decode16(B[ob], typeAB);
      acc += p;
      bd += fabs(p);
    }
    double c = alpha * acc;
    if (beta != 0.0) c += beta * orc_decode_c(Cin, b * sC + i * ldc + j, typeC);
    cref[s] = c;
    if (bnd) bnd[s] = bd;
  }
  return ORC_OK;
}

/* ------------------------------------------------- attention-pair input */

typedef struct {
  const uint16_t* Q;
  const uint16_t* Kt;
  uint16_t* P;
  int64_t L, D;
  double alpha;
  int64_t lo, hi; /* flat rows (b*L + i) */
  int rc;
} orc_sm_job;

static void* orc_softmax_worker(void* p) {
  orc_sm_job* j = (orc_sm_job*)p;
  const int64_t L = j->L, D = j->D;
  double* s = (double*)malloc((size_t)L * sizeof(double));
  double* q = (double*)malloc((size_t)D * sizeof(double));
  if (!s || !q) { free(s); free(q); j->rc = ORC_ENOMEM; return NULL; }
  for (int64_t r = j->lo; r < j->hi; ++r) {
    const int64_t b = r / L, i = r % L;
    for (int64_t k = 0; k < D; ++k) q[k] = orc_bf16_to_f64(j->Q[(b * L + i) * D + k]);
    double mx = -INFINITY;
    for (int64_t c = 0; c < L; ++c) {
      double acc = 0.0;
      for (int64_t k = 0; k < D; ++k) acc += q[k] * orc_bf16_to_f64(j->Kt[(b * L + c) * D + k]);
      s[c] = j->alpha * acc;
      if (s[c] > mx) mx = s[c];
    }
    double sum = 0.0;
    for (int64_t c = 0; c < L; ++c) { s[c] = exp(s[c] - mx); sum += s[c]; }
    for (int64_t c = 0; c < L; ++c) j->P[(b * L + i) * L + c] = oracle_round_bf16(s[c] / sum);
  }
  free(s); free(q);
  return NULL;
}

/*
 * Input recipe for the second half of the attention-shaped pair:
 *   S[b] = alpha * Q[b] * K[b]^T   (Q, K: [batch][L][D] bf16 bits, dense)
 *   P[b,i,:] = softmax over the row S[b,i,:], in fp64, rounded once to bf16.
 * P is written as [batch][L][L] bf16 bits.  The row maximum is subtracted
 * before exp(), which leaves the softmax unchanged and keeps exp() finite.
 */
int oracle_attention_probs_bf16(int64_t batch, int64_t L, int64_t D, double alpha,
                                const uint16_t* Q, const uint16_t* Kt, uint16_t* P,
                                int nthreads) {
  if (batch < 0 || L < 0 || D < 0 || !P) return ORC_EINVAL;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  int64_t rows = batch * L;
  if (rows == 0) return ORC_OK;
  pthread_t th[256];
  int started[256];
  orc_sm_job jobs[256];
  int64_t per = (rows + nthreads - 1) / nthreads;
  for (int t = nthreads - 1; t >= 0; --t) {
    orc_sm_job jb = {Q, Kt, P, L, D, alpha, t * per < rows ? t * per : rows,
                     (t + 1) * per < rows ? (t + 1) * per : rows, ORC_OK};
    jobs[t] = jb;
    started[t] = 0;
    if (jobs[t].lo >= jobs[t].hi) continue;
    if (t == 0 || pthread_create(&th[t], NULL, orc_softmax_worker, &jobs[t]) != 0)
      orc_softmax_worker(&jobs[t]);
    else
      started[t] = 1;
  }
  int rc = ORC_OK;
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) pthread_join(th[t], NULL);
    if (jobs[t].rc != ORC_OK) rc = jobs[t].rc;
  }
  return rc;
}

/* ------------------------------------------------- fused attention */

typedef struct {
  const uint16_t *Q, *K, *V;
  double *O, *Bnd;
  int64_t Lq, Lk, D;
  double alpha;
  int64_t lo, hi; /* flat query rows (b*Lq + i) */
  int rc;
} orc_att_job;

static void* orc_attention_worker(void* p) {
  orc_att_job* j = (orc_att_job*)p;
  const int64_t Lq = j->Lq, Lk = j->Lk, D = j->D;
  double* s = (double*)malloc((size_t)(Lk > 0 ? Lk : 1) * sizeof(double));
  double* q = (double*)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
  if (!s || !q) { free(s); free(q); j->rc = ORC_ENOMEM; return NULL; }
  for (int64_t r = j->lo; r < j->hi; ++r) {
    const int64_t b = r / Lq, i = r % Lq;
    for (int64_t k = 0; k < D; ++k) q[k] = orc_bf16_to_f64(j->Q[(b * Lq + i) * D + k]);
    double mx = -INFINITY;
    for (int64_t c = 0; c < Lk; ++c) {
      double acc = 0.0;
      for (int64_t k = 0; k < D; ++k) acc += q[k] * orc_bf16_to_f64(j->K[(b * Lk + c) * D + k]);
      s[c] = j->alpha * acc;
      if (s[c] > mx) mx = s[c];
    }
    double sum = 0.0;
    for (int64_t c = 0; c < Lk; ++c) { s[c] = exp(s[c] - mx); sum += s[c]; }
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0, bnd = 0.0;
      for (int64_t c = 0; c < Lk; ++c) {
        const double pv = (s[c] / sum) * orc_bf16_to_f64(j->V[(b * Lk + c) * D + d]);
        acc += pv;
        bnd += fabs(pv);
      }
      j->O[(b * Lq + i) * D + d] = acc;
      if (j->Bnd) j->Bnd[(b * Lq + i) * D + d] = bnd;
    }
  }
  free(s); free(q);
  return NULL;
}

/*
 * The attention-shaped contraction in one piece, from its definition:
 *   O[b,i,:] = sum_c softmax_c(alpha * Q[b,i,:] . K[b,c,:]) * V[b,c,:]
 * with the softmax over c in fp64 (row maximum subtracted before exp(), which
 * leaves it unchanged).  Q: [batch][Lq][D], K and V: [batch][Lk][D], dense
 * bf16 bits.  Writes O and Bnd[b,i,d] = sum_c p_ic * |V[b,c,d]| (the scale of
 * the sum, for tolerances) as [batch][Lq][D] fp64; Bnd may be NULL.
 */
int oracle_attention_f64(int64_t batch, int64_t Lq, int64_t Lk, int64_t D, double alpha,
                         const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                         double* O, double* Bnd, int nthreads) {
  if (batch < 0 || Lq < 0 || Lk < 1 || D < 0 || !O) return ORC_EINVAL;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  const int64_t rows = batch * Lq;
  if (rows == 0) return ORC_OK;
  pthread_t th[256];
  int started[256];
  orc_att_job jobs[256];
  const int64_t per = (rows + nthreads - 1) / nthreads;
  for (int t = nthreads - 1; t >= 0; --t) {
    orc_att_job jb = {Q, K, V, O, Bnd, Lq, Lk, D, alpha, t * per < rows ? t * per : rows,
                      (t + 1) * per < rows ? (t + 1) * per : rows, ORC_OK};
    jobs[t] = jb;
    started[t] = 0;
    if (jobs[t].lo >= jobs[t].hi) continue;
    if (t == 0 || pthread_create(&th[t], NULL, orc_attention_worker, &jobs[t]) != 0)
      orc_attention_worker(&jobs[t]);
    else
      started[t] = 1;
  }
  int rc = ORC_OK;
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) pthread_join(th[t], NULL);
    if (jobs[t].rc != ORC_OK) rc = jobs[t].rc;
  }
  return rc;
}

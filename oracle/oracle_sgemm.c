/*
 * oracle_sgemm.c -- plain, slow, obviously-correct CPU oracle for single
 * precision GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into its own shared library
 * (liboracle_sgemm.so) and is loaded only by the test-suite, by the package's
 * smoke check and by the CPU-baseline leg of the benchmark.  The GPU library
 * shares no code, header, table or helper with it, and the product path never
 * calls it.
 *
 * What it computes
 * ----------------
 *   R[i][j] = alpha * sum_{k=0}^{K-1} opA(i,k) * opB(k,j)  +  beta * C[i][j]
 *
 * with every matrix row-major and
 *   opA(i,k) = A[i*lda + k]  (transA == 0, A stored M x K)
 *            = A[k*lda + i]  (transA == 1, A stored K x M)
 *   opB(k,j) = B[k*ldb + j]  (transB == 0, B stored K x N)
 *            = B[j*ldb + k]  (transB == 1, B stored N x K).
 *
 * This is the definition printed as the naive kernel of
 * "CUDA矩阵乘法性能优化实战：从朴素内核到寄存器分块与Nsight剖析" (section 1.1, the
 * statement C(MxN) = A(MxK) x B(KxN) with each C[i][j] a K-term multiply-add;
 * section 2.1, matmul_naive: sum over k of A[row*K+k] * B[k*N+col]), widened to
 * the alpha/beta/transposed-B form D = alpha * A * B^T + beta * C that the
 * cloud.baidu.com article 9456745 (naive vs. 2D block-tiled shared-memory
 * matmul, its worked formula in the naive-implementation paragraph) states.
 *
 * Arithmetic
 * ----------
 *  - every product opA(i,k)*opB(k,j) of two FP32 values is exact in double
 *    (24+24 = 48 significant bits <= 53), so fused or unfused multiply-add give
 *    the same double;
 *  - the K products of one output are added in ascending k into a double that
 *    starts at 0.0 -- the order the definition writes;
 *  - R = (double)alpha * s + (double)beta * (double)C[i][j], both terms in double;
 *  - beta == 0 means C is never read (a NaN there has no effect);
 *  - alpha == 0 or K == 0 means A and B are never read and R = beta * C.
 *    (The pages are silent on these three degenerate cases; the reading taken
 *    is the usual BLAS one.)
 *
 * The result is returned in double; callers round it to FP32 (round to
 * nearest even) when they want the single-precision answer.
 *
 * Loop order: for op(B) == N the i-k-j order keeps a double row accumulator so
 * that B is walked along rows; for op(B) == T each output is a dot product
 * over contiguous k.  In both orders every output's sum runs over k ascending,
 * so the two give bit-identical doubles.  Rows are split across POSIX threads;
 * that changes nothing in any output's arithmetic.
 *
 * Build: gcc -O2 -fno-fast-math -fPIC -shared -pthread (no -ffast-math, no
 * -Ofast: the oracle must keep IEEE double semantics).
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

static inline double op_a(const float *A, int64_t lda, int transA, int64_t i, int64_t k) {
  return transA ? (double)A[k * lda + i] : (double)A[i * lda + k];
}

static inline double op_b(const float *B, int64_t ldb, int transB, int64_t k, int64_t j) {
  return transB ? (double)B[j * ldb + k] : (double)B[k * ldb + j];
}

typedef struct {
  int transA, transB;
  int64_t M, N, K;
  double alpha, beta;
  const float *A, *B, *C;
  int64_t lda, ldb, ldc;
  double *R;
  int64_t ldr;
  int64_t row_begin, row_end;
  int status;
} oracle_job;

/* One block of output rows [row_begin, row_end). */
static void *oracle_rows(void *arg) {
  oracle_job *job = (oracle_job *)arg;
  const int64_t N = job->N, K = job->K;
  const int skip_product = (job->alpha == 0.0) || (K == 0);
  double *acc = NULL;
  if (!skip_product && !job->transB) {
    acc = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!acc) {
      job->status = ORACLE_ENOMEM;
      return NULL;
    }
  }
  for (int64_t i = job->row_begin; i < job->row_end; ++i) {
    double *r = job->R + i * job->ldr;
    if (skip_product) {
      for (int64_t j = 0; j < N; ++j) r[j] = 0.0;
    } else if (!job->transB) {
      /* i-k-j: acc[j] collects sum_k opA(i,k)*B[k][j], k ascending. */
      for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double a = op_a(job->A, job->lda, job->transA, i, k);
        const float *brow = job->B + k * job->ldb;
        for (int64_t j = 0; j < N; ++j) acc[j] += a * (double)brow[j];
      }
      for (int64_t j = 0; j < N; ++j) r[j] = job->alpha * acc[j];
    } else {
      /* i-j-k: one dot product per output, k ascending. */
      for (int64_t j = 0; j < N; ++j) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
          s += op_a(job->A, job->lda, job->transA, i, k) * op_b(job->B, job->ldb, 1, k, j);
        r[j] = job->alpha * s;
      }
    }
    if (job->beta != 0.0) {
      const float *crow = job->C + i * job->ldc;
      for (int64_t j = 0; j < N; ++j) r[j] += job->beta * (double)crow[j];
    }
  }
  free(acc);
  return NULL;
}

static int check_args(int transA, int transB, int64_t M, int64_t N, int64_t K,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      float beta, const float *C, int64_t ldc) {
  if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return ORACLE_EINVAL;
  if (M < 0 || N < 0 || K < 0) return ORACLE_EINVAL;
  /* stored widths: A is (transA ? K x M : M x K), B is (transB ? N x K : K x N) */
  if (lda < (transA ? (M > 1 ? M : 1) : (K > 1 ? K : 1))) return ORACLE_EINVAL;
  if (ldb < (transB ? (K > 1 ? K : 1) : (N > 1 ? N : 1))) return ORACLE_EINVAL;
  if (beta != 0.0f && ldc < (N > 1 ? N : 1)) return ORACLE_EINVAL;
  if (M > 0 && N > 0 && K > 0 && (A == NULL || B == NULL)) return ORACLE_EINVAL;
  if (M > 0 && N > 0 && beta != 0.0f && C == NULL) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/*
 * Full product.  R is an M x N row-major double matrix with leading dimension
 * ldr >= N.  nthreads <= 1 runs on the calling thread.
 */
int oracle_sgemm_f64(int transA, int transB, int64_t M, int64_t N, int64_t K,
                     float alpha, const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     float beta, const float *C, int64_t ldc,
                     double *R, int64_t ldr, int nthreads) {
  int st = check_args(transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc);
  if (st != ORACLE_OK) return st;
  if (M == 0 || N == 0) return ORACLE_OK;
  if (R == NULL || ldr < N) return ORACLE_EINVAL;
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > M) nthreads = (int)M;

  oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  char *started = (char *)calloc((size_t)nthreads, 1);
  if (!jobs || !tids || !started) {
    free(jobs);
    free(tids);
    free(started);
    return ORACLE_ENOMEM;
  }
  const int64_t per = (M + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    oracle_job *j = &jobs[t];
    j->transA = transA;
    j->transB = transB;
    j->M = M;
    j->N = N;
    j->K = K;
    j->alpha = (double)alpha;
    j->beta = (double)beta;
    j->A = A;
    j->B = B;
    j->C = C;
    j->lda = lda;
    j->ldb = ldb;
    j->ldc = ldc;
    j->R = R;
    j->ldr = ldr;
    j->row_begin = (int64_t)t * per < M ? (int64_t)t * per : M;
    j->row_end = j->row_begin + per < M ? j->row_begin + per : M;
    j->status = ORACLE_OK;
    /* block 0 runs on the calling thread; empty blocks run nowhere */
    if (t == 0 || j->row_begin >= j->row_end) continue;
    if (pthread_create(&tids[t], NULL, oracle_rows, j) == 0)
      started[t] = 1;
    else
      oracle_rows(j); /* could not spawn: do the block here */
  }
  oracle_rows(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (started[t]) pthread_join(tids[t], NULL);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].status != ORACLE_OK) st = jobs[t].status;
  free(started);
  free(jobs);
  free(tids);
  return st;
}

/*
 * Selected outputs only: R[e] = the (I[e], J[e]) entry of the full product.
 * Each entry is computed on its own with the same arithmetic as above; used to
 * check sampled outputs of products too large to compute whole on the CPU.
 */
int oracle_sgemm_entries_f64(int transA, int transB, int64_t M, int64_t N, int64_t K,
                             float alpha, const float *A, int64_t lda,
                             const float *B, int64_t ldb,
                             float beta, const float *C, int64_t ldc,
                             int64_t n_entries, const int64_t *I, const int64_t *J,
                             double *R) {
  int st = check_args(transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc);
  if (st != ORACLE_OK) return st;
  if (n_entries < 0 || (n_entries > 0 && (I == NULL || J == NULL || R == NULL))) return ORACLE_EINVAL;
  const int skip_product = (alpha == 0.0f) || (K == 0);
  for (int64_t e = 0; e < n_entries; ++e) {
    const int64_t i = I[e], j = J[e];
    if (i < 0 || i >= M || j < 0 || j >= N) return ORACLE_EINVAL;
    double s = 0.0;
    if (!skip_product)
      for (int64_t k = 0; k < K; ++k)
        s += op_a(A, lda, transA, i, k) * op_b(B, ldb, transB, k, j);
    double r = skip_product ? 0.0 : (double)alpha * s;
    if (beta != 0.0f) r += (double)beta * (double)C[i * ldc + j];
    R[e] = r;
  }
  return ORACLE_OK;
}

/*
 * Matrix transpose, the workload of "现代 CUDA 工具箱实战：从朴素代码到硬件极限的优化之路"
 * (hankli.space; its naive kernel in "代码实现 / Baseline" reads element
 * (y, x) of the N x N input and writes it to (x, y) of the output):
 *
 *   out[c * ld_out + r] = in[r * ld_in + c]     for r < rows, c < cols,
 *
 * widened from a square N x N matrix to a rows x cols input with leading
 * dimensions (out is cols x rows).  A copy of each value: no arithmetic, so
 * the result is bit-exact by construction.  Elements of out outside the
 * cols x rows block are not touched.
 */
int oracle_transpose_f32(int64_t rows, int64_t cols, const float *in, int64_t ld_in,
                         float *out, int64_t ld_out) {
  if (rows < 0 || cols < 0) return ORACLE_EINVAL;
  if (rows == 0 || cols == 0) return ORACLE_OK;
  if (in == NULL || out == NULL || ld_in < cols || ld_out < rows) return ORACLE_EINVAL;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) out[c * ld_out + r] = in[r * ld_in + c];
  return ORACLE_OK;
}

/*
 * ttt_kernels.h -- kernel-level entry points of libttt (C ABI).
 *
 * These expose the individual CUDA kernels that make up one TTT-E2E
 * inner-loop step, so that each can be checked on its own against the float64
 * oracle.  All pointers are DEVICE pointers owned by the caller; nothing is
 * allocated, retained or synchronised; every call enqueues on `stream`
 * (a cudaStream_t, NULL = legacy default stream) and returns 0, or a negative
 * TTT_ERR_* code (ttt.h) when an argument is rejected or the launch fails.
 *
 * bf16 operands are stored as uint16 bit patterns.  In "split" mode an fp32
 * value v travels as a pair hi = bf16(v), lo = bf16(v - hi); the *_lo pointers
 * are NULL otherwise.
 */
#ifndef TTT_KERNELS_H
#define TTT_KERNELS_H

#include <stddef.h>
#include <stdint.h>

#include "ttt.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Epilogue selector of ttt_k_gemm (applied to each fp32 accumulator value acc). */
enum {
  TTT_EPI_F32 = 0,      /* out32[r][c] = acc                                          */
  TTT_EPI_OPND = 1,     /* out_hi/lo[r][c] = split(acc)                               */
  TTT_EPI_RESID = 2,    /* out32[r][c] = resid[r][c] + acc   (may alias)              */
  TTT_EPI_GELU = 3,     /* out32 = acc (if out32); out_hi/lo = gelu_tanh(acc)         */
  TTT_EPI_GELU_BWD = 4, /* out_hi/lo = acc * gelu_tanh'(aux[r][c])                    */
  TTT_EPI_SGD = 5,      /* w32 -= eta*acc; w_hi/lo = split(w32)                       */
  TTT_EPI_CE_FWD = 6,   /* part[ntile*M + r] = (max, sum exp(acc - max)) over the
                           columns of N-tile ntile; zt[r] = acc at column tgt[r]      */
  TTT_EPI_CE_BWD = 7    /* out_hi/lo = tgt[r] < 0 ? 0 :
                           (exp(acc - lse[r]) - [c == tgt[r]]) * scale               */
};

/* Epilogue operands of ttt_k_gemm.  Row pitches (ld*) are in elements and must
 * be multiples of 8; unused fields may be zero. */
typedef struct {
  float* out32;  int64_t ldo32;
  void* out_hi;  void* out_lo;  int64_t ldo;
  const float* resid;  int64_t ldr;
  const float* aux;  int64_t ldaux;
  float* w32;  void* w_hi;  void* w_lo;  int64_t ldw;  float eta;
  const int32_t* tgt;  float* part;  float* zt;  const float* lse;  float scale;
  int32_t* err;   /* device int, set non-zero if a bounded wait in the kernel expired */
  int32_t allow_ksplit; /* F32 / RESID only: non-zero lets the product be cut into K slices
                           whose partial sums are added atomically into out32 (cleared,
                           or loaded with resid, first); the summation order then varies */
} ttt_gemm_epilogue;

/*
 * C[M][N] = A[M][K] . B^T[K][N] on the tcgen05 tensor cores (bf16 x bf16,
 * fp32 accumulate), then epilogue `epi`.
 *   A, K-major (a_mn = 0): row-major [M][lda], K in the columns.
 *   A, MN-major (a_mn = 1): row-major [K][lda], M in the columns (A^T stored).
 *   B, K-major (b_mn = 0): row-major [N][ldb], K in the columns.
 *   B, MN-major (b_mn = 1): row-major [K][ldb], N in the columns (x.W with
 *   W stored [K][N] row-major).
 * split != 0: a_lo / b_lo hold the bf16 remainders; three products per step.
 * Base pointers must be 16-byte aligned and pitches multiples of 8 elements.
 */
TTT_API int ttt_k_gemm(int epi, int M, int N, int K,
               const void* a_hi, const void* a_lo, int64_t lda, int a_mn,
               const void* b_hi, const void* b_lo, int64_t ldb, int b_mn,
               int split, const ttt_gemm_epilogue* e, void* stream);

/*
 * Windowed causal attention forward for one chunk (all heads), tcgen05.
 * Token-major bf16 [rows][d] arrays, d = H*dh, head h in columns h*dh..h*dh+dh-1:
 *   q       [n][d]       queries at absolute positions pos0 .. pos0+n-1 (post-RoPE)
 *   kc, vc  [window][d]  window cache: slot (p mod window) holds position p, for
 *                        the positions max(0, pos0-window) .. pos0-1
 *   ko, vo  [n][d]       the chunk's own keys/values
 * A query at p attends to the keys at positions j with p - window < j <= p.
 * Outputs: o [n][d] (bf16 hi/lo), lse [H][n] (log2-sum-exp of the scaled scores,
 * may be NULL).  dh in {32, 64, 96, 128} ({32, 64} with split), window % 128 == 0,
 * n <= window.  *_lo are the bf16 remainders (split != 0) or NULL.
 */
TTT_API int ttt_k_attn_fwd(int n, int H, int dh, int window, int64_t pos0, int split,
                           const void* q_hi, const void* q_lo, const void* kc_hi, const void* kc_lo,
                           const void* vc_hi, const void* vc_lo, const void* ko_hi, const void* ko_lo,
                           const void* vo_hi, const void* vo_lo, void* o_hi, void* o_lo, float* lse,
                           int32_t* err, void* stream);

/*
 * Attention backward for the same geometry: given dO [n][d] (bf16 hi/lo), the
 * forward's lse [H][n] and D [H][n] = rowsum(dO * O) per head, writes fp32
 * token-major dq [n][d] (through every key in the window) and dk, dv [n][d]
 * for the chunk's own keys (cached keys are constants).
 */
TTT_API int ttt_k_attn_bwd(int n, int H, int dh, int window, int64_t pos0, int split,
                           const void* q_hi, const void* q_lo, const void* kc_hi, const void* kc_lo,
                           const void* vc_hi, const void* vc_lo, const void* ko_hi, const void* ko_lo,
                           const void* vo_hi, const void* vo_lo, const void* do_hi, const void* do_lo,
                           const float* lse, const float* D, float* dq, float* dk, float* dv,
                           int32_t* err, void* stream);

/* D[h][t] = sum_i dO[t][h*dh+i] * O[t][h*dh+i] (hi + lo values). */
TTT_API int ttt_k_attn_rowdot(int n, int H, int dh, const void* do_hi, const void* do_lo, const void* o_hi,
                              const void* o_lo, float* D, void* stream);

/*
 * Failure detection, exercised without a fault: one CTA in which two threads
 * wait on an mbarrier phase that nothing completes, through the bounded wait
 * every kernel of the library uses.  Thread 0 of warp 0 starts at once, thread
 * 0 of warp 1 100 ms later.  After the wait limit (4 s) warp 0's wait gives up:
 * it raises the CTA abort flag and writes 3 (an epilogue-side wait ran out)
 * into *err if *err was 0; warp 1's wait then stops at its next check of the
 * flag, without writing *err.  status[2w] = 1 if warp w's wait succeeded (never)
 * else 0; status[2w+1] = milliseconds warp w waited.  err and status (4 ints)
 * are caller-owned DEVICE memory.  Returns TTT_ERR_ARG for a null pointer,
 * TTT_ERR_CUDA if the launch fails, else 0; the kernel runs about 4 s, and the
 * context stays usable afterwards.
 */
TTT_API int ttt_k_wait_limit_probe(int32_t* err, int32_t* status, void* stream);

/*
 * LM-head cross-entropy statistics WITHOUT ANY DEVICE ALLOCATION.  The paper
 * has no counterpart: this entry point exists for callers that cannot call
 * cudaMalloc, for example a process whose device memory is owned up front by
 * another allocator, or a latency-bound caller that cannot take cudaMalloc's
 * implicit device synchronisation.  It computes what ttt_k_gemm with
 * TTT_EPI_CE_FWD followed by the per-row combine computes, for bf16 operands:
 *   z = x . W_lm          x    [M][ldx] bf16 (K-major, K used columns)
 *                        W_lm [K][ldw] bf16 (row-major, V used columns)
 *   lse[r]  = log sum_c exp(z[r][c])                        (natural log)
 *   loss[r] = tgt[r] >= 0 ? lse[r] - z[r][tgt[r]] : 0        tgt[r] in {-1} U [0, V)
 * x, W_lm, tgt, lse and loss are caller-owned DEVICE memory; err is an
 * optional device int that a kernel sets if one of its bounded waits expires.
 *
 * Scratch: the partial (max, sum) pairs of every (row, vocab tile) and the
 * target logits live in one file-scope __device__ array of
 * TTT_CE_STATIC_SCRATCH_ENTRIES float2 (4 MiB).  The CUDA runtime loads the
 * library's modules lazily, so the array is allocated on a device by the
 * first call there (the symbol lookup below loads its module) and is held
 * until the process exits; a caller whose memory another allocator reserves
 * up front should make its first call before that reservation.  Every scratch element a call reads is
 * written earlier in the same call, so nothing needs clearing between calls.
 * All calls share that one array: calls whose work overlaps on the GPU (other
 * streams, other host threads) race and give wrong results; serialise them.
 * Limit: ceil(V / 128) * M + ceil(M / 2) <= TTT_CE_STATIC_SCRATCH_ENTRIES
 * (e.g. M = 1024 rows with V up to 65,408); larger sizes return
 * TTT_ERR_SCRATCH before anything is enqueued.
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (once per device, with that device current); make that
 * first call before any stream capture.  Like the rest of the library (ttt.h),
 * one process drives one GPU: launch settings are cached per process.  Returns 0, TTT_ERR_ARG (null
 * pointer, size < 1, pitch < width or not a multiple of 8), TTT_ERR_SCRATCH,
 * or TTT_ERR_CUDA (symbol lookup or launch failure).
 */
#define TTT_CE_STATIC_SCRATCH_ENTRIES 524288
#define TTT_ERR_SCRATCH (-7)     /* the call needs more static scratch than the library holds */
TTT_API int ttt_k_lmhead_ce_static(int M, int K, int V, const void* x, int64_t ldx, const void* w_lm,
                                   int64_t ldw, const int32_t* tgt, float* lse, float* loss, int32_t* err,
                                   void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TTT_KERNELS_H */

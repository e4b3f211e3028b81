// Row-wise kernels (rowops.cu).  All return 0 or a cudaError_t value.
#pragma once
#include "kernels.h"

namespace ttt {

int rows_embed(const int* tok, int n, const float* E, int V, int d, float* x, int* err, cudaStream_t st);
int rows_targets(const int* tok, int n, const int* next, int V, int* tgt, int* err, cudaStream_t st);
// x_copy (optional, not x): also receives x, the start value of a K-sliced residual product
int rows_rmsnorm(const float* x, const float* g, float eps, int n, int d, bf16* yh, bf16* yl, float* rstd,
                 cudaStream_t st, float* x_copy = nullptr);
// clear_dy: dy is set to zero once read (dy must be none of x, resid, out)
int rows_rmsnorm_bwd(const float* dy, const float* x, const float* g, const float* rstd, const float* resid, int n,
                     int d, float* out, bf16* oh, bf16* ol, cudaStream_t st, bool clear_dy = false);
int rows_rope_table(long pos0, int n, int dh, const double* inv_freq, float* cs, float* sn, cudaStream_t st);
int rows_rope_qkv(const float* qkv, const float* cs, const float* sn, int n, int H, int dh, bf16* qh, bf16* ql,
                  bf16* kh, bf16* kl, bf16* vh, bf16* vl, cudaStream_t st);
int rows_commit(const bf16* own, bf16* ring, long own_layer_stride, long ring_layer_stride, int n_layers, long pos0,
                int n, int window, int d, cudaStream_t st);
int rows_ce_combine(const float2* part, const float* zt, const int* tgt, int n, int ntiles, float* lse,
                    float* loss_row, cudaStream_t st);
// out = mean of loss_row over rows with tgt >= 0; inv_count = 1 / that count (0 if none)
int rows_loss_mean(const float* loss_row, const int* tgt, int n, float* out, float* inv_count, cudaStream_t st);
int rows_convert(const float* src, long rows, int cols, long src_ld, bf16* dh, bf16* dl, long dst_ld,
                 cudaStream_t st);
// next token from logits z[V]: sample = 0 greedy (first largest), 1 inverse CDF of softmax(z / temp) at *u
int rows_pick(const float* z, int V, int sample, float temp, const float* u, int* out, cudaStream_t st);
int rows_attn_rowdot(const bf16* doh, const bf16* dol, const bf16* oh, const bf16* ol, int n, int H, int dh, float* D,
                     cudaStream_t st);

}  // namespace ttt

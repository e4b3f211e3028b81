// Internal C++ interface between the host orchestrator and the CUDA kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace ttt {

using bf16 = __nv_bfloat16;

// Launch with programmatic stream serialisation: the kernel may begin while
// its predecessor drains (every kernel here calls pdl_wait() before touching
// global memory).  Returns the launch's cudaError_t.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------------ GEMM
// C[M,N] = A[M,K] . B[N,K]^T on tcgen05 (bf16 operands, fp32 accumulate in
// TMEM), followed by one of these epilogues on each fp32 accumulator value.
enum Epi : int {
  EPI_F32 = 0,      // out32 = acc
  EPI_OPND = 1,     // (oh, ol) = split(acc)                 -> next GEMM operand
  EPI_RESID = 2,    // out32 = resid + acc                   (residual stream)
  EPI_GELU = 3,     // out32 = acc (skipped when out32 is null) ; (oh, ol) = gelu_tanh(acc)
  EPI_GELU_BWD = 4, // (oh, ol) = acc * gelu_tanh'(aux)
  EPI_SGD = 5,      // w32 -= eta*acc ; (wh, wl) = split(w32)  (fused SGD step)
  EPI_CE_FWD = 6,   // per (row, N-tile): (max, sum exp) of logits; zt[row] = logit of target
  EPI_CE_BWD = 7,   // (oh, ol) = (softmax(acc) - onehot(tgt)) * scale, softmax from lse
  EPI_QKV_ROPE = 8, // [q | k | v] product: RoPE on q, k; q, k, v written as bf16 operands (gemm_qkv_rope)
  EPI_COUNT = 9
};

struct GemmArgs {
  int M = 0, N = 0, K = 0;
  int a_mn = 0, b_mn = 0;
  float* out32 = nullptr; long ldo32 = 0;
  bf16* oh = nullptr; bf16* ol = nullptr; long ldo = 0;
  const float* resid = nullptr; long ldr = 0;
  const float* aux = nullptr; long ldaux = 0;
  float* w32 = nullptr; bf16* wh = nullptr; bf16* wl = nullptr; long ldw = 0; float eta = 0.f;
  const int* tgt = nullptr; float2* part = nullptr; float* zt = nullptr; const float* lse = nullptr;
  float scale = 0.f;
  const float* scale_dev = nullptr;  // CE_BWD: device copy of the scale (used when non-null)
  // QKV_ROPE: outputs [M][rd] (hi, lo) for q, k, v; angle tables [M][dh/2]; rd = section width d
  bf16 *rq_h = nullptr, *rq_l = nullptr, *rk_h = nullptr, *rk_l = nullptr, *rv_h = nullptr, *rv_l = nullptr;
  const float *rcs = nullptr, *rsn = nullptr;
  int rd = 0;
  int* err = nullptr;
  // F32 / RESID: the product may be cut into K slices whose partial sums are added
  // atomically into out32 (gemm_run clears it, or copies resid into it, first);
  // the sum order then varies from run to run.
  bool allow_ksplit = false;
  int ksplit = 1;  // set by gemm_run
  // K slices: out32 already holds their start value (zero for F32, the residual for
  // RESID), set by an earlier kernel, so gemm_run enqueues no clear or copy
  bool out32_ready = false;
};

// One GEMM operand in HBM.  K-major: row-major [rows][ld] holding the K index
// in its columns.  MN-major: row-major [K][ld] holding the M (or N) index in
// its columns.  lo is the bf16 remainder of the fp32 value (split mode) or null.
struct Opnd {
  const bf16* hi = nullptr;
  const bf16* lo = nullptr;
  long ld = 0;
  int mn = 0;
};

// Returns 0 or a cudaError_t value.
int gemm_run(int epi, const Opnd& A, const Opnd& B, GemmArgs args, bool split, cudaStream_t st);
int num_sms();
int pick_bn(int M, int N);   // tile width gemm_run will use for an M x N product
// [q | k | v] = A.B with RoPE applied to q and k in the epilogue (head width dh);
// returns cudaErrorInvalidValue when no tile width fits whole heads (qkv_rope_bn == 0).
int gemm_qkv_rope(const Opnd& A, const Opnd& B, GemmArgs args, int dh, bool split, cudaStream_t st);
int qkv_rope_bn(int dh, int d, bool split);

}  // namespace ttt

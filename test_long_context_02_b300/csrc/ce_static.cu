// LM-head cross-entropy statistics with no device allocation at all.
//
// Same computation as ttt_k_gemm with the CE_FWD epilogue followed by the
// per-row combine, but the per-(row, vocab tile) partial (max, sum) pairs and
// the target logits live in a file-scope __device__ array instead of caller
// memory.  For callers that cannot call cudaMalloc: processes whose device
// memory is owned up front by another allocator, and latency-bound callers
// that cannot take cudaMalloc's implicit device synchronisation.
#include <mutex>

#include "kernels.h"
#include "rowops.h"
#include "ttt.h"
#include "ttt_kernels.h"

using namespace ttt;

namespace {

// 4 MiB: (max, sum) pairs for M rows x ceil(V / tile) vocab tiles, then M
// target logits packed two per entry.  Module loading is lazy, so a device
// allocates the array when the first call there looks up its address, and
// holds it until the process exits.
constexpr long kScratchEntries = TTT_CE_STATIC_SCRATCH_ENTRIES;
static __device__ __align__(256) float2 g_ce_scratch[kScratchEntries];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float2* g_addr[kMaxDevices] = {};

// Device address of g_ce_scratch on the current device (looked up once per device).
int scratch_address(float2** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TTT_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ce_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return TTT_ERR_CUDA;
    }
    g_addr[dev] = static_cast<float2*>(p);
  }
  *out = g_addr[dev];
  return TTT_OK;
}

}  // namespace

extern "C" int ttt_k_lmhead_ce_static(int M, int K, int V, const void* x, int64_t ldx, const void* w_lm,
                                      int64_t ldw, const int32_t* tgt, float* lse, float* loss, int32_t* err,
                                      void* stream) {
  if (M < 1 || K < 1 || V < 1 || !x || !w_lm || !tgt || !lse || !loss) return TTT_ERR_ARG;
  if (ldx < K || ldw < V || (ldx % 8) || (ldw % 8)) return TTT_ERR_ARG;
  // The bound is taken at the narrowest vocab tile (128), so it does not depend on the device.
  if (((long)V + 127) / 128 * (long)M + ((long)M + 1) / 2 > kScratchEntries) return TTT_ERR_SCRATCH;
  const long bn = pick_bn(M, V);
  const long ntiles = (V + bn - 1) / bn;
  float2* scratch = nullptr;
  const int r = scratch_address(&scratch);
  if (r != TTT_OK) return r;
  GemmArgs g;
  g.M = M; g.N = V; g.K = K;
  g.tgt = tgt;
  g.part = scratch;                                             // [ntiles][M]: written for every row and tile
  g.zt = reinterpret_cast<float*>(scratch + ntiles * (long)M);  // [M]: read only where tgt >= 0, written there
  g.err = err;
  Opnd A, B;
  A.hi = static_cast<const bf16*>(x); A.ld = (long)ldx; A.mn = 0;
  B.hi = static_cast<const bf16*>(w_lm); B.ld = (long)ldw; B.mn = 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (gemm_run(EPI_CE_FWD, A, B, g, false, st) != 0) return TTT_ERR_CUDA;
  if (rows_ce_combine(g.part, g.zt, tgt, M, (int)ntiles, lse, loss, st) != 0) return TTT_ERR_CUDA;
  return TTT_OK;
}

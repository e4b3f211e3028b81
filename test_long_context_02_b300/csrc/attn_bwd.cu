// Windowed attention backward: dQ over every key in the window (attn_dq2.cuh),
// dK / dV for the chunk's own keys only (attn_dkv2.cuh), in ONE launch.
//
// In the TTT-E2E inner loop the keys/values cached from earlier chunks were
// computed with earlier weights and are constants of the current step, so
// gradients flow into the queries and the chunk's own keys/values only (pages:
// "把 Transformer 做成“终身学习者”", §4.2; the backward runs through the
// last-quarter blocks, whose attention weights are frozen but pass activation
// gradients).
//
// The two parts read the same inputs and write disjoint outputs, and each alone
// has one CTA per (128-row tile, head): 128 CTAs at a 1024-token chunk with 16
// heads, short of the 148 SMs.  One grid holds both: the dQ CTAs first (about
// the same work each: every query tile sees the whole window), then the dK/dV
// CTAs ordered by key tile, the key tiles that meet the most query tiles first,
// so they fill the SMs the dQ CTAs leave free and the short ones come last.
#include "attn.h"
#include "attn_dkv2.cuh"
#include "attn_dq2.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {

namespace {

constexpr int kBwdThreads = 320;
static_assert(kBwdThreads == kQ2Threads && kBwdThreads == kK2Threads, "both parts use the same block");

// mode bit 0: dQ CTAs (nq * H, first); bit 1: dK/dV CTAs (nq * H, after them)
template <int DH, bool SPLIT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tQl,
                    const __grid_constant__ CUtensorMap tDO, const __grid_constant__ CUtensorMap tDOl,
                    const __grid_constant__ CUtensorMap tKr, const __grid_constant__ CUtensorMap tKrl,
                    const __grid_constant__ CUtensorMap tVr, const __grid_constant__ CUtensorMap tVrl,
                    const __grid_constant__ CUtensorMap tKo, const __grid_constant__ CUtensorMap tKol,
                    const __grid_constant__ CUtensorMap tVo, const __grid_constant__ CUtensorMap tVol,
                    const AttnBwdArgs a, const int mode) {
  const int nq = (a.g.n + 127) / 128, H = a.g.H;
  const int ndq = (mode & 1) ? nq * H : 0;
  const int bid = (int)blockIdx.x;
  if (bid < ndq) {
    dq2_body<DH, SPLIT>(&tQ, &tQl, &tDO, &tDOl, &tKr, &tKrl, &tVr, &tVrl, &tKo, &tKol, &tVo, &tVol, a, bid % nq,
                        bid / nq);
  } else {
    const int j = bid - ndq;
    dkv2_body<DH, SPLIT>(&tQ, &tQl, &tDO, &tDOl, &tKo, &tKol, &tVo, &tVol, a, j / H, j % H);
  }
}

template <int DH, bool SPLIT>
int launch_bwd(const AttnBwdMaps& m, const AttnBwdArgs& a, int mode, cudaStream_t st) {
  constexpr int SMEM = Q2Cfg<DH, SPLIT>::SMEM > K2Cfg<DH, SPLIT>::SMEM ? Q2Cfg<DH, SPLIT>::SMEM
                                                                       : K2Cfg<DH, SPLIT>::SMEM;
  auto kern = attn_bwd_kernel<DH, SPLIT>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return (int)e;
    attr = true;
  }
  const int per = ((a.g.n + 127) / 128) * a.g.H;
  const int blocks = ((mode & 1) ? per : 0) + ((mode & 2) ? per : 0);
  if (blocks == 0) return 0;
  const AttnMaps& f = m.f;
  return (int)launch_k(kern, dim3(blocks), dim3(kBwdThreads), SMEM, st, f.q, f.ql, m.dO, m.dOl, f.kr, f.krl, f.vr,
                       f.vrl, f.ko, f.kol, f.vo, f.vol, a, mode);
}

}  // namespace

int attn_bwd_run(const AttnBwdMaps& m, const AttnBwdArgs& a, bool split, cudaStream_t st, int which) {
  if (a.g.n <= 0) return 0;
  const int mode = which == 1 ? 1 : (which == 2 ? 2 : 3);
  if (split) {
    switch (a.g.dh) {
      case 32: return launch_bwd<32, true>(m, a, mode, st);
      case 64: return launch_bwd<64, true>(m, a, mode, st);
    }
    return (int)cudaErrorInvalidValue;
  }
  switch (a.g.dh) {
    case 32: return launch_bwd<32, false>(m, a, mode, st);
    case 64: return launch_bwd<64, false>(m, a, mode, st);
    case 96: return launch_bwd<96, false>(m, a, mode, st);
    case 128: return launch_bwd<128, false>(m, a, mode, st);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace ttt

// Windowed attention backward: dQ over every key in the window (attn_dq2.cu),
// dK / dV for the chunk's own keys only (attn_dkv2.cu).
//
// In the TTT-E2E inner loop the keys/values cached from earlier chunks were
// computed with earlier weights and are constants of the current step, so
// gradients flow into the queries and the chunk's own keys/values only (pages:
// "把 Transformer 做成“终身学习者”", §4.2; the backward runs through the
// last-quarter blocks, whose attention weights are frozen but pass activation
// gradients).
#include "attn.h"
#include "kernels.h"

namespace ttt {

int attn_bwd_run(const AttnBwdMaps& m, const AttnBwdArgs& a, bool split, cudaStream_t st, int which) {
  if (a.g.n <= 0) return 0;
  if (which != 2) {
    const int r = attn_dq2_run(m, a, split, st);
    if (r != 0) return r;
  }
  return which != 1 ? attn_dkv2_run(m, a, split, st) : 0;
}

}  // namespace ttt

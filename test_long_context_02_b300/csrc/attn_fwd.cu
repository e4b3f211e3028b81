// Windowed attention forward: choice of kernel.
//
// Both kernels compute, for the chunk's queries at absolute positions
// pos0 .. pos0+n-1, softmax attention over the keys at positions j with
// p - k < j <= p (pages: "把 Transformer 做成“终身学习者”", §4.2, the key/value
// cache holds only the window; §8 FAQ Q4, any k >= b), keys before the chunk
// from the k-slot cache and the chunk's own keys from its own K/V buffer, and
// write O (bf16 hi [+ lo]) and the per-row log2-sum-exp for the backward.
//   attn_fwd5.cu: bf16 operands; one 128-query tile per CTA, two softmax
//                 warpgroups on alternate key tiles, each with its own O
//                 accumulator in tensor memory;
//   attn_fwd3.cu: split (fp32) mode; one 128-query tile per CTA, two threads
//                 per query row, P and O in tensor memory.
#include "attn.h"
#include "kernels.h"

namespace ttt {

int attn_fwd_run(const AttnMaps& m, const AttnArgs& a, bool split, cudaStream_t st) {
  if (a.n <= 0) return 0;
  if (!split) return attn_fwd5_run(m, a, st);
  return attn_fwd3_run(m, a, split, st);
}

}  // namespace ttt

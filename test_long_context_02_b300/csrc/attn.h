// Sliding-window attention kernels (attn_fwd.cu, attn_bwd.cu).
#pragma once
#include <cuda.h>
#include "kernels.h"

namespace ttt {

// Geometry of one chunk's attention for one sequence and layer.  Activations
// are token-major [rows][d] (head h in columns h*dh .. h*dh+dh-1).
struct AttnArgs {
  int n = 0;            // queries = the chunk's own tokens
  int H = 0, dh = 0;
  int window = 0;       // k (multiple of 128); also the number of cache slots
  long pos0 = 0;        // absolute position of the chunk's first token
  float scale_log2 = 0; // log2(e) / sqrt(dh)
  bf16* o_hi = nullptr; bf16* o_lo = nullptr; long ldo = 0;   // forward output [n][d]
  float* lse = nullptr; // [H][n] log2-sum-exp of the scaled scores (optional)
  int* err = nullptr;
  int qt0 = 0;          // forward only: first query tile computed (earlier rows are left as they are)
};

// TMA maps (box {64, 128}) of: queries [n][d]; cache keys/values [k][d];
// the chunk's own keys/values [n][d].  *_l: the bf16 remainders (split mode).
struct AttnMaps {
  CUtensorMap q, ql, kr, krl, vr, vrl, ko, kol, vo, vol;
};

int attn_fwd_run(const AttnMaps& m, const AttnArgs& a, bool split, cudaStream_t st);
// One query tile per CTA, P and O kept in TMEM (attn_fwd3.cu).
int attn_fwd3_run(const AttnMaps& m, const AttnArgs& a, bool split, cudaStream_t st);
// bf16 operands only: one query tile per CTA, two softmax warpgroups on alternate key
// tiles, each with its own O accumulator in TMEM (attn_fwd5.cu).
int attn_fwd5_run(const AttnMaps& m, const AttnArgs& a, cudaStream_t st);

// Backward: geometry from g; lse ([H][n], log2 domain) from the forward;
// D[h][t] = rowsum(dO * O); outputs dq (all keys) and dk, dv (own keys only),
// fp32 token-major [n][ldg].
struct AttnBwdArgs {
  AttnArgs g;
  const float* lse = nullptr;
  const float* D = nullptr;
  float* dq = nullptr; float* dk = nullptr; float* dv = nullptr; long ldg = 0;
  float scale = 0.f;  // 1/sqrt(dh)
  // Fused output (when qkv_h is set; dq / dk / dv are then not written): the gradient
  // [dq | dk | dv] with RoPE's rotation transposed on dq and dk, as the bf16 operand
  // (+ remainder in split mode) of the QKV dX product, row-major [n][ld_qkv]; section
  // offsets k_off, v_off (columns); angle tables cs / sn [n][dh/2] of the chunk's rows.
  bf16* qkv_h = nullptr; bf16* qkv_l = nullptr; long ld_qkv = 0, k_off = 0, v_off = 0;
  const float* cs = nullptr; const float* sn = nullptr;
};
struct AttnBwdMaps {
  AttnMaps f;          // q, cache k/v, own k/v as in the forward
  CUtensorMap dO, dOl; // output gradient [n][d]
};

// dQ (dS kept in TMEM, attn_dq2.cuh) and dK/dV (P^T, dS^T kept in TMEM,
// attn_dkv2.cuh) in one launch (attn_bwd.cu); which: 0 = both, 1 = dQ only,
// 2 = dK/dV only.
int attn_bwd_run(const AttnBwdMaps& m, const AttnBwdArgs& a, bool split, cudaStream_t st, int which = 0);


}  // namespace ttt

// Output stage shared by the two CTA bodies of the attention backward
// (attn_dq2.cuh, attn_dkv2.cuh): the fused write of the QKV-product operand.
#pragma once
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {
namespace {

// The 256 softmax / epilogue threads (warps 2-9) meet at named barrier 1.
TTT_DEV void epilogue_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// HO (a multiple of 8) values as bf16 (+ remainders), 16-byte stores.
template <int HO, bool SPLIT>
TTT_DEV void store_row_opnd(bf16* hi, bf16* lo, const float* v) {
#pragma unroll
  for (int u = 0; u < HO / 8; ++u) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 t = __floats2bfloat162_rn(v[8 * u + 2 * e], v[8 * u + 2 * e + 1]);
      h[e] = *reinterpret_cast<uint32_t*>(&t);
      if (SPLIT) {
        const float2 f = __bfloat1622float2(t);
        l[e] = pack_bf16(v[8 * u + 2 * e] - f.x, v[8 * u + 2 * e + 1] - f.y);
      }
    }
    *reinterpret_cast<uint4*>(hi + 8 * u) = make_uint4(h[0], h[1], h[2], h[3]);
    if (SPLIT) *reinterpret_cast<uint4*>(lo + 8 * u) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// Shared-memory floats rope_bwd_store needs (row stride HO + 1 keeps the per-row
// accesses of a warp on distinct banks): the two halves of every row, then the
// tile's cos and sin rows.
template <int HO>
constexpr int rope_bwd_smem_floats() { return 4 * 128 * (HO + 1); }

// Row r of a 128-row tile of dQ or dK is held by two threads: hf = 0 owns columns
// [0, HO), hf = 1 owns [HO, 2 HO), which are exactly the rotate-half pairs (i, i + HO).
// The transpose of the rotation, d1' = d1 c + d2 s, d2' = d2 c - d1 s (c, s of the
// row's position), needs the partner's half: each thread puts its half into shared
// memory, the 256 epilogue threads (tid = 0..255) copy the tile's angle rows
// (cs_tile / sn_tile [rows][HO], coalesced) beside them, and after the barrier each
// thread reads the other half and its row's angles.  Every epilogue thread calls this
// (valid = false: take part only).
template <int HO, bool SPLIT>
TTT_DEV void rope_bwd_store(float* sm, int tid, int r, int hf, const float (&v)[HO], bool valid,
                            const float* cs_tile, const float* sn_tile, int rows, bf16* hi, bf16* lo) {
  constexpr int P = HO + 1;
  float* half = sm;                   // [2][128][P]
  float* cs_s = sm + 2 * 128 * P;     // [128][P]
  float* sn_s = cs_s + 128 * P;       // [128][P]
  float* mine = half + (hf * 128 + r) * P;
#pragma unroll
  for (int i = 0; i < HO; ++i) mine[i] = v[i];
  for (int idx = tid; idx < 128 * HO; idx += 256) {
    const int rr = idx / HO, i = idx - rr * HO;
    const bool in = rr < rows;
    cs_s[rr * P + i] = in ? cs_tile[idx] : 0.f;
    sn_s[rr * P + i] = in ? sn_tile[idx] : 0.f;
  }
  epilogue_sync();
  if (!valid) return;
  const float* other = half + ((hf ^ 1) * 128 + r) * P;
  const float* c = cs_s + r * P;
  const float* s = sn_s + r * P;
  const float sg = hf == 0 ? 1.f : -1.f;
  float out[HO];
#pragma unroll
  for (int i = 0; i < HO; ++i) out[i] = v[i] * c[i] + sg * other[i] * s[i];
  store_row_opnd<HO, SPLIT>(hi, lo, out);
}

}  // namespace
}  // namespace ttt

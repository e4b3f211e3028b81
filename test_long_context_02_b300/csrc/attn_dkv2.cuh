// dK / dV of the windowed attention for the chunk's own keys, with P^T and dS^T
// kept in tensor memory.
//
// In the TTT-E2E inner loop the keys/values cached from earlier chunks were
// computed with earlier weights and are constants of the current step, so only
// the chunk's own keys receive gradients (pages: "把 Transformer 做成“终身学习者”",
// §4.2; the backward runs through the last-quarter blocks, whose attention
// weights are frozen but pass activation gradients).  With P = softmax(S),
// S = Q K^T / sqrt(dh), D = rowsum(dO * O):  dV = P^T dO,  dK = dS^T Q / sqrt(dh),
// dS = P * (dP - D).  A chunk's own key at row i is seen by the chunk's queries
// at rows >= i only (n <= k), so the key tile kt meets query tiles kt .. nq-1.
//
// CTA = (128 own keys, head).  Warp 0 loads K, V once and (Q_i, dO_i) through a
// 2-stage TMA ring, its 32 lanes staging the query tile's log2-sum-exp and D in
// shared memory.  Warp 1 issues S^T = K Q_i^T and dP^T = V dO_i^T into TMEM,
// then dV += P^T dO_i and dK += dS^T Q_i with P^T and dS^T read from TMEM.
// Warps 2-9 (two threads per key row, 64 query columns each) form P^T from S^T
// and the stored statistics, write it as bf16 over their own S^T columns, then
// dS^T over their own dP^T columns.
#pragma once
#include "attn.h"
#include "attn_bwd_out.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {

namespace {

constexpr int kK2Threads = 320;  // warp 0 TMA + statistics, warp 1 MMA, warps 2-9 two threads per key row

template <int DH, bool SPLIT>
struct K2Cfg {
  static constexpr int DP = DH <= 64 ? 64 : 128;
  static constexpr int NATOM = DP / 64;
  static constexpr int TILE = 128 * DP * 2;
  static constexpr int NOP = SPLIT ? 2 : 1;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = NOP * TILE;
  static constexpr int Q_OFF = 2 * NOP * TILE;     // 2 stages x (Q, dO)
  static constexpr int STAGE = 2 * NOP * TILE;
  static constexpr int ST_OFF = Q_OFF + 2 * STAGE;  // statistics: [2 stages][lse, D][128] fp32
  static constexpr int BAR_OFF = ST_OFF + 2 * 2 * 128 * 4;
  static constexpr int SMEM = BAR_OFF + 256;
  static_assert(SMEM <= 232448, "dK/dV kernel exceeds shared memory");
};

TTT_DEV bool drain_k2(uint64_t* bar, uint32_t parity, int* err) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      if (err) atomicCAS(err, 0, (int)DERR_TIMEOUT_DRAIN);
      return false;
    }
  }
  return true;
}

template <int NATOM>
TTT_DEV void load_tile_k2(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int a = 0; a < NATOM; ++a) tma_load_2d(dst + a * 16384, map, bar, col0 + 64 * a, row0);
}
TTT_DEV uint64_t kdesc_k2(uint32_t base, int kk) { return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024); }
TTT_DEV uint64_t mndesc_k2(uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 16384, 1024); }

template <int N>
TTT_DEV void ld_cols_k2(uint32_t a, float* v) {
  if constexpr (N >= 32) {
    float t[32];
    tmem_ld32(a, t);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = t[i];
    ld_cols_k2<N - 32>(a + 32, v + 32);
  } else if constexpr (N == 16) {
    float t[16];
    tmem_ld16(a, t);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = t[i];
  }
}

// 64 values -> 32 bf16 pairs (hi) and, in split mode, 32 pairs of remainders.
template <bool SPLIT>
TTT_DEV void pack64(const float* x, uint32_t (&hi)[32], uint32_t (&lo)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    __nv_bfloat162 t = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    hi[e] = *reinterpret_cast<uint32_t*>(&t);
    if (SPLIT) {
      const float2 f = __bfloat1622float2(t);
      lo[e] = pack_bf16(x[2 * e] - f.x, x[2 * e + 1] - f.y);
    }
  }
}

// One CTA of dK / dV: own-key tile kt of head h.
template <int DH, bool SPLIT>
TTT_DEV void dkv2_body(const CUtensorMap* tQ, const CUtensorMap* tQl, const CUtensorMap* tDO, const CUtensorMap* tDOl,
                       const CUtensorMap* tKo, const CUtensorMap* tKol, const CUtensorMap* tVo, const CUtensorMap* tVol,
                       const AttnBwdArgs& a, const int kt, const int h) {
  using C = K2Cfg<DH, SPLIT>;
  constexpr int HO = DH / 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0 && a.g.err) atomicCAS(a.g.err, 0, (int)DERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* kv_full = bars;       // 1
  uint64_t* qd_full = bars + 1;   // 2
  uint64_t* qd_empty = bars + 3;  // 2
  uint64_t* st_full = bars + 5;   // 2: statistics staged (32 producer lanes)
  uint64_t* s_full = bars + 7;    // 1
  uint64_t* p_full = bars + 8;    // 1
  uint64_t* ds_full = bars + 9;   // 1
  uint64_t* acc_full = bars + 10; // 1
  uint64_t* drain = bars + 11;    // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* stats = reinterpret_cast<float*>(smem + C::ST_OFF);

  const AttnArgs& g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = (g.n + 127) / 128;
  const int I = nq - kt;  // causal query tiles kt .. nq-1
  const int col0 = h * DH;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
      mbar_init(&st_full[i], 32);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 256);
    mbar_init(ds_full, 256);
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the predecessor kernel's outputs are complete and visible from here on
  pdl_launch_dependents();
  const uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + C::DP;

  if (warp == 0) {  // ---------------------------------------------- TMA producer + statistics
    uint32_t iss = 0, ipar = 0;
    if (lane == 0) {
      mbar_expect_tx(kv_full, 2 * C::NOP * C::TILE);
      load_tile_k2<C::NATOM>(smem + C::K_OFF, tKo, kv_full, col0, 128 * kt);
      load_tile_k2<C::NATOM>(smem + C::V_OFF, tVo, kv_full, col0, 128 * kt);
      if (SPLIT) {
        load_tile_k2<C::NATOM>(smem + C::K_OFF + C::TILE, tKol, kv_full, col0, 128 * kt);
        load_tile_k2<C::NATOM>(smem + C::V_OFF + C::TILE, tVol, kv_full, col0, 128 * kt);
      }
    }
    for (int i = 0; i < I; ++i) {
      const int s = i & 1;
      const uint32_t par = (uint32_t)((i >> 1) & 1);
      const bool got = mbar_wait(&qd_empty[s], par ^ 1u, abort_flag, g.err, DERR_TIMEOUT_PRODUCER);
      if (!__all_sync(0xffffffffu, got)) break;
      const int q0 = 128 * (kt + i);
      if (lane == 0) {
        uint8_t* st = smem + C::Q_OFF + s * C::STAGE;
        mbar_expect_tx(&qd_full[s], 2 * C::NOP * C::TILE);
        load_tile_k2<C::NATOM>(st, tQ, &qd_full[s], col0, q0);
        load_tile_k2<C::NATOM>(st + C::NOP * C::TILE, tDO, &qd_full[s], col0, q0);
        if (SPLIT) {
          load_tile_k2<C::NATOM>(st + C::TILE, tQl, &qd_full[s], col0, q0);
          load_tile_k2<C::NATOM>(st + C::NOP * C::TILE + C::TILE, tDOl, &qd_full[s], col0, q0);
        }
        iss |= 1u << s;
        ipar = (ipar & ~(1u << s)) | (par << s);
      }
      float* sl = stats + s * 256;  // [lse | D] of the query tile's 128 rows
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = lane + 32 * e, q = q0 + c;
        sl[c] = q < g.n ? a.lse[(long)h * g.n + q] : 0.f;
        sl[128 + c] = q < g.n ? a.D[(long)h * g.n + q] : 0.f;
      }
      mbar_arrive(&st_full[s]);
    }
    if (lane == 0) {  // no TMA write may still be in flight when the CTA exits
      drain_k2(kv_full, 0, g.err);
      for (int s = 0; s < 2; ++s)
        if (iss & (1u << s)) drain_k2(&qd_full[s], (ipar >> s) & 1u, g.err);
    }
  } else if (warp == 1) {  // MMA issuer: the whole warp, one elected lane issues
    auto wait_all = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, g.err, DERR_TIMEOUT_MMA));
    };
    constexpr uint32_t idSS = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idAcc = idesc_bf16(128, DH, 0, 1);
    const uint32_t kb = smem_u32(smem + C::K_OFF), vb = smem_u32(smem + C::V_OFF);
    auto xy = [&](uint32_t d, uint32_t xb, uint32_t yb) {  // d = X Y^T over the head dim
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        mma_bf16_w(d, kdesc_k2(xb, kk), kdesc_k2(yb, kk), idSS, kk ? 1u : 0u);
        if (SPLIT) {
          mma_bf16_w(d, kdesc_k2(xb, kk), kdesc_k2(yb + C::TILE, kk), idSS, 1u);
          mma_bf16_w(d, kdesc_k2(xb + C::TILE, kk), kdesc_k2(yb, kk), idSS, 1u);
        }
      }
    };
    // d (+)= A Y with A (128 keys x 128 queries, bf16) in TMEM: query columns 0-63 at
    // [a0, a0+32) (+ remainders [a0+32, a0+64)), 64-127 at [a0+64, a0+96) (+ [a0+96, a0+128))
    auto acc = [&](uint32_t d, uint32_t a0, uint32_t yb, bool first) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t pa = a0 + (uint32_t)((kk < 4 ? 0 : 64) + 8 * (kk & 3));
        mma_bf16_ts_w(d, pa, mndesc_k2(yb, kk), idAcc, (!first || kk) ? 1u : 0u);
        if (SPLIT) {
          mma_bf16_ts_w(d, pa, mndesc_k2(yb + C::TILE, kk), idAcc, 1u);
          mma_bf16_ts_w(d, pa + 32u, mndesc_k2(yb, kk), idAcc, 1u);
        }
      }
    };
    bool ok = I > 0 && wait_all(kv_full, 0);
    for (int i = 0; i < I && ok; ++i) {
      const int s = i & 1;
      if (!wait_all(&qd_full[s], (uint32_t)((i >> 1) & 1))) break;
      tc_fence_after();
      const uint32_t qb = smem_u32(smem + C::Q_OFF + s * C::STAGE);
      const uint32_t dob = qb + C::NOP * C::TILE;
      xy(tmem + T_S, kb, qb);    // S^T = K Q^T   (P^T, dS^T of tile i-1 were consumed above)
      xy(tmem + T_DP, vb, dob);  // dP^T = V dO^T
      mma_commit_w(s_full);
      if (!wait_all(p_full, (uint32_t)(i & 1))) break;
      tc_fence_after();
      acc(tmem + T_DV, tmem + T_S, dob, i == 0);  // dV += P^T dO
      if (!wait_all(ds_full, (uint32_t)(i & 1))) break;
      tc_fence_after();
      acc(tmem + T_DK, tmem + T_DP, qb, i == 0);  // dK += dS^T Q
      mma_commit_w(&qd_empty[s]);
    }
    mma_commit_w(acc_full);
    mma_commit_w(drain);
    drain_k2(drain, 0, g.err);
  } else {  // ------------------------------------------- softmax: two threads per key row (64 queries)
    const int hf = (warp - 2) >> 2, qd = warp & 3, r = qd * 32 + lane;
    const int krow = 128 * kt + r;
    const bool kvalid = krow < g.n;
    const float sl2 = g.scale_log2;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const int b0 = hf * 64;
    bool ok = true;
    for (int i = 0; i < I; ++i) {
      const int s = i & 1;
      const int q0 = 128 * (kt + i);
      // query column c is valid iff q0 + c < n and it is not before the key (causal)
      const int c_lo = kvalid ? krow - q0 : 128;
      const int c_hi = min(127, g.n - 1 - q0);
      const bool full = __all_sync(0xffffffffu, c_lo <= b0 && c_hi >= b0 + 63);
      bool got = mbar_wait(&st_full[s], (uint32_t)((i >> 1) & 1), abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      got = got && mbar_wait(s_full, (uint32_t)(i & 1), abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* sl = stats + s * 256 + b0;  // this thread's 64 query columns
      const float* sd = sl + 128;
      float pv[64];
      tmem_ld64(trow + T_S + b0, pv);  // S^T row
      const uint64_t sc2 = f32x2(sl2, sl2);
#pragma unroll
      for (int e = 0; e < 64; e += 2) {  // pairs of query columns in packed f32x2 arithmetic
        const float2 a = f32x2_split(ffma2(f32x2(pv[e], pv[e + 1]), sc2, f32x2(-sl[e], -sl[e + 1])));
        const float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
        pv[e] = (full || (b0 + e >= c_lo && b0 + e <= c_hi)) ? p0 : 0.f;
        pv[e + 1] = (full || (b0 + e + 1 >= c_lo && b0 + e + 1 <= c_hi)) ? p1 : 0.f;
      }
      {
        uint32_t hi[32], lo[32];
        pack64<SPLIT>(pv, hi, lo);
        tmem_st32(trow + T_S + b0, hi);  // over this thread's own (already read) S^T columns
        if (SPLIT) tmem_st32(trow + T_S + b0 + 32, lo);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full);
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // dS^T = P^T (dP^T - D), in place over pv, 32 columns at a time
        float dp[32];
        tmem_ld32(trow + T_DP + (uint32_t)(b0 + 32 * c), dp);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int i = 32 * c + e;
          const float2 x = f32x2_split(fmul2(f32x2(pv[i], pv[i + 1]),
                                             fadd2(f32x2(dp[e], dp[e + 1]), f32x2(-sd[i], -sd[i + 1]))));
          pv[i] = x.x;
          pv[i + 1] = x.y;
        }
      }
      {
        uint32_t hi[32], lo[32];
        pack64<SPLIT>(pv, hi, lo);
        tmem_st32(trow + T_DP + b0, hi);
        if (SPLIT) tmem_st32(trow + T_DP + b0 + 32, lo);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    bool got = ok && mbar_wait(acc_full, 0, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
    const bool have = __all_sync(0xffffffffu, got);
    float v[HO], w[HO];
#pragma unroll
    for (int e = 0; e < HO; ++e) v[e] = w[e] = 0.f;
    if (have) {
      tc_fence_after();
      ld_cols_k2<HO>(trow + T_DV + hf * HO, v);
      ld_cols_k2<HO>(trow + T_DK + hf * HO, w);
#pragma unroll
      for (int e = 0; e < HO; ++e) w[e] *= a.scale;
    }
    if (a.qkv_h) {  // dV as is, dK rotated back; the K, V and Q / dO stages are free now
      const long o = (long)krow * a.ld_qkv + col0 + hf * HO;
      if (have && kvalid) store_row_opnd<HO, SPLIT>(a.qkv_h + o + a.v_off, SPLIT ? a.qkv_l + o + a.v_off : nullptr, v);
      static_assert(rope_bwd_smem_floats<HO>() * 4 <= C::ST_OFF - C::K_OFF, "rope exchange exceeds the stages");
      const long t0 = 128L * kt;
      rope_bwd_store<HO, SPLIT>(reinterpret_cast<float*>(smem + C::K_OFF), (warp - 2) * 32 + lane, r, hf, w,
                                have && kvalid, a.cs + t0 * HO, a.sn + t0 * HO, (int)min(128L, g.n - t0),
                                a.qkv_h + o + a.k_off, SPLIT ? a.qkv_l + o + a.k_off : nullptr);
    } else if (have && kvalid) {
      float4* dv = reinterpret_cast<float4*>(a.dv + (long)krow * a.ldg + col0 + hf * HO);
      float4* dk = reinterpret_cast<float4*>(a.dk + (long)krow * a.ldg + col0 + hf * HO);
#pragma unroll
      for (int e = 0; e < HO / 4; ++e) {
        dv[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        dk[e] = make_float4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

}  // namespace ttt

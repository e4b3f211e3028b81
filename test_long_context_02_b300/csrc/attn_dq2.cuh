// dQ of the windowed attention over every key in the window, with dS kept in
// tensor memory.
//
// Same geometry as the forward (pages: "把 Transformer 做成“终身学习者”", §4.2):
// a query at p sees keys j with p - k < j <= p, from the k-slot cache before the
// chunk and from the chunk's own K/V after it.  With P = softmax(S), S = Q K^T
// / sqrt(dh), D = rowsum(dO * O): dP = dO V^T, dS = P * (dP - D), dQ = dS K /
// sqrt(dh); P is recomputed from S and the forward's log2-sum-exp.
//
// CTA = (128 queries, head).  Warp 0 loads Q, dO once and K/V tiles through
// 2-stage TMA rings.  Warp 1 issues dP_j = dO V_j^T, S_{j+1} = Q K_{j+1}^T into
// the other of two TMEM score buffers, then dQ += dS_j K_j with dS_j read from
// TMEM.  Warps 2-9 (two threads per query row, 64 key columns each) form dS_j
// from S_j, dP_j and the row statistics and write it as bf16 over their own
// columns of S_j.
#pragma once
#include "attn.h"
#include "attn_bwd_out.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {

namespace {

constexpr int kQ2Threads = 320;

template <int DH, bool SPLIT>
struct Q2Cfg {
  static constexpr int DP = DH <= 64 ? 64 : 128;
  static constexpr int NATOM = DP / 64;
  static constexpr int TILE = 128 * DP * 2;
  static constexpr int NOP = SPLIT ? 2 : 1;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = NOP * TILE;
  static constexpr int KST = 3;                         // key stages
  static constexpr int K_OFF = 2 * NOP * TILE;
  static constexpr int V_OFF = K_OFF + KST * NOP * TILE;  // 2 stages
  static constexpr int BAR_OFF = V_OFF + 2 * NOP * TILE;
  static constexpr int SMEM = BAR_OFF + 256;
  static_assert(SMEM <= 232448, "dQ kernel exceeds shared memory");
};

TTT_DEV bool drain_q2(uint64_t* bar, uint32_t parity, int* err) {
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
TTT_DEV void load_tile_q2(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int a = 0; a < NATOM; ++a) tma_load_2d(dst + a * 16384, map, bar, col0 + 64 * a, row0);
}
TTT_DEV uint64_t kdesc_q2(uint32_t base, int kk) { return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024); }
TTT_DEV uint64_t mndesc_q2(uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 16384, 1024); }

template <int N>
TTT_DEV void ld_cols_q2(uint32_t a, float* v) {
  if constexpr (N >= 32) {
    float t[32];
    tmem_ld32(a, t);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = t[i];
    ld_cols_q2<N - 32>(a + 32, v + 32);
  } else if constexpr (N == 16) {
    float t[16];
    tmem_ld16(a, t);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = t[i];
  }
}

struct RangeQ2 {
  int n_ring, m_lo, J;
};
TTT_DEV RangeQ2 range_q2(const AttnArgs& a, int qt) {
  RangeQ2 r;
  const long qlo = a.pos0 + 128L * qt;
  const int qend = min(a.n, 128 * qt + 128);
  if (a.pos0 > 0) {
    const long lo = max(0L, qlo - a.window + 1);
    r.m_lo = (int)(lo / 128);
    r.n_ring = (int)((a.pos0 - 1) / 128) - r.m_lo + 1;
  } else {
    r.m_lo = 0;
    r.n_ring = 0;
  }
  r.J = r.n_ring + (qend - 1) / 128 + 1;
  return r;
}

// One CTA of dQ: query tile qt of head h.  The tensor maps are the kernel's
// __grid_constant__ parameters.
template <int DH, bool SPLIT>
TTT_DEV void dq2_body(const CUtensorMap* tQ, const CUtensorMap* tQl, const CUtensorMap* tDO, const CUtensorMap* tDOl,
                      const CUtensorMap* tKr, const CUtensorMap* tKrl, const CUtensorMap* tVr, const CUtensorMap* tVrl,
                      const CUtensorMap* tKo, const CUtensorMap* tKol, const CUtensorMap* tVo, const CUtensorMap* tVol,
                      const AttnBwdArgs& a, const int qt, const int h) {
  using C = Q2Cfg<DH, SPLIT>;
  constexpr int HO = DH / 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0 && a.g.err) atomicCAS(a.g.err, 0, (int)DERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;        // 1 (Q and dO)
  uint64_t* k_full = bars + 1;    // 3
  uint64_t* k_empty = bars + 4;   // 3
  uint64_t* v_full = bars + 7;    // 2
  uint64_t* v_empty = bars + 9;   // 2
  uint64_t* s_full = bars + 11;   // 2 (per score buffer: S_j and dP_j landed)
  uint64_t* ds_full = bars + 13;  // 2 (per score buffer)
  uint64_t* dq_full = bars + 15;  // 1
  uint64_t* drain = bars + 16;    // 1
  uint64_t* dp_free = bars + 17;  // 1 (the softmax of the last tile has read dP out of TMEM)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const AttnArgs& g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RangeQ2 tr = range_q2(g, qt);
  const int J = tr.J;
  const int col0 = h * DH;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::KST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&ds_full[i], 256);
    }
    mbar_init(dq_full, 1);
    mbar_init(drain, 1);
    mbar_init(dp_free, 256);
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
  const uint32_t T_DP = 256, T_DQ = 384;  // score buffers at 0 and 128

  auto tile_row0 = [&](int j, bool& own) -> int {
    if (j < tr.n_ring) {
      own = false;
      return (int)(((long)(tr.m_lo + j) * 128) % g.window);
    }
    own = true;
    return 128 * (j - tr.n_ring);
  };

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------------- TMA producer
      uint32_t kiss = 0, kpar = 0, viss = 0, vpar = 0;
      mbar_expect_tx(q_full, 2 * C::NOP * C::TILE);
      load_tile_q2<C::NATOM>(smem + C::Q_OFF, tQ, q_full, col0, 128 * qt);
      load_tile_q2<C::NATOM>(smem + C::DO_OFF, tDO, q_full, col0, 128 * qt);
      if (SPLIT) {
        load_tile_q2<C::NATOM>(smem + C::Q_OFF + C::TILE, tQl, q_full, col0, 128 * qt);
        load_tile_q2<C::NATOM>(smem + C::DO_OFF + C::TILE, tDOl, q_full, col0, 128 * qt);
      }
      for (int j = 0; j < J; ++j) {
        const int s = j & 1;
        const uint32_t par = (uint32_t)((j >> 1) & 1);
        const int ks = j % C::KST;
        const uint32_t kp = (uint32_t)((j / C::KST) & 1);
        bool own;
        const int row0 = tile_row0(j, own);
        if (!mbar_wait(&k_empty[ks], kp ^ 1u, abort_flag, g.err, DERR_TIMEOUT_PRODUCER)) break;
        uint8_t* kd = smem + C::K_OFF + ks * C::NOP * C::TILE;
        mbar_expect_tx(&k_full[ks], C::NOP * C::TILE);
        load_tile_q2<C::NATOM>(kd, own ? tKo : tKr, &k_full[ks], col0, row0);
        if (SPLIT) load_tile_q2<C::NATOM>(kd + C::TILE, own ? tKol : tKrl, &k_full[ks], col0, row0);
        kiss |= 1u << ks;
        kpar = (kpar & ~(1u << ks)) | (kp << ks);
        if (!mbar_wait(&v_empty[s], par ^ 1u, abort_flag, g.err, DERR_TIMEOUT_PRODUCER)) break;
        uint8_t* vd = smem + C::V_OFF + s * C::NOP * C::TILE;
        mbar_expect_tx(&v_full[s], C::NOP * C::TILE);
        load_tile_q2<C::NATOM>(vd, own ? tVo : tVr, &v_full[s], col0, row0);
        if (SPLIT) load_tile_q2<C::NATOM>(vd + C::TILE, own ? tVol : tVrl, &v_full[s], col0, row0);
        viss |= 1u << s;
        vpar = (vpar & ~(1u << s)) | (par << s);
      }
      drain_q2(q_full, 0, g.err);
      for (int s = 0; s < C::KST; ++s)
        if (kiss & (1u << s)) drain_q2(&k_full[s], (kpar >> s) & 1u, g.err);
      for (int s = 0; s < 2; ++s)
        if (viss & (1u << s)) drain_q2(&v_full[s], (vpar >> s) & 1u, g.err);
    }
  } else if (warp == 1) {  // MMA issuer: the whole warp, one elected lane issues
    auto wait_all = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, g.err, DERR_TIMEOUT_MMA));
    };
    constexpr uint32_t idSS = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idDQ = idesc_bf16(128, DH, 0, 1);
    const uint32_t qb = smem_u32(smem + C::Q_OFF), dob = smem_u32(smem + C::DO_OFF);
    auto xk = [&](uint32_t d, uint32_t xb, uint32_t kb) {  // d = X K^T over the head dim
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        mma_bf16_w(d, kdesc_q2(xb, kk), kdesc_q2(kb, kk), idSS, kk ? 1u : 0u);
        if (SPLIT) {
          mma_bf16_w(d, kdesc_q2(xb, kk), kdesc_q2(kb + C::TILE, kk), idSS, 1u);
          mma_bf16_w(d, kdesc_q2(xb + C::TILE, kk), kdesc_q2(kb, kk), idSS, 1u);
        }
      }
    };
    auto kstage = [&](int j) { return smem_u32(smem + C::K_OFF + (j % C::KST) * C::NOP * C::TILE); };
    // dQ += dS_j K_j; dS_j: keys 0-63 in columns [0,32) (+ remainders [32,64)), keys 64-127 in
    // [64,96) (+ [96,128)) of score buffer j & 1
    auto dq_mma = [&](int j) {
      const uint32_t kb = kstage(j);
      const uint32_t pb = tmem + (uint32_t)((j & 1) * 128);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t pa = pb + (uint32_t)((kk < 4 ? 0 : 64) + 8 * (kk & 3));
        mma_bf16_ts_w(tmem + T_DQ, pa, mndesc_q2(kb, kk), idDQ, (j | kk) ? 1u : 0u);
        if (SPLIT) {
          mma_bf16_ts_w(tmem + T_DQ, pa, mndesc_q2(kb + C::TILE, kk), idDQ, 1u);
          mma_bf16_ts_w(tmem + T_DQ, pa + 32u, mndesc_q2(kb, kk), idDQ, 1u);
        }
      }
      mma_commit_w(&k_empty[j % C::KST]);
    };
    // Tensor-pipe order per key tile j: dP_j, dQ_{j-1}, S_{j+1}.  dP_j goes into the one dP
    // buffer as soon as the softmax of tile j-1 has loaded dP_{j-1} into registers (dp_free),
    // so it executes during that softmax; the softmax of tile j then finds S_j (issued a
    // tile earlier) and dP_j ready, and runs while dQ_{j-1} and S_{j+1} execute.  dQ_{j-1}
    // waits for dS_{j-1} (ds_full).  S_{j+1} overwrites the score buffer of dS_{j-1}, after
    // dQ_{j-1} in issue order; K_{j+1} has a stage of its own (three key stages), so its
    // load does not wait for dQ_{j-1} to release K_{j-1}.
    bool ok = J > 0 && wait_all(q_full, 0) && wait_all(&k_full[0], 0);
    if (ok) {
      tc_fence_after();
      xk(tmem, qb, kstage(0));  // S_0
    }
    for (int j = 0; j < J && ok; ++j) {
      const int s = j & 1;
      if (!wait_all(&v_full[s], (uint32_t)((j >> 1) & 1))) {
        ok = false;
        break;
      }
      // the softmax of tile j-1 has read dP_{j-1} out of the dP buffer
      if (j > 0 && !wait_all(dp_free, (uint32_t)((j - 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      xk(tmem + T_DP, dob, smem_u32(smem + C::V_OFF + s * C::NOP * C::TILE));  // dP_j = dO V_j^T
      mma_commit_w(&s_full[s]);
      mma_commit_w(&v_empty[s]);
      if (j > 0) {  // dQ_{j-1} once the softmax of tile j-1 has written dS_{j-1}
        if (!wait_all(&ds_full[s ^ 1], (uint32_t)(((j - 1) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        dq_mma(j - 1);
      }
      if (j + 1 < J) {  // S_{j+1} into the other score buffer
        if (!wait_all(&k_full[(j + 1) % C::KST], (uint32_t)(((j + 1) / C::KST) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        xk(tmem + (uint32_t)((s ^ 1) * 128), qb, kstage(j + 1));
      }
    }
    if (ok && wait_all(&ds_full[(J - 1) & 1], (uint32_t)(((J - 1) >> 1) & 1))) {
      tc_fence_after();
      dq_mma(J - 1);
    }
    mma_commit_w(dq_full);
    mma_commit_w(drain);
    drain_q2(drain, 0, g.err);
  } else {  // ------------------------------------------------- softmax: two threads per query row
    const int hf = (warp - 2) >> 2, qd = warp & 3, r = qd * 32 + lane;
    const long p = g.pos0 + 128L * qt + r;
    const bool rvalid = 128 * qt + r < g.n;
    const float sl2 = g.scale_log2;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const float lse2 = rvalid ? a.lse[(long)h * g.n + 128 * qt + r] : 0.f;
    const float Dr = rvalid ? a.D[(long)h * g.n + 128 * qt + r] : 0.f;
    const int b0 = hf * 64;
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      const int s = j & 1;
      const bool own = j >= tr.n_ring;
      const long kpos0 = own ? g.pos0 + 128L * (j - tr.n_ring) : 128L * (tr.m_lo + j);
      int c_lo, c_hi;
      if (!rvalid) { c_lo = 0; c_hi = -1; }
      else if (own) { c_lo = 0; c_hi = (int)min(127L, p - kpos0); }
      else { c_lo = (int)max(0L, p - g.window + 1 - kpos0); c_hi = (int)min(127L, g.pos0 - 1 - kpos0); }
      const bool full = __all_sync(0xffffffffu, c_lo <= b0 && c_hi >= b0 + 63);
      const bool got = mbar_wait(&s_full[s], (uint32_t)((j >> 1) & 1), abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sd[128];  // [0,64): S row, [64,128): dP row, under one wait
      tmem_ld64x2(trow + (uint32_t)(s * 128 + b0), trow + T_DP + (uint32_t)b0, sd);
      tc_fence_before();
      mbar_arrive(dp_free);  // the dP buffer may take dP_{j+1} now
      const float* sv = sd;
      const float* dp = sd + 64;
      uint32_t hi[32], lo[32];
      // dS = P (dP - D), P = 2^(S scale_log2 - lse2): pairs of columns in packed f32x2
      // arithmetic (each lane rounded as the scalar instruction would round it)
      const uint64_t sc2 = f32x2(sl2, sl2), nl2 = f32x2(-lse2, -lse2), nd2 = f32x2(-Dr, -Dr);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float2 a = f32x2_split(ffma2(f32x2(sv[2 * e], sv[2 * e + 1]), sc2, nl2));
        float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
        if (!full) {
          const int col = b0 + 2 * e;
          p0 = (col >= c_lo && col <= c_hi) ? p0 : 0.f;
          p1 = (col + 1 >= c_lo && col + 1 <= c_hi) ? p1 : 0.f;
        }
        const float2 xx = f32x2_split(fmul2(f32x2(p0, p1), fadd2(f32x2(dp[2 * e], dp[2 * e + 1]), nd2)));
        const float x[2] = {xx.x, xx.y};
        __nv_bfloat162 t = __floats2bfloat162_rn(x[0], x[1]);
        hi[e] = *reinterpret_cast<uint32_t*>(&t);
        if (SPLIT) {
          const float2 f = __bfloat1622float2(t);
          lo[e] = pack_bf16(x[0] - f.x, x[1] - f.y);
        }
      }
      tmem_st32(trow + (uint32_t)(s * 128 + b0), hi);  // over this thread's own (already read) S columns
      if (SPLIT) tmem_st32(trow + (uint32_t)(s * 128 + b0 + 32), lo);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ds_full[s]);
    }
    bool got = ok && mbar_wait(dq_full, 0, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
    const bool have = __all_sync(0xffffffffu, got);
    float v[HO];
#pragma unroll
    for (int e = 0; e < HO; ++e) v[e] = 0.f;
    if (have) {
      tc_fence_after();
      ld_cols_q2<HO>(trow + T_DQ + (uint32_t)(hf * HO), v);
#pragma unroll
      for (int e = 0; e < HO; ++e) v[e] *= a.scale;
    }
    const long row = 128L * qt + r;
    if (a.qkv_h) {  // rotated back and written as the QKV product's operand; the K / V stages are free now
      static_assert(rope_bwd_smem_floats<HO>() * 4 <= C::BAR_OFF - C::K_OFF, "rope exchange exceeds the stages");
      const long o = row * a.ld_qkv + col0 + hf * HO;
      const long t0 = 128L * qt;
      rope_bwd_store<HO, SPLIT>(reinterpret_cast<float*>(smem + C::K_OFF), (warp - 2) * 32 + lane, r, hf, v,
                                have && rvalid, a.cs + t0 * HO, a.sn + t0 * HO, (int)min(128L, g.n - t0),
                                a.qkv_h + o, SPLIT ? a.qkv_l + o : nullptr);
    } else if (have && rvalid) {
      float4* dst = reinterpret_cast<float4*>(a.dq + row * a.ldg + col0 + hf * HO);
#pragma unroll
      for (int e = 0; e < HO / 4; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
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

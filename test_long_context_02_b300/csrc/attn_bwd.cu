// Sliding-window attention backward on tcgen05: dQ over every key in the
// window, dK / dV only for the chunk's own keys.
//
// In the TTT-E2E inner loop the keys/values cached from earlier chunks were
// computed with earlier weights and are constants of the current step, so
// gradients flow into the queries and into the chunk's own keys/values only
// (pages: "把 Transformer 做成“终身学习者”", §4.2; the backward runs through the
// last-quarter blocks, whose attention weights are frozen but pass activation
// gradients).  With P = softmax(S), S = Q K^T / sqrt(dh), D = rowsum(dO * O):
//     dP = dO V^T,  dS = P * (dP - D),  dQ = dS K / sqrt(dh),
//     dK = dS^T Q / sqrt(dh),  dV = P^T dO.
// P is recomputed from S and the forward's per-row log2-sum-exp.
//
// attn_dq_kernel  : CTA = (128 queries, head).  Per key tile: S and dP into
//   TMEM (S double-buffered, issued one tile ahead), softmax warps form dS as
//   bf16 in shared memory, dQ += dS K accumulates in TMEM.
// attn_dkv_kernel : CTA = (128 own keys, head).  Per causal query tile:
//   S^T = K Q^T and dP^T = V dO^T into TMEM, P^T written to shared memory for
//   dV += P^T dO, then dS^T (same buffer) for dK += dS^T Q; both in TMEM.
#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {

namespace {

template <int DH, bool SPLIT>
struct BCfg {
  static constexpr int DP = DH <= 64 ? 64 : 128;
  static constexpr int NATOM = DP / 64;
  static constexpr int TILE = 128 * DP * 2;
  static constexpr int NOP = SPLIT ? 2 : 1;
  static constexpr int PB = 128 * 128 * 2;
  // dQ kernel
  static constexpr int KST = 2;
  static constexpr int NDS = SPLIT ? 1 : 2;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = NOP * TILE;
  static constexpr int K_OFF = 2 * NOP * TILE;
  static constexpr int V_OFF = K_OFF + KST * NOP * TILE;
  static constexpr int DS_OFF = V_OFF + NOP * TILE;
  static constexpr int BAR_OFF = DS_OFF + NDS * NOP * PB;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;
  static_assert(SMEM <= 232448, "dQ kernel exceeds shared memory");
  // dK/dV kernel
  static constexpr int X_K = 0;
  static constexpr int X_V = NOP * TILE;
  static constexpr int X_Q = 2 * NOP * TILE;
  static constexpr int X_DO = 3 * NOP * TILE;
  static constexpr int X_P = 4 * NOP * TILE;
  static constexpr int X_BAR = X_P + NOP * PB;
  static constexpr int XSMEM = X_BAR + 256 + 1024;
  static_assert(XSMEM <= 232448, "dK/dV kernel exceeds shared memory");
};

TTT_DEV bool wait_drain(uint64_t* bar, uint32_t parity, int* err) {
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
TTT_DEV void load_head_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int a = 0; a < NATOM; ++a) tma_load_2d(dst + a * 16384, map, bar, col0 + 64 * a, row0);
}
TTT_DEV uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
TTT_DEV uint64_t mnmajor_desc(uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 16384, 1024); }

// Write 32 fp32 values (columns 32c..32c+31 of one 64-column atom) as bf16 (and
// remainders) into a 128-B swizzled row; rowp = atom base + r * 128.
template <bool SPLIT>
TTT_DEV void put_half_row32(uint8_t* rowp, int r, int c, const float (&v)[32], int lo_off) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int ch = (c * 4 + u) ^ (r & 7);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = v[u * 8 + 2 * e], x1 = v[u * 8 + 2 * e + 1];
      __nv_bfloat162 t = __floats2bfloat162_rn(x0, x1);
      hw[e] = *reinterpret_cast<uint32_t*>(&t);
      if (SPLIT) {
        float2 f = __bfloat1622float2(t);
        lw[e] = pack_bf16(x0 - f.x, x1 - f.y);
      }
    }
    uint8_t* dst = rowp + ch * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (SPLIT) *reinterpret_cast<uint4*>(dst + lo_off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

template <int N>
TTT_DEV void tmem_ldn(uint32_t a, float* v) {
  if constexpr (N >= 32) {
    float t[32];
    tmem_ld32(a, t);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = t[i];
    tmem_ldn<N - 32>(a + 32, v + 32);
  } else if constexpr (N == 16) {
    float t[16];
    tmem_ld16(a, t);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = t[i];
  }
}

constexpr int kBwdThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 two threads per row

struct TileRange {
  int n_ring, m_lo, J;
};
TTT_DEV TileRange tiles_for(const AttnArgs& a, int qt) {
  TileRange r;
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

// ================================================================ dQ kernel
template <int DH, bool SPLIT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_dq_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tQl,
                   const __grid_constant__ CUtensorMap tDO, const __grid_constant__ CUtensorMap tDOl,
                   const __grid_constant__ CUtensorMap tKr, const __grid_constant__ CUtensorMap tKrl,
                   const __grid_constant__ CUtensorMap tVr, const __grid_constant__ CUtensorMap tVrl,
                   const __grid_constant__ CUtensorMap tKo, const __grid_constant__ CUtensorMap tKol,
                   const __grid_constant__ CUtensorMap tVo, const __grid_constant__ CUtensorMap tVol,
                   const AttnBwdArgs a) {
  using C = BCfg<DH, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + C::KST;
  uint64_t* v_full = k_empty + C::KST;
  uint64_t* v_empty = v_full + 1;
  uint64_t* s_full = v_empty + 1;
  uint64_t* ds_full = s_full + 2;
  uint64_t* ds_empty = ds_full + C::NDS;
  uint64_t* dq_full = ds_empty + C::NDS;
  uint64_t* drain = dq_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y;
  const AttnArgs& g = a.g;
  const TileRange tr = tiles_for(g, qt);
  const int J = tr.J;
  const int col0 = h * DH;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::KST; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    for (int i = 0; i < C::NDS; ++i) { mbar_init(&ds_full[i], 256); mbar_init(&ds_empty[i], 1); }
    mbar_init(dq_full, 1);
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
  const uint32_t T_DP = 256, T_DQ = 384;

  auto tile_row0 = [&](int j, bool& own) -> int {
    if (j < tr.n_ring) {
      own = false;
      return (int)(((long)(tr.m_lo + j) * 128) % g.window);
    }
    own = true;
    return 128 * (j - tr.n_ring);
  };

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------------- producer
      uint32_t kiss = 0, kpar = 0;
      bool viss = false;
      uint32_t vpar = 0;
      mbar_expect_tx(q_full, 2 * C::NOP * C::TILE);
      load_head_tile<C::NATOM>(smem + C::Q_OFF, &tQ, q_full, col0, 128 * qt);
      load_head_tile<C::NATOM>(smem + C::DO_OFF, &tDO, q_full, col0, 128 * qt);
      if (SPLIT) {
        load_head_tile<C::NATOM>(smem + C::Q_OFF + C::TILE, &tQl, q_full, col0, 128 * qt);
        load_head_tile<C::NATOM>(smem + C::DO_OFF + C::TILE, &tDOl, q_full, col0, 128 * qt);
      }
      for (int j = 0; j < J; ++j) {
        bool own;
        const int row0 = tile_row0(j, own);
        const int s = j % C::KST;
        if (!mbar_wait(&k_empty[s], ((j / C::KST) & 1) ^ 1, abort_flag, g.err, DERR_TIMEOUT_PRODUCER)) break;
        uint8_t* kd = smem + C::K_OFF + s * C::NOP * C::TILE;
        mbar_expect_tx(&k_full[s], C::NOP * C::TILE);
        load_head_tile<C::NATOM>(kd, own ? &tKo : &tKr, &k_full[s], col0, row0);
        if (SPLIT) load_head_tile<C::NATOM>(kd + C::TILE, own ? &tKol : &tKrl, &k_full[s], col0, row0);
        kiss |= 1u << s;
        kpar = (kpar & ~(1u << s)) | ((uint32_t)((j / C::KST) & 1) << s);
        if (!mbar_wait(v_empty, (j & 1) ^ 1, abort_flag, g.err, DERR_TIMEOUT_PRODUCER)) break;
        uint8_t* vd = smem + C::V_OFF;
        mbar_expect_tx(v_full, C::NOP * C::TILE);
        load_head_tile<C::NATOM>(vd, own ? &tVo : &tVr, v_full, col0, row0);
        if (SPLIT) load_head_tile<C::NATOM>(vd + C::TILE, own ? &tVol : &tVrl, v_full, col0, row0);
        viss = true;
        vpar = (uint32_t)(j & 1);
      }
      wait_drain(q_full, 0, g.err);
      for (int s = 0; s < C::KST; ++s)
        if (kiss & (1u << s)) wait_drain(&k_full[s], (kpar >> s) & 1u, g.err);
      if (viss) wait_drain(v_full, vpar, g.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------------ MMA
      constexpr uint32_t idSS = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idDQ = idesc_bf16(128, DH, 0, 1);
      const uint32_t qb = smem_u32(smem + C::Q_OFF), dob = smem_u32(smem + C::DO_OFF);
      auto qk = [&](uint32_t d, uint32_t xb, uint32_t kb) {  // d = X . K^T over the head dim
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          mma_bf16(d, kmajor_desc(xb, kk), kmajor_desc(kb, kk), idSS, kk ? 1u : 0u);
          if (SPLIT) {
            mma_bf16(d, kmajor_desc(xb, kk), kmajor_desc(kb + C::TILE, kk), idSS, 1u);
            mma_bf16(d, kmajor_desc(xb + C::TILE, kk), kmajor_desc(kb, kk), idSS, 1u);
          }
        }
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, g.err, DERR_TIMEOUT_MMA) &&
                mbar_wait(&k_full[0], 0, abort_flag, g.err, DERR_TIMEOUT_MMA);
      if (ok) {
        tc_fence_after();
        qk(tmem + 0, qb, smem_u32(smem + C::K_OFF));
      }
      for (int j = 0; j < J && ok; ++j) {
        if (!mbar_wait(v_full, j & 1, abort_flag, g.err, DERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        qk(tmem + T_DP, dob, smem_u32(smem + C::V_OFF));  // dP_j = dO V_j^T
        mma_commit(&s_full[j & 1]);
        mma_commit(v_empty);
        if (j + 1 < J) {
          const int s = (j + 1) % C::KST;
          if (!mbar_wait(&k_full[s], ((j + 1) / C::KST) & 1, abort_flag, g.err, DERR_TIMEOUT_MMA)) break;
          tc_fence_after();
          qk(tmem + (uint32_t)(((j + 1) & 1) * 128), qb, smem_u32(smem + C::K_OFF + s * C::NOP * C::TILE));
        }
        const int b = j % C::NDS;
        if (!mbar_wait(&ds_full[b], (j / C::NDS) & 1, abort_flag, g.err, DERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        const uint32_t dsb = smem_u32(smem + C::DS_OFF + b * C::NOP * C::PB);
        const uint32_t kb = smem_u32(smem + C::K_OFF + (j % C::KST) * C::NOP * C::TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_bf16(tmem + T_DQ, kmajor_desc(dsb, kk), mnmajor_desc(kb, kk), idDQ, (j | kk) ? 1u : 0u);
          if (SPLIT) {
            mma_bf16(tmem + T_DQ, kmajor_desc(dsb, kk), mnmajor_desc(kb + C::TILE, kk), idDQ, 1u);
            mma_bf16(tmem + T_DQ, kmajor_desc(dsb + C::PB, kk), mnmajor_desc(kb, kk), idDQ, 1u);
          }
        }
        mma_commit(&ds_empty[b]);
        mma_commit(&k_empty[j % C::KST]);
      }
      mma_commit(dq_full);
      mma_commit(drain);
      wait_drain(drain, 0, g.err);
    }
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
      const bool own = j >= tr.n_ring;
      const long kpos0 = own ? g.pos0 + 128L * (j - tr.n_ring) : 128L * (tr.m_lo + j);
      int c_lo, c_hi;
      if (!rvalid) { c_lo = 0; c_hi = -1; }
      else if (own) { c_lo = 0; c_hi = (int)min(127L, p - kpos0); }
      else { c_lo = (int)max(0L, p - g.window + 1 - kpos0); c_hi = (int)min(127L, g.pos0 - 1 - kpos0); }
      const bool full = __all_sync(0xffffffffu, c_lo <= b0 && c_hi >= b0 + 63);
      bool got = mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      const int b = j % C::NDS, u = j / C::NDS;
      if (got && u >= 1) got = mbar_wait(&ds_empty[b], (u - 1) & 1, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      uint8_t* dsrow = smem + C::DS_OFF + b * C::NOP * C::PB + hf * 16384 + r * 128;
      const uint32_t sb = trow + (uint32_t)((j & 1) * 128 + b0);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float sv[32], dp[32];
        tmem_ld32(sb + c * 32, sv);
        tmem_ld32(trow + T_DP + b0 + c * 32, dp);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int col = b0 + c * 32 + i;
          float pr = ex2_approx(fmaf(sv[i], sl2, -lse2));
          if (!full) pr = (col >= c_lo && col <= c_hi) ? pr : 0.f;
          sv[i] = pr * (dp[i] - Dr);
        }
        put_half_row32<SPLIT>(dsrow, r, c, sv, C::PB);
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&ds_full[b]);
    }
    bool got = ok && mbar_wait(dq_full, 0, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
    if (__all_sync(0xffffffffu, got)) {
      tc_fence_after();
      constexpr int HO = DH / 2;
      float v[HO];
      tmem_ldn<HO>(trow + T_DQ + hf * HO, v);
      if (rvalid) {
        const float sc = a.scale;
        float4* dst = reinterpret_cast<float4*>(a.dq + (long)(128 * qt + r) * a.ldg + col0 + hf * HO);
#pragma unroll
        for (int e = 0; e < HO / 4; ++e)
          dst[e] = make_float4(v[4 * e] * sc, v[4 * e + 1] * sc, v[4 * e + 2] * sc, v[4 * e + 3] * sc);
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

// ============================================================ dK / dV kernel
template <int DH, bool SPLIT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_dkv_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tQl,
                    const __grid_constant__ CUtensorMap tDO, const __grid_constant__ CUtensorMap tDOl,
                    const __grid_constant__ CUtensorMap tKo, const __grid_constant__ CUtensorMap tKol,
                    const __grid_constant__ CUtensorMap tVo, const __grid_constant__ CUtensorMap tVol,
                    const AttnBwdArgs a) {
  using C = BCfg<DH, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + C::X_BAR);
  uint64_t* qd_full = kv_full + 1;
  uint64_t* qd_empty = qd_full + 1;
  uint64_t* s_full = qd_empty + 1;
  uint64_t* p_full = s_full + 1;
  uint64_t* p_free = p_full + 1;
  uint64_t* ds_full = p_free + 1;
  uint64_t* buf_free = ds_full + 1;
  uint64_t* acc_full = buf_free + 1;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, h = blockIdx.y;
  const AttnArgs& g = a.g;
  const int nq = (g.n + 127) / 128;
  const int I = nq - kt;  // causal query tiles kt .. nq-1
  const int col0 = h * DH;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(qd_full, 1);
    mbar_init(qd_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 256);
    mbar_init(p_free, 1);
    mbar_init(ds_full, 256);
    mbar_init(buf_free, 1);
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
  const uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + C::DP;

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------------- producer
      mbar_expect_tx(kv_full, 2 * C::NOP * C::TILE);
      load_head_tile<C::NATOM>(smem + C::X_K, &tKo, kv_full, col0, 128 * kt);
      load_head_tile<C::NATOM>(smem + C::X_V, &tVo, kv_full, col0, 128 * kt);
      if (SPLIT) {
        load_head_tile<C::NATOM>(smem + C::X_K + C::TILE, &tKol, kv_full, col0, 128 * kt);
        load_head_tile<C::NATOM>(smem + C::X_V + C::TILE, &tVol, kv_full, col0, 128 * kt);
      }
      bool iss = false;
      uint32_t par = 0;
      for (int i = 0; i < I; ++i) {
        if (!mbar_wait(qd_empty, (i & 1) ^ 1, abort_flag, g.err, DERR_TIMEOUT_PRODUCER)) break;
        const int row0 = 128 * (kt + i);
        mbar_expect_tx(qd_full, 2 * C::NOP * C::TILE);
        load_head_tile<C::NATOM>(smem + C::X_Q, &tQ, qd_full, col0, row0);
        load_head_tile<C::NATOM>(smem + C::X_DO, &tDO, qd_full, col0, row0);
        if (SPLIT) {
          load_head_tile<C::NATOM>(smem + C::X_Q + C::TILE, &tQl, qd_full, col0, row0);
          load_head_tile<C::NATOM>(smem + C::X_DO + C::TILE, &tDOl, qd_full, col0, row0);
        }
        iss = true;
        par = (uint32_t)(i & 1);
      }
      wait_drain(kv_full, 0, g.err);
      if (iss) wait_drain(qd_full, par, g.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------------ MMA
      constexpr uint32_t idSS = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idAcc = idesc_bf16(128, DH, 0, 1);
      const uint32_t kb = smem_u32(smem + C::X_K), vb = smem_u32(smem + C::X_V);
      const uint32_t qb = smem_u32(smem + C::X_Q), dob = smem_u32(smem + C::X_DO);
      const uint32_t pb = smem_u32(smem + C::X_P);
      auto xy = [&](uint32_t d, uint32_t xb, uint32_t yb) {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          mma_bf16(d, kmajor_desc(xb, kk), kmajor_desc(yb, kk), idSS, kk ? 1u : 0u);
          if (SPLIT) {
            mma_bf16(d, kmajor_desc(xb, kk), kmajor_desc(yb + C::TILE, kk), idSS, 1u);
            mma_bf16(d, kmajor_desc(xb + C::TILE, kk), kmajor_desc(yb, kk), idSS, 1u);
          }
        }
      };
      auto acc = [&](uint32_t d, uint32_t yb, bool first) {  // d += Pbuf . Y (Y MN-major over queries)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_bf16(d, kmajor_desc(pb, kk), mnmajor_desc(yb, kk), idAcc, (!first || kk) ? 1u : 0u);
          if (SPLIT) {
            mma_bf16(d, kmajor_desc(pb, kk), mnmajor_desc(yb + C::TILE, kk), idAcc, 1u);
            mma_bf16(d, kmajor_desc(pb + C::PB, kk), mnmajor_desc(yb, kk), idAcc, 1u);
          }
        }
      };
      bool ok = mbar_wait(kv_full, 0, abort_flag, g.err, DERR_TIMEOUT_MMA);
      for (int i = 0; i < I && ok; ++i) {
        if (!mbar_wait(qd_full, i & 1, abort_flag, g.err, DERR_TIMEOUT_MMA)) break;
        if (i > 0 && !mbar_wait(ds_full, (i - 1) & 1, abort_flag, g.err, DERR_TIMEOUT_MMA)) break;  // S/dP TMEM read
        tc_fence_after();
        xy(tmem + T_S, kb, qb);    // S^T = K Q^T
        xy(tmem + T_DP, vb, dob);  // dP^T = V dO^T
        mma_commit(s_full);
        if (!mbar_wait(p_full, i & 1, abort_flag, g.err, DERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        acc(tmem + T_DV, dob, i == 0);  // dV += P^T dO
        mma_commit(p_free);
        if (!mbar_wait(ds_full, i & 1, abort_flag, g.err, DERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        acc(tmem + T_DK, qb, i == 0);   // dK += dS^T Q
        mma_commit(buf_free);
        mma_commit(qd_empty);
      }
      mma_commit(acc_full);
      mma_commit(drain);
      wait_drain(drain, 0, g.err);
    }
  } else {  // --------------------------------------- softmax: two threads per key row (64 queries each)
    const int hf = (warp - 2) >> 2, qd = warp & 3, r = qd * 32 + lane;
    const int krow = 128 * kt + r;
    const bool kvalid = krow < g.n;
    const float sl2 = g.scale_log2;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const int b0 = hf * 64;
    uint8_t* prow = smem + C::X_P + hf * 16384 + r * 128;
    bool ok = true;
    for (int i = 0; i < I; ++i) {
      const int q0 = 128 * (kt + i);
      // per-column statistics of the query tile, read straight from global memory
      // (warp-uniform addresses: one broadcast transaction each)
      const float* sl = a.lse + (long)h * g.n + q0;
      const float* sd = a.D + (long)h * g.n + q0;
      const int clast = g.n - 1 - q0;  // columns beyond it are masked and read a clamped index
      // query column c is valid iff q0 + c < n and key position <= query position
      const int c_lo = kvalid ? krow - q0 : 128;
      const int c_hi = min(127, g.n - 1 - q0);
      const bool full = __all_sync(0xffffffffu, c_lo <= b0 && c_hi >= b0 + 63);
      bool got = mbar_wait(s_full, i & 1, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      if (got && i > 0) got = mbar_wait(buf_free, (i - 1) & 1, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // pass A: P^T
        float pv[32];
        tmem_ld32(trow + T_S + b0 + c * 32, pv);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = b0 + c * 32 + e;
          const float pr = ex2_approx(fmaf(pv[e], sl2, -sl[min(col, clast)]));
          pv[e] = (full || (col >= c_lo && col <= c_hi)) ? pr : 0.f;
        }
        put_half_row32<SPLIT>(prow, r, c, pv, C::PB);
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(p_full);
      got = mbar_wait(p_free, i & 1, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // pass B: dS^T = P^T (dP^T - D)
        float dp[32], dv[32];
        tmem_ld32(trow + T_S + b0 + c * 32, dv);
        tmem_ld32(trow + T_DP + b0 + c * 32, dp);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = b0 + c * 32 + e;
          const int cc = min(col, clast);
          float pr = ex2_approx(fmaf(dv[e], sl2, -sl[cc]));
          pr = (full || (col >= c_lo && col <= c_hi)) ? pr : 0.f;
          dv[e] = pr * (dp[e] - sd[cc]);
        }
        put_half_row32<SPLIT>(prow, r, c, dv, C::PB);
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    bool got = ok && mbar_wait(acc_full, 0, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
    if (__all_sync(0xffffffffu, got)) {
      tc_fence_after();
      constexpr int HO = DH / 2;
      float v[HO], w[HO];
      tmem_ldn<HO>(trow + T_DV + hf * HO, v);
      tmem_ldn<HO>(trow + T_DK + hf * HO, w);
      if (kvalid) {
        const float sc = a.scale;
        float4* dv = reinterpret_cast<float4*>(a.dv + (long)krow * a.ldg + col0 + hf * HO);
        float4* dk = reinterpret_cast<float4*>(a.dk + (long)krow * a.ldg + col0 + hf * HO);
#pragma unroll
        for (int e = 0; e < HO / 4; ++e) {
          dv[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          dk[e] = make_float4(w[4 * e] * sc, w[4 * e + 1] * sc, w[4 * e + 2] * sc, w[4 * e + 3] * sc);
        }
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

template <int DH, bool SPLIT>
int launch_bwd(const AttnBwdMaps& m, const AttnBwdArgs& a, cudaStream_t st, int which) {
  using C = BCfg<DH, SPLIT>;
  auto kq = attn_dq_kernel<DH, SPLIT>;
  auto kkv = attn_dkv_kernel<DH, SPLIT>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::XSMEM);
    if (e != cudaSuccess) return (int)e;
    attr = true;
  }
  dim3 grid((a.g.n + 127) / 128, a.g.H);
  const AttnMaps& f = m.f;
  if (which != 2) {
    kq<<<grid, kBwdThreads, C::SMEM, st>>>(f.q, f.ql, m.dO, m.dOl, f.kr, f.krl, f.vr, f.vrl, f.ko, f.kol, f.vo, f.vol, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  if (which != 1) kkv<<<grid, kBwdThreads, C::XSMEM, st>>>(f.q, f.ql, m.dO, m.dOl, f.ko, f.kol, f.vo, f.vol, a);
  return (int)cudaGetLastError();
}

}  // namespace

int attn_bwd_run(const AttnBwdMaps& m, const AttnBwdArgs& a, bool split, cudaStream_t st, int which) {
  if (a.g.n <= 0) return 0;
  if (which != 2) {
    const int r = attn_dq2_run(m, a, split, st);
    if (r != 0) return r;
  }
  return which != 1 ? attn_dkv2_run(m, a, split, st) : 0;
}

// The earlier kernels (dS and P^T through shared memory).
int attn_bwd1_run(const AttnBwdMaps& m, const AttnBwdArgs& a, bool split, cudaStream_t st, int which) {
  if (a.g.n <= 0) return 0;
  if (split) {
    switch (a.g.dh) {
      case 32: return launch_bwd<32, true>(m, a, st, which);
      case 64: return launch_bwd<64, true>(m, a, st, which);
    }
    return (int)cudaErrorInvalidValue;
  }
  switch (a.g.dh) {
    case 32: return launch_bwd<32, false>(m, a, st, which);
    case 64: return launch_bwd<64, false>(m, a, st, which);
    case 96: return launch_bwd<96, false>(m, a, st, which);
    case 128: return launch_bwd<128, false>(m, a, st, which);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace ttt

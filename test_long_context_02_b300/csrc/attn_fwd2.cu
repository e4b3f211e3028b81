// Sliding-window causal attention forward, bf16 operands, two query tiles per CTA.
//
// Same operation and geometry as attn_fwd.cu (pages: "把 Transformer 做成“终身学习者”",
// §4.2, the key/value cache holds only the window; §8 FAQ Q4, any k >= b): a
// query at absolute position p sees the keys at positions j with p - k < j <= p,
// keys before the chunk come from the k-slot cache (slot = position mod k), the
// chunk's own keys from its own K/V buffer; key tiles are 128 positions aligned
// to multiples of 128 in absolute position.
//
// CTA = one head x 256 queries as two 128-row tiles Q0, Q1 that share every K/V
// tile.  Warp 0 loads Q0, Q1 once and K/V tiles through a 2-stage TMA ring;
// warp 1 issues, per key tile j, S0 = Q0 K_j^T, S1 = Q1 K_j^T, O0 += P0 V_j,
// O1 += P1 V_j, ping-ponging so the tensor core works on one tile's products
// while the other tile's softmax runs.  Warps 2-5 (tile 0) and 6-9 (tile 1)
// run the softmax with one thread per query row: the row of S is read from
// TMEM, P = exp2(S*c - m) is written back over S as bf16 and read by the PV
// product straight from TMEM, and O accumulates in TMEM.  The running max m
// is updated lazily: O and the row sum are rescaled only when the max grows by
// more than 2^8, so P stays below 256 and the rescale is rare.
#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {

namespace {

constexpr float kLazyLog2 = 8.0f;
constexpr int kF2Threads = 320;

template <int DH>
struct F2Cfg {
  static constexpr int DP = DH <= 64 ? 64 : 128;  // head width padded to whole 128-B atoms
  static constexpr int NATOM = DP / 64;
  static constexpr int TILE = 128 * DP * 2;
  static constexpr int Q_OFF = 0;                  // Q0, Q1
  static constexpr int K_OFF = 2 * TILE;           // 2 stages
  static constexpr int V_OFF = K_OFF + 2 * TILE;   // 2 stages
  static constexpr int BAR_OFF = V_OFF + 2 * TILE;
  static constexpr int SMEM = BAR_OFF + 256;
  static_assert(SMEM <= 232448, "attention forward exceeds shared memory");
};

TTT_DEV bool wait_drain2(uint64_t* bar, uint32_t parity, int* err) {
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
TTT_DEV void load_tile2(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int a = 0; a < NATOM; ++a) tma_load_2d(dst + a * 16384, map, bar, col0 + 64 * a, row0);
}
TTT_DEV uint64_t kdesc(uint32_t base, int kk) { return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024); }
TTT_DEV uint64_t mndesc(uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 16384, 1024); }

// Key tiles of a 256-query block: cache tiles [m_lo, m_lo + n_ring) then own tiles.
struct Range2 {
  int n_ring, m_lo, J;
};
TTT_DEV Range2 range_for(const AttnArgs& a, int qb) {
  Range2 r;
  const long qlo = a.pos0 + 256L * qb;
  const int qend = min(a.n, 256 * qb + 256);
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

template <int DH>
__global__ void __launch_bounds__(kF2Threads, 1)
    attn_fwd2_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tKr,
                     const __grid_constant__ CUtensorMap tVr, const __grid_constant__ CUtensorMap tKo,
                     const __grid_constant__ CUtensorMap tVo, const AttnArgs a) {
  using C = F2Cfg<DH>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // swizzled tiles need a 1024-B aligned base; report, do nothing else
    if (threadIdx.x == 0 && a.err) atomicCAS(a.err, 0, (int)DERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;          // 1
  uint64_t* k_full = bars + 1;      // 2
  uint64_t* k_empty = bars + 3;     // 2
  uint64_t* v_full = bars + 5;      // 2
  uint64_t* v_empty = bars + 7;     // 2
  uint64_t* s_full = bars + 9;      // 2 (per query tile)
  uint64_t* p_full = bars + 11;     // 2
  uint64_t* o_final = bars + 13;    // 2: the last P V product of each query tile
  uint64_t* drain = bars + 15;      // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = blockIdx.x, h = blockIdx.y;
  const Range2 tr = range_for(a, qb);
  const int J = tr.J;
  const int col0 = h * DH;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_final[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512)
  pdl_wait();  // the predecessor kernel's outputs are complete and visible from here on
  pdl_launch_dependents();

  auto tile_row0 = [&](int j, bool& own) -> int {
    if (j < tr.n_ring) {
      own = false;
      return (int)(((long)(tr.m_lo + j) * 128) % a.window);
    }
    own = true;
    return 128 * (j - tr.n_ring);
  };

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------------ TMA producer
      uint32_t kiss = 0, kpar = 0, viss = 0, vpar = 0;
      mbar_expect_tx(q_full, 2 * C::TILE);
      load_tile2<C::NATOM>(smem + C::Q_OFF, &tQ, q_full, col0, 256 * qb);
      load_tile2<C::NATOM>(smem + C::Q_OFF + C::TILE, &tQ, q_full, col0, 256 * qb + 128);
      for (int j = 0; j < J; ++j) {
        const int s = j & 1;
        const uint32_t par = (uint32_t)((j >> 1) & 1);
        bool own;
        const int row0 = tile_row0(j, own);
        if (!mbar_wait(&k_empty[s], par ^ 1u, abort_flag, a.err, DERR_TIMEOUT_PRODUCER)) break;
        mbar_expect_tx(&k_full[s], C::TILE);
        load_tile2<C::NATOM>(smem + C::K_OFF + s * C::TILE, own ? &tKo : &tKr, &k_full[s], col0, row0);
        kiss |= 1u << s;
        kpar = (kpar & ~(1u << s)) | (par << s);
        if (!mbar_wait(&v_empty[s], par ^ 1u, abort_flag, a.err, DERR_TIMEOUT_PRODUCER)) break;
        mbar_expect_tx(&v_full[s], C::TILE);
        load_tile2<C::NATOM>(smem + C::V_OFF + s * C::TILE, own ? &tVo : &tVr, &v_full[s], col0, row0);
        viss |= 1u << s;
        vpar = (vpar & ~(1u << s)) | (par << s);
      }
      // no TMA write may still be in flight when the CTA exits
      wait_drain2(q_full, 0, a.err);
      for (int s = 0; s < 2; ++s) {
        if (kiss & (1u << s)) wait_drain2(&k_full[s], (kpar >> s) & 1u, a.err);
        if (viss & (1u << s)) wait_drain2(&v_full[s], (vpar >> s) & 1u, a.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // -------------------------------------------------------- MMA issuer
      constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(128, DH, 0, 1);
      const uint32_t q0 = smem_u32(smem + C::Q_OFF), q1 = q0 + C::TILE;
      auto issue_s = [&](int i, int j) {  // S_i = Q_i K_j^T over the head dim
        const uint32_t kb = smem_u32(smem + C::K_OFF + (j & 1) * C::TILE);
        const uint32_t qi = i ? q1 : q0;
        const uint32_t d = tmem + (uint32_t)(i * 128);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) mma_bf16(d, kdesc(qi, kk), kdesc(kb, kk), idS, kk ? 1u : 0u);
        mma_commit(&s_full[i]);
      };
      auto issue_pv = [&](int i, int j) {  // O_i (+)= P_i V_j, P_i from TMEM (over S_i)
        const uint32_t vb = smem_u32(smem + C::V_OFF + (j & 1) * C::TILE);
        const uint32_t p = tmem + (uint32_t)(i * 128);
        const uint32_t d = tmem + 256u + (uint32_t)(i * 128);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_bf16_ts(d, p + (uint32_t)(kk * 8), mndesc(vb, kk), idPV, (j | kk) ? 1u : 0u);
        if (j == J - 1) mma_commit(&o_final[i]);
      };
      bool ok = J > 0 && mbar_wait(q_full, 0, abort_flag, a.err, DERR_TIMEOUT_MMA) &&
                mbar_wait(&k_full[0], 0, abort_flag, a.err, DERR_TIMEOUT_MMA);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        mma_commit(&k_empty[0]);
      }
      for (int j = 0; j < J && ok; ++j) {
        const int s = j & 1;
        const uint32_t par = (uint32_t)((j >> 1) & 1);
        const bool more = j + 1 < J;
        if (!mbar_wait(&v_full[s], par, abort_flag, a.err, DERR_TIMEOUT_MMA)) break;
        if (!mbar_wait(&p_full[0], (uint32_t)(j & 1), abort_flag, a.err, DERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        issue_pv(0, j);
        if (more) {
          if (!mbar_wait(&k_full[s ^ 1], (uint32_t)(((j + 1) >> 1) & 1), abort_flag, a.err, DERR_TIMEOUT_MMA)) break;
          tc_fence_after();
          issue_s(0, j + 1);  // after PV_0(j) in issue order: S_0 reuses the columns P_0 occupied
        }
        if (!mbar_wait(&p_full[1], (uint32_t)(j & 1), abort_flag, a.err, DERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        issue_pv(1, j);
        mma_commit(&v_empty[s]);
        if (more) {
          issue_s(1, j + 1);
          mma_commit(&k_empty[s ^ 1]);
        }
      }
      mma_commit(drain);  // every MMA issued above has finished once this arrives
      wait_drain2(drain, 0, a.err);
    }
  } else {  // ------------------------------------------------ softmax: one thread per query row
    const int i = (warp - 2) >> 2;   // query tile of this warpgroup
    const int qd = warp & 3;          // TMEM lane quadrant of this warp
    const int r = qd * 32 + lane;     // row within the tile
    const int qrow = 256 * qb + 128 * i + r;
    const long p = a.pos0 + qrow;
    const bool rvalid = qrow < a.n;
    const float sl2 = a.scale_log2;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t sS = tmem + lane_off + (uint32_t)(i * 128);
    const uint32_t sO = tmem + lane_off + 256u + (uint32_t)(i * 128);
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      const bool own = j >= tr.n_ring;
      const long kpos0 = own ? a.pos0 + 128L * (j - tr.n_ring) : 128L * (tr.m_lo + j);
      int c_lo, c_hi;  // visible key columns [c_lo, c_hi] of this tile for this row
      if (!rvalid) {
        c_lo = 0;
        c_hi = -1;
      } else if (own) {
        c_lo = 0;
        c_hi = (int)min(127L, p - kpos0);
      } else {
        c_lo = (int)max(0L, p - a.window + 1 - kpos0);
        c_hi = (int)min(127L, a.pos0 - 1 - kpos0);
      }
      const bool full = __all_sync(0xffffffffu, c_lo == 0 && c_hi == 127);
      const bool got = mbar_wait(&s_full[i], (uint32_t)(j & 1), abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // pass 1: row max over the tile, eight independent chains (S is re-read in pass 2
      // rather than held, which keeps registers below the 320-thread limit)
      float mx;
      {
        float t[128];
        tmem_ld128(sS, t);
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
        if (full) {
#pragma unroll
          for (int e = 0; e < 128; ++e) m8[e & 7] = fmaxf(m8[e & 7], t[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 128; ++e) m8[e & 7] = fmaxf(m8[e & 7], (e >= c_lo && e <= c_hi) ? t[e] : -INFINITY);
        }
        mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      }
      const float m_tile = mx * sl2;
      // lazy max: move it only when the tile's max exceeds it by more than 2^8
      const bool grow = m_tile > m_used + kLazyLog2;
      if (__any_sync(0xffffffffu, grow) && j > 0) {
        // O_i is complete up to tile j-1: S_i(j) was issued after P_i V_{j-1}, and its
        // completion (s_full) covers every earlier product.  Rescale O_i in place.
        tc_fence_after();
        const float alpha = grow ? ex2_approx(m_used - m_tile) : 1.0f;
#pragma unroll
        for (int c = 0; c < DH / 32; ++c) {
          float t[32];
          tmem_ld32(sO + (uint32_t)(c * 32), t);
          uint32_t u[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(t[e] * alpha);
          tmem_st32(sO + (uint32_t)(c * 32), u);
        }
        l_run *= alpha;
      }
      if (grow) m_used = m_tile;
      const float m_use = (m_used == -INFINITY) ? 0.f : m_used;
      float r8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) r8[e] = 0.f;
      // pass 2: P as bf16 pairs written over the first 64 columns of S_i.  Chunk c
      // reads S columns 32c.. before it writes P columns 16c.., which only overlap
      // S columns already read (16c + 16 <= 32c for c >= 1; c = 0 reads first).
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float t[32];
        tmem_ld32(sS + (uint32_t)(c * 32), t);
        uint32_t u[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float y0 = t[2 * e], y1 = t[2 * e + 1];
          if (!full) {
            const int k0 = 32 * c + 2 * e;
            y0 = (k0 >= c_lo && k0 <= c_hi) ? y0 : -INFINITY;
            y1 = (k0 + 1 >= c_lo && k0 + 1 <= c_hi) ? y1 : -INFINITY;
          }
          const float x0 = ex2_approx(fmaf(y0, sl2, -m_use));
          const float x1 = ex2_approx(fmaf(y1, sl2, -m_use));
          r8[(2 * e) & 7] += x0;
          r8[(2 * e + 1) & 7] += x1;
          u[e] = pack_bf16(x0, x1);
        }
        tmem_st16(sS + (uint32_t)(c * 16), u);
      }
      const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[i]);
      l_run += rs;
    }
    // epilogue: O_i / l after the last P V product
    bool got = ok && J > 0 && mbar_wait(&o_final[i], 0, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
    if (__all_sync(0xffffffffu, got)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        float t[32];
        tmem_ld32(sO + (uint32_t)(c * 32), t);
        if (rvalid) {
          uint32_t hw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) hw[e] = pack_bf16(t[2 * e] * inv, t[2 * e + 1] * inv);
          uint4* dst = reinterpret_cast<uint4*>(a.o_hi + (long)qrow * a.ldo + col0 + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(hw[4 * v], hw[4 * v + 1], hw[4 * v + 2], hw[4 * v + 3]);
        }
      }
      if (rvalid && a.lse) a.lse[(long)h * a.n + qrow] = (m_used == -INFINITY ? 0.f : m_used) + log2f(l_run);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DH>
int launch_fwd2(const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  using C = F2Cfg<DH>;
  auto kern = attn_fwd2_kernel<DH>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return (int)e;
    attr = true;
  }
  dim3 grid((a.n + 255) / 256, a.H);
  return (int)launch_k(kern, grid, dim3(kF2Threads), C::SMEM, st, m.q, m.kr, m.vr, m.ko, m.vo, a);
}

}  // namespace

int attn_fwd2_run(const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  if (a.n <= 0) return 0;
  switch (a.dh) {
    case 32: return launch_fwd2<32>(m, a, st);
    case 64: return launch_fwd2<64>(m, a, st);
    case 96: return launch_fwd2<96>(m, a, st);
    case 128: return launch_fwd2<128>(m, a, st);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace ttt

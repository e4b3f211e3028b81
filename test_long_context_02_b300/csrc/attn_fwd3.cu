// Sliding-window causal attention forward, one 128-query tile per CTA, with P
// and O kept in tensor memory.
//
// Same operation and geometry as attn_fwd.cu (pages: "把 Transformer 做成“终身学习者”",
// §4.2, the key/value cache holds only the window; §8 FAQ Q4, any k >= b): a
// query at absolute position p sees the keys at positions j with p - k < j <= p;
// keys before the chunk come from the k-slot cache (slot = position mod k), the
// chunk's own keys from its own K/V buffer; key tiles are 128 positions aligned
// to multiples of 128 in absolute position.
//
// Warp 0 loads Q once and K/V tiles through 2-stage TMA rings.  Warp 1 issues
// S_{j+1} = Q K_{j+1}^T into one of two TMEM score buffers while the softmax
// works on S_j, then O += P_j V_j with P_j read from TMEM.  Warps 2-9 run the
// softmax, two threads per query row (64 key columns each): the row max is
// exchanged through shared memory, P = exp2(S*c - m) is written as bf16 over
// the thread's own columns of S_j, and O accumulates in TMEM.  The running max
// m is lazy: O (each thread its half of the head dimension) and the row sum are
// rescaled only when the max grows by more than 2^8.  In split mode (fp32
// compute) every operand is a bf16 pair and each product is hi*hi + hi*lo + lo*hi.
#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {

namespace {

constexpr float kLazy = 8.0f;       // log2 of the largest P value a stale max may produce
constexpr int kF3Threads = 320;     // warp 0 TMA, warp 1 MMA, warps 2-9 softmax

template <int DH, bool SPLIT>
struct F3Cfg {
  static constexpr int DP = DH <= 64 ? 64 : 128;  // head width padded to whole 128-B atoms
  static constexpr int NATOM = DP / 64;
  static constexpr int TILE = 128 * DP * 2;
  static constexpr int NOP = SPLIT ? 2 : 1;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = NOP * TILE;              // 2 stages
  static constexpr int V_OFF = K_OFF + 2 * NOP * TILE;  // 2 stages
  static constexpr int BAR_OFF = V_OFF + 2 * NOP * TILE;
  static constexpr int XCH_OFF = BAR_OFF + 256;         // [2 parities][2 halves][128 rows] fp32
  static constexpr int SMEM = XCH_OFF + 2048;
  static_assert(SMEM <= 232448, "attention forward exceeds shared memory");
};

TTT_DEV bool drain3(uint64_t* bar, uint32_t parity, int* err) {
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
TTT_DEV void load_tile3(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int a = 0; a < NATOM; ++a) tma_load_2d(dst + a * 16384, map, bar, col0 + 64 * a, row0);
}
TTT_DEV uint64_t kdesc3(uint32_t base, int kk) { return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024); }
TTT_DEV uint64_t mndesc3(uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 16384, 1024); }

// N (multiple of 16) consecutive 32-bit TMEM columns <-> registers.
template <int N>
TTT_DEV void ld_cols(uint32_t a, float* v) {
  if constexpr (N >= 32) {
    float t[32];
    tmem_ld32(a, t);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = t[i];
    ld_cols<N - 32>(a + 32, v + 32);
  } else if constexpr (N == 16) {
    float t[16];
    tmem_ld16(a, t);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = t[i];
  }
}
template <int N>
TTT_DEV void st_cols(uint32_t a, const float* v) {
  if constexpr (N >= 32) {
    uint32_t t[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(v[i]);
    tmem_st32(a, t);
    st_cols<N - 32>(a + 32, v + 32);
  } else if constexpr (N == 16) {
    uint32_t t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(v[i]);
    tmem_st16(a, t);
  }
}

struct Range3 {
  int n_ring, m_lo, J;
};
TTT_DEV Range3 range3(const AttnArgs& a, int qt) {
  Range3 r;
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

template <int DH, bool SPLIT>
__global__ void __launch_bounds__(kF3Threads, 1)
    attn_fwd3_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tQl,
                     const __grid_constant__ CUtensorMap tKr, const __grid_constant__ CUtensorMap tKrl,
                     const __grid_constant__ CUtensorMap tVr, const __grid_constant__ CUtensorMap tVrl,
                     const __grid_constant__ CUtensorMap tKo, const __grid_constant__ CUtensorMap tKol,
                     const __grid_constant__ CUtensorMap tVo, const __grid_constant__ CUtensorMap tVol,
                     const AttnArgs a) {
  using C = F3Cfg<DH, SPLIT>;
  constexpr int HO = DH / 2;  // output columns per softmax thread
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // swizzled tiles need a 1024-B aligned base; report, do nothing else
    if (threadIdx.x == 0 && a.err) atomicCAS(a.err, 0, (int)DERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;         // 1
  uint64_t* k_full = bars + 1;     // 2
  uint64_t* k_empty = bars + 3;    // 2
  uint64_t* v_full = bars + 5;     // 2
  uint64_t* v_empty = bars + 7;    // 2
  uint64_t* s_full = bars + 9;     // 2 (per score buffer)
  uint64_t* p_full = bars + 11;    // 2 (per score buffer)
  uint64_t* o_done = bars + 13;    // 1: one phase per P V product
  uint64_t* o_final = bars + 14;   // 1: the last P V product
  uint64_t* pairbar = bars + 15;   // 4: the two softmax warps of one TMEM lane quadrant
  uint64_t* drain = bars + 19;     // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem + C::XCH_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = (int)blockIdx.x + a.qt0, h = blockIdx.y;
  const Range3 tr = range3(a, qt);
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
      mbar_init(&p_full[i], 256);
    }
    mbar_init(o_done, 1);
    mbar_init(o_final, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&pairbar[i], 64);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S buffers [0,128) and [128,256); O [256, 256 + DH)
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
      mbar_expect_tx(q_full, C::NOP * C::TILE);
      load_tile3<C::NATOM>(smem + C::Q_OFF, &tQ, q_full, col0, 128 * qt);
      if (SPLIT) load_tile3<C::NATOM>(smem + C::Q_OFF + C::TILE, &tQl, q_full, col0, 128 * qt);
      for (int j = 0; j < J; ++j) {
        const int s = j & 1;
        const uint32_t par = (uint32_t)((j >> 1) & 1);
        bool own;
        const int row0 = tile_row0(j, own);
        if (!mbar_wait(&k_empty[s], par ^ 1u, abort_flag, a.err, DERR_TIMEOUT_PRODUCER)) break;
        uint8_t* kd = smem + C::K_OFF + s * C::NOP * C::TILE;
        mbar_expect_tx(&k_full[s], C::NOP * C::TILE);
        load_tile3<C::NATOM>(kd, own ? &tKo : &tKr, &k_full[s], col0, row0);
        if (SPLIT) load_tile3<C::NATOM>(kd + C::TILE, own ? &tKol : &tKrl, &k_full[s], col0, row0);
        kiss |= 1u << s;
        kpar = (kpar & ~(1u << s)) | (par << s);
        if (!mbar_wait(&v_empty[s], par ^ 1u, abort_flag, a.err, DERR_TIMEOUT_PRODUCER)) break;
        uint8_t* vd = smem + C::V_OFF + s * C::NOP * C::TILE;
        mbar_expect_tx(&v_full[s], C::NOP * C::TILE);
        load_tile3<C::NATOM>(vd, own ? &tVo : &tVr, &v_full[s], col0, row0);
        if (SPLIT) load_tile3<C::NATOM>(vd + C::TILE, own ? &tVol : &tVrl, &v_full[s], col0, row0);
        viss |= 1u << s;
        vpar = (vpar & ~(1u << s)) | (par << s);
      }
      // no TMA write may still be in flight when the CTA exits
      drain3(q_full, 0, a.err);
      for (int s = 0; s < 2; ++s) {
        if (kiss & (1u << s)) drain3(&k_full[s], (kpar >> s) & 1u, a.err);
        if (viss & (1u << s)) drain3(&v_full[s], (vpar >> s) & 1u, a.err);
      }
    }
  } else if (warp == 1) {  // MMA issuer: the whole warp, one elected lane issues
    auto wait_all = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, a.err, DERR_TIMEOUT_MMA));
    };
    constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idPV = idesc_bf16(128, DH, 0, 1);
    const uint32_t q0 = smem_u32(smem + C::Q_OFF);
    auto issue_s = [&](int j) {  // S_j = Q K_j^T into score buffer j & 1
      const int s = j & 1;
      const uint32_t kb = smem_u32(smem + C::K_OFF + s * C::NOP * C::TILE);
      const uint32_t d = tmem + (uint32_t)(s * 128);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        mma_bf16_w(d, kdesc3(q0, kk), kdesc3(kb, kk), idS, kk ? 1u : 0u);
        if (SPLIT) {
          mma_bf16_w(d, kdesc3(q0, kk), kdesc3(kb + C::TILE, kk), idS, 1u);
          mma_bf16_w(d, kdesc3(q0 + C::TILE, kk), kdesc3(kb, kk), idS, 1u);
        }
      }
      mma_commit_w(&s_full[s]);
      mma_commit_w(&k_empty[s]);
    };
    bool ok = J > 0 && wait_all(q_full, 0) &&
              wait_all(&k_full[0], 0);
    if (ok) {
      tc_fence_after();
      issue_s(0);
    }
    for (int j = 0; j < J && ok; ++j) {
      const int s = j & 1;
      if (j + 1 < J) {  // next scores into the other buffer, whose P V product was issued last round
        if (!wait_all(&k_full[s ^ 1], (uint32_t)(((j + 1) >> 1) & 1))) break;
        tc_fence_after();
        issue_s(j + 1);
      }
      if (!wait_all(&p_full[s], (uint32_t)((j >> 1) & 1))) break;
      if (!wait_all(&v_full[s], (uint32_t)((j >> 1) & 1))) break;
      tc_fence_after();
      // O += P_j V_j; P_j: keys 0-63 in columns [0,32) (+ remainders [32,64)), keys 64-127 in
      // columns [64,96) (+ [96,128)) of score buffer s
      const uint32_t pb = tmem + (uint32_t)(s * 128);
      const uint32_t vb = smem_u32(smem + C::V_OFF + s * C::NOP * C::TILE);
      const uint32_t d = tmem + 256u;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t pa = pb + (uint32_t)((kk < 4 ? 0 : 64) + 8 * (kk & 3));
        mma_bf16_ts_w(d, pa, mndesc3(vb, kk), idPV, (j | kk) ? 1u : 0u);
        if (SPLIT) {
          mma_bf16_ts_w(d, pa, mndesc3(vb + C::TILE, kk), idPV, 1u);
          mma_bf16_ts_w(d, pa + 32u, mndesc3(vb, kk), idPV, 1u);
        }
      }
      mma_commit_w(o_done);
      mma_commit_w(&v_empty[s]);
      if (j == J - 1) mma_commit_w(o_final);
    }
    mma_commit_w(drain);  // every MMA issued above has finished once this arrives
    drain3(drain, 0, a.err);
  } else {  // --------------------------------------------------- softmax: two threads per query row
    const int hf = (warp - 2) >> 2;  // which 64 key columns (and which half of the head dim)
    const int qd = warp & 3;         // TMEM lane quadrant of this warp
    const int r = qd * 32 + lane;    // query row within the tile
    const long p = a.pos0 + 128L * qt + r;
    const bool rvalid = 128 * qt + r < a.n;
    const float sl2 = a.scale_log2;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const uint32_t tO = trow + 256u + (uint32_t)(hf * HO);
    const int b0 = hf * 64;
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;

    // exchange a per-row value with the partner thread (same row, other half); phase ph
    auto exchange = [&](float mine, int ph, float& other) -> bool {
      xch[(ph & 1) * 256 + hf * 128 + r] = mine;
      mbar_arrive(&pairbar[qd]);
      const bool got = mbar_wait(&pairbar[qd], ph & 1, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) return false;
      other = xch[(ph & 1) * 256 + (hf ^ 1) * 128 + r];
      return true;
    };

    for (int j = 0; j < J; ++j) {
      const int s = j & 1;
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
      const bool full = __all_sync(0xffffffffu, c_lo <= b0 && c_hi >= b0 + 63);
      const bool got = mbar_wait(&s_full[s], (uint32_t)((j >> 1) & 1), abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = trow + (uint32_t)(s * 128 + b0);
      float v[64];
      tmem_ld64(tS, v);  // one load, one wait
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
      if (full) {
#pragma unroll
        for (int e = 0; e < 64; ++e) m8[e & 7] = fmaxf(m8[e & 7], v[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          v[e] = (b0 + e >= c_lo && b0 + e <= c_hi) ? v[e] : -INFINITY;
          m8[e & 7] = fmaxf(m8[e & 7], v[e]);
        }
      }
      const float mx =
          fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      float mo;
      if (!exchange(mx, j, mo)) {
        ok = false;
        break;
      }
      const float m_tile = fmaxf(mx, mo) * sl2;
      const bool grow = m_tile > m_used + kLazy;  // the same on both halves of a row
      if (__any_sync(0xffffffffu, grow) && j > 0) {
        // O holds the products up to tile j-2 for sure; wait for P_{j-1} V_{j-1}, then rescale
        const bool g2 = mbar_wait(o_done, (uint32_t)((j - 1) & 1), abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
        if (!__all_sync(0xffffffffu, g2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float alpha = grow ? ex2_approx(m_used - m_tile) : 1.0f;
        float o[HO];
        ld_cols<HO>(tO, o);
#pragma unroll
        for (int e = 0; e < HO; ++e) o[e] *= alpha;
        st_cols<HO>(tO, o);
        l_run *= alpha;
      }
      if (grow) m_used = m_tile;
      const float m_use = (m_used == -INFINITY) ? 0.f : m_used;
      float r4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t ph[32], pl[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x0 = ex2_approx(fmaf(v[2 * e], sl2, -m_use));
        const float x1 = ex2_approx(fmaf(v[2 * e + 1], sl2, -m_use));
        r4[e & 3] += x0 + x1;
        __nv_bfloat162 t = __floats2bfloat162_rn(x0, x1);
        ph[e] = *reinterpret_cast<uint32_t*>(&t);
        if (SPLIT) {
          const float2 f = __bfloat1622float2(t);
          pl[e] = pack_bf16(x0 - f.x, x1 - f.y);
        }
      }
      tmem_st32(trow + (uint32_t)(s * 128 + b0), ph);  // over this thread's own (already read) S columns
      if (SPLIT) tmem_st32(trow + (uint32_t)(s * 128 + b0 + 32), pl);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[s]);
      l_run += (r4[0] + r4[1]) + (r4[2] + r4[3]);
    }
    float l_other = 0.f;
    if (J > 0 && ok && exchange(l_run, J, l_other)) {
      const bool got = mbar_wait(o_final, 0, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (__all_sync(0xffffffffu, got)) {
        tc_fence_after();
        float o[HO];
        ld_cols<HO>(tO, o);
        const float lt = l_run + l_other;
        const float inv = lt > 0.f ? 1.0f / lt : 0.f;
        if (rvalid) {
          const long orow = (long)(128 * qt + r) * a.ldo + col0 + hf * HO;
#pragma unroll
          for (int c = 0; c < HO / 8; ++c) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float x0 = o[c * 8 + 2 * e] * inv, x1 = o[c * 8 + 2 * e + 1] * inv;
              __nv_bfloat162 t = __floats2bfloat162_rn(x0, x1);
              hw[e] = *reinterpret_cast<uint32_t*>(&t);
              const float2 f = __bfloat1622float2(t);
              lw[e] = pack_bf16(x0 - f.x, x1 - f.y);
            }
            *reinterpret_cast<uint4*>(a.o_hi + orow + c * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            if (a.o_lo) *reinterpret_cast<uint4*>(a.o_lo + orow + c * 8) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
          if (a.lse && hf == 0) a.lse[(long)h * a.n + 128 * qt + r] = (m_used == -INFINITY ? 0.f : m_used) + log2f(lt);
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
int launch_fwd3(const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  using C = F3Cfg<DH, SPLIT>;
  auto kern = attn_fwd3_kernel<DH, SPLIT>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return (int)e;
    attr = true;
  }
  dim3 grid((a.n + 127) / 128 - a.qt0, a.H);
  return (int)launch_k(kern, grid, dim3(kF3Threads), C::SMEM, st, m.q, m.ql, m.kr, m.krl, m.vr, m.vrl, m.ko, m.kol,
                       m.vo, m.vol, a);
}

}  // namespace

int attn_fwd3_run(const AttnMaps& m, const AttnArgs& a, bool split, cudaStream_t st) {
  if (a.n <= 0) return 0;
  if (split) {
    switch (a.dh) {
      case 32: return launch_fwd3<32, true>(m, a, st);
      case 64: return launch_fwd3<64, true>(m, a, st);
    }
    return (int)cudaErrorInvalidValue;
  }
  switch (a.dh) {
    case 32: return launch_fwd3<32, false>(m, a, st);
    case 64: return launch_fwd3<64, false>(m, a, st);
    case 96: return launch_fwd3<96, false>(m, a, st);
    case 128: return launch_fwd3<128, false>(m, a, st);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace ttt

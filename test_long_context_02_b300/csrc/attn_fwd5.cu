// Sliding-window causal attention forward, bf16 operands: one 128-query tile per
// CTA, two softmax warpgroups that take alternate key tiles.
//
// Same operation and geometry as attn_fwd.cu (pages: "把 Transformer 做成“终身学习者”",
// §4.2, the key/value cache holds only the window; §8 FAQ Q4, any k >= b): a
// query at absolute position p sees the keys at positions j with p - k < j <= p;
// keys before the chunk come from the k-slot cache (slot = position mod k), the
// chunk's own keys from its own K/V buffer; key tiles are 128 positions aligned
// to multiples of 128 in absolute position.
//
// The key tiles are split between two softmax warpgroups: warps 2-5 take the
// even tiles, warps 6-9 the odd ones, one thread per query row each.  Each
// warpgroup has its own TMEM score buffer (S_j of its tiles, overwritten by
// P_j as bf16 and read by the P V product from TMEM), its own output
// accumulator O_w and its own lazy running max m_w and row sum l_w, so the two
// softmax chains run concurrently and need no exchange until the end, where
// warps 2-5 merge the two partial results:
//   m = max(m_0, m_1),  O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)).
// Warp 0 loads Q once and K/V tiles through 2-stage TMA rings; warp 1 issues
// S_j = Q K_j^T into buffer j & 1 and O_{j&1} += P_j V_j, and S_{j+2} right after
// P_j V_j (which frees the buffer).
#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {

namespace {

constexpr float kLazy5 = 8.0f;
constexpr int kF5Threads = 320;

template <int DH>
struct F5Cfg {
  static constexpr int DP = DH <= 64 ? 64 : 128;
  static constexpr int NATOM = DP / 64;
  static constexpr int TILE = 128 * DP * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = TILE;             // 2 stages
  static constexpr int V_OFF = K_OFF + 2 * TILE; // 2 stages
  static constexpr int BAR_OFF = V_OFF + 2 * TILE;
  static constexpr int XCH_OFF = BAR_OFF + 256;  // [m_1 | l_1] of each row, fp32
  static constexpr int SMEM = XCH_OFF + 1024;
  static_assert(SMEM <= 232448, "attention forward exceeds shared memory");
};

TTT_DEV bool drain5(uint64_t* bar, uint32_t parity, int* err) {
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
TTT_DEV void load_tile5(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int a = 0; a < NATOM; ++a) tma_load_2d(dst + a * 16384, map, bar, col0 + 64 * a, row0);
}
TTT_DEV uint64_t kdesc5(uint32_t base, int kk) { return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024); }
TTT_DEV uint64_t mndesc5(uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 16384, 1024); }

struct Range5 {
  int n_ring, m_lo, J;
};
TTT_DEV Range5 range5(const AttnArgs& a, int qt) {
  Range5 r;
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

template <int DH>
__global__ void __launch_bounds__(kF5Threads, 1)
    attn_fwd5_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tKr,
                     const __grid_constant__ CUtensorMap tVr, const __grid_constant__ CUtensorMap tKo,
                     const __grid_constant__ CUtensorMap tVo, const AttnArgs a) {
  using C = F5Cfg<DH>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0 && a.err) atomicCAS(a.err, 0, (int)DERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;         // 1
  uint64_t* k_full = bars + 1;     // 2
  uint64_t* k_empty = bars + 3;    // 2
  uint64_t* v_full = bars + 5;     // 2
  uint64_t* v_empty = bars + 7;    // 2
  uint64_t* s_full = bars + 9;     // 2: per warpgroup (score buffer)
  uint64_t* p_full = bars + 11;    // 2
  uint64_t* o_final = bars + 13;   // 2: the last P V product of each warpgroup
  uint64_t* ml_full = bars + 15;   // 1: warpgroup 1's (m, l) are in shared memory
  uint64_t* drain = bars + 16;     // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem + C::XCH_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = (int)blockIdx.x + a.qt0, h = blockIdx.y;
  const Range5 tr = range5(a, qt);
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
    mbar_init(ml_full, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S_0 [0,128), S_1 [128,256), O_0 [256, 256+DH), O_1 [384, 384+DH)
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
      // order K_0, K_1, then V_j, K_{j+2}: K_{j+2} is needed right after P_j V_j, and only
      // waits for S_j to have been issued, so it must not queue behind V_{j+1}
      uint32_t kiss = 0, kpar = 0, viss = 0, vpar = 0;
      mbar_expect_tx(q_full, C::TILE);
      load_tile5<C::NATOM>(smem + C::Q_OFF, &tQ, q_full, col0, 128 * qt);
      auto load_k = [&](int j) -> bool {
        const int s = j & 1;
        const uint32_t par = (uint32_t)((j >> 1) & 1);
        bool own;
        const int row0 = tile_row0(j, own);
        if (!mbar_wait(&k_empty[s], par ^ 1u, abort_flag, a.err, DERR_TIMEOUT_PRODUCER)) return false;
        mbar_expect_tx(&k_full[s], C::TILE);
        load_tile5<C::NATOM>(smem + C::K_OFF + s * C::TILE, own ? &tKo : &tKr, &k_full[s], col0, row0);
        kiss |= 1u << s;
        kpar = (kpar & ~(1u << s)) | (par << s);
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j & 1;
        const uint32_t par = (uint32_t)((j >> 1) & 1);
        bool own;
        const int row0 = tile_row0(j, own);
        if (!mbar_wait(&v_empty[s], par ^ 1u, abort_flag, a.err, DERR_TIMEOUT_PRODUCER)) return false;
        mbar_expect_tx(&v_full[s], C::TILE);
        load_tile5<C::NATOM>(smem + C::V_OFF + s * C::TILE, own ? &tVo : &tVr, &v_full[s], col0, row0);
        viss |= 1u << s;
        vpar = (vpar & ~(1u << s)) | (par << s);
        return true;
      };
      bool ok = load_k(0) && (J < 2 || load_k(1));
      for (int j = 0; j < J && ok; ++j) ok = load_v(j) && (j + 2 >= J || load_k(j + 2));
      drain5(q_full, 0, a.err);
      for (int s = 0; s < 2; ++s) {
        if (kiss & (1u << s)) drain5(&k_full[s], (kpar >> s) & 1u, a.err);
        if (viss & (1u << s)) drain5(&v_full[s], (vpar >> s) & 1u, a.err);
      }
    }
  } else if (warp == 1) {  // ----------------------------- MMA issuer: the whole warp, one elected lane issues
    constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idPV = idesc_bf16(128, DH, 0, 1);
    const uint32_t q0 = smem_u32(smem + C::Q_OFF);
    auto wait_all = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, a.err, DERR_TIMEOUT_MMA));
    };
    auto issue_s = [&](int j) {  // S_j = Q K_j^T into buffer j & 1 (key stage j & 1)
      const int s = j & 1;
      const uint32_t kb = smem_u32(smem + C::K_OFF + s * C::TILE);
      const uint32_t d = tmem + (uint32_t)(s * 128);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) mma_bf16_w(d, kdesc5(q0, kk), kdesc5(kb, kk), idS, kk ? 1u : 0u);
      mma_commit_w(&s_full[s]);
      mma_commit_w(&k_empty[s]);
    };
    bool ok = J > 0 && wait_all(q_full, 0);
    for (int j = 0; j < 2 && j < J && ok; ++j) {
      ok = wait_all(&k_full[j], 0);
      if (ok) {
        tc_fence_after();
        issue_s(j);
      }
    }
    for (int j = 0; j < J && ok; ++j) {
      const int w = j & 1;
      const uint32_t par = (uint32_t)((j >> 1) & 1);
      if (!wait_all(&p_full[w], par)) break;
      if (!wait_all(&v_full[w], par)) break;
      tc_fence_after();
      const uint32_t pb = tmem + (uint32_t)(w * 128);  // P_j as bf16 pairs over the first 64 columns of S_w
      const uint32_t vb = smem_u32(smem + C::V_OFF + w * C::TILE);
      const uint32_t d = tmem + 256u + (uint32_t)(w * 128);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_bf16_ts_w(d, pb + (uint32_t)(kk * 8), mndesc5(vb, kk), idPV, (j >= 2 || kk) ? 1u : 0u);
      mma_commit_w(&v_empty[w]);
      if (j + 2 >= J) mma_commit_w(&o_final[w]);
      if (j + 2 < J) {  // after P_j V_j in issue order: S_{j+2} reuses buffer w
        if (!wait_all(&k_full[w], (uint32_t)(((j + 2) >> 1) & 1))) break;
        tc_fence_after();
        issue_s(j + 2);
      }
    }
    mma_commit_w(drain);
    drain5(drain, 0, a.err);
  } else {  // ---------------------------------- softmax: warpgroup w takes key tiles w, w+2, ...
    const int w = (warp - 2) >> 2;
    const int qd = warp & 3;
    const int r = qd * 32 + lane;
    const long p = a.pos0 + 128L * qt + r;
    const bool rvalid = 128 * qt + r < a.n;
    const float sl2 = a.scale_log2;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)(w * 128);
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(w * 128);
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = w, t = 0; j < J; j += 2, ++t) {
      const bool own = j >= tr.n_ring;
      const long kpos0 = own ? a.pos0 + 128L * (j - tr.n_ring) : 128L * (tr.m_lo + j);
      int c_lo, c_hi;
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
      const bool got = mbar_wait(&s_full[w], (uint32_t)(t & 1), abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[128];
      tmem_ld128(tS, sv);  // the whole score row, one load and one wait
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
      if (full) {  // eight chains of three-input max
#pragma unroll
        for (int e = 0; e < 64; ++e) m8[e & 7] = fmax3(m8[e & 7], sv[2 * e], sv[2 * e + 1]);
      } else {
#pragma unroll
        for (int e = 0; e < 128; ++e) {
          sv[e] = (e >= c_lo && e <= c_hi) ? sv[e] : -INFINITY;
          m8[e & 7] = fmaxf(m8[e & 7], sv[e]);
        }
      }
      const float mx =
          fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float m_tile = mx * sl2;
      const bool grow = m_tile > m_used + kLazy5;
      const float alpha = grow ? ex2_approx(m_used - m_tile) : 1.0f;  // 0 while m_used is -inf
      if (grow) m_used = m_tile;
      const float m_use = (m_used == -INFINITY) ? 0.f : m_used;
      // P_j as bf16 pairs over the first 64 columns of S_w (keys 2q, 2q+1 in column q);
      // every score is already in registers
      // exp2(s * scale - m) on packed pairs: one fma.f32x2, two ex2, one add.f32x2 into
      // four packed row-sum chains, one bf16x2 conversion per pair of keys
      const uint64_t sc2 = f32x2(sl2, sl2), nm2 = f32x2(-m_use, -m_use);
      uint64_t r4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) r4[e] = f32x2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t u[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 y = f32x2_split(ffma2(f32x2(sv[32 * c + 2 * e], sv[32 * c + 2 * e + 1]), sc2, nm2));
          const float x0 = ex2_approx(y.x), x1 = ex2_approx(y.y);
          r4[e & 3] = fadd2(r4[e & 3], f32x2(x0, x1));
          u[e] = pack_bf16(x0, x1);
        }
        tmem_st16(tS + (uint32_t)(c * 16), u);
      }
      float r8[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 v = f32x2_split(r4[e]);
        r8[2 * e] = v.x;
        r8[2 * e + 1] = v.y;
      }
      if (__any_sync(0xffffffffu, grow) && t > 0) {
        // O_w holds every product of this warpgroup's earlier tiles: S_j was issued after
        // the last of them, and its completion (s_full) covers every earlier MMA
#pragma unroll
        for (int c = 0; c < DH / 32; ++c) {
          float o[32];
          tmem_ld32(tO + (uint32_t)(c * 32), o);
          uint32_t u[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(o[e] * alpha);
          tmem_st32(tO + (uint32_t)(c * 32), u);
        }
      }
      l_run = l_run * alpha + (((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7])));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[w]);
    }
    if (w == 1) {  // hand (m_1, l_1) to warpgroup 0
      xch[r] = ok ? m_used : -INFINITY;
      xch[128 + r] = ok ? l_run : 0.f;
      mbar_arrive(ml_full);
    } else {
      bool got = ok && mbar_wait(ml_full, 0, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      got = got && mbar_wait(&o_final[0], 0, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (J > 1) got = got && mbar_wait(&o_final[1], 0, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (__all_sync(0xffffffffu, got)) {
        tc_fence_after();
        const float m1 = xch[r], l1 = xch[128 + r];
        const float m = fmaxf(m_used, m1);
        const float mu = (m == -INFINITY) ? 0.f : m;
        const float a0 = ex2_approx(m_used - mu), a1 = (J > 1) ? ex2_approx(m1 - mu) : 0.f;
        const float lt = l_run * a0 + l1 * a1;
        const float inv = lt > 0.f ? 1.0f / lt : 0.f;
        const float s0 = a0 * inv, s1 = a1 * inv;
        const uint32_t tO1 = tmem + lane_off + 384u;
#pragma unroll
        for (int c = 0; c < DH / 32; ++c) {
          float o0[32], o1[32];
          tmem_ld32(tO + (uint32_t)(c * 32), o0);
          if (J > 1) {
            tmem_ld32(tO1 + (uint32_t)(c * 32), o1);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o1[e] = 0.f;
          }
          if (rvalid) {
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float x0 = o0[2 * e] * s0 + o1[2 * e] * s1, x1 = o0[2 * e + 1] * s0 + o1[2 * e + 1] * s1;
              __nv_bfloat162 t2 = __floats2bfloat162_rn(x0, x1);
              hw[e] = *reinterpret_cast<uint32_t*>(&t2);
              const float2 f = __bfloat1622float2(t2);
              lw[e] = pack_bf16(x0 - f.x, x1 - f.y);
            }
            const long orow = (long)(128 * qt + r) * a.ldo + col0 + c * 32;
            uint4* dst = reinterpret_cast<uint4*>(a.o_hi + orow);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(hw[4 * v], hw[4 * v + 1], hw[4 * v + 2], hw[4 * v + 3]);
            if (a.o_lo) {
              uint4* dl = reinterpret_cast<uint4*>(a.o_lo + orow);
#pragma unroll
              for (int v = 0; v < 4; ++v) dl[v] = make_uint4(lw[4 * v], lw[4 * v + 1], lw[4 * v + 2], lw[4 * v + 3]);
            }
          }
        }
        if (rvalid && a.lse) a.lse[(long)h * a.n + 128 * qt + r] = mu + log2f(lt);
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

template <int DH>
int launch_fwd5(const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  using C = F5Cfg<DH>;
  auto kern = attn_fwd5_kernel<DH>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return (int)e;
    attr = true;
  }
  dim3 grid((a.n + 127) / 128 - a.qt0, a.H);
  return (int)launch_k(kern, grid, dim3(kF5Threads), C::SMEM, st, m.q, m.kr, m.vr, m.ko, m.vo, a);
}

}  // namespace

int attn_fwd5_run(const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  if (a.n <= 0) return 0;
  switch (a.dh) {
    case 32: return launch_fwd5<32>(m, a, st);
    case 64: return launch_fwd5<64>(m, a, st);
    case 96: return launch_fwd5<96>(m, a, st);
    case 128: return launch_fwd5<128>(m, a, st);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace ttt

// Sliding-window causal attention forward on tcgen05 (one head, 128 queries per CTA).
//
// The queries are the chunk's own positions pos0 .. pos0+n-1; a query at p sees
// the keys at positions j with p - k < j <= p (pages: "把 Transformer 做成“终身学习者”",
// §4.2, the key/value cache holds an 8K window; §8 FAQ Q4, any k >= b).  Keys
// before pos0 come from the k-slot window cache (slot = position mod k); keys
// of the chunk itself come from the chunk's own K/V buffer.  Key tiles are 128
// positions wide and aligned to multiples of 128 in absolute position, so a
// cache tile never wraps (k % 128 == 0); masking is by absolute position.
//
// Warp roles: warp 0 loads Q once and K/V tiles by TMA (K one tile ahead of V),
// warp 1 issues S = Q K^T into one of two TMEM score buffers and O_j = P_j V_j
// into one of two TMEM output buffers, warps 2-5 (one query row per thread) run
// the online softmax in base 2: row max over S_j, P_j = exp2(S_j*c - m) written
// as bf16 to shared memory for the PV product, and O accumulated in registers
// as O <- (O + O_{j-1}) * exp2(m_{j-1} - m_j).  Output: O / l as bf16 rows, and
// the per-row log2-sum-exp m + log2(l) used by the backward.
#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace ttt {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int DH, bool SPLIT>
struct FCfg {
  static constexpr int DP = DH <= 64 ? 64 : 128;  // head width padded to whole 128-B atoms
  static constexpr int NATOM = DP / 64;
  static constexpr int TILE = 128 * DP * 2;
  static constexpr int NOP = SPLIT ? 2 : 1;
  static constexpr int KST = SPLIT ? 1 : 2;
  static constexpr int VST = SPLIT ? 1 : 2;
  static constexpr int NP = SPLIT ? 1 : 2;
  static constexpr int PB = 128 * 128 * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = NOP * TILE;
  static constexpr int V_OFF = K_OFF + KST * NOP * TILE;
  static constexpr int P_OFF = V_OFF + VST * NOP * TILE;
  static constexpr int BAR_OFF = P_OFF + NP * NOP * PB;
  static constexpr int XCH_OFF = BAR_OFF + 256;       // row-max / row-sum exchange, [2][2][128] fp32
  static constexpr int SMEM = XCH_OFF + 2048;          // dynamic smem must start 1024-aligned (checked)
  static_assert(SMEM <= 232448, "attention forward exceeds shared memory");
};

constexpr int kFwdThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 softmax (two per query row)

// Load N consecutive fp32 TMEM columns (N a multiple of 16) into v.
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

// Load a 128-row tile of one head: NATOM boxes of {64 cols, 128 rows}.
template <int NATOM>
TTT_DEV void load_head_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int a = 0; a < NATOM; ++a) tma_load_2d(dst + a * 16384, map, bar, col0 + 64 * a, row0);
}

// K-major operand (128 rows, 128-B swizzled atoms of 64 columns, 16 KB apart): k-step kk of 16.
TTT_DEV uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
// The same tile read as an MN-major operand (N = head dim), k-step kk of 16 rows.
TTT_DEV uint64_t mnmajor_desc(uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 16384, 1024); }

struct TileRange {
  int n_ring, m_lo;  // cache tiles: absolute positions [128(m_lo+j), +128)
  int J;             // total tiles (cache then own)
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

template <int DH, bool SPLIT>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tQl,
                    const __grid_constant__ CUtensorMap tKr, const __grid_constant__ CUtensorMap tKrl,
                    const __grid_constant__ CUtensorMap tVr, const __grid_constant__ CUtensorMap tVrl,
                    const __grid_constant__ CUtensorMap tKo, const __grid_constant__ CUtensorMap tKol,
                    const __grid_constant__ CUtensorMap tVo, const __grid_constant__ CUtensorMap tVol,
                    const AttnArgs a) {
  using C = FCfg<DH, SPLIT>;
  constexpr int HO = DH / 2;  // output columns per softmax thread
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the swizzled tiles need a 1024-B aligned base; report, do nothing else
    if (threadIdx.x == 0 && a.err) atomicCAS(a.err, 0, (int)DERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + C::KST;
  uint64_t* v_full = k_empty + C::KST;
  uint64_t* v_empty = v_full + C::VST;
  uint64_t* s_full = v_empty + C::VST;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + C::NP;
  uint64_t* o_empty = o_full + 2;
  uint64_t* pairbar = o_empty + 2;  // [4]: the two softmax warps of one TMEM lane quadrant
  uint64_t* drain = pairbar + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem + C::XCH_OFF);  // [parity][half][row]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y;
  const TileRange tr = tiles_for(a, qt);
  const int J = tr.J;
  const int col0 = h * DH;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::KST; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < C::VST; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&o_full[i], 1); mbar_init(&o_empty[i], 256); }
    for (int i = 0; i < C::NP; ++i) mbar_init(&p_full[i], 256);
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
  const uint32_t tmem = *tmem_slot;

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
      uint32_t kpar_iss = 0, vpar_iss = 0, kiss = 0, viss = 0;
      mbar_expect_tx(q_full, C::NOP * C::TILE);
      load_head_tile<C::NATOM>(smem + C::Q_OFF, &tQ, q_full, col0, 128 * qt);
      if (SPLIT) load_head_tile<C::NATOM>(smem + C::Q_OFF + C::TILE, &tQl, q_full, col0, 128 * qt);
      bool ok = true;
      for (int j = 0; j <= J && ok; ++j) {
        if (j < J) {
          const int s = j % C::KST;
          if (!mbar_wait(&k_empty[s], ((j / C::KST) & 1) ^ 1, abort_flag, a.err, DERR_TIMEOUT_PRODUCER)) break;
          bool own;
          const int row0 = tile_row0(j, own);
          uint8_t* dst = smem + C::K_OFF + s * C::NOP * C::TILE;
          mbar_expect_tx(&k_full[s], C::NOP * C::TILE);
          load_head_tile<C::NATOM>(dst, own ? &tKo : &tKr, &k_full[s], col0, row0);
          if (SPLIT) load_head_tile<C::NATOM>(dst + C::TILE, own ? &tKol : &tKrl, &k_full[s], col0, row0);
          kiss |= 1u << s;
          kpar_iss = (kpar_iss & ~(1u << s)) | (((uint32_t)(j / C::KST) & 1u) << s);
        }
        if (j >= 1) {
          const int jj = j - 1, s = jj % C::VST;
          if (!mbar_wait(&v_empty[s], ((jj / C::VST) & 1) ^ 1, abort_flag, a.err, DERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          bool own;
          const int row0 = tile_row0(jj, own);
          uint8_t* dst = smem + C::V_OFF + s * C::NOP * C::TILE;
          mbar_expect_tx(&v_full[s], C::NOP * C::TILE);
          load_head_tile<C::NATOM>(dst, own ? &tVo : &tVr, &v_full[s], col0, row0);
          if (SPLIT) load_head_tile<C::NATOM>(dst + C::TILE, own ? &tVol : &tVrl, &v_full[s], col0, row0);
          viss |= 1u << s;
          vpar_iss = (vpar_iss & ~(1u << s)) | (((uint32_t)(jj / C::VST) & 1u) << s);
        }
      }
      wait_drain(q_full, 0, a.err);
      for (int s = 0; s < C::KST; ++s)
        if (kiss & (1u << s)) wait_drain(&k_full[s], (kpar_iss >> s) & 1u, a.err);
      for (int s = 0; s < C::VST; ++s)
        if (viss & (1u << s)) wait_drain(&v_full[s], (vpar_iss >> s) & 1u, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // -------------------------------------------------------- MMA issuer
      constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(128, DH, 0, 1);
      const uint32_t q_base = smem_u32(smem + C::Q_OFF);
      auto issue_s = [&](int j) {
        const int s = j % C::KST;
        const uint32_t kb = smem_u32(smem + C::K_OFF + s * C::NOP * C::TILE);
        const uint32_t d = tmem + (uint32_t)((j & 1) * 128);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          mma_bf16(d, kmajor_desc(q_base, kk), kmajor_desc(kb, kk), idS, kk ? 1u : 0u);
          if (SPLIT) {
            mma_bf16(d, kmajor_desc(q_base, kk), kmajor_desc(kb + C::TILE, kk), idS, 1u);
            mma_bf16(d, kmajor_desc(q_base + C::TILE, kk), kmajor_desc(kb, kk), idS, 1u);
          }
        }
        mma_commit(&s_full[j & 1]);
        mma_commit(&k_empty[s]);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, a.err, DERR_TIMEOUT_MMA);
      if (ok) ok = mbar_wait(&k_full[0], 0, abort_flag, a.err, DERR_TIMEOUT_MMA);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; j < J && ok; ++j) {
        if (j + 1 < J) {
          const int s = (j + 1) % C::KST;
          if (!mbar_wait(&k_full[s], ((j + 1) / C::KST) & 1, abort_flag, a.err, DERR_TIMEOUT_MMA)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        const int pb = j % C::NP, vs = j % C::VST;
        if (!mbar_wait(&p_full[pb], (j / C::NP) & 1, abort_flag, a.err, DERR_TIMEOUT_MMA)) break;
        if (!mbar_wait(&v_full[vs], (j / C::VST) & 1, abort_flag, a.err, DERR_TIMEOUT_MMA)) break;
        if (!mbar_wait(&o_empty[j & 1], ((j >> 1) & 1) ^ 1, abort_flag, a.err, DERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        const uint32_t pbase = smem_u32(smem + C::P_OFF + pb * C::NOP * C::PB);
        const uint32_t vbase = smem_u32(smem + C::V_OFF + vs * C::NOP * C::TILE);
        const uint32_t d = tmem + 256u + (uint32_t)((j & 1) * C::DP);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_bf16(d, kmajor_desc(pbase, kk), mnmajor_desc(vbase, kk), idPV, kk ? 1u : 0u);
          if (SPLIT) {
            mma_bf16(d, kmajor_desc(pbase, kk), mnmajor_desc(vbase + C::TILE, kk), idPV, 1u);
            mma_bf16(d, kmajor_desc(pbase + C::PB, kk), mnmajor_desc(vbase, kk), idPV, 1u);
          }
        }
        mma_commit(&o_full[j & 1]);
        mma_commit(&v_empty[vs]);
      }
      mma_commit(drain);
      wait_drain(drain, 0, a.err);
    }
  } else {  // --------------------------------------------------- softmax: two threads per query row
    const int sw = warp - 2;
    const int hf = sw >> 2;          // which 64 key columns of each tile (and half of the head dim)
    const int qd = warp & 3;         // TMEM lane quadrant of this warp
    const int r = qd * 32 + lane;    // query row within the tile
    const long p = a.pos0 + 128L * qt + r;
    const bool rvalid = 128 * qt + r < a.n;
    const float sl2 = a.scale_log2;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    float o[HO];
#pragma unroll
    for (int i = 0; i < HO; ++i) o[i] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;

    auto accumulate = [&](int jp, float alpha) -> bool {  // O <- (O + O_jp) * alpha on this thread's columns
      const bool got = mbar_wait(&o_full[jp & 1], (jp >> 1) & 1, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) return false;
      tc_fence_after();
      float v[HO];
      tmem_ldn<HO>(trow + 256u + (uint32_t)((jp & 1) * C::DP + hf * HO), v);
#pragma unroll
      for (int i = 0; i < HO; ++i) o[i] = (o[i] + v[i]) * alpha;
      tc_fence_before();
      mbar_arrive(&o_empty[jp & 1]);
      return true;
    };
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
      long kpos0;
      const bool own = j >= tr.n_ring;
      kpos0 = own ? a.pos0 + 128L * (j - tr.n_ring) : 128L * (tr.m_lo + j);
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
      const int b0 = hf * 64;
      const bool full = __all_sync(0xffffffffu, c_lo <= b0 && c_hi >= b0 + 63);
      const bool got = mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[64];
      {
        const uint32_t sb = trow + (uint32_t)((j & 1) * 128 + b0);
        tmem_ldn<64>(sb, v);
      }
      float m8[8];  // eight independent max chains
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
      if (full) {
#pragma unroll
        for (int i = 0; i < 64; ++i) m8[i & 7] = fmaxf(m8[i & 7], v[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const bool valid = (b0 + i >= c_lo) && (b0 + i <= c_hi);
          v[i] = valid ? v[i] : -INFINITY;
          m8[i & 7] = fmaxf(m8[i & 7], v[i]);
        }
      }
      const float mx =
          fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      float mo;
      if (!exchange(mx, j, mo)) {
        ok = false;
        break;
      }
      const float m_new = fmaxf(m_run, fmaxf(mx, mo) * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m_run - m_use);
      if (C::NP == 1 && j > 0) {
        if (!accumulate(j - 1, alpha)) {
          ok = false;
          break;
        }
      }
      const int pb = j % C::NP;
      uint8_t* pbuf = smem + C::P_OFF + pb * C::NOP * C::PB + hf * 16384 + r * 128;
      float r4[4] = {0.f, 0.f, 0.f, 0.f};  // independent sum chains
#pragma unroll
      for (int u = 0; u < 8; ++u) {  // 8 x 16-B chunks: columns b0 + 8u .. b0 + 8u + 7 (128-B swizzle)
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = ex2_approx(fmaf(v[8 * u + 2 * e], sl2, -m_use));
          const float x1 = ex2_approx(fmaf(v[8 * u + 2 * e + 1], sl2, -m_use));
          r4[e] += x0 + x1;
          __nv_bfloat162 t = __floats2bfloat162_rn(x0, x1);
          hw[e] = *reinterpret_cast<uint32_t*>(&t);
          if (SPLIT) {
            float2 f = __bfloat1622float2(t);
            lw[e] = pack_bf16(x0 - f.x, x1 - f.y);
          }
        }
        uint8_t* dst = pbuf + ((u ^ (r & 7)) * 16);
        *reinterpret_cast<uint4*>(dst) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if (SPLIT) *reinterpret_cast<uint4*>(dst + C::PB) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&p_full[pb]);
      const float rs = (r4[0] + r4[1]) + (r4[2] + r4[3]);
      l_run = l_run * alpha + rs;
      if (C::NP == 2 && j > 0) {
        if (!accumulate(j - 1, alpha)) {
          ok = false;
          break;
        }
      }
      m_run = m_new;
    }
    float l_other = 0.f;
    if (J > 0 && ok && accumulate(J - 1, 1.0f) && exchange(l_run, J, l_other) && rvalid) {
      const float inv = 1.0f / (l_run + l_other);
      const long orow = (long)(128 * qt + r) * a.ldo + col0 + hf * HO;
#pragma unroll
      for (int c = 0; c < HO / 8; ++c) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = o[c * 8 + 2 * e] * inv, x1 = o[c * 8 + 2 * e + 1] * inv;
          __nv_bfloat162 t = __floats2bfloat162_rn(x0, x1);
          hw[e] = *reinterpret_cast<uint32_t*>(&t);
          float2 f = __bfloat1622float2(t);
          lw[e] = pack_bf16(x0 - f.x, x1 - f.y);
        }
        *reinterpret_cast<uint4*>(a.o_hi + orow + c * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if (a.o_lo) *reinterpret_cast<uint4*>(a.o_lo + orow + c * 8) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      if (a.lse && hf == 0) a.lse[(long)h * a.n + 128 * qt + r] = m_run + log2f(l_run + l_other);
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
int launch_fwd(const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  using C = FCfg<DH, SPLIT>;
  auto kern = attn_fwd_kernel<DH, SPLIT>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return (int)e;
    attr = true;
  }
  dim3 grid((a.n + 127) / 128, a.H);
  kern<<<grid, kFwdThreads, C::SMEM, st>>>(m.q, m.ql, m.kr, m.krl, m.vr, m.vrl, m.ko, m.kol, m.vo, m.vol, a);
  return (int)cudaGetLastError();
}

}  // namespace

int attn_fwd_run(const AttnMaps& m, const AttnArgs& a, bool split, cudaStream_t st) {
  if (a.n <= 0) return 0;
  // bf16 operands: the two-query-tile kernel when its grid makes two full waves
  if (!split && (long)((a.n + 255) / 256) * a.H >= 2L * num_sms()) return attn_fwd2_run(m, a, st);
  return attn_fwd3_run(m, a, split, st);
}

// The earlier one-tile kernel (P through shared memory, O in registers).
int attn_fwd1_run(const AttnMaps& m, const AttnArgs& a, bool split, cudaStream_t st) {
  if (a.n <= 0) return 0;
  if (split) {
    switch (a.dh) {
      case 32: return launch_fwd<32, true>(m, a, st);
      case 64: return launch_fwd<64, true>(m, a, st);
    }
    return (int)cudaErrorInvalidValue;
  }
  switch (a.dh) {
    case 32: return launch_fwd<32, false>(m, a, st);
    case 64: return launch_fwd<64, false>(m, a, st);
    case 96: return launch_fwd<96, false>(m, a, st);
    case 128: return launch_fwd<128, false>(m, a, st);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace ttt

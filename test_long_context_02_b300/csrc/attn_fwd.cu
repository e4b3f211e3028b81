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
  static constexpr int SMEM = BAR_OFF + 256 + 1024;
  static_assert(SMEM <= 232448, "attention forward exceeds shared memory");
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
__global__ void __launch_bounds__(192, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tQl,
                    const __grid_constant__ CUtensorMap tKr, const __grid_constant__ CUtensorMap tKrl,
                    const __grid_constant__ CUtensorMap tVr, const __grid_constant__ CUtensorMap tVrl,
                    const __grid_constant__ CUtensorMap tKo, const __grid_constant__ CUtensorMap tKol,
                    const __grid_constant__ CUtensorMap tVo, const __grid_constant__ CUtensorMap tVol,
                    const AttnArgs a) {
  using C = FCfg<DH, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
  uint64_t* drain = o_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y;
  const TileRange tr = tiles_for(a, qt);
  const int J = tr.J;
  const int col0 = h * DH;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::KST; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < C::VST; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&o_full[i], 1); mbar_init(&o_empty[i], 128); }
    for (int i = 0; i < C::NP; ++i) mbar_init(&p_full[i], 128);
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
  } else {  // -------------------------------------------------------------- softmax warps
    const int qd = warp & 3;
    const int r = qd * 32 + lane;
    const long p = a.pos0 + 128L * qt + r;
    const bool rvalid = 128 * qt + r < a.n;
    const float sl2 = a.scale_log2;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    float o[DH];
#pragma unroll
    for (int i = 0; i < DH; ++i) o[i] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;

    auto accumulate = [&](int jp, float alpha) -> bool {  // O <- (O + O_jp) * alpha
      const bool got = mbar_wait(&o_full[jp & 1], (jp >> 1) & 1, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) return false;
      tc_fence_after();
      const uint32_t ob = trow + 256u + (uint32_t)((jp & 1) * C::DP);
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        float v[32];
        tmem_ld32(ob + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c * 32 + i] = (o[c * 32 + i] + v[i]) * alpha;
      }
      tc_fence_before();
      mbar_arrive(&o_empty[jp & 1]);
      return true;
    };

    for (int j = 0; j < J && ok; ++j) {
      bool own;
      long kpos0;
      if (j < tr.n_ring) {
        own = false;
        kpos0 = 128L * (tr.m_lo + j);
      } else {
        own = true;
        kpos0 = a.pos0 + 128L * (j - tr.n_ring);
      }
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
      const bool full = (c_lo <= 0 && c_hi >= 127);
      const bool got = mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, a.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sb = trow + (uint32_t)((j & 1) * 128);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(sb + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int col = c * 32 + i;
          if (full || (col >= c_lo && col <= c_hi)) mx = fmaxf(mx, v[i]);
        }
      }
      const float m_new = fmaxf(m_run, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m_run - m_use);
      if (C::NP == 1 && j > 0) {
        if (!accumulate(j - 1, alpha)) {
          ok = false;
          break;
        }
      }
      const int pb = j % C::NP;
      uint8_t* pbuf = smem + C::P_OFF + pb * C::NOP * C::PB;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(sb + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int col = c * 32 + i;
          const bool valid = full || (col >= c_lo && col <= c_hi);
          v[i] = valid ? exp2f(v[i] * sl2 - m_use) : 0.f;
          rs += v[i];
        }
        // 4 x 16-B chunks of row r, columns 32c .. 32c+31 (128-B swizzle)
        const int atom = c >> 1;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ch = ((c & 1) * 4 + u) ^ (r & 7);
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
          uint8_t* dst = pbuf + atom * 16384 + r * 128 + ch * 16;
          *reinterpret_cast<uint4*>(dst) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          if (SPLIT) *reinterpret_cast<uint4*>(dst + C::PB) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&p_full[pb]);
      l_run = l_run * alpha + rs;
      if (C::NP == 2 && j > 0) {
        if (!accumulate(j - 1, alpha)) {
          ok = false;
          break;
        }
      }
      m_run = m_new;
    }
    if (J > 0 && ok) {
      if (accumulate(J - 1, 1.0f) && rvalid) {
        const float inv = 1.0f / l_run;
        const long orow = (long)(128 * qt + r) * a.ldo + col0;
#pragma unroll
        for (int c = 0; c < DH / 8; ++c) {
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
        if (a.lse) a.lse[(long)h * a.n + 128 * qt + r] = m_run + log2f(l_run);
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
  kern<<<grid, 192, C::SMEM, st>>>(m.q, m.ql, m.kr, m.krl, m.vr, m.vrl, m.ko, m.kol, m.vo, m.vol, a);
  return (int)cudaGetLastError();
}

}  // namespace

int attn_fwd_run(const AttnMaps& m, const AttnArgs& a, bool split, cudaStream_t st) {
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

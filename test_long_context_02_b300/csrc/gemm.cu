// Persistent warp-specialised tcgen05 GEMM with fused epilogues.
//
// Every dense contraction of the TTT-E2E inner-loop step runs here: the
// frozen QKV / O / MLP projections of the forward, the LM head (fused with the
// vocab-tiled softmax statistics of the cross-entropy and, in the backward,
// with the logit gradient), the activation-gradient (dX) products of the
// suffix blocks, and the fast-weight gradients dW = X^T dY whose epilogue
// applies the SGD step W <- W - eta*dW in place (pages: "把 Transformer 做成
// “终身学习者”", §4.2, one mini-batch gradient step on the last-quarter MLPs;
// "测试时训练：长上下文的持续学习", §2.1.2, theta <- theta - eta*grad).
//
// CTA = 10 warps: warp 0 issues TMA loads into a ring of shared-memory stages;
// warp 1 owns the TMEM accumulators and issues tcgen05.mma (the whole warp
// runs the loop, one lane chosen by elect.sync issues); warps 2-9 drain a
// 128 x BN fp32 accumulator from TMEM, two warps per 32-lane quadrant taking
// alternate 32-column chunks, and apply the epilogue while the MMA warp fills
// the other accumulator.
// Tiles are 128 x BN x 64 (bf16, 128-byte swizzle); operands are K-major or
// MN-major per call, so weights stay in one row-major copy for both x.W
// (MN-major B) and dY.W^T (K-major B), and dW = X^T dY reads activations
// MN-major without a transpose.  In split mode each operand is a bf16 pair
// (hi, lo) and every k-step issues hi*hi + hi*lo + lo*hi.
#include <cstdio>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace ttt {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kSmemBudget = 192 * 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kGeluC = 0.7978845608028654f;  // sqrt(2/pi)

template <int BN, bool SPLIT>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int NOP = SPLIT ? 2 : 1;
  static constexpr int STAGE = NOP * (A_BYTES + B_BYTES);
  static constexpr int STAGES = kSmemBudget / STAGE;
  static constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;  // power of two >= 2 accumulators
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
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

// tanh: the documented tanh.approx.f32 (about 2^-11 relative) when the result is
// rounded to one bf16, tanhf when a bf16 remainder keeps ~2^-17 of it.
TTT_DEV float tanh_sel(float u, bool exact) {
  if (exact) return tanhf(u);
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(u));
  return y;
}
TTT_DEV float gelu_f(float a, bool exact) {
  return 0.5f * a * (1.f + tanh_sel(kGeluC * (a + 0.044715f * a * a * a), exact));
}
TTT_DEV float gelu_grad_f(float a, bool exact) {
  const float t = tanh_sel(kGeluC * (a + 0.044715f * a * a * a), exact);
  return 0.5f * (1.f + t) + 0.5f * a * (1.f - t * t) * kGeluC * (1.f + 3.f * 0.044715f * a * a);
}

// Load one operand tile (rows x 64 of K) for K index k0 and M/N origin r0.
template <int ROWS>
TTT_DEV void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int r0, int k0, int mn) {
  if (!mn) {
    tma_load_2d(dst, map, bar, k0, r0);  // box {64 K, ROWS}
  } else {
#pragma unroll
    for (int j = 0; j < ROWS / 64; ++j) tma_load_2d(dst + j * (BK * 128), map, bar, r0 + 64 * j, k0);  // box {64, 64 K}
  }
}

TTT_DEV uint64_t tile_desc(uint32_t base, int kk, int mn) {
  return mn ? sdesc_sw128(base + kk * 2048, BK * 128, 1024) : sdesc_sw128(base + kk * 32, 16, 1024);
}

TTT_DEV void store_opnd(bf16* hi, bf16* lo, long off, float v) {
  bf16 h = __float2bfloat16_rn(v);
  hi[off] = h;
  if (lo) lo[off] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// 32 consecutive values of one row: vector path when the whole fragment is in range.
TTT_DEV void store_opnd32(bf16* hi, bf16* lo, long base, const float (&v)[32], int ncols) {
  if (ncols == 32) {
    uint32_t h[16], l[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      __nv_bfloat162 t = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      h[i] = *reinterpret_cast<uint32_t*>(&t);
      if (lo) {
        float2 f = __bfloat1622float2(t);
        l[i] = pack_bf16(v[2 * i] - f.x, v[2 * i + 1] - f.y);
      }
    }
    uint4* ph = reinterpret_cast<uint4*>(hi + base);
#pragma unroll
    for (int i = 0; i < 4; ++i) ph[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    if (lo) {
      uint4* pl = reinterpret_cast<uint4*>(lo + base);
#pragma unroll
      for (int i = 0; i < 4; ++i) pl[i] = make_uint4(l[4 * i], l[4 * i + 1], l[4 * i + 2], l[4 * i + 3]);
    }
  } else {  // ragged edge: predicated, fully unrolled (v stays in registers)
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) store_opnd(hi, lo, base + i, v[i]);
  }
}

// N (multiple of 8) consecutive values of one row as bf16 (+ remainders), 16-byte stores.
template <int N>
TTT_DEV void store_opnd_n(bf16* hi, bf16* lo, long base, const float* v) {
#pragma unroll
  for (int u = 0; u < N / 8; ++u) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 t = __floats2bfloat162_rn(v[8 * u + 2 * e], v[8 * u + 2 * e + 1]);
      h[e] = *reinterpret_cast<uint32_t*>(&t);
      if (lo) {
        float2 f = __bfloat1622float2(t);
        l[e] = pack_bf16(v[8 * u + 2 * e] - f.x, v[8 * u + 2 * e + 1] - f.y);
      }
    }
    *reinterpret_cast<uint4*>(hi + base + 8 * u) = make_uint4(h[0], h[1], h[2], h[3]);
    if (lo) *reinterpret_cast<uint4*>(lo + base + 8 * u) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

TTT_DEV void store_f32_32(float* p, const float (&v)[32], int ncols) {
  if (ncols == 32) {
    float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) p[i] = v[i];
  }
}

// out[i] += v[i] for 32 consecutive fp32 values (vector reductions when the fragment is whole).
TTT_DEV void red_add_f32_32(float* p, const float (&v)[32], int ncols) {
  if (ncols == 32) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p + 4 * i), "f"(v[4 * i]), "f"(v[4 * i + 1]),
                   "f"(v[4 * i + 2]), "f"(v[4 * i + 3])
                   : "memory");
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) atomicAdd(p + i, v[i]);
  }
}

TTT_DEV void load_f32_32(const float* p, float (&v)[32], int ncols) {
  if (ncols == 32) {
    const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 t = q[i];
      v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = i < ncols ? p[i] : 0.f;
  }
}

constexpr int kGemmThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue (two per TMEM lane quadrant)
constexpr int kXposeBytes = 8 * 32 * 33 * 4;  // elementwise epilogues: a 32 x 33 fp32 buffer per epilogue warp

template <int BN, bool SPLIT, int EPI, int DH>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tAl,
                const __grid_constant__ CUtensorMap tB, const __grid_constant__ CUtensorMap tBl, const GemmArgs g) {
  using C = Cfg<BN, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // elementwise epilogues: one 32 x 33 fp32 transpose buffer per epilogue warp, after the barriers
  float* xpose = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE + 256);
  constexpr bool kCoalesced = EPI == EPI_F32 || EPI == EPI_OPND || EPI == EPI_RESID || EPI == EPI_GELU ||
                              EPI == EPI_GELU_BWD || EPI == EPI_SGD;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (g.M + BM - 1) / BM, nt = (g.N + BN - 1) / BN, ntiles = mt * nt;
  const int nk = (g.K + BK - 1) / BK;
  // work unit u = (output tile u % ntiles, K slice u / ntiles); slices > 1 only for
  // the F32 / RESID epilogues, which then add their partial sums atomically
  const int ks = g.ksplit > 1 ? g.ksplit : 1;
  const int nunits = ntiles * ks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 256);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tA);
    tma_prefetch(&tB);
    if (SPLIT) {
      tma_prefetch(&tAl);
      tma_prefetch(&tBl);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the predecessor kernel's outputs are complete and visible from here on
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------- TMA producer
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      uint32_t issued = 0;  // bit s: stage s has a fill in flight or landed
      uint32_t iss_par = 0; // bit s: parity of that fill
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int t = u % ntiles, sl = u / ntiles;
        const int m0 = (t % mt) * BM, n0 = (t / mt) * BN;
        const int kb0 = (int)((long)sl * nk / ks), kb1 = (int)((long)(sl + 1) * nk / ks);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, g.err, DERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::STAGE;
          mbar_expect_tx(&full[s], C::STAGE);
          load_tile<BM>(st, &tA, &full[s], m0, kb * BK, g.a_mn);
          load_tile<BN>(st + C::A_BYTES, &tB, &full[s], n0, kb * BK, g.b_mn);
          if (SPLIT) {
            load_tile<BM>(st + C::A_BYTES + C::B_BYTES, &tAl, &full[s], m0, kb * BK, g.a_mn);
            load_tile<BN>(st + 2 * C::A_BYTES + C::B_BYTES, &tBl, &full[s], n0, kb * BK, g.b_mn);
          }
          issued |= 1u << s;
          iss_par = (iss_par & ~(1u << s)) | (ph << s);
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // no TMA write may still be in flight when the CTA exits
      for (int i = 0; i < C::STAGES; ++i)
        if (issued & (1u << i)) wait_drain(&full[i], (iss_par >> i) & 1u, g.err);
    }
  } else if (warp == 1) {  // --------------------- MMA issuer: the whole warp, one elected lane issues
    const uint32_t idesc = idesc_bf16(BM, BN, g.a_mn, g.b_mn);
    auto wait_all = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, g.err, DERR_TIMEOUT_MMA));
    };
    int s = 0;
    uint32_t ph = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++it) {
      const int sl = u / ntiles;
      const int kb0 = (int)((long)sl * nk / ks), kb1 = (int)((long)(sl + 1) * nk / ks);
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!wait_all(&tempty[buf], (use & 1u) ^ 1u)) break;
      tc_fence_after();
      const uint32_t dt = tmem + (uint32_t)(buf * BN);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_all(&full[s], ph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + s * C::STAGE);
        const uint32_t b = a + C::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t da = tile_desc(a, kk, g.a_mn), db = tile_desc(b, kk, g.b_mn);
          mma_bf16_w(dt, da, db, idesc, (kb > kb0 || kk) ? 1u : 0u);
          if (SPLIT) {
            const uint64_t dal = tile_desc(a + C::A_BYTES + C::B_BYTES, kk, g.a_mn);
            const uint64_t dbl = tile_desc(a + 2 * C::A_BYTES + C::B_BYTES, kk, g.b_mn);
            mma_bf16_w(dt, da, dbl, idesc, 1u);
            mma_bf16_w(dt, dal, db, idesc, 1u);
          }
        }
        mma_commit_w(&empty[s]);
        if (++s == C::STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit_w(&tfull[buf]);
    }
    mma_commit_w(drain);  // every MMA issued above has finished once this arrives
    wait_drain(drain, 0, g.err);
  } else {  // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;   // the two warps of a quadrant take alternate column chunks
    const bool exact = g.ol != nullptr; // bf16 remainders are kept: full-precision transcendentals
    int it = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++it) {
      const int t = u % ntiles;
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      const bool got = mbar_wait(&tfull[buf], use & 1u, abort_flag, g.err, DERR_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) break;  // warp-uniform: tcgen05.ld below is .sync.aligned
      tc_fence_after();
      const int mtile = t % mt, ntile = t / mt;
      const int row = mtile * BM + q * 32 + lane;
      const int n0 = ntile * BN;
      const bool rok = row < g.M;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      float ce_m = -INFINITY, ce_s = 0.f;
      int tg = -1;
      float lse_r = 0.f;
      if (EPI == EPI_CE_FWD || EPI == EPI_CE_BWD) {
        if (rok) tg = g.tgt[row];
        if (EPI == EPI_CE_BWD && rok) lse_r = g.lse[row];
        if (EPI == EPI_CE_BWD) ce_s = g.scale_dev ? *g.scale_dev : g.scale;
      }
      if constexpr (EPI == EPI_QKV_ROPE) {
        // The tile holds BN / DH whole heads of one section (q, k or v) of the
        // [q | k | v] product; q and k are rotated (rotate-half pairs i, i + DH/2,
        // angle table row = token row) and all three written as bf16 operands.
        const int sec = n0 / g.rd;
        const int scol = n0 - sec * g.rd;
        bf16* oh = sec == 0 ? g.rq_h : (sec == 1 ? g.rk_h : g.rv_h);
        bf16* ol = sec == 0 ? g.rq_l : (sec == 1 ? g.rk_l : g.rv_l);
#pragma unroll 1
        for (int hh = half; hh < BN / DH; hh += 2) {
          float v[DH];
#pragma unroll
          for (int c = 0; c < DH / 32; ++c) {
            float t[32];
            tmem_ld32(taddr + (uint32_t)(hh * DH + c * 32), t);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 * c + i] = t[i];
          }
          if (!rok) continue;
          if (sec < 2) {
            const float4* c4 = reinterpret_cast<const float4*>(g.rcs + (long)row * (DH / 2));
            const float4* s4 = reinterpret_cast<const float4*>(g.rsn + (long)row * (DH / 2));
#pragma unroll
            for (int i4 = 0; i4 < DH / 8; ++i4) {
              const float4 cc = c4[i4], ss = s4[i4];
              const float cv[4] = {cc.x, cc.y, cc.z, cc.w}, sv[4] = {ss.x, ss.y, ss.z, ss.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 4 * i4 + e;
                const float x1 = v[i], x2 = v[i + DH / 2];
                v[i] = x1 * cv[e] - x2 * sv[e];
                v[i + DH / 2] = x2 * cv[e] + x1 * sv[e];
              }
            }
          }
          store_opnd_n<DH>(oh, ol, (long)row * g.rd + scol + hh * DH, v);
        }
      } else if constexpr (kCoalesced) {
        // Elementwise epilogues with coalesced global traffic: the accumulator (one row
        // per lane) goes through a 32 x 33 shared-memory transpose so that each lane then
        // owns 4 consecutive columns of rows lr, lr+4, ..., lr+28 of the warp's 32 rows,
        // and every load, store or reduction of the warp covers four whole 128-B row
        // segments.  The epilogue's fp32 operand (residual, GELU argument, weights) is
        // fetched one chunk ahead in the same layout.
        float* xs = xpose + (warp - 2) * (32 * 33);
        const int r0 = mtile * BM + q * 32;
        const int lr = lane >> 3, lc = (lane & 7) * 4;
        const bool sliced = (EPI == EPI_F32 || EPI == EPI_RESID) && ks > 1;
        constexpr bool kIn = EPI == EPI_RESID || EPI == EPI_GELU_BWD || EPI == EPI_SGD;
        const float* gin = EPI == EPI_RESID ? g.resid : (EPI == EPI_GELU_BWD ? g.aux : g.w32);
        const long ldin = EPI == EPI_RESID ? g.ldr : (EPI == EPI_GELU_BWD ? g.ldaux : g.ldw);
        float4 pn[8] = {};
        auto load_in = [&](int c0) {
          if constexpr (kIn) {
            if (sliced) return;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = r0 + lr + 4 * i;
              pn[i] = (rr < g.M && c0 + lc + 3 < g.N)
                          ? *reinterpret_cast<const float4*>(gin + (long)rr * ldin + c0 + lc)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        };
        // one element of the epilogue: acc -> (fp32 result, bf16-operand result)
        auto elem = [&](float acc, float in, float& f32, float& opnd) {
          if (EPI == EPI_F32) { f32 = acc; }
          else if (EPI == EPI_OPND) { opnd = acc; }
          else if (EPI == EPI_RESID) { f32 = in + acc; }
          else if (EPI == EPI_GELU) { f32 = acc; opnd = gelu_f(acc, exact); }
          else if (EPI == EPI_GELU_BWD) { opnd = acc * gelu_grad_f(in, exact); }
          else if (EPI == EPI_SGD) { f32 = in - g.eta * acc; opnd = f32; }
        };
        float* out32 = EPI == EPI_SGD ? g.w32 : g.out32;
        const long ld32 = EPI == EPI_SGD ? g.ldw : g.ldo32;
        bf16* oh = EPI == EPI_SGD ? g.wh : g.oh;
        bf16* ol = EPI == EPI_SGD ? g.wl : g.ol;
        const long ldh = EPI == EPI_SGD ? g.ldw : g.ldo;
        constexpr bool kF32Out = EPI == EPI_F32 || EPI == EPI_RESID || EPI == EPI_GELU || EPI == EPI_SGD;
        constexpr bool kOpndOut = EPI == EPI_OPND || EPI == EPI_GELU || EPI == EPI_GELU_BWD || EPI == EPI_SGD;
        load_in(n0 + half * 32);
#pragma unroll 1
        for (int c = half; c < BN / 32; c += 2) {
          const int c0 = n0 + c * 32;
          float v[32];
          tmem_ld32(taddr + (uint32_t)(c * 32), v);
#pragma unroll
          for (int j = 0; j < 32; ++j) xs[lane * 33 + j] = v[j];
          __syncwarp();
          float4 in4[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) in4[i] = pn[i];
          if (c + 2 < BN / 32) load_in(c0 + 64);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = lr + 4 * i, rr = r0 + rl;
            if (rr >= g.M || c0 + lc >= g.N) continue;
            const float* a4 = xs + rl * 33 + lc;
            const long o32 = (long)rr * ld32 + c0 + lc, oh_off = (long)rr * ldh + c0 + lc;
            if (c0 + lc + 3 < g.N) {
              const float inv[4] = {in4[i].x, in4[i].y, in4[i].z, in4[i].w};
              float f[4] = {0.f, 0.f, 0.f, 0.f}, o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int e = 0; e < 4; ++e) elem(a4[e], inv[e], f[e], o[e]);
              if (sliced) {
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(g.out32 + o32), "f"(a4[0]),
                             "f"(a4[1]), "f"(a4[2]), "f"(a4[3])
                             : "memory");
                continue;
              }
              if (kF32Out && out32) *reinterpret_cast<float4*>(out32 + o32) = make_float4(f[0], f[1], f[2], f[3]);
              if (kOpndOut) {
                __nv_bfloat162 t0 = __floats2bfloat162_rn(o[0], o[1]), t1 = __floats2bfloat162_rn(o[2], o[3]);
                uint2 hv;
                hv.x = *reinterpret_cast<uint32_t*>(&t0);
                hv.y = *reinterpret_cast<uint32_t*>(&t1);
                *reinterpret_cast<uint2*>(oh + oh_off) = hv;
                if (ol) {
                  const float2 f0 = __bfloat1622float2(t0), f1 = __bfloat1622float2(t1);
                  uint2 lv;
                  lv.x = pack_bf16(o[0] - f0.x, o[1] - f0.y);
                  lv.y = pack_bf16(o[2] - f1.x, o[3] - f1.y);
                  *reinterpret_cast<uint2*>(ol + oh_off) = lv;
                }
              }
            } else {  // ragged right edge: scalar, the operand read directly
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (c0 + lc + e >= g.N) continue;
                if (sliced) {
                  atomicAdd(g.out32 + o32 + e, a4[e]);
                  continue;
                }
                const float in = kIn ? gin[(long)rr * ldin + c0 + lc + e] : 0.f;
                float f = 0.f, o = 0.f;
                elem(a4[e], in, f, o);
                if (kF32Out && out32) out32[o32 + e] = f;
                if (kOpndOut) store_opnd(oh, ol, oh_off + e, o);
              }
            }
          }
          __syncwarp();
        }
      } else {
      // Global operand of the epilogue (residual, GELU argument, fp32 weights), fetched
      // one chunk ahead so that its latency overlaps the current chunk's work.
      constexpr bool kLoads = EPI == EPI_RESID || EPI == EPI_GELU_BWD || EPI == EPI_SGD;
      const float* gsrc = EPI == EPI_RESID ? g.resid : (EPI == EPI_GELU_BWD ? g.aux : g.w32);
      const long gld = EPI == EPI_RESID ? g.ldr : (EPI == EPI_GELU_BWD ? g.ldaux : g.ldw);
      const bool do_loads = kLoads && !(EPI == EPI_RESID && ks > 1);
      float nxt[32];
      if (do_loads && rok && n0 + half * 32 < g.N)
        load_f32_32(gsrc + (long)row * gld + n0 + half * 32, nxt, min(32, g.N - n0 - half * 32));
      // CE_FWD keeps one running (max, sum) per row: the first warp of each quadrant does all chunks
      const int c_first = EPI == EPI_CE_FWD ? 0 : half;
      const int c_step = EPI == EPI_CE_FWD ? 1 : 2;
#pragma unroll 1
      for (int c = c_first; c < BN / 32 && !(EPI == EPI_CE_FWD && half); c += c_step) {
        float v[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), v);
        const int c0 = n0 + c * 32;
        const int ncols = min(32, g.N - c0);
        float cur[32];
        if (do_loads) {
#pragma unroll
          for (int i = 0; i < 32; ++i) cur[i] = nxt[i];
          const int cn = n0 + (c + 2) * 32;
          if (rok && c + 2 < BN / 32 && cn < g.N) load_f32_32(gsrc + (long)row * gld + cn, nxt, min(32, g.N - cn));
        }
        if (!rok || ncols <= 0) continue;
        if ((EPI == EPI_F32 || EPI == EPI_RESID) && ks > 1) {
          // K slice: add the partial sum (out32 holds 0, or the residual, before the first slice lands)
          red_add_f32_32(g.out32 + (long)row * g.ldo32 + c0, v, ncols);
        } else if (EPI == EPI_F32) {
          store_f32_32(g.out32 + (long)row * g.ldo32 + c0, v, ncols);
        } else if (EPI == EPI_OPND) {
          store_opnd32(g.oh, g.ol, (long)row * g.ldo + c0, v, ncols);
        } else if (EPI == EPI_RESID) {
#pragma unroll
          for (int i = 0; i < 32; ++i) cur[i] += v[i];
          store_f32_32(g.out32 + (long)row * g.ldo32 + c0, cur, ncols);
        } else if (EPI == EPI_GELU) {
          if (g.out32) store_f32_32(g.out32 + (long)row * g.ldo32 + c0, v, ncols);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i], exact);
          store_opnd32(g.oh, g.ol, (long)row * g.ldo + c0, v, ncols);
        } else if (EPI == EPI_GELU_BWD) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= gelu_grad_f(cur[i], exact);
          store_opnd32(g.oh, g.ol, (long)row * g.ldo + c0, v, ncols);
        } else if (EPI == EPI_SGD) {
          float* wp = g.w32 + (long)row * g.ldw + c0;
#pragma unroll
          for (int i = 0; i < 32; ++i) cur[i] -= g.eta * v[i];
          store_f32_32(wp, cur, ncols);
          store_opnd32(g.wh, g.wl, (long)row * g.ldw + c0, cur, ncols);
        } else if (EPI == EPI_CE_FWD) {
          float mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < ncols) mx = fmaxf(mx, v[i]);
          const float mn = fmaxf(ce_m, mx);
          float s = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < ncols) s += exp2f((v[i] - mn) * kLog2e);
          ce_s = ce_s * exp2f((ce_m - mn) * kLog2e) + s;
          ce_m = mn;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c0 + i == tg) g.zt[row] = v[i];
        } else if (EPI == EPI_CE_BWD) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p = exp2f((v[i] - lse_r) * kLog2e);
            v[i] = (tg >= 0) ? (p - ((c0 + i == tg) ? 1.f : 0.f)) * ce_s : 0.f;
          }
          store_opnd32(g.oh, g.ol, (long)row * g.ldo + c0, v, ncols);
        }
      }
      }
      if (EPI == EPI_CE_FWD && rok && half == 0) g.part[(long)ntile * g.M + row] = make_float2(ce_m, ce_s);
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
// Operand rows along M (or N) = `rows`, reduction length K.
bool operand_map(CUtensorMap* m, const bf16* p, const Opnd& o, int rows, int K, int box_rows) {
  if (!o.mn) return make_map(m, p, (uint64_t)K, (uint64_t)rows, (uint64_t)o.ld, (uint32_t)box_rows);
  return make_map(m, p, (uint64_t)rows, (uint64_t)K, (uint64_t)o.ld, 64u);
}

template <int BN, bool SPLIT, int EPI, int DH = 0>
int launch(const CUtensorMap& a, const CUtensorMap& al, const CUtensorMap& b, const CUtensorMap& bl,
           const GemmArgs& g, cudaStream_t st) {
  using C = Cfg<BN, SPLIT>;
  auto kern = gemm_kernel<BN, SPLIT, EPI, DH>;
  constexpr bool kCo = EPI == EPI_F32 || EPI == EPI_OPND || EPI == EPI_RESID || EPI == EPI_GELU ||
                      EPI == EPI_GELU_BWD || EPI == EPI_SGD;
  constexpr int SMEM = C::SMEM + (kCo ? kXposeBytes : 0);
  static_assert(SMEM <= 232448, "GEMM exceeds shared memory");
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return (int)e;
    attr_set = true;
  }
  const int tiles = ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN) * (g.ksplit > 1 ? g.ksplit : 1);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return (int)launch_k(kern, dim3(grid), dim3(kGemmThreads), SMEM, st, a, al, b, bl, g);
}

template <int BN, bool SPLIT>
int dispatch_epi(int epi, const CUtensorMap& a, const CUtensorMap& al, const CUtensorMap& b,
                 const CUtensorMap& bl, const GemmArgs& g, cudaStream_t st) {
  switch (epi) {
    case EPI_F32: return launch<BN, SPLIT, EPI_F32>(a, al, b, bl, g, st);
    case EPI_OPND: return launch<BN, SPLIT, EPI_OPND>(a, al, b, bl, g, st);
    case EPI_RESID: return launch<BN, SPLIT, EPI_RESID>(a, al, b, bl, g, st);
    case EPI_GELU: return launch<BN, SPLIT, EPI_GELU>(a, al, b, bl, g, st);
    case EPI_GELU_BWD: return launch<BN, SPLIT, EPI_GELU_BWD>(a, al, b, bl, g, st);
    case EPI_SGD: return launch<BN, SPLIT, EPI_SGD>(a, al, b, bl, g, st);
    case EPI_CE_FWD: return launch<BN, SPLIT, EPI_CE_FWD>(a, al, b, bl, g, st);
    case EPI_CE_BWD: return launch<BN, SPLIT, EPI_CE_BWD>(a, al, b, bl, g, st);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace

// Tile width for N: the one that needs the fewest tile-columns of work per SM
// (waves x BN), preferring the wider tile on a tie.
// Weight of a tile width in the cost model: its MMA rate per byte of shared memory
// against the 256-wide tile (measured ~0.6 for 128 wide; 192 wide reads 11 % more
// operand bytes per product).
double bn_weight(int bn) { return bn == 256 ? 1.0 : (bn == 192 ? 1.1 : 1.6); }

int pick_bn(int M, int N) {
  const int sms = num_sms();
  const long mt = (M + BM - 1) / BM;
  if (N <= 128) return 128;
  int best = 256;
  double bc = -1;
  for (int bn : {256, 192, 128}) {  // waves x tile width x weight; the wider tile on a tie
    const long t = mt * ((N + bn - 1) / bn);
    const double c = (double)((t + sms - 1) / sms) * bn * bn_weight(bn);
    if (bc < 0 || c < bc) {
      bc = c;
      best = bn;
    }
  }
  return best;
}

// Tile width of the fused QKV + RoPE product for head width dh and model width d
// (whole heads per tile, tiles never straddle the q / k / v sections), 0 if none.
int qkv_rope_bn(int dh, int d, bool split) {
  if (split && dh > 64) return 0;
  const int cand[3] = {256, 192, 128};
  for (int bn : cand) {
    if (bn % dh || d % bn) continue;
    if (bn == 192 && dh != 96) continue;
    if (dh != 32 && dh != 64 && dh != 96 && dh != 128) continue;
    return bn;
  }
  return 0;
}

template <bool SPLIT>
int launch_qkv_rope(int bn, int dh, const CUtensorMap& a, const CUtensorMap& al, const CUtensorMap& b,
                    const CUtensorMap& bl, const GemmArgs& g, cudaStream_t st) {
  if (bn == 256 && dh == 32) return launch<256, SPLIT, EPI_QKV_ROPE, 32>(a, al, b, bl, g, st);
  if (bn == 256 && dh == 64) return launch<256, SPLIT, EPI_QKV_ROPE, 64>(a, al, b, bl, g, st);
  if (bn == 128 && dh == 32) return launch<128, SPLIT, EPI_QKV_ROPE, 32>(a, al, b, bl, g, st);
  if (bn == 128 && dh == 64) return launch<128, SPLIT, EPI_QKV_ROPE, 64>(a, al, b, bl, g, st);
  if constexpr (!SPLIT) {
    if (bn == 192 && dh == 96) return launch<192, false, EPI_QKV_ROPE, 96>(a, al, b, bl, g, st);
    if (bn == 256 && dh == 128) return launch<256, false, EPI_QKV_ROPE, 128>(a, al, b, bl, g, st);
    if (bn == 128 && dh == 128) return launch<128, false, EPI_QKV_ROPE, 128>(a, al, b, bl, g, st);
  }
  return (int)cudaErrorInvalidValue;
}

int gemm_qkv_rope(const Opnd& A, const Opnd& B, GemmArgs g, int dh, bool split, cudaStream_t st) {
  if (g.M <= 0) return 0;
  const int bn = qkv_rope_bn(dh, g.rd, split);
  if (bn == 0 || g.N != 3 * g.rd || !g.rcs || !g.rsn || !g.rq_h || !g.rk_h || !g.rv_h)
    return (int)cudaErrorInvalidValue;
  if (split && (!A.lo || !B.lo || !g.rq_l || !g.rk_l || !g.rv_l)) return (int)cudaErrorInvalidValue;
  g.a_mn = A.mn;
  g.b_mn = B.mn;
  CUtensorMap a, al, b, bl;
  if (!operand_map(&a, A.hi, A, g.M, g.K, BM) || !operand_map(&b, B.hi, B, g.N, g.K, bn))
    return (int)cudaErrorInvalidValue;
  al = a;
  bl = b;
  if (split && (!operand_map(&al, A.lo, A, g.M, g.K, BM) || !operand_map(&bl, B.lo, B, g.N, g.K, bn)))
    return (int)cudaErrorInvalidValue;
  return split ? launch_qkv_rope<true>(bn, dh, a, al, b, bl, g, st) : launch_qkv_rope<false>(bn, dh, a, al, b, bl, g, st);
}

// Tile width and K slices for an M x N x K product: the fewest (waves x tile width x
// k-blocks per unit) per SM, preferring the wider tile and fewer slices on ties.
// Slices only when allowed (F32 / RESID epilogues) and each keeps >= 4 k-blocks;
// they pay off where the tiles fill the last wave poorly.
void choose_tiling(int M, int N, int K, bool allow_slices, int* bn_out, int* ks_out) {
  const long sms = num_sms();
  const long mt = (M + BM - 1) / BM, nk = (K + BK - 1) / BK;
  double best = -1;
  for (int bn : {256, 192, 128}) {
    if (bn > 128 && N <= 128) continue;
    const long tiles = mt * ((N + bn - 1) / bn);
    for (int ks = 1; ks <= (allow_slices ? 8 : 1); ++ks) {
      if (ks > 1 && nk / ks < 4) break;
      const long units = tiles * ks;
      // per unit: its k-blocks, plus about two k-blocks' worth for the atomic epilogue of a slice;
      // tile widths weighted as in pick_bn
      const double cost = (double)((units + sms - 1) / sms) * bn * bn_weight(bn) *
                          ((nk + ks - 1) / ks + (ks > 1 ? 2 : 0));
      if (best < 0 || cost < best) {
        best = cost;
        *bn_out = bn;
        *ks_out = ks;
      }
    }
  }
}

int gemm_run(int epi, const Opnd& A, const Opnd& B, GemmArgs g, bool split, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return 0;
  if (epi < 0 || epi >= EPI_COUNT || epi == EPI_QKV_ROPE) return (int)cudaErrorInvalidValue;
  if (split && (!A.lo || !B.lo)) return (int)cudaErrorInvalidValue;
  g.a_mn = A.mn;
  g.b_mn = B.mn;
  int bn = pick_bn(g.M, g.N), ks = 1;
  if ((epi == EPI_F32 || epi == EPI_RESID) && g.allow_ksplit) choose_tiling(g.M, g.N, g.K, true, &bn, &ks);
  g.ksplit = ks;
  if (ks > 1 && !g.out32_ready) {  // the slices add into out32: start it at 0 (F32) or at the residual (RESID)
    cudaError_t e;
    if (epi == EPI_F32)
      e = cudaMemset2DAsync(g.out32, (size_t)g.ldo32 * 4, 0, (size_t)g.N * 4, (size_t)g.M, st);
    else if (g.out32 != g.resid)
      e = cudaMemcpy2DAsync(g.out32, (size_t)g.ldo32 * 4, g.resid, (size_t)g.ldr * 4, (size_t)g.N * 4, (size_t)g.M,
                            cudaMemcpyDeviceToDevice, st);
    else
      e = cudaSuccess;
    if (e != cudaSuccess) return (int)e;
  }
  CUtensorMap a, al, b, bl;
  if (!operand_map(&a, A.hi, A, g.M, g.K, BM) || !operand_map(&b, B.hi, B, g.N, g.K, bn))
    return (int)cudaErrorInvalidValue;
  al = a;
  bl = b;
  if (split && (!operand_map(&al, A.lo, A, g.M, g.K, BM) || !operand_map(&bl, B.lo, B, g.N, g.K, bn)))
    return (int)cudaErrorInvalidValue;
  if (bn == 128)
    return split ? dispatch_epi<128, true>(epi, a, al, b, bl, g, st) : dispatch_epi<128, false>(epi, a, al, b, bl, g, st);
  if (bn == 192)
    return split ? dispatch_epi<192, true>(epi, a, al, b, bl, g, st) : dispatch_epi<192, false>(epi, a, al, b, bl, g, st);
  return split ? dispatch_epi<256, true>(epi, a, al, b, bl, g, st) : dispatch_epi<256, false>(epi, a, al, b, bl, g, st);
}

}  // namespace ttt

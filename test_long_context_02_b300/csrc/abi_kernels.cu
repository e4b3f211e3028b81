// C-ABI entry points of the individual kernels (include/ttt_kernels.h).
#include "ttt.h"
#include "ttt_kernels.h"
#include "kernels.h"
#include "attn.h"
#include "rowops.h"
#include "tmap.h"

#include <cmath>

using namespace ttt;

extern "C" int ttt_k_gemm(int epi, int M, int N, int K, const void* a_hi, const void* a_lo, int64_t lda, int a_mn,
                          const void* b_hi, const void* b_lo, int64_t ldb, int b_mn, int split,
                          const ttt_gemm_epilogue* e, void* stream) {
  if (!a_hi || !b_hi || !e || M < 0 || N < 0 || K < 0 || lda <= 0 || ldb <= 0) return TTT_ERR_ARG;
  if ((lda % 8) || (ldb % 8)) return TTT_ERR_ARG;
  if (split && (!a_lo || !b_lo)) return TTT_ERR_ARG;
  GemmArgs g;
  g.M = M; g.N = N; g.K = K;
  g.out32 = e->out32; g.ldo32 = (long)e->ldo32;
  g.oh = (bf16*)e->out_hi; g.ol = (bf16*)e->out_lo; g.ldo = (long)e->ldo;
  g.resid = e->resid; g.ldr = (long)e->ldr;
  g.aux = e->aux; g.ldaux = (long)e->ldaux;
  g.w32 = e->w32; g.wh = (bf16*)e->w_hi; g.wl = (bf16*)e->w_lo; g.ldw = (long)e->ldw; g.eta = e->eta;
  g.tgt = e->tgt; g.part = (float2*)e->part; g.zt = e->zt; g.lse = e->lse; g.scale = e->scale;
  g.err = e->err;
  g.allow_ksplit = e->allow_ksplit != 0;
  Opnd A, B;
  A.hi = (const bf16*)a_hi; A.lo = (const bf16*)a_lo; A.ld = (long)lda; A.mn = a_mn ? 1 : 0;
  B.hi = (const bf16*)b_hi; B.lo = (const bf16*)b_lo; B.ld = (long)ldb; B.mn = b_mn ? 1 : 0;
  const int r = gemm_run(epi, A, B, g, split != 0, (cudaStream_t)stream);
  return r == 0 ? TTT_OK : TTT_ERR_CUDA;
}

namespace {

bool map2(CUtensorMap* m, const void* p, int d, int rows) {
  return make_map(m, p, (uint64_t)d, (uint64_t)rows, (uint64_t)d, 128u);
}

bool attn_kernel_maps(AttnMaps* m, int n, int d, int window, bool split, const void* qh, const void* ql,
                      const void* kch, const void* kcl, const void* vch, const void* vcl, const void* koh,
                      const void* kol, const void* voh, const void* vol) {
  if (!map2(&m->q, qh, d, n) || !map2(&m->kr, kch, d, window) || !map2(&m->vr, vch, d, window) ||
      !map2(&m->ko, koh, d, n) || !map2(&m->vo, voh, d, n))
    return false;
  if (split)
    return map2(&m->ql, ql, d, n) && map2(&m->krl, kcl, d, window) && map2(&m->vrl, vcl, d, window) &&
           map2(&m->kol, kol, d, n) && map2(&m->vol, vol, d, n);
  m->ql = m->q; m->krl = m->kr; m->vrl = m->vr; m->kol = m->ko; m->vol = m->vo;
  return true;
}

int attn_check(int n, int H, int dh, int window, int64_t pos0, int split) {
  if (n < 1 || H < 1 || window < 1 || pos0 < 0 || n > window || window % 128) return TTT_ERR_ARG;
  if (dh % 16 || (dh != 32 && dh != 64 && dh != 96 && dh != 128) || (split && dh > 64)) return TTT_ERR_UNSUPPORTED;
  return TTT_OK;
}

}  // namespace

extern "C" int ttt_k_attn_fwd(int n, int H, int dh, int window, int64_t pos0, int split, const void* q_hi,
                              const void* q_lo, const void* kc_hi, const void* kc_lo, const void* vc_hi,
                              const void* vc_lo, const void* ko_hi, const void* ko_lo, const void* vo_hi,
                              const void* vo_lo, void* o_hi, void* o_lo, float* lse, int32_t* err, void* stream) {
  int r = attn_check(n, H, dh, window, pos0, split);
  if (r) return r;
  if (!q_hi || !kc_hi || !vc_hi || !ko_hi || !vo_hi || !o_hi) return TTT_ERR_ARG;
  const int d = H * dh;
  AttnMaps m;
  if (!attn_kernel_maps(&m, n, d, window, split, q_hi, q_lo, kc_hi, kc_lo, vc_hi, vc_lo, ko_hi, ko_lo, vo_hi, vo_lo))
    return TTT_ERR_ARG;
  AttnArgs a;
  a.n = n; a.H = H; a.dh = dh; a.window = window; a.pos0 = (long)pos0;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)dh));
  a.o_hi = (bf16*)o_hi; a.o_lo = (bf16*)o_lo; a.ldo = d; a.lse = lse; a.err = err;
  return attn_fwd_run(m, a, split != 0, (cudaStream_t)stream) == 0 ? TTT_OK : TTT_ERR_CUDA;
}

extern "C" int ttt_k_attn_bwd(int n, int H, int dh, int window, int64_t pos0, int split, const void* q_hi,
                              const void* q_lo, const void* kc_hi, const void* kc_lo, const void* vc_hi,
                              const void* vc_lo, const void* ko_hi, const void* ko_lo, const void* vo_hi,
                              const void* vo_lo, const void* do_hi, const void* do_lo, const float* lse,
                              const float* D, float* dq, float* dk, float* dv, int32_t* err, void* stream) {
  int r = attn_check(n, H, dh, window, pos0, split);
  if (r) return r;
  if (!q_hi || !kc_hi || !vc_hi || !ko_hi || !vo_hi || !do_hi || !lse || !D || !dq || !dk || !dv) return TTT_ERR_ARG;
  const int d = H * dh;
  AttnBwdMaps m;
  if (!attn_kernel_maps(&m.f, n, d, window, split, q_hi, q_lo, kc_hi, kc_lo, vc_hi, vc_lo, ko_hi, ko_lo, vo_hi,
                        vo_lo) ||
      !map2(&m.dO, do_hi, d, n))
    return TTT_ERR_ARG;
  if (split) {
    if (!map2(&m.dOl, do_lo, d, n)) return TTT_ERR_ARG;
  } else {
    m.dOl = m.dO;
  }
  AttnBwdArgs a;
  a.g.n = n; a.g.H = H; a.g.dh = dh; a.g.window = window; a.g.pos0 = (long)pos0;
  a.g.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)dh));
  a.g.err = err;
  a.lse = lse; a.D = D; a.dq = dq; a.dk = dk; a.dv = dv; a.ldg = d;
  a.scale = (float)(1.0 / std::sqrt((double)dh));
  return attn_bwd_run(m, a, split != 0, (cudaStream_t)stream) == 0 ? TTT_OK : TTT_ERR_CUDA;
}

extern "C" int ttt_k_attn_rowdot(int n, int H, int dh, const void* do_hi, const void* do_lo, const void* o_hi,
                                 const void* o_lo, float* D, void* stream) {
  if (n < 1 || H < 1 || dh % 8 || !do_hi || !o_hi || !D) return TTT_ERR_ARG;
  return rows_attn_rowdot((const bf16*)do_hi, (const bf16*)do_lo, (const bf16*)o_hi, (const bf16*)o_lo, n, H, dh, D,
                          (cudaStream_t)stream) == 0
             ? TTT_OK
             : TTT_ERR_CUDA;
}

// libttt host orchestrator: the C ABI of include/ttt.h.
//
// One context = one model (frozen weights in bf16, plus the bf16 remainders in
// the fp32-compute mode) and n_seqs independent sequences, each with its own
// k-slot key/value window cache per layer and its own fp32 fast weights
// (W_up, W_down of the last S blocks) with bf16 shadows used as GEMM operands.
// Up to kMaxLanes sequences run side by side, each on a lane: its own working
// buffers and streams, forked from the context stream and joined back into it.
//
// One inner-loop step of one sequence (pages: "把 Transformer 做成“终身学习者”：
// TTT-E2E 如何让大模型边用边学？", §4.2 and §4.4; "TTT-E2E技术：突破大语言模型上下文限制的新范式",
// §2.1), all on the lane's main stream unless noted:
//   forward  : embed; per block RMSNorm, QKV product, RoPE (+ own K/V), windowed
//              attention, O product + residual, RMSNorm, up product + GELU,
//              down product + residual; final RMSNorm; LM head fused with the
//              vocab-tiled cross-entropy statistics; mean loss.
//   backward : logit gradient (LM head recomputed) and its product with W_lm^T;
//              final RMSNorm backward; for the trainable blocks, last first:
//              dU = dY W_down^T (x GELU'), dW_down = U^T dY with the SGD step in
//              its epilogue, dXn = dA W_up^T, dW_up = Xn^T dA with the SGD step,
//              then (except for the first trainable block) RMSNorm backward,
//              dO = dH Wo^T, attention backward (which writes dQKV with RoPE's
//              rotation transposed), dXn = dQKV Wqkv^T, RMSNorm backward.  The
//              dW + SGD products run on the lane's third stream; every dX
//              product reads the weights before the step (the events order it
//              first); all gradients of the step are taken at the chunk's
//              starting weights.
//   commit   : the chunk's keys/values of every layer go into the window cache.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"
#include "rowops.h"
#include "tmap.h"
#include "ttt.h"

using namespace ttt;

namespace {

struct Pair {  // bf16 operand (hi) and remainder (lo, split mode only)
  bf16* hi = nullptr;
  bf16* lo = nullptr;
  Pair at(long off) const { return Pair{hi + off, lo ? lo + off : nullptr}; }
};

struct Seq {
  long pos = 0;
  Pair ring_k, ring_v;          // [L][k][d]
  float* up32 = nullptr;        // [S][d][f]
  float* down32 = nullptr;      // [S][f][d]
  Pair up16, down16;            // shadows
};

// Per-sequence working set of the chunk loop.  A lane runs one sequence at a
// time; a context with several sequences runs them on several lanes, each on
// its own streams, side by side on the GPU (lane 0's main stream is the
// context stream; the others fork from it and join back into it).
struct Lane {
  cudaStream_t st = nullptr;  // main stream of the lane
  bool own_st = false;        // st was created for the lane (lanes other than 0)
  int* tgt = nullptr;
  float *cs = nullptr, *sn = nullptr;
  float *x = nullptr, *xp = nullptr, *qkv = nullptr;
  Pair xn, q, o, u;
  // frozen-prefix pass outputs, double-buffered so the pass of the next group of chunks
  // can run on a second stream while the current group's trainable steps read theirs
  float* xpb[2] = {nullptr, nullptr};   // [R][d] residual stream after the frozen blocks (xpb[0] == xp)
  float* csb[2] = {nullptr, nullptr};   // angle tables [R][dh/2] (csb[0] == cs, snb[0] == sn)
  float* snb[2] = {nullptr, nullptr};
  Pair sxn;                             // [b][d] normalised attention input of the trainable blocks
  cudaStream_t st2 = nullptr;           // the frozen-prefix passes run ahead on this stream
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_pass[2] = {nullptr, nullptr}, ev_suf[2] = {nullptr, nullptr};
  // the fast-weight gradient products with their SGD step run on a third stream beside
  // the rest of the chunk's backward (nothing in it reads the updated weights)
  cudaStream_t st3 = nullptr;
  cudaEvent_t ev_dx = nullptr, ev_wu = nullptr;
  Pair kown, vown;           // [L][R][d]
  float *sx = nullptr, *sh = nullptr, *srs_a = nullptr, *srs_m = nullptr, *slse = nullptr, *sa = nullptr;
  Pair sq, so, sxm, su;
  Pair xf, dz;
  float *rs_f = nullptr, *zt = nullptr, *lse_row = nullptr, *loss_row = nullptr, *inv_nvalid = nullptr;
  float2* part = nullptr;
  float *dy = nullptr, *dxn = nullptr, *dh32 = nullptr, *D = nullptr;
  Pair dy16, da, dh16, do16, dqkv;
  float* sa_s = nullptr;     // dual-MLP: static pre-activations [S][b][f]
  Pair us, da_s;             // dual-MLP: static GELU output and its gradient [b][f]
};

}  // namespace

struct ttt_ctx {
  ttt_config cfg{};
  cudaStream_t st = nullptr;
  bool split = false, loaded = false, dual = false;
  std::string err;
  int L = 0, S = 0, d = 0, H = 0, dh = 0, f = 0, V = 0, k = 0, b = 0, B = 0;
  int G = 1, R = 0;  // chunks per frozen-prefix pass, and its rows G*b
  std::vector<void*> allocs;
  // frozen weights
  float* E = nullptr;        // [V][d]
  float* gains = nullptr;    // [2L+1][d]: g_attn(l), g_mlp(l), g_final
  Pair Wqkv, Wo, Wup, Wdown, Wlm;  // [L][d][3d], [L][d][d], [L-S][d][f], [L-S][f][d], [d][V]
  Pair Wup_s, Wdown_s;             // dual-MLP variant: static pair of the trainable blocks [S][d][f], [S][f][d]
  std::vector<Seq> seqs;
  std::vector<Lane> lanes;         // min(n_seqs, kMaxLanes) working sets
  bool concurrent = true;  // side streams and parallel lanes (ttt_set_concurrency)
  // per-call device scratch shared by the lanes
  int *tok = nullptr, *next = nullptr, *minus1 = nullptr, *derr = nullptr;
  float* loss_dev = nullptr;
  double* inv_freq = nullptr;
  float* zdec = nullptr;     // decoding: one row of logits [V]
  cudaEvent_t ev_fork = nullptr;  // lanes and side streams start after the context stream's earlier work
  // host whole-sequence entry point: device staging of tokens and losses (grown on demand)
  int* seq_tok = nullptr;
  float* seq_loss = nullptr;
  size_t seq_tok_cap = 0, seq_loss_cap = 0;
  // initial fast weights (device copy) for ttt_reset
  float *init_up = nullptr, *init_down = nullptr;
  // launch counting and optional per-class event timing
  int64_t launches = 0;
  uint64_t prof_mask = 0;   // bit i: bracket launches of kernel class i with events
  int prof_every = 1;       // ... one launch in prof_every of each such class
  int64_t prof_seen[64] = {};
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  struct ProfRec {
    int cls;
    cudaEvent_t a, b;
    double alg, exec, bytes;
    int nkern;
  };
  std::vector<ProfRec> recs;
  struct ProfAcc {
    int64_t launches = 0;
    double ms = 0, alg = 0, exec = 0, bytes = 0;
  };
  std::vector<ProfAcc> acc;
};
using ProfRec = ttt_ctx::ProfRec;

namespace {

// Rows of one frozen-prefix pass (whole chunks): large enough for full GEMM waves.
constexpr int kPrefixRows = 8192;
// Sequences of one context that run side by side (each lane holds one working set).
constexpr int kMaxLanes = 4;

int fail(ttt_ctx* c, int code, const std::string& msg) {
  if (c) c->err = msg;
  return code;
}

#define CK(expr)                                                                                  \
  do {                                                                                            \
    int _r = (int)(expr);                                                                         \
    if (_r != 0)                                                                                  \
      return fail(c, TTT_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString((cudaError_t)_r)); \
  } while (0)

template <typename T>
T* dalloc(ttt_ctx* c, size_t count, bool& ok) {
  void* p = nullptr;
  if (!ok) return nullptr;
  if (cudaMalloc(&p, count * sizeof(T) + 256) != cudaSuccess) {
    ok = false;
    cudaGetLastError();
    return nullptr;
  }
  cudaMemset(p, 0, count * sizeof(T) + 256);
  c->allocs.push_back(p);
  return static_cast<T*>(p);
}

Pair palloc(ttt_ctx* c, size_t count, bool& ok) {
  Pair p;
  p.hi = dalloc<bf16>(c, count, ok);
  if (c->split) p.lo = dalloc<bf16>(c, count, ok);
  return p;
}

Opnd opnd(const Pair& p, long ld, int mn) {
  Opnd o;
  o.hi = p.hi;
  o.lo = p.lo;
  o.ld = ld;
  o.mn = mn;
  return o;
}

bool attn_maps(AttnMaps* m, const Pair& q, const Pair& kr, const Pair& vr, const Pair& ko, const Pair& vo, int n,
               int d, int window) {
  auto mk = [&](CUtensorMap* t, const bf16* p, int rows) { return make_map(t, p, (uint64_t)d, (uint64_t)rows, d, 128); };
  bool ok = mk(&m->q, q.hi, n) && mk(&m->kr, kr.hi, window) && mk(&m->vr, vr.hi, window) && mk(&m->ko, ko.hi, n) &&
            mk(&m->vo, vo.hi, n);
  if (!ok) return false;
  if (q.lo) {
    ok = mk(&m->ql, q.lo, n) && mk(&m->krl, kr.lo, window) && mk(&m->vrl, vr.lo, window) && mk(&m->kol, ko.lo, n) &&
         mk(&m->vol, vo.lo, n);
  } else {
    m->ql = m->q;
    m->krl = m->kr;
    m->vrl = m->vr;
    m->kol = m->ko;
    m->vol = m->vo;
  }
  return ok;
}

// Kernel classes timed by the optional profiler (names exported by ttt_profile_read).
enum Cls : int {
  K_GEMM_QKV, K_ATTN_FWD, K_GEMM_O, K_GEMM_UP, K_GEMM_DOWN, K_CE_FWD, K_CE_BWD, K_LM_DX, K_MLP_DX, K_DW_SGD,
  K_ATTN_DX, K_ATTN_BWD, K_RMSNORM, K_ROPE, K_COMMIT, K_MISC, K_NCLS
};
const char* const kClsName[K_NCLS] = {
    "gemm_qkv", "attn_fwd", "gemm_o_resid", "gemm_up_gelu", "gemm_down_resid", "lmhead_ce_fwd",
    "lmhead_ce_bwd", "lmhead_dx", "gemm_mlp_dx", "gemm_dw_sgd", "gemm_attn_dx", "attn_bwd",
    "rmsnorm", "rope", "kv_commit", "misc"};

cudaEvent_t next_event(ttt_ctx* c) {
  if (c->ev_used == c->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    c->ev_pool.push_back(e);
  }
  return c->ev_pool[c->ev_used++];
}

// Run one launch site: count its kernels and, when profiling, bracket it with events
// recorded on the stream the site launches on.
template <class F>
int site(ttt_ctx* c, int cls, cudaStream_t sst, int nkern, double alg, double exec, double bytes, F&& f) {
  cudaEvent_t a = nullptr;
  if (((c->prof_mask >> cls) & 1u) && c->prof_seen[cls]++ % c->prof_every == 0 && (a = next_event(c)))
    cudaEventRecord(a, sst);
  const int r = f();
  if (a) {
    cudaEvent_t b = next_event(c);
    if (b) {
      cudaEventRecord(b, sst);
      c->recs.push_back(ProfRec{cls, a, b, alg, exec, bytes, nkern});
    }
  }
  c->launches += nkern;
  return r;
}

// RUN launches on the stream `st` of the enclosing scope; RUN_ON names the stream.
#define RUN_ON(sst, cls, nk, alg, exec, bytes, expr) \
  CK(site(c, cls, sst, nk, alg, exec, bytes, [&]() { return (int)(expr); }))
#define RUN(cls, nk, alg, exec, bytes, expr) RUN_ON(st, cls, nk, alg, exec, bytes, expr)

// Tiles of 128 keys visited by the attention kernels for query tile qt (as the kernels enumerate them).
long attn_tiles(long pos0, int n, int k, int qt) {
  long ring = 0;
  if (pos0 > 0) {
    const long lo = std::max(0L, pos0 + 128L * qt - k + 1);
    ring = (pos0 - 1) / 128 - lo / 128 + 1;
  }
  const int qend = std::min(n, 128 * qt + 128);
  return ring + (qend - 1) / 128 + 1;
}

// Window pairs (query, visible key) of n queries starting at absolute position pos0.
double window_pairs(long pos0, int n, int k) {
  double pairs = 0;
  for (long p = pos0; p < pos0 + n; ++p) pairs += (double)std::min<long>(p + 1, k);
  return pairs;
}
double tile_pairs(long pos0, int n, int k) {
  double t = 0;
  for (int qt = 0; qt < (n + 127) / 128; ++qt) t += 128.0 * 128.0 * attn_tiles(pos0, n, k, qt);
  return t;
}

// Forward of block l over the n chunk rows r0 .. r0+n-1 (absolute positions
// pos0+r0 ..., pos0 = the chunk's first position).  Blocks run with save =
// false (the frozen blocks, and the trainable ones during decoding) update the
// residual stream in place through the prefix-pass buffers; trainable blocks
// run with save = true (r0 = 0) keep what their backward needs in the suffix
// buffers and write xout.  si >= 0 selects the sequence's fast weights.
// xin / xout and the angle tables cs / sn point at row r0.
int layer_forward(ttt_ctx* c, Lane& ln, Seq& sq_, int l, int si, bool save, int n, int r0, long pos0, float* xin,
                  float* xout, const float* cs, const float* sn, cudaStream_t st) {
  const int d = c->d, H = c->H, dh = c->dh, f = c->f, k = c->k, b = c->b, R = c->R;
  const bool fast = si >= 0, suf = fast && save, sp = c->split;
  const double nn = n, dd = d, ff = f;
  const double ops = sp ? 3.0 : 1.0, eb = sp ? 4.0 : 2.0;
  const long ro = (long)r0 * d, rf = (long)r0 * f;
  float* hbuf = suf ? ln.sh + (long)si * b * d : xin;
  Pair xn_a = suf ? ln.sxn : ln.xn.at(ro);
  Pair q0 = suf ? ln.sq.at((long)si * b * d) : ln.q;  // row 0 of the chunk's queries / outputs
  Pair o0 = suf ? ln.so.at((long)si * b * d) : ln.o;
  Pair xn_m = suf ? ln.sxm.at((long)si * b * d) : ln.xn.at(ro);
  Pair ub = suf ? ln.su.at((long)si * b * f) : ln.u.at(rf);
  Pair ko0 = ln.kown.at((long)l * R * d), vo0 = ln.vown.at((long)l * R * d);
  Pair kr = sq_.ring_k.at((long)l * k * d), vr = sq_.ring_v.at((long)l * k * d);

  // with a separate output buffer, the norm also copies its input there: the start value
  // of the O product's K slices (x + o.Wo), so the product needs no copy of its own
  RUN(K_RMSNORM, 1, 0, 0, nn * dd * (4 + eb + (hbuf != xin ? 4 : 0)),
      rows_rmsnorm(xin, c->gains + (long)(2 * l) * d, c->cfg.rms_eps, n, d, xn_a.hi, xn_a.lo,
                   suf ? ln.srs_a + (long)si * b : nullptr, st, hbuf != xin ? hbuf : nullptr));
  Pair qw = q0.at(ro), kw = ko0.at(ro), vw = vo0.at(ro);
  if (qkv_rope_bn(dh, d, sp)) {  // RoPE and the q / own k / own v writes fused into the product's epilogue
    GemmArgs g;
    g.M = n; g.N = 3 * d; g.K = d; g.err = c->derr;
    g.rq_h = qw.hi; g.rq_l = qw.lo; g.rk_h = kw.hi; g.rk_l = kw.lo; g.rv_h = vw.hi; g.rv_l = vw.lo;
    g.rcs = cs; g.rsn = sn; g.rd = d;
    RUN(K_GEMM_QKV, 1, 6 * nn * dd * dd, 6 * nn * dd * dd * ops, 0,
        gemm_qkv_rope(opnd(xn_a, d, 0), opnd(c->Wqkv.at((long)l * d * 3 * d), 3 * d, 1), g, dh, sp, st));
  } else {
    GemmArgs g;
    g.M = n; g.N = 3 * d; g.K = d;
    g.out32 = ln.qkv; g.ldo32 = 3 * d; g.err = c->derr;
    RUN(K_GEMM_QKV, 1, 6 * nn * dd * dd, 6 * nn * dd * dd * ops, 0,
        gemm_run(EPI_F32, opnd(xn_a, d, 0), opnd(c->Wqkv.at((long)l * d * 3 * d), 3 * d, 1), g, sp, st));
    RUN(K_ROPE, 1, 0, 0, nn * dd * (12 + 3 * eb),
        rows_rope_qkv(ln.qkv, cs, sn, n, H, dh, qw.hi, qw.lo, kw.hi, kw.lo, vw.hi, vw.lo, st));
  }
  {  // queries r0 .. r0+n-1 over the cache and own keys 0 .. r0+n-1 (tiles before r0's are skipped)
    const int na = r0 + n;
    AttnMaps m;
    if (!attn_maps(&m, q0, kr, vr, ko0, vo0, na, d, k)) return fail(c, TTT_ERR_CUDA, "attention tensor maps");
    AttnArgs a;
    a.n = na; a.H = H; a.dh = dh; a.window = k; a.pos0 = pos0; a.qt0 = r0 / 128;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)dh));
    a.o_hi = o0.hi; a.o_lo = o0.lo; a.ldo = d;
    a.lse = suf ? ln.slse + (long)si * H * b : nullptr;
    a.err = c->derr;
    RUN(K_ATTN_FWD, 1, 4 * dd * window_pairs(pos0 + r0, n, k), 4 * dd * tile_pairs(pos0, na, k) * ops, 0,
        attn_fwd_run(m, a, sp, st));
  }
  {
    GemmArgs g;
    g.M = n; g.N = d; g.K = d;
    g.out32 = hbuf; g.ldo32 = d; g.resid = xin; g.ldr = d; g.err = c->derr; g.allow_ksplit = true;
    g.out32_ready = hbuf != xin;  // holds xin (the norm above copied it)
    RUN(K_GEMM_O, 1, 2 * nn * dd * dd, 2 * nn * dd * dd * ops, 0,
        gemm_run(EPI_RESID, opnd(o0.at(ro), d, 0), opnd(c->Wo.at((long)l * d * d), d, 1), g, sp, st));
  }
  RUN(K_RMSNORM, 1, 0, 0, nn * dd * (4 + eb + (xout != hbuf ? 4 : 0)),
      rows_rmsnorm(hbuf, c->gains + (long)(2 * l + 1) * d, c->cfg.rms_eps, n, d, xn_m.hi, xn_m.lo,
                   suf ? ln.srs_m + (long)si * b : nullptr, st, xout != hbuf ? xout : nullptr));
  {
    GemmArgs g;
    g.M = n; g.N = f; g.K = d;
    g.out32 = suf ? ln.sa + (long)si * b * f : nullptr;  // pre-activation kept for GELU' only when trainable
    g.ldo32 = f; g.oh = ub.hi; g.ol = ub.lo; g.ldo = f; g.err = c->derr;
    Pair w = fast ? sq_.up16.at((long)si * d * f) : c->Wup.at((long)l * d * f);
    RUN(K_GEMM_UP, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 0,
        gemm_run(EPI_GELU, opnd(xn_m, d, 0), opnd(w, f, 1), g, sp, st));
  }
  {
    GemmArgs g;
    g.M = n; g.N = d; g.K = f;
    g.out32 = xout; g.ldo32 = d; g.resid = hbuf; g.ldr = d; g.err = c->derr; g.allow_ksplit = true;
    g.out32_ready = xout != hbuf;  // holds h (the norm above copied it)
    Pair w = fast ? sq_.down16.at((long)si * f * d) : c->Wdown.at((long)l * f * d);
    RUN(K_GEMM_DOWN, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 0,
        gemm_run(EPI_RESID, opnd(ub, f, 0), opnd(w, d, 1), g, sp, st));
  }
  if (fast && c->dual) {  // the frozen static MLP of a trainable block, on the same normalised input
    Pair usb = ln.us.at(rf);
    GemmArgs g;
    g.M = n; g.N = f; g.K = d;
    g.out32 = suf ? ln.sa_s + (long)si * b * f : nullptr; g.ldo32 = f; g.oh = usb.hi; g.ol = usb.lo; g.ldo = f;
    g.err = c->derr;
    RUN(K_GEMM_UP, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 0,
        gemm_run(EPI_GELU, opnd(xn_m, d, 0), opnd(c->Wup_s.at((long)si * d * f), f, 1), g, sp, st));
    GemmArgs g2;  // y += u_s . W_down_s, in place over the block output
    g2.M = n; g2.N = d; g2.K = f;
    g2.out32 = xout; g2.ldo32 = d; g2.resid = xout; g2.ldr = d; g2.err = c->derr; g2.allow_ksplit = true;
    RUN(K_GEMM_DOWN, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 0,
        gemm_run(EPI_RESID, opnd(usb, f, 0), opnd(c->Wdown_s.at((long)si * f * d), d, 1), g2, sp, st));
  }
  return TTT_OK;
}

// The frozen blocks 0..L-S-1 of sequence s over n tokens (whole chunks, n <= R)
// starting at absolute position pos0.  Their outputs do not depend on the fast
// weights, so several chunks go through them in one pass; the suffix steps of
// those chunks then read their rows of ln.xp.  The frozen blocks' keys/values
// of all n tokens enter the window cache at the end of the pass (every query of
// the pass has already read the cache).
int prefix_pass(ttt_ctx* c, Lane& ln, int s, const int* tok, int n, long pos0, cudaStream_t st, int buf) {
  Seq& sq_ = c->seqs[s];
  float* xp = ln.xpb[buf];
  const int d = c->d, dh = c->dh, k = c->k, R = c->R;
  const int P0 = c->L - c->S;
  const double nn = n, dd = d;
  RUN(K_MISC, 1, 0, 0, nn * dd * 8, rows_embed(tok, n, c->E, c->V, d, xp, c->derr, st));
  RUN(K_ROPE, 1, 0, 0, nn * dh * 4, rows_rope_table(pos0, n, dh, c->inv_freq, ln.csb[buf], ln.snb[buf], st));
  for (int l = 0; l < P0; ++l) {
    const int r = layer_forward(c, ln, sq_, l, -1, false, n, 0, pos0, xp, xp, ln.csb[buf], ln.snb[buf], st);
    if (r != TTT_OK) return r;
  }
  if (P0 > 0) {
    const double cb = (double)P0 * nn * dd * 2 * 2;
    RUN(K_COMMIT, 1, 0, 0, cb, rows_commit(ln.kown.hi, sq_.ring_k.hi, (long)R * d, (long)k * d, P0, pos0, n, k, d, st));
    RUN(K_COMMIT, 1, 0, 0, cb, rows_commit(ln.vown.hi, sq_.ring_v.hi, (long)R * d, (long)k * d, P0, pos0, n, k, d, st));
    if (c->split) {
      RUN(K_COMMIT, 1, 0, 0, cb,
          rows_commit(ln.kown.lo, sq_.ring_k.lo, (long)R * d, (long)k * d, P0, pos0, n, k, d, st));
      RUN(K_COMMIT, 1, 0, 0, cb,
          rows_commit(ln.vown.lo, sq_.ring_v.lo, (long)R * d, (long)k * d, P0, pos0, n, k, d, st));
    }
  }
  return TTT_OK;
}

// One inner-loop step of sequence s for the chunk whose rows start at `row`
// within the last prefix pass: tokens tok[n], next target next[1] (device).
// Runs the trainable blocks forward, the loss, the backward through them with
// the fused SGD step, and commits their keys/values; the position advances by n.
int suffix_step(ttt_ctx* c, Lane& ln, int s, int row, const int* tok, int n, const int* next, float* loss_out, int buf = 0) {
  Seq& sq_ = c->seqs[s];
  cudaStream_t st = ln.st;
  const int L = c->L, S = c->S, d = c->d, H = c->H, dh = c->dh, f = c->f, V = c->V, k = c->k, b = c->b, R = c->R;
  const long pos0 = sq_.pos;
  const bool sp = c->split;
  const int P0 = L - S;  // first trainable block
  const float eta = c->cfg.eta;
  const double nn = n, dd = d, ff = f, VV = V;
  const double ops = sp ? 3.0 : 1.0;             // products per multiply in split mode
  const double eb = sp ? 4.0 : 2.0;              // bytes per operand element (hi [+ lo])
  const double pairs = window_pairs(pos0, n, k), tpairs = tile_pairs(pos0, n, k);
  const double own_pairs = nn * (nn + 1) / 2;
  const int nq = (n + 127) / 128;
  const double own_tile_pairs = 128.0 * 128.0 * nq * (nq + 1) / 2;
  const float* cs = ln.csb[buf] + (long)row * (dh / 2);
  const float* sn = ln.snb[buf] + (long)row * (dh / 2);

  RUN(K_MISC, 1, 0, 0, nn * 8, rows_targets(tok, n, next, V, ln.tgt, c->derr, st));

  // ------------------------------------------------------------------ forward
  for (int l = P0; l < L; ++l) {
    const int si = l - P0;
    float* xin = si == 0 ? ln.xpb[buf] + (long)row * d : ln.sx + (long)si * b * d;
    float* xout = (l + 1 < L) ? ln.sx + (long)(si + 1) * b * d : ln.x;
    const int r = layer_forward(c, ln, sq_, l, si, true, n, 0, pos0, xin, xout, cs, sn, st);
    if (r != TTT_OK) return r;
  }
  // final norm + LM head + cross-entropy statistics
  RUN(K_RMSNORM, 1, 0, 0, nn * dd * (4 + eb),
      rows_rmsnorm(ln.x, c->gains + (long)(2 * L) * d, c->cfg.rms_eps, n, d, ln.xf.hi, ln.xf.lo, ln.rs_f, st));
  const int bn = pick_bn(n, V);
  const int ntiles = (V + bn - 1) / bn;
  {
    GemmArgs g;
    g.M = n; g.N = V; g.K = d;
    g.tgt = ln.tgt; g.part = ln.part; g.zt = ln.zt; g.err = c->derr;
    RUN(K_CE_FWD, 1, 2 * nn * dd * VV, 2 * nn * dd * VV * ops, 0,
        gemm_run(EPI_CE_FWD, opnd(ln.xf, d, 0), opnd(c->Wlm, V, 1), g, sp, st));
  }
  RUN(K_MISC, 1, 0, 0, nn * ntiles * 8,
      rows_ce_combine(ln.part, ln.zt, ln.tgt, n, ntiles, ln.lse_row, ln.loss_row, st));
  RUN(K_MISC, 1, 0, 0, nn * 8, rows_loss_mean(ln.loss_row, ln.tgt, n, loss_out, ln.inv_nvalid, st));

  // ----------------------------------------------------------------- backward
  {  // dZ = (softmax(Z) - onehot(target)) / n_valid, logits recomputed tile by tile
    GemmArgs g;
    g.M = n; g.N = V; g.K = d;
    g.tgt = ln.tgt; g.lse = ln.lse_row; g.scale_dev = ln.inv_nvalid;
    g.oh = ln.dz.hi; g.ol = ln.dz.lo; g.ldo = V; g.err = c->derr;
    RUN(K_CE_BWD, 1, 0, 2 * nn * dd * VV * ops, 0,
        gemm_run(EPI_CE_BWD, opnd(ln.xf, d, 0), opnd(c->Wlm, V, 1), g, sp, st));
  }
  {
    GemmArgs g;
    g.M = n; g.N = d; g.K = V;
    g.out32 = ln.dxn; g.ldo32 = d; g.err = c->derr; g.allow_ksplit = true;
    g.out32_ready = true;  // dxn is zero between its uses (each reader clears it)
    RUN(K_LM_DX, 1, 2 * nn * dd * VV, 2 * nn * dd * VV * ops, 0,
        gemm_run(EPI_F32, opnd(ln.dz, V, 0), opnd(c->Wlm, V, 0), g, sp, st));
  }
  RUN(K_RMSNORM, 1, 0, 0, nn * dd * (12 + eb),
      rows_rmsnorm_bwd(ln.dxn, ln.x, c->gains + (long)(2 * L) * d, ln.rs_f, nullptr, n, d, ln.dy, ln.dy16.hi,
                       ln.dy16.lo, st, true));
  // The block's two dW + SGD products go to the third stream, after dXn (the last product
  // that reads the old W_up; dA read the old W_down before it), behind one event; one
  // wait brings them back before dY is overwritten (they read dY and dA), and a last one
  // before the commit (the next chunk's forward reads the weights).  Fewer stream
  // operations between the chain's kernels keep more launch overlap.
  const bool side = ln.st3 != nullptr && c->concurrent;
  cudaStream_t sw = side ? ln.st3 : st;
  bool steps_pending = false;
  for (int si = S - 1; si >= 0; --si) {
    const int l = P0 + si;
    Pair up16 = sq_.up16.at((long)si * d * f), down16 = sq_.down16.at((long)si * f * d);
    {  // dA = (dY W_down^T) * gelu'(a)
      GemmArgs g;
      g.M = n; g.N = f; g.K = d;
      g.aux = ln.sa + (long)si * b * f; g.ldaux = f;
      g.oh = ln.da.hi; g.ol = ln.da.lo; g.ldo = f; g.err = c->derr;
      RUN(K_MLP_DX, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 0,
          gemm_run(EPI_GELU_BWD, opnd(ln.dy16, d, 0), opnd(down16, d, 0), g, sp, st));
    }
    if (si > 0) {  // dXn_m = dA W_up^T  (before W_up changes)
      GemmArgs g;
      g.M = n; g.N = d; g.K = f;
      g.out32 = ln.dxn; g.ldo32 = d; g.err = c->derr; g.allow_ksplit = true;
      g.out32_ready = true;
      RUN(K_MLP_DX, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 0,
          gemm_run(EPI_F32, opnd(ln.da, f, 0), opnd(up16, f, 0), g, sp, st));
    }
    if (si > 0 && c->dual) {  // the static MLP passes gradient to its input: dXn_m += dA_s W_up_s^T
      GemmArgs g;
      g.M = n; g.N = f; g.K = d;
      g.aux = ln.sa_s + (long)si * b * f; g.ldaux = f;
      g.oh = ln.da_s.hi; g.ol = ln.da_s.lo; g.ldo = f; g.err = c->derr;
      RUN(K_MLP_DX, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 0,
          gemm_run(EPI_GELU_BWD, opnd(ln.dy16, d, 0), opnd(c->Wdown_s.at((long)si * f * d), d, 0), g, sp, st));
      GemmArgs g2;
      g2.M = n; g2.N = d; g2.K = f;
      g2.out32 = ln.dxn; g2.ldo32 = d; g2.resid = ln.dxn; g2.ldr = d; g2.err = c->derr; g2.allow_ksplit = true;
      RUN(K_MLP_DX, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 0,
          gemm_run(EPI_RESID, opnd(ln.da_s, f, 0), opnd(c->Wup_s.at((long)si * d * f), f, 0), g2, sp, st));
    }
    if (side) {
      CK(cudaEventRecord(ln.ev_dx, st));
      CK(cudaStreamWaitEvent(sw, ln.ev_dx, 0));
    }
    {  // W_down -= eta U^T dY
      GemmArgs g;
      g.M = f; g.N = d; g.K = n;
      g.w32 = sq_.down32 + (long)si * f * d; g.wh = down16.hi; g.wl = down16.lo; g.ldw = d; g.eta = eta;
      g.err = c->derr;
      RUN_ON(sw, K_DW_SGD, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 8 * dd * ff,
             gemm_run(EPI_SGD, opnd(ln.su.at((long)si * b * f), f, 1), opnd(ln.dy16, d, 1), g, sp, sw));
    }
    {  // W_up -= eta Xn_m^T dA
      GemmArgs g;
      g.M = d; g.N = f; g.K = n;
      g.w32 = sq_.up32 + (long)si * d * f; g.wh = up16.hi; g.wl = up16.lo; g.ldw = f; g.eta = eta;
      g.err = c->derr;
      RUN_ON(sw, K_DW_SGD, 1, 2 * nn * dd * ff, 2 * nn * dd * ff * ops, 8 * dd * ff,
             gemm_run(EPI_SGD, opnd(ln.sxm.at((long)si * b * d), d, 1), opnd(ln.da, f, 1), g, sp, sw));
    }
    if (side) {
      CK(cudaEventRecord(ln.ev_wu, sw));
      steps_pending = true;
    }
    if (si == 0) break;  // the first trainable block's attention needs no gradient
    // dH = dY + RMSNorm_m^T(dXn_m)
    RUN(K_RMSNORM, 1, 0, 0, nn * dd * (20 + eb),
        rows_rmsnorm_bwd(ln.dxn, ln.sh + (long)si * b * d, c->gains + (long)(2 * l + 1) * d,
                         ln.srs_m + (long)si * b, ln.dy, n, d, ln.dh32, ln.dh16.hi, ln.dh16.lo, st, true));
    {  // dO = dH Wo^T
      GemmArgs g;
      g.M = n; g.N = d; g.K = d;
      g.oh = ln.do16.hi; g.ol = ln.do16.lo; g.ldo = d; g.err = c->derr;
      RUN(K_ATTN_DX, 1, 2 * nn * dd * dd, 2 * nn * dd * dd * ops, 0,
          gemm_run(EPI_OPND, opnd(ln.dh16, d, 0), opnd(c->Wo.at((long)l * d * d), d, 0), g, sp, st));
    }
    Pair qb = ln.sq.at((long)si * b * d), ob = ln.so.at((long)si * b * d);
    RUN(K_MISC, 1, 0, 0, nn * dd * 2 * eb,
        rows_attn_rowdot(ln.do16.hi, ln.do16.lo, ob.hi, ob.lo, n, H, dh, ln.D, st));
    {
      AttnBwdMaps m;
      Pair ko = ln.kown.at((long)l * R * d), vo = ln.vown.at((long)l * R * d);
      Pair kr = sq_.ring_k.at((long)l * k * d), vr = sq_.ring_v.at((long)l * k * d);
      if (!attn_maps(&m.f, qb, kr, vr, ko, vo, n, d, k) ||
          !make_map(&m.dO, ln.do16.hi, (uint64_t)d, (uint64_t)n, d, 128))
        return fail(c, TTT_ERR_CUDA, "attention backward tensor maps");
      if (sp) {
        if (!make_map(&m.dOl, ln.do16.lo, (uint64_t)d, (uint64_t)n, d, 128))
          return fail(c, TTT_ERR_CUDA, "attention backward tensor maps");
      } else {
        m.dOl = m.dO;
      }
      AttnBwdArgs ba;
      ba.g.n = n; ba.g.H = H; ba.g.dh = dh; ba.g.window = k; ba.g.pos0 = pos0;
      ba.g.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)dh));
      ba.g.ldo = d; ba.g.err = c->derr;
      ba.lse = ln.slse + (long)si * H * b;
      ba.D = ln.D;
      ba.scale = (float)(1.0 / std::sqrt((double)dh));
      // written straight into the QKV dX product's operand, RoPE's rotation transposed
      ba.qkv_h = ln.dqkv.hi; ba.qkv_l = ln.dqkv.lo; ba.ld_qkv = 3L * d; ba.k_off = d; ba.v_off = 2L * d;
      ba.cs = cs; ba.sn = sn;
      RUN(K_ATTN_BWD, 1, 4 * dd * (pairs + own_pairs), (6 * dd * tpairs + 8 * dd * own_tile_pairs) * ops, 0,
          attn_bwd_run(m, ba, sp, st, 0));
    }
    {  // dXn_a = dQKV Wqkv^T
      GemmArgs g;
      g.M = n; g.N = d; g.K = 3 * d;
      g.out32 = ln.dxn; g.ldo32 = d; g.err = c->derr; g.allow_ksplit = true;
      g.out32_ready = true;
      RUN(K_ATTN_DX, 1, 6 * nn * dd * dd, 6 * nn * dd * dd * ops, 0,
          gemm_run(EPI_F32, opnd(ln.dqkv, 3 * d, 0), opnd(c->Wqkv.at((long)l * d * 3 * d), 3 * d, 0), g, sp, st));
    }
    if (steps_pending) {  // the block's steps have read dY and dA
      CK(cudaStreamWaitEvent(st, ln.ev_wu, 0));
      steps_pending = false;
    }
    // dY_{l-1} = dH + RMSNorm_a^T(dXn_a)
    RUN(K_RMSNORM, 1, 0, 0, nn * dd * (20 + eb),
        rows_rmsnorm_bwd(ln.dxn, ln.sx + (long)si * b * d, c->gains + (long)(2 * l) * d, ln.srs_a + (long)si * b,
                         ln.dh32, n, d, ln.dy, ln.dy16.hi, ln.dy16.lo, st, true));
  }
  if (steps_pending) CK(cudaStreamWaitEvent(st, ln.ev_wu, 0));  // every step is in place before the weights are read
  // ------------------------------------------------------------------- commit
  const double cb = (double)S * nn * dd * 2 * 2;
  const long os = (long)R * d, rs = (long)k * d;
  RUN(K_COMMIT, 1, 0, 0, cb,
      rows_commit(ln.kown.hi + (long)P0 * os, sq_.ring_k.hi + (long)P0 * rs, os, rs, S, pos0, n, k, d, st));
  RUN(K_COMMIT, 1, 0, 0, cb,
      rows_commit(ln.vown.hi + (long)P0 * os, sq_.ring_v.hi + (long)P0 * rs, os, rs, S, pos0, n, k, d, st));
  if (sp) {
    RUN(K_COMMIT, 1, 0, 0, cb,
        rows_commit(ln.kown.lo + (long)P0 * os, sq_.ring_k.lo + (long)P0 * rs, os, rs, S, pos0, n, k, d, st));
    RUN(K_COMMIT, 1, 0, 0, cb,
        rows_commit(ln.vown.lo + (long)P0 * os, sq_.ring_v.lo + (long)P0 * rs, os, rs, S, pos0, n, k, d, st));
  }
  sq_.pos = pos0 + n;
  return TTT_OK;
}
}  // namespace

// ============================================================================ C ABI
extern "C" int ttt_create(const ttt_config* cfg, void* cuda_stream, ttt_ctx** out) {
  if (!cfg || !out) return TTT_ERR_ARG;
  *out = nullptr;
  const ttt_config& g = *cfg;
  if (g.n_layers <= 0 || g.n_trainable <= 0 || g.n_trainable > g.n_layers || g.d_model <= 0 || g.n_heads <= 0 ||
      g.d_ff <= 0 || g.vocab <= 0 || g.window <= 0 || g.chunk <= 0 || g.n_seqs <= 0 || g.chunk > g.window ||
      g.d_model % g.n_heads != 0 || !(g.rope_theta > 0) || !(g.rms_eps >= 0) || (g.compute != 0 && g.compute != 1) ||
      (g.dual_mlp != 0 && g.dual_mlp != 1))
    return TTT_ERR_ARG;
  const int dh = g.d_model / g.n_heads;
  const bool split = g.compute == 0;
  if (dh % 16 || dh > 128 || (split && dh > 64) || g.d_model % 64 || g.d_model > 4096 || g.d_ff % 64 ||
      g.vocab % 8 || g.window % 128)
    return TTT_ERR_UNSUPPORTED;
  ttt_ctx* c = new ttt_ctx();
  c->cfg = g;
  c->st = (cudaStream_t)cuda_stream;
  c->split = split;
  c->dual = g.dual_mlp == 1;
  c->L = g.n_layers; c->S = g.n_trainable; c->d = g.d_model; c->H = g.n_heads; c->dh = dh; c->f = g.d_ff;
  c->V = g.vocab; c->k = g.window; c->b = g.chunk; c->B = g.n_seqs;
  // the frozen blocks run ahead over up to kPrefixRows tokens of whole chunks, never more than the window
  c->G = std::max(1, std::min(kPrefixRows / c->b, c->k / c->b));
  c->R = c->G * c->b;
  const long L = c->L, S = c->S, d = c->d, f = c->f, V = c->V, k = c->k, b = c->b, H = c->H;
  bool ok = true;
  c->E = dalloc<float>(c, V * d, ok);
  c->gains = dalloc<float>(c, (2 * L + 1) * d, ok);
  c->Wqkv = palloc(c, L * d * 3 * d, ok);
  c->Wo = palloc(c, L * d * d, ok);
  c->Wup = palloc(c, (L - S) * d * f, ok);
  c->Wdown = palloc(c, (L - S) * f * d, ok);
  c->Wlm = palloc(c, d * V, ok);
  if (c->dual) {
    c->Wup_s = palloc(c, S * d * f, ok);
    c->Wdown_s = palloc(c, S * f * d, ok);
  }
  c->seqs.resize(g.n_seqs);
  for (auto& s : c->seqs) {
    s.ring_k = palloc(c, L * k * d, ok);
    s.ring_v = palloc(c, L * k * d, ok);
    s.up32 = dalloc<float>(c, S * d * f, ok);
    s.down32 = dalloc<float>(c, S * f * d, ok);
    s.up16 = palloc(c, S * d * f, ok);
    s.down16 = palloc(c, S * f * d, ok);
  }
  c->init_up = dalloc<float>(c, S * d * f, ok);
  c->init_down = dalloc<float>(c, S * f * d, ok);
  c->acc.resize(K_NCLS);
  c->tok = dalloc<int>(c, (size_t)g.n_seqs * b, ok);
  c->next = dalloc<int>(c, g.n_seqs, ok);
  c->minus1 = dalloc<int>(c, 1, ok);
  c->derr = dalloc<int>(c, 1, ok);
  c->loss_dev = dalloc<float>(c, g.n_seqs, ok);
  c->inv_freq = dalloc<double>(c, dh / 2, ok);
  c->zdec = dalloc<float>(c, V, ok);
  const long R = c->R;
  const bool fused_qkv = qkv_rope_bn(dh, (int)d, split) != 0;
  c->lanes.resize(std::min(g.n_seqs, kMaxLanes));
  for (Lane& ln : c->lanes) {
    ln.tgt = dalloc<int>(c, b, ok);
    ln.cs = dalloc<float>(c, R * dh / 2, ok);
    ln.sn = dalloc<float>(c, R * dh / 2, ok);
    ln.x = dalloc<float>(c, b * d, ok);
    ln.xp = dalloc<float>(c, R * d, ok);
    ln.xpb[0] = ln.xp;
    ln.xpb[1] = dalloc<float>(c, R * d, ok);
    ln.csb[0] = ln.cs;
    ln.snb[0] = ln.sn;
    ln.csb[1] = dalloc<float>(c, R * dh / 2, ok);
    ln.snb[1] = dalloc<float>(c, R * dh / 2, ok);
    ln.sxn = palloc(c, b * d, ok);
    if (!fused_qkv) ln.qkv = dalloc<float>(c, R * 3 * d, ok);
    ln.xn = palloc(c, R * d, ok);
    ln.q = palloc(c, R * d, ok);
    ln.o = palloc(c, R * d, ok);
    ln.u = palloc(c, R * f, ok);
    ln.kown = palloc(c, L * R * d, ok);
    ln.vown = palloc(c, L * R * d, ok);
    ln.sx = dalloc<float>(c, S * b * d, ok);
    ln.sh = dalloc<float>(c, S * b * d, ok);
    ln.srs_a = dalloc<float>(c, S * b, ok);
    ln.srs_m = dalloc<float>(c, S * b, ok);
    ln.slse = dalloc<float>(c, S * H * b, ok);
    ln.sa = dalloc<float>(c, S * b * f, ok);
    ln.sq = palloc(c, S * b * d, ok);
    ln.so = palloc(c, S * b * d, ok);
    ln.sxm = palloc(c, S * b * d, ok);
    ln.su = palloc(c, S * b * f, ok);
    ln.xf = palloc(c, b * d, ok);
    ln.dz = palloc(c, b * V, ok);
    ln.rs_f = dalloc<float>(c, b, ok);
    ln.zt = dalloc<float>(c, b, ok);
    ln.lse_row = dalloc<float>(c, b, ok);
    ln.loss_row = dalloc<float>(c, b, ok);
    ln.inv_nvalid = dalloc<float>(c, 1, ok);
    ln.part = dalloc<float2>(c, ((V + 127) / 128) * b, ok);
    ln.dy = dalloc<float>(c, b * d, ok);
    ln.dxn = dalloc<float>(c, b * d, ok);
    ln.dh32 = dalloc<float>(c, b * d, ok);
    ln.D = dalloc<float>(c, H * b, ok);
    ln.dy16 = palloc(c, b * d, ok);
    ln.da = palloc(c, b * f, ok);
    ln.dh16 = palloc(c, b * d, ok);
    ln.do16 = palloc(c, b * d, ok);
    ln.dqkv = palloc(c, b * 3 * d, ok);
    if (c->dual) {
      ln.sa_s = dalloc<float>(c, S * b * f, ok);
      ln.us = palloc(c, b * f, ok);
      ln.da_s = palloc(c, b * f, ok);
    }
  }
  if (!ok) {
    ttt_destroy(c);
    return TTT_ERR_OOM;
  }
  auto mk_ev = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
  auto mk_st = [](cudaStream_t* t) { return cudaStreamCreateWithFlags(t, cudaStreamNonBlocking) == cudaSuccess; };
  bool made = mk_ev(&c->ev_fork);
  for (size_t i = 0; i < c->lanes.size() && made; ++i) {
    Lane& ln = c->lanes[i];
    if (i == 0) {
      ln.st = c->st;
    } else {
      made = mk_st(&ln.st);
      ln.own_st = made;
    }
    made = made && mk_st(&ln.st2) && mk_st(&ln.st3) && mk_ev(&ln.ev_dx) &&
           mk_ev(&ln.ev_wu) && mk_ev(&ln.ev_fork) && mk_ev(&ln.ev_join) && mk_ev(&ln.ev_pass[0]) &&
           mk_ev(&ln.ev_pass[1]) && mk_ev(&ln.ev_suf[0]) && mk_ev(&ln.ev_suf[1]);
  }
  if (!made) {
    cudaGetLastError();
    ttt_destroy(c);
    return TTT_ERR_CUDA;
  }
  std::vector<double> invf(dh / 2);
  for (int i = 0; i < dh / 2; ++i) invf[i] = std::pow(g.rope_theta, -2.0 * i / (double)dh);
  int m1 = -1;
  if (cudaMemcpy(c->inv_freq, invf.data(), invf.size() * sizeof(double), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(c->minus1, &m1, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    ttt_destroy(c);
    return TTT_ERR_CUDA;
  }
  *out = c;
  return TTT_OK;
}

extern "C" void ttt_destroy(ttt_ctx* c) {
  if (!c) return;
  if (c->st) cudaStreamSynchronize(c->st);
  for (Lane& ln : c->lanes)
    for (cudaStream_t t : {ln.own_st ? ln.st : nullptr, ln.st2, ln.st3})
      if (t) cudaStreamSynchronize(t);
  cudaDeviceSynchronize();
  for (Lane& ln : c->lanes) {
    for (cudaStream_t t : {ln.own_st ? ln.st : nullptr, ln.st2, ln.st3})
      if (t) cudaStreamDestroy(t);
    for (cudaEvent_t e : {ln.ev_fork, ln.ev_join, ln.ev_pass[0], ln.ev_pass[1], ln.ev_suf[0], ln.ev_suf[1],
                          ln.ev_dx, ln.ev_wu})
      if (e) cudaEventDestroy(e);
  }
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  for (void* p : c->allocs) cudaFree(p);
  if (c->seq_tok) cudaFree(c->seq_tok);
  if (c->seq_loss) cudaFree(c->seq_loss);
  for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
  delete c;
}

extern "C" const char* ttt_last_error(const ttt_ctx* c) { return c ? c->err.c_str() : "null context"; }

extern "C" int64_t ttt_position(const ttt_ctx* c) { return (c && !c->seqs.empty()) ? c->seqs[0].pos : -1; }

extern "C" int ttt_load_weights(ttt_ctx* c, const float* blob, size_t n_floats) {
  if (!c || !blob) return TTT_ERR_ARG;
  const long L = c->L, S = c->S, d = c->d, f = c->f, V = c->V;
  const size_t need = (size_t)(V * d + L * (2 * d + 4 * d * d + 2 * d * f) + d + d * V) +
                      (c->dual ? (size_t)(S * 2 * d * f) : 0);
  if (n_floats != need) return fail(c, TTT_ERR_ARG, "blob size " + std::to_string(n_floats) + " != " + std::to_string(need));
  c->loaded = false;
  cudaStream_t st = c->st;
  float* stage = nullptr;
  if (cudaMalloc(&stage, need * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    return fail(c, TTT_ERR_OOM, "weight staging buffer");
  }
  auto body = [&]() -> int {
    CK(cudaMemcpyAsync(stage, blob, need * sizeof(float), cudaMemcpyHostToDevice, st));
    long off = 0;
    CK(cudaMemcpyAsync(c->E, stage, (size_t)V * d * 4, cudaMemcpyDeviceToDevice, st));
    off += V * d;
    for (long l = 0; l < L; ++l) {
      CK(cudaMemcpyAsync(c->gains + (2 * l) * d, stage + off, (size_t)d * 4, cudaMemcpyDeviceToDevice, st));
      off += d;
      for (int part = 0; part < 3; ++part) {  // Wq | Wk | Wv -> columns of Wqkv[l]
        Pair dst = c->Wqkv.at(l * d * 3 * d + part * d);
        CK(rows_convert(stage + off, d, (int)d, d, dst.hi, dst.lo, 3 * d, st));
        off += d * d;
      }
      Pair wo = c->Wo.at(l * d * d);
      CK(rows_convert(stage + off, d, (int)d, d, wo.hi, wo.lo, d, st));
      off += d * d;
      CK(cudaMemcpyAsync(c->gains + (2 * l + 1) * d, stage + off, (size_t)d * 4, cudaMemcpyDeviceToDevice, st));
      off += d;
      const float* up = stage + off;
      const float* down = stage + off + d * f;
      off += 2 * d * f;
      if (l < L - S) {
        Pair wu = c->Wup.at(l * d * f), wd = c->Wdown.at(l * f * d);
        CK(rows_convert(up, d, (int)f, f, wu.hi, wu.lo, f, st));
        CK(rows_convert(down, f, (int)d, d, wd.hi, wd.lo, d, st));
      } else {
        const long si = l - (L - S);
        CK(cudaMemcpyAsync(c->init_up + si * d * f, up, (size_t)d * f * 4, cudaMemcpyDeviceToDevice, st));
        CK(cudaMemcpyAsync(c->init_down + si * f * d, down, (size_t)f * d * 4, cudaMemcpyDeviceToDevice, st));
        for (auto& s : c->seqs) {
          CK(cudaMemcpyAsync(s.up32 + si * d * f, up, (size_t)d * f * 4, cudaMemcpyDeviceToDevice, st));
          CK(cudaMemcpyAsync(s.down32 + si * f * d, down, (size_t)f * d * 4, cudaMemcpyDeviceToDevice, st));
          Pair wu = s.up16.at(si * d * f), wd = s.down16.at(si * f * d);
          CK(rows_convert(up, d, (int)f, f, wu.hi, wu.lo, f, st));
          CK(rows_convert(down, f, (int)d, d, wd.hi, wd.lo, d, st));
        }
        if (c->dual) {  // the static pair follows the block's W_down
          Pair su = c->Wup_s.at(si * d * f), sd = c->Wdown_s.at(si * f * d);
          CK(rows_convert(stage + off, d, (int)f, f, su.hi, su.lo, f, st));
          CK(rows_convert(stage + off + d * f, f, (int)d, d, sd.hi, sd.lo, d, st));
          off += 2 * d * f;
        }
      }
    }
    CK(cudaMemcpyAsync(c->gains + (2 * L) * d, stage + off, (size_t)d * 4, cudaMemcpyDeviceToDevice, st));
    off += d;
    CK(rows_convert(stage + off, d, (int)V, V, c->Wlm.hi, c->Wlm.lo, V, st));
    off += d * V;
    for (auto& s : c->seqs) {
      s.pos = 0;
      const size_t rb = (size_t)L * c->k * d * sizeof(bf16);
      CK(cudaMemsetAsync(s.ring_k.hi, 0, rb, st));
      CK(cudaMemsetAsync(s.ring_v.hi, 0, rb, st));
      if (c->split) {
        CK(cudaMemsetAsync(s.ring_k.lo, 0, rb, st));
        CK(cudaMemsetAsync(s.ring_v.lo, 0, rb, st));
      }
    }
    // the K-sliced dX products add into dxn, which its readers leave at zero; a chunk cut
    // short by an error may not have, so start from zero
    for (Lane& ln : c->lanes) CK(cudaMemsetAsync(ln.dxn, 0, (size_t)c->b * d * sizeof(float), st));
    CK(cudaMemsetAsync(c->derr, 0, sizeof(int), st));
    CK(cudaStreamSynchronize(st));
    return TTT_OK;
  };
  const int r = body();
  cudaStreamSynchronize(st);
  cudaFree(stage);
  if (r == TTT_OK) {
    c->loaded = true;
    c->err.clear();
  }
  return r;
}

namespace {
int check_device_error(ttt_ctx* c) {
  int e = 0;
  if (cudaMemcpy(&e, c->derr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(c, TTT_ERR_CUDA, "reading the device error word");
  if (e != 0) {
    c->loaded = false;
    return fail(c, TTT_ERR_DEVICE, e == DERR_BAD_TOKEN ? "token id outside [0, vocab)"
                                                        : "bounded wait expired in a kernel (code " + std::to_string(e) + ")");
  }
  return TTT_OK;
}
}  // namespace

extern "C" int ttt_sync(ttt_ctx* c) {
  if (!c) return TTT_ERR_ARG;
  cudaError_t e = cudaStreamSynchronize(c->st);
  if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
  return check_device_error(c);
}

namespace {
// Lanes 0 .. nl-1, side streams included, start after everything already enqueued
// on the context stream.
int fork_lanes(ttt_ctx* c, int nl) {
  CK(cudaEventRecord(c->ev_fork, c->st));
  for (int i = 0; i < nl; ++i) {
    Lane& ln = c->lanes[i];
    if (ln.own_st) CK(cudaStreamWaitEvent(ln.st, c->ev_fork, 0));
    CK(cudaStreamWaitEvent(ln.st2, c->ev_fork, 0));
    CK(cudaStreamWaitEvent(ln.st3, c->ev_fork, 0));
  }
  return TTT_OK;
}

// The context stream waits for everything lanes 0 .. nl-1 enqueued on any of their streams.
int join_lanes(ttt_ctx* c, int nl) {
  for (int i = 0; i < nl; ++i) {
    Lane& ln = c->lanes[i];
    for (cudaStream_t t : {ln.st2, ln.st3, ln.own_st ? ln.st : nullptr}) {
      if (!t) continue;
      CK(cudaEventRecord(ln.ev_join, t));
      CK(cudaStreamWaitEvent(c->st, ln.ev_join, 0));
    }
  }
  return TTT_OK;
}

// Lanes side by side when concurrency is on, else one lane for every sequence in turn.
int lanes_in_use(const ttt_ctx* c) { return c->concurrent ? (int)c->lanes.size() : 1; }
}  // namespace

extern "C" int ttt_prefill_chunk_dev(ttt_ctx* c, const int32_t* d_tokens, int32_t n, const int32_t* d_next,
                                     float* d_loss) {
  if (!c || !d_tokens || !d_next || !d_loss) return TTT_ERR_ARG;
  if (!c->loaded) return fail(c, TTT_ERR_STATE, "weights not loaded");
  if (n < 1 || n > c->b) return fail(c, TTT_ERR_ARG, "n outside 1..chunk");
  const int nl = lanes_in_use(c);
  for (int s0 = 0; s0 < c->B; s0 += nl) {
    const int m = std::min(nl, c->B - s0);
    int r = fork_lanes(c, m);
    for (int i = 0; i < m && r == TTT_OK; ++i) {
      Lane& ln = c->lanes[i];
      const int s = s0 + i;
      const int32_t* tk = d_tokens + (long)s * n;
      r = prefix_pass(c, ln, s, tk, n, c->seqs[s].pos, ln.st, 0);
      if (r == TTT_OK) r = suffix_step(c, ln, s, 0, tk, n, d_next + s, d_loss + s);
    }
    const int rj = join_lanes(c, m);
    if (r != TTT_OK) return r;
    if (rj != TTT_OK) return rj;
  }
  return TTT_OK;
}

extern "C" int ttt_prefill_chunk(ttt_ctx* c, const int32_t* tokens, int32_t n, const int32_t* next_tokens,
                                 float* chunk_loss) {
  if (!c || !tokens || !next_tokens || !chunk_loss) return TTT_ERR_ARG;
  if (!c->loaded) return fail(c, TTT_ERR_STATE, "weights not loaded");
  if (n < 1 || n > c->b) return fail(c, TTT_ERR_ARG, "n outside 1..chunk");
  for (long i = 0; i < (long)c->B * n; ++i)
    if (tokens[i] < 0 || tokens[i] >= c->V) return fail(c, TTT_ERR_ARG, "token id outside [0, vocab)");
  for (int s = 0; s < c->B; ++s)
    if (next_tokens[s] < -1 || next_tokens[s] >= c->V) return fail(c, TTT_ERR_ARG, "next token outside [-1, vocab)");
  if (cudaMemcpyAsync(c->tok, tokens, (size_t)c->B * n * sizeof(int), cudaMemcpyHostToDevice, c->st) != cudaSuccess ||
      cudaMemcpyAsync(c->next, next_tokens, (size_t)c->B * sizeof(int), cudaMemcpyHostToDevice, c->st) != cudaSuccess)
    return fail(c, TTT_ERR_CUDA, "token upload");
  int r = ttt_prefill_chunk_dev(c, c->tok, n, c->next, c->loss_dev);
  if (r != TTT_OK) return r;
  if (cudaMemcpyAsync(chunk_loss, c->loss_dev, (size_t)c->B * sizeof(float), cudaMemcpyDeviceToHost, c->st) !=
      cudaSuccess)
    return fail(c, TTT_ERR_CUDA, "loss download");
  return ttt_sync(c);
}

namespace {
// Sequences s0 .. s0+nl-1 over T tokens each (device ids toks[B][T]), sequence
// s0+i on lane i: the frozen blocks run ahead over groups of G chunks, the
// trainable blocks step chunk by chunk; losses[B][ceil(T/b)] (device).  With
// more than one group, the frozen pass of group g+1 runs on the lane's second
// stream while group g's trainable steps run on its main stream: the pass
// outputs are double-buffered, the steps of group g wait for pass g, and pass
// g+2 waits for the steps of group g (the last readers of its buffer).  The two
// sides share no other buffer: the steps touch only the trainable blocks'
// keys/values and window caches.  The lanes' work is enqueued chunk by chunk in
// turn, so every lane has launches queued while the others run.
int prefill_lanes(ttt_ctx* c, int s0, int nl, const int32_t* toks, int T, float* losses) {
  const int b = c->b, G = c->G;
  const int nc = (T + b - 1) / b, ng = (nc + G - 1) / G;
  const bool overlap = ng > 1 && c->concurrent && qkv_rope_bn(c->dh, c->d, c->split) != 0;
  std::vector<long> base(nl);
  for (int i = 0; i < nl; ++i) base[i] = c->seqs[s0 + i].pos;
  auto seq = [&](int i) { return toks + (long)(s0 + i) * T; };
  auto pass = [&](int i, int g, cudaStream_t st, int buf) -> int {
    const int t0 = g * G * b, t1 = std::min(T, (g + 1) * G * b);
    return prefix_pass(c, c->lanes[i], s0 + i, seq(i) + t0, t1 - t0, base[i] + t0, st, buf);
  };
  auto ahead = [&](int i, int g) -> int {
    Lane& ln = c->lanes[i];
    if (g >= 2) CK(cudaStreamWaitEvent(ln.st2, ln.ev_suf[g & 1], 0));
    const int r = pass(i, g, ln.st2, g & 1);
    if (r != TTT_OK) return r;
    CK(cudaEventRecord(ln.ev_pass[g & 1], ln.st2));
    return TTT_OK;
  };
  auto body = [&]() -> int {
    if (overlap)
      for (int i = 0; i < nl; ++i) {
        const int r = ahead(i, 0);
        if (r != TTT_OK) return r;
      }
    for (int g = 0; g < ng; ++g) {
      for (int i = 0; i < nl; ++i) {
        Lane& ln = c->lanes[i];
        const int r = !overlap ? pass(i, g, ln.st, 0) : (g + 1 < ng ? ahead(i, g + 1) : TTT_OK);
        if (r != TTT_OK) return r;
        if (overlap) CK(cudaStreamWaitEvent(ln.st, ln.ev_pass[g & 1], 0));
      }
      const int g0 = g * G, g1 = std::min(nc, g0 + G), t0 = g0 * b;
      for (int ci = g0; ci < g1; ++ci) {
        const int p0 = ci * b, n = std::min(b, T - p0);
        for (int i = 0; i < nl; ++i) {
          const int32_t* sq = seq(i);
          const int32_t* nx = (p0 + n < T) ? sq + p0 + n : c->minus1;
          const int r = suffix_step(c, c->lanes[i], s0 + i, p0 - t0, sq + p0, n, nx,
                                    losses + (long)(s0 + i) * nc + ci, overlap ? (g & 1) : 0);
          if (r != TTT_OK) return r;
        }
      }
      if (overlap)
        for (int i = 0; i < nl; ++i) CK(cudaEventRecord(c->lanes[i].ev_suf[g & 1], c->lanes[i].st));
    }
    return TTT_OK;
  };
  int r = fork_lanes(c, nl);
  if (r == TTT_OK) r = body();
  const int rj = join_lanes(c, nl);  // also on failure: later work stays behind what was queued
  return r != TTT_OK ? r : rj;
}
}  // namespace

extern "C" int ttt_prefill_sequence_dev(ttt_ctx* c, const int32_t* d_tokens, int32_t T, float* d_losses) {
  if (!c || !d_tokens || !d_losses || T < 1) return TTT_ERR_ARG;
  if (!c->loaded) return fail(c, TTT_ERR_STATE, "weights not loaded");
  const int nl = lanes_in_use(c);
  for (int s0 = 0; s0 < c->B; s0 += nl) {
    const int r = prefill_lanes(c, s0, std::min(nl, c->B - s0), d_tokens, T, d_losses);
    if (r != TTT_OK) return r;
  }
  return TTT_OK;
}

namespace {
// Logits of one row of the final normalised hidden state: z[V] = xf_row . W_lm.
int logits_row(ttt_ctx* c, const Pair& xf_row, float* z) {
  const double dd = c->d, VV = c->V;
  GemmArgs g;
  g.M = 1; g.N = c->V; g.K = c->d;
  g.out32 = z; g.ldo32 = c->V; g.err = c->derr;
  RUN_ON(c->st, K_CE_FWD, 1, 2 * dd * VV, 2 * dd * VV * (c->split ? 3 : 1), 0,
         gemm_run(EPI_F32, opnd(xf_row, c->d, 0), opnd(c->Wlm, c->V, 1), g, c->split, c->st));
  return TTT_OK;
}
}  // namespace

extern "C" int ttt_decode_dev(ttt_ctx* c, const int32_t* d_prompt, int32_t T, int32_t n_new, int32_t sample,
                              float temp, const float* d_u, int32_t* d_out, float* d_prefill_losses,
                              float* d_gen_losses, float* d_logits) {
  if (!c || !d_prompt || !d_out || !d_prefill_losses || T < 1 || n_new < 0) return TTT_ERR_ARG;
  if ((sample != 0 && sample != 1) || (sample && (!d_u || !(temp > 0.f)))) return TTT_ERR_ARG;
  if (n_new >= c->b && !d_gen_losses) return TTT_ERR_ARG;
  if (!c->loaded) return fail(c, TTT_ERR_STATE, "weights not loaded");
  Lane& ln = c->lanes[0];  // decoding runs every sequence on the first lane in turn
  cudaStream_t st = ln.st;
  const int b = c->b, L = c->L, P0 = c->L - c->S, d = c->d, dh = c->dh, V = c->V;
  const int ncp = (T + b - 1) / b, ncg = n_new / b;
  const double dd = d;
  for (int s = 0; s < c->B; ++s) {
    Seq& sq_ = c->seqs[s];
    int32_t* out = d_out + (long)s * (n_new + 1);
    const float* u = d_u ? d_u + (long)s * (n_new + 1) : nullptr;
    auto zrow = [&](int i) { return d_logits ? d_logits + ((long)s * (n_new + 1) + i) * V : c->zdec; };
    // the prompt goes through the chunked inner loop; its last position has no target
    int r = prefill_lanes(c, s, 1, d_prompt, T, d_prefill_losses);
    if (r != TTT_OK) return r;
    // the first token comes from the prompt's last position, as the last prompt chunk's
    // forward computed it (before that chunk's update): the final hidden rows are still in xf
    const int nl = T - (ncp - 1) * b;
    r = logits_row(c, ln.xf.at((long)(nl - 1) * d), zrow(0));
    if (r != TTT_OK) return r;
    RUN(K_MISC, 1, 0, 0, (double)V * 4, rows_pick(zrow(0), V, sample, temp, u, out, st));
    for (int i = 0; i < n_new; ++i) {
      const int rr = i % b;           // row of the token in its generated chunk
      const long pos0 = sq_.pos;      // first position of that chunk
      if (rr == 0) RUN(K_ROPE, 1, 0, 0, (double)b * dh * 4, rows_rope_table(pos0, b, dh, c->inv_freq, ln.cs, ln.sn, st));
      // one-token forward with the chunk's starting fast weights; its keys/values go to row
      // rr of the chunk's own buffers, the window cache is untouched until the chunk's step
      float* x = ln.xp + (long)rr * d;
      RUN(K_MISC, 1, 0, 0, dd * 8, rows_embed(out + i, 1, c->E, V, d, x, c->derr, st));
      for (int l = 0; l < L; ++l) {
        r = layer_forward(c, ln, sq_, l, l >= P0 ? l - P0 : -1, false, 1, rr, pos0, x, x, ln.cs + (long)rr * (dh / 2),
                          ln.sn + (long)rr * (dh / 2), st);
        if (r != TTT_OK) return r;
      }
      Pair xf = ln.xf.at((long)rr * d);
      RUN(K_RMSNORM, 1, 0, 0, dd * 8,
          rows_rmsnorm(x, c->gains + (long)(2 * L) * d, c->cfg.rms_eps, 1, d, xf.hi, xf.lo, nullptr, st));
      r = logits_row(c, xf, zrow(i + 1));
      if (r != TTT_OK) return r;
      RUN(K_MISC, 1, 0, 0, (double)V * 4, rows_pick(zrow(i + 1), V, sample, temp, u ? u + i + 1 : nullptr, out + i + 1, st));
      if (rr == b - 1) {  // a complete generated chunk takes one inner-loop step; its last target is the pick above
        const int32_t* ids = out + i - (b - 1);
        r = prefix_pass(c, ln, s, ids, b, pos0, st, 0);
        if (r == TTT_OK) r = suffix_step(c, ln, s, 0, ids, b, out + i + 1, d_gen_losses + (long)s * ncg + i / b);
        if (r != TTT_OK) return r;
      }
    }
  }
  return TTT_OK;
}

extern "C" int ttt_prefill_sequence(ttt_ctx* c, const int32_t* tokens, int32_t T, float* losses) {
  if (!c || !tokens || !losses || T < 1) return TTT_ERR_ARG;
  if (!c->loaded) return fail(c, TTT_ERR_STATE, "weights not loaded");
  const size_t ntok = (size_t)c->B * T, nloss = (size_t)c->B * ((T + c->b - 1) / c->b);
  for (size_t i = 0; i < ntok; ++i)
    if (tokens[i] < 0 || tokens[i] >= c->V) return fail(c, TTT_ERR_ARG, "token id outside [0, vocab)");
  if (ntok > c->seq_tok_cap || nloss > c->seq_loss_cap) {  // grow the staging buffers (synchronises)
    if (cudaStreamSynchronize(c->st) != cudaSuccess) return fail(c, TTT_ERR_CUDA, "stream synchronize");
    if (c->seq_tok) cudaFree(c->seq_tok);
    if (c->seq_loss) cudaFree(c->seq_loss);
    c->seq_tok = nullptr;
    c->seq_loss = nullptr;
    c->seq_tok_cap = c->seq_loss_cap = 0;
    if (cudaMalloc(&c->seq_tok, ntok * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&c->seq_loss, nloss * sizeof(float)) != cudaSuccess) {
      cudaGetLastError();
      return fail(c, TTT_ERR_OOM, "sequence staging buffers");
    }
    c->seq_tok_cap = ntok;
    c->seq_loss_cap = nloss;
  }
  if (cudaMemcpyAsync(c->seq_tok, tokens, ntok * sizeof(int32_t), cudaMemcpyHostToDevice, c->st) != cudaSuccess)
    return fail(c, TTT_ERR_CUDA, "token upload");
  const int r = ttt_prefill_sequence_dev(c, c->seq_tok, T, c->seq_loss);
  if (r != TTT_OK) return r;
  if (cudaMemcpyAsync(losses, c->seq_loss, nloss * sizeof(float), cudaMemcpyDeviceToHost, c->st) != cudaSuccess)
    return fail(c, TTT_ERR_CUDA, "loss download");
  return ttt_sync(c);
}

extern "C" int ttt_get_fast_weights(ttt_ctx* c, int32_t seq, int32_t sl, float* w_up, float* w_down) {
  if (!c || seq < 0 || seq >= c->B || sl < 0 || sl >= c->S) return TTT_ERR_ARG;
  const long d = c->d, f = c->f;
  cudaError_t e = cudaStreamSynchronize(c->st);
  if (e == cudaSuccess && w_up)
    e = cudaMemcpy(w_up, c->seqs[seq].up32 + sl * d * f, (size_t)d * f * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && w_down)
    e = cudaMemcpy(w_down, c->seqs[seq].down32 + sl * f * d, (size_t)f * d * 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
  return TTT_OK;
}

extern "C" int ttt_get_window(ttt_ctx* c, int32_t seq, int32_t layer, float* k_out, float* v_out, int64_t* pos_out) {
  if (!c || seq < 0 || seq >= c->B || layer < 0 || layer >= c->L) return TTT_ERR_ARG;
  const long d = c->d, k = c->k;
  const Seq& s = c->seqs[seq];
  cudaError_t e = cudaStreamSynchronize(c->st);
  if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
  if (pos_out) {  // slot i holds the latest position p < pos with p mod k == i (-1: never written)
    for (long i = 0; i < k; ++i) {
      long p = s.pos - 1 - ((s.pos - 1 - i) % k + k) % k;
      pos_out[i] = (s.pos > 0 && p >= 0) ? p : -1;
    }
  }
  std::vector<uint16_t> hi((size_t)k * d), lo(c->split ? (size_t)k * d : 0);
  const Pair* rings[2] = {&s.ring_k, &s.ring_v};
  float* outs[2] = {k_out, v_out};
  for (int w = 0; w < 2; ++w) {
    if (!outs[w]) continue;
    const Pair r = rings[w]->at((long)layer * k * d);
    e = cudaMemcpy(hi.data(), r.hi, hi.size() * 2, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && r.lo) e = cudaMemcpy(lo.data(), r.lo, lo.size() * 2, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
    for (size_t i = 0; i < hi.size(); ++i) {
      uint32_t bits = (uint32_t)hi[i] << 16;
      float v;
      std::memcpy(&v, &bits, 4);
      if (r.lo) {
        uint32_t lb = (uint32_t)lo[i] << 16;
        float l;
        std::memcpy(&l, &lb, 4);
        v += l;
      }
      outs[w][i] = v;
    }
  }
  return TTT_OK;
}

// ------------------------------------------------------------------ state export / import
// One sequence's resumable state, as raw bytes: a header, the fp32 fast
// weights, then the window cache exactly as the device holds it (bf16 bits,
// remainders too in the fp32 mode).  The bf16 shadows of the fast weights are
// not stored: import derives them with the rounding the SGD step uses.
namespace {
struct StateHeader {
  char magic[8];  // "TTTSTAT1"
  int32_t L, S, d, f, k, split, dual, pad;
  int64_t pos;
};
static_assert(sizeof(StateHeader) == 48, "state header layout");

size_t state_parts(const ttt_ctx* c, size_t* fw, size_t* ring) {
  *fw = (size_t)c->S * c->d * c->f * sizeof(float);                  // one of W_up, W_down
  *ring = (size_t)c->L * c->k * c->d * sizeof(bf16);                 // one of K, V (hi or lo)
  return sizeof(StateHeader) + 2 * *fw + (c->split ? 4 : 2) * *ring;
}
}  // namespace

extern "C" int64_t ttt_state_bytes(const ttt_ctx* c) {
  if (!c) return -1;
  size_t fw, ring;
  return (int64_t)state_parts(c, &fw, &ring);
}

extern "C" int ttt_export_state(ttt_ctx* c, int32_t seq, void* buf, size_t bytes) {
  if (!c || !buf || seq < 0 || seq >= c->B) return TTT_ERR_ARG;
  size_t fw, ring;
  if (bytes != state_parts(c, &fw, &ring)) return fail(c, TTT_ERR_ARG, "state buffer size");
  cudaError_t e = cudaStreamSynchronize(c->st);
  if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
  const Seq& s = c->seqs[seq];
  StateHeader h{};
  std::memcpy(h.magic, "TTTSTAT1", 8);
  h.L = c->L; h.S = c->S; h.d = c->d; h.f = c->f; h.k = c->k; h.split = c->split; h.dual = c->dual;
  h.pos = s.pos;
  uint8_t* p = static_cast<uint8_t*>(buf);
  std::memcpy(p, &h, sizeof(h));
  p += sizeof(h);
  const void* src[6] = {s.up32, s.down32, s.ring_k.hi, s.ring_v.hi, s.ring_k.lo, s.ring_v.lo};
  const size_t len[6] = {fw, fw, ring, ring, ring, ring};
  for (int i = 0; i < (c->split ? 6 : 4); ++i) {
    e = cudaMemcpy(p, src[i], len[i], cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
    p += len[i];
  }
  return TTT_OK;
}

extern "C" int ttt_import_state(ttt_ctx* c, int32_t seq, const void* buf, size_t bytes) {
  if (!c || !buf || seq < 0 || seq >= c->B) return TTT_ERR_ARG;
  if (!c->loaded) return fail(c, TTT_ERR_STATE, "weights not loaded");
  size_t fw, ring;
  if (bytes != state_parts(c, &fw, &ring)) return fail(c, TTT_ERR_ARG, "state buffer size");
  StateHeader h;
  std::memcpy(&h, buf, sizeof(h));
  if (std::memcmp(h.magic, "TTTSTAT1", 8) != 0 || h.L != c->L || h.S != c->S || h.d != c->d || h.f != c->f ||
      h.k != c->k || h.split != (int)c->split || h.dual != (int)c->dual || h.pos < 0)
    return fail(c, TTT_ERR_ARG, "state was exported from a context of another shape");
  cudaError_t e = cudaStreamSynchronize(c->st);
  if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
  Seq& s = c->seqs[seq];
  const uint8_t* p = static_cast<const uint8_t*>(buf) + sizeof(h);
  void* dst[6] = {s.up32, s.down32, s.ring_k.hi, s.ring_v.hi, s.ring_k.lo, s.ring_v.lo};
  const size_t len[6] = {fw, fw, ring, ring, ring, ring};
  for (int i = 0; i < (c->split ? 6 : 4); ++i) {
    e = cudaMemcpy(dst[i], p, len[i], cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
    p += len[i];
  }
  const long S = c->S, d = c->d, f = c->f;
  CK(rows_convert(s.up32, S * d, (int)f, f, s.up16.hi, s.up16.lo, f, c->st));
  CK(rows_convert(s.down32, S * f, (int)d, d, s.down16.hi, s.down16.lo, d, c->st));
  c->launches += 2;
  s.pos = h.pos;
  return ttt_sync(c);
}

extern "C" int ttt_reset(ttt_ctx* c) {
  if (!c) return TTT_ERR_ARG;
  if (!c->loaded) return fail(c, TTT_ERR_STATE, "weights not loaded");
  const long L = c->L, S = c->S, d = c->d, f = c->f, k = c->k;
  cudaStream_t st = c->st;
  for (auto& s : c->seqs) {
    s.pos = 0;
    CK(cudaMemcpyAsync(s.up32, c->init_up, (size_t)S * d * f * 4, cudaMemcpyDeviceToDevice, st));
    CK(cudaMemcpyAsync(s.down32, c->init_down, (size_t)S * f * d * 4, cudaMemcpyDeviceToDevice, st));
    CK(rows_convert(c->init_up, S * d, (int)f, f, s.up16.hi, s.up16.lo, f, st));
    CK(rows_convert(c->init_down, S * f, (int)d, d, s.down16.hi, s.down16.lo, d, st));
    const size_t rb = (size_t)L * k * d * sizeof(bf16);
    CK(cudaMemsetAsync(s.ring_k.hi, 0, rb, st));
    CK(cudaMemsetAsync(s.ring_v.hi, 0, rb, st));
    if (c->split) {
      CK(cudaMemsetAsync(s.ring_k.lo, 0, rb, st));
      CK(cudaMemsetAsync(s.ring_v.lo, 0, rb, st));
    }
  }
  c->launches += 2 * (long)c->seqs.size();
  return TTT_OK;
}

extern "C" int64_t ttt_launch_count(const ttt_ctx* c) { return c ? c->launches : -1; }

extern "C" int ttt_set_concurrency(ttt_ctx* c, int32_t on) {
  if (!c || (on != 0 && on != 1)) return TTT_ERR_ARG;
  if (cudaStreamSynchronize(c->st) != cudaSuccess) return fail(c, TTT_ERR_CUDA, "stream synchronize");
  c->concurrent = on == 1;
  return TTT_OK;
}

extern "C" int ttt_profile(ttt_ctx* c, int64_t class_mask) {
  if (!c) return TTT_ERR_ARG;
  if (cudaStreamSynchronize(c->st) != cudaSuccess) return fail(c, TTT_ERR_CUDA, "stream synchronize");
  c->recs.clear();
  c->ev_used = 0;
  for (auto& a : c->acc) a = ttt_ctx::ProfAcc();
  for (auto& n : c->prof_seen) n = 0;
  c->prof_mask = (uint64_t)class_mask & ((1ull << K_NCLS) - 1);
  return TTT_OK;
}

extern "C" int ttt_profile_sample(ttt_ctx* c, int32_t every) {
  if (!c || every < 1) return TTT_ERR_ARG;
  c->prof_every = every;
  for (auto& n : c->prof_seen) n = 0;
  return TTT_OK;
}

extern "C" const char* ttt_profile_class_name(int cls) {
  return (cls >= 0 && cls < K_NCLS) ? kClsName[cls] : nullptr;
}

extern "C" int ttt_profile_read(ttt_ctx* c, ttt_kernel_stat* out, int max_out, int* n_out) {
  if (!c || !n_out || (max_out > 0 && !out)) return TTT_ERR_ARG;
  cudaError_t e = cudaStreamSynchronize(c->st);
  if (e != cudaSuccess) return fail(c, TTT_ERR_CUDA, cudaGetErrorString(e));
  for (const auto& r : c->recs) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return fail(c, TTT_ERR_CUDA, "event elapsed time");
    auto& a = c->acc[r.cls];
    a.launches += r.nkern;
    a.ms += ms;
    a.alg += r.alg;
    a.exec += r.exec;
    a.bytes += r.bytes;
  }
  c->recs.clear();
  c->ev_used = 0;
  int n = 0;
  for (int i = 0; i < K_NCLS; ++i) {
    if (c->acc[i].launches == 0) continue;
    if (n < max_out) {
      ttt_kernel_stat& o = out[n];
      std::memset(&o, 0, sizeof(o));
      std::snprintf(o.name, sizeof(o.name), "%s", kClsName[i]);
      o.launches = c->acc[i].launches;
      o.ms = c->acc[i].ms;
      o.alg_flops = c->acc[i].alg;
      o.exec_flops = c->acc[i].exec;
      o.bytes = c->acc[i].bytes;
    }
    ++n;
  }
  *n_out = n;
  return TTT_OK;
}

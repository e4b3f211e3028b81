// Row-wise kernels of the TTT-E2E inner-loop step: token embedding, RMSNorm
// forward/backward, RoPE (angle table; rotation of q/k with the write of the
// chunk's own k/v where the QKV product's epilogue cannot do it), the commit of
// the chunk's keys/values into the k-slot window cache, the cross-entropy
// combine/mean, the rowsum(dO * O) term of the attention backward, and the
// token pick of decoding.  (RoPE's transpose runs in the attention backward.)
//
// All are HBM-bound: one warp per row, 16-byte vector loads/stores, fp32
// arithmetic; operands for the tensor-core kernels are written as bf16
// (plus the bf16 remainder in split mode).
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"
#include "rowops.h"

namespace ttt {

namespace {

TTT_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 8 consecutive fp32 values -> 8 bf16 (hi) [+ 8 bf16 remainders], one 16-B store each.
TTT_DEV void store8(bf16* hi, bf16* lo, long off, const float (&v)[8]) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 t = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    h[i] = *reinterpret_cast<uint32_t*>(&t);
    float2 f = __bfloat1622float2(t);
    l[i] = pack_bf16(v[2 * i] - f.x, v[2 * i + 1] - f.y);
  }
  *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
  if (lo) *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

TTT_DEV void load8(const float* p, float (&v)[8]) {
  float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

TTT_DEV void load8_bf(const bf16* hi, const bf16* lo, long off, float (&v)[8]) {
  uint4 h = *reinterpret_cast<const uint4*>(hi + off);
  const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&h);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(hp[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
  if (lo) {
    uint4 l = *reinterpret_cast<const uint4*>(lo + off);
    const __nv_bfloat162* lp = reinterpret_cast<const __nv_bfloat162*>(&l);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(lp[i]);
      v[2 * i] += f.x;
      v[2 * i + 1] += f.y;
    }
  }
}

// x[t][:] = E[tok[t]][:]; bad ids are reported and read row 0.
__global__ void embed_kernel(const int* __restrict__ tok, int n, const float* __restrict__ E, int V, int d,
                             float* __restrict__ x, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n) return;
  int id = tok[row];
  if (id < 0 || id >= V) {
    if (lane == 0 && err) atomicCAS(err, 0, (int)DERR_BAD_TOKEN);
    id = 0;
  }
  const float4* src = reinterpret_cast<const float4*>(E + (long)id * d);
  float4* dst = reinterpret_cast<float4*>(x + (long)row * d);
  for (int i = lane; i < d / 4; i += 32) dst[i] = src[i];
}

// Next-token targets of the chunk: tgt[i] = tok[i+1] (i < n-1), tgt[n-1] = *next (-1: none).
__global__ void targets_kernel(const int* __restrict__ tok, int n, const int* __restrict__ next, int V,
                               int* __restrict__ tgt, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int t = (i + 1 < n) ? tok[i + 1] : *next;
  if (t >= V || t < -1) {
    if (err) atomicCAS(err, 0, (int)DERR_BAD_TOKEN);
    t = -1;
  }
  tgt[i] = t;
}

// y = x * g / sqrt(mean(x^2) + eps) -> bf16 (hi, lo); rstd saved when requested; x
// also copied to x_copy when given (the start value of a K-sliced residual product).
// One warp per row; lane l holds columns l*8 + 256*i (i < NCH) in registers, so
// the row is read from HBM once and every load of the row is in flight at once.
template <int NCH>
__global__ void __launch_bounds__(128) rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ g,
                                                      float eps, int n, int d, bf16* __restrict__ yh,
                                                      bf16* __restrict__ yl, float* __restrict__ rstd,
                                                      float* __restrict__ x_copy) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n) return;
  const float* xr = x + (long)row * d;
  float v[NCH][8];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = lane * 8 + 256 * i;
    if (c < d) {
      load8(xr + c, v[i]);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss += v[i][e] * v[i][e];
    }
  }
  if (x_copy) {
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int c = lane * 8 + 256 * i;
      if (c < d) {
        float4* o = reinterpret_cast<float4*>(x_copy + (long)row * d + c);
        o[0] = make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
        o[1] = make_float4(v[i][4], v[i][5], v[i][6], v[i][7]);
      }
    }
  }
  ss = warp_sum(ss);
  const float r = 1.0f / sqrtf(ss / (float)d + eps);
  if (rstd && lane == 0) rstd[row] = r;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = lane * 8 + 256 * i;
    if (c < d) {
      float gg[8];
      load8(g + c, gg);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[i][e] = v[i][e] * r * gg[e];
      store8(yh, yl, (long)row * d + c, v[i]);
    }
  }
}

// out = resid + [r g dy - x r^3/d * sum(dy g x)]  (gradient of RMSNorm w.r.t. its input, gain frozen)
// Same register layout as the forward: dy and x of the row are read once.  With
// clear_dy, dy's row is set to zero once read (the next K-sliced product into that
// buffer adds onto zeros).
template <int NCH>
__global__ void __launch_bounds__(128) rmsnorm_bwd_kernel(const float* dy, const float* __restrict__ x,
                                                          const float* __restrict__ g, const float* __restrict__ rstd,
                                                          const float* resid, int n, int d, float* out,
                                                          bf16* __restrict__ oh, bf16* __restrict__ ol,
                                                          float* clear_dy) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n) return;
  const long base = (long)row * d;
  float a[NCH][8], b[NCH][8], q[NCH][8];  // dy, x and the residual of the row, all loads in flight at once
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = lane * 8 + 256 * i;
    if (c < d) {
      float gg[8];
      load8(dy + base + c, a[i]);
      load8(x + base + c, b[i]);
      if (resid) {
        load8(resid + base + c, q[i]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) q[i][e] = 0.f;
      }
      load8(g + c, gg);
#pragma unroll
      for (int e = 0; e < 8; ++e) s += a[i][e] * gg[e] * b[i][e];
    }
  }
  if (clear_dy) {  // each lane clears only the columns it has loaded
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int c = lane * 8 + 256 * i;
      if (c < d) {
        float4* z = reinterpret_cast<float4*>(clear_dy + base + c);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  s = warp_sum(s);
  const float r = rstd[row];
  const float k = r * r * r * s / (float)d;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = lane * 8 + 256 * i;
    if (c < d) {
      float gg[8], rr[8];
      load8(g + c, gg);
#pragma unroll
      for (int e = 0; e < 8; ++e) rr[e] = q[i][e] + (r * gg[e] * a[i][e] - b[i][e] * k);
      float4* o = reinterpret_cast<float4*>(out + base + c);
      o[0] = make_float4(rr[0], rr[1], rr[2], rr[3]);
      o[1] = make_float4(rr[4], rr[5], rr[6], rr[7]);
      if (oh) store8(oh, ol, base + c, rr);
    }
  }
}

// cos/sin of pos * theta^(-2i/dh) for the chunk, angles formed and reduced in fp64.
__global__ void rope_table_kernel(long pos0, int n, int half, const double* __restrict__ inv_freq,
                                  float* __restrict__ cs, float* __restrict__ sn) {
  pdl_wait();
  pdl_launch_dependents();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * half) return;
  const int t = idx / half, i = idx % half;
  double s, c;
  sincos((double)(pos0 + t) * inv_freq[i], &s, &c);
  cs[idx] = (float)c;
  sn[idx] = (float)s;
}

// q' = rope(q), k' = rope(k), v from qkv[t][3d] (fp32); rotate-half pairs (i, i+dh/2).
// One thread per (token, head, 4 pairs).
__global__ void rope_qkv_kernel(const float* __restrict__ qkv, const float* __restrict__ cs,
                                const float* __restrict__ sn, int n, int H, int dh, bf16* qh, bf16* ql, bf16* kh,
                                bf16* kl, bf16* vh, bf16* vl) {
  pdl_wait();
  pdl_launch_dependents();
  const int half = dh / 2, groups = half / 4;
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)n * H * groups) return;
  const int gi = (int)(idx % groups);
  const int h = (int)((idx / groups) % H);
  const int t = (int)(idx / ((long)groups * H));
  const int d = H * dh, i0 = gi * 4;
  const float* row = qkv + (long)t * 3 * d;
  const float4 c4 = *reinterpret_cast<const float4*>(cs + (long)t * half + i0);
  const float4 s4 = *reinterpret_cast<const float4*>(sn + (long)t * half + i0);
  const float c[4] = {c4.x, c4.y, c4.z, c4.w}, s[4] = {s4.x, s4.y, s4.z, s4.w};
  const long o1 = (long)t * d + h * dh + i0, o2 = o1 + half;
#pragma unroll
  for (int part = 0; part < 2; ++part) {  // 0: q, 1: k
    const float* src = row + part * d + h * dh + i0;
    const float4 a4 = *reinterpret_cast<const float4*>(src);
    const float4 b4 = *reinterpret_cast<const float4*>(src + half);
    const float a[4] = {a4.x, a4.y, a4.z, a4.w}, b[4] = {b4.x, b4.y, b4.z, b4.w};
    bf16* oh = part ? kh : qh;
    bf16* ol = part ? kl : ql;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 r;
      r.x = a[j] * c[j] - b[j] * s[j];
      r.y = b[j] * c[j] + a[j] * s[j];
      __nv_bfloat16 x1h, x1l, x2h, x2l;
      split_bf16(r.x, x1h, x1l);
      split_bf16(r.y, x2h, x2l);
      oh[o1 + j] = x1h;
      oh[o2 + j] = x2h;
      if (ol) {
        ol[o1 + j] = x1l;
        ol[o2 + j] = x2l;
      }
    }
  }
  const float* vs = row + 2 * d + h * dh + i0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat16 h1, l1, h2, l2;
    split_bf16(vs[j], h1, l1);
    split_bf16(vs[j + half], h2, l2);
    vh[o1 + j] = h1;
    vh[o2 + j] = h2;
    if (vl) {
      vl[o1 + j] = l1;
      vl[o2 + j] = l2;
    }
  }
}

// ring[(pos0 + t) mod k][:] = own[t][:] for the keys and values of every layer.
// grid = (tokens, layers)
__global__ void commit_kernel(const bf16* __restrict__ own, bf16* __restrict__ ring, long own_layer_stride,
                              long ring_layer_stride, long pos0, int n, int window, int d) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int l = blockIdx.y;
  if (t >= n) return;
  const long slot = (pos0 + t) % window;
  const uint4* src = reinterpret_cast<const uint4*>(own + l * own_layer_stride + (long)t * d);
  uint4* dst = reinterpret_cast<uint4*>(ring + l * ring_layer_stride + slot * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = src[i];
}

// lse[r] = log sum_tiles s_i exp(m_i); loss_row[r] = lse - z_target (0 when no target).
__global__ void ce_combine_kernel(const float2* __restrict__ part, const float* __restrict__ zt,
                                  const int* __restrict__ tgt, int n, int ntiles, float* __restrict__ lse,
                                  float* __restrict__ loss_row) {
  pdl_wait();
  pdl_launch_dependents();
  // one warp per row: lane i merges the (max, sum) pairs of tiles i, i+32, ..., then the warp merges the lanes
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= n) return;
  float m = -INFINITY, s = 0.f;
  for (int i = lane; i < ntiles; i += 32) {
    const float2 p = part[(long)i * n + r];
    if (p.x > m) {
      s = s * expf(m - p.x) + p.y;
      m = p.x;
    } else {
      s += p.y * expf(p.x - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
    const float mm = fmaxf(m, om);
    s = (m == -INFINITY ? 0.f : s * expf(m - mm)) + (om == -INFINITY ? 0.f : os * expf(om - mm));
    m = mm;
  }
  if (lane == 0) {
    const float l = m + logf(s);
    lse[r] = l;
    loss_row[r] = (tgt[r] >= 0) ? (l - zt[r]) : 0.f;
  }
}

// Mean over the rows with a target, fixed reduction order (bit-reproducible).
__global__ void loss_mean_kernel(const float* __restrict__ loss_row, const int* __restrict__ tgt, int n,
                                 float* __restrict__ out, float* __restrict__ inv_count) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float ssum[32];
  __shared__ int scnt[32];
  float s = 0.f;
  int c = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    if (tgt[i] >= 0) {
      s += loss_row[i];
      ++c;
    }
  s = warp_sum(s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) {
    ssum[threadIdx.x >> 5] = s;
    scnt[threadIdx.x >> 5] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float ts = 0.f;
    int tc = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      ts += ssum[w];
      tc += scnt[w];
    }
    *out = tc > 0 ? ts / (float)tc : 0.f;
    if (inv_count) *inv_count = tc > 0 ? 1.0f / (float)tc : 0.f;
  }
}

// D[h][t] = sum_i dO[t][h dh + i] * O[t][h dh + i]  (one warp per (t, h))
__global__ void attn_rowdot_kernel(const bf16* __restrict__ doh, const bf16* __restrict__ dol,
                                   const bf16* __restrict__ oh, const bf16* __restrict__ ol, int n, int H,
                                   int dh, float* __restrict__ D) {
  pdl_wait();
  pdl_launch_dependents();
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= n * H) return;
  const int t = w / H, h = w % H;
  const long base = (long)t * H * dh + h * dh;
  float s = 0.f;
  for (int c = lane * 8; c < dh; c += 256) {
    float a[8], b[8];
    load8_bf(doh, dol, base + c, a);
    load8_bf(oh, ol, base + c, b);
#pragma unroll
    for (int i = 0; i < 8; ++i) s += a[i] * b[i];
  }
  s = warp_sum(s);
  if (lane == 0) D[(long)h * n + t] = s;
}

// dst[r][c] = split(src[r][c]) for r < rows, c < cols (weight upload / layout change).
__global__ void convert_kernel(const float* __restrict__ src, long rows, int cols, long src_ld, bf16* dh, bf16* dl,
                               long dst_ld) {
  pdl_wait();
  pdl_launch_dependents();
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * cols) return;
  const long r = idx / cols;
  const int c = (int)(idx % cols);
  __nv_bfloat16 h, l;
  split_bf16(src[r * src_ld + c], h, l);
  dh[r * dst_ld + c] = h;
  if (dl) dl[r * dst_ld + c] = l;
}

constexpr int kRowWarps = 8;
inline int row_grid(int n) { return (n + kRowWarps - 1) / kRowWarps; }

// Next token from one row of logits z[V] (decode-phase TTT).  Greedy: the first
// index of the largest logit.  Sampling: inverse CDF of softmax(z / temp) at the
// caller's uniform *u: the first index whose running sum of exp(z/temp - max)
// exceeds *u times the total.  One block; thread t owns the contiguous run
// [t*per, (t+1)*per) of the vocabulary, so running sums follow index order.
constexpr int kPickThreads = 1024;
__global__ void __launch_bounds__(kPickThreads)
    pick_kernel(const float* __restrict__ z, int V, int sample, float temp, const float* __restrict__ u,
                int* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float s_v[32];
  __shared__ int s_i[32];
  __shared__ float s_sum[32];
  __shared__ int s_pick;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int per = (V + kPickThreads - 1) / kPickThreads;
  const int j0 = min(V, t * per), j1 = min(V, j0 + per);
  auto val = [&](int j) { return sample ? z[j] / temp : z[j]; };
  // largest value, first index on ties
  float mv = -INFINITY;
  int mi = V;
  for (int j = j0; j < j1; ++j) {
    const float y = val(j);
    if (y > mv) { mv = y; mi = j; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, mv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
    if (ov > mv || (ov == mv && oi < mi)) { mv = ov; mi = oi; }
  }
  if (lane == 0) { s_v[w] = mv; s_i[w] = mi; }
  if (t == 0) s_pick = V;
  __syncthreads();
  if (w == 0) {
    mv = s_v[lane];
    mi = s_i[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, mv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
      if (ov > mv || (ov == mv && oi < mi)) { mv = ov; mi = oi; }
    }
    if (lane == 0) { s_v[0] = mv; s_i[0] = mi; }
  }
  __syncthreads();
  if (!sample) {
    if (t == 0) *out = min(s_i[0], V - 1);
    return;
  }
  const float m = s_v[0];
  float loc = 0.f;
  for (int j = j0; j < j1; ++j) loc += expf(val(j) - m);
  // exclusive prefix of the runs' sums in thread order
  float inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float x = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += x;
  }
  if (lane == 31) s_sum[w] = inc;
  __syncthreads();
  if (w == 0) {
    float ws = s_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float x = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += x;
    }
    s_sum[lane] = ws;  // inclusive sum up to warp `lane`
  }
  __syncthreads();
  const float total = s_sum[31];
  const float target = *u * total;
  float c = (w > 0 ? s_sum[w - 1] : 0.f) + (inc - loc);
  for (int j = j0; j < j1; ++j) {
    c += expf(val(j) - m);
    if (c > target) {
      atomicMin(&s_pick, j);
      break;
    }
  }
  __syncthreads();
  if (t == 0) *out = min(s_pick, V - 1);
}

}  // namespace

int rows_pick(const float* z, int V, int sample, float temp, const float* u, int* out, cudaStream_t st) {
  return (int)launch_k(pick_kernel, dim3(1), dim3(kPickThreads), 0, st, z, V, sample, temp, u, out);
}

int rows_embed(const int* tok, int n, const float* E, int V, int d, float* x, int* err, cudaStream_t st) {
  return (int)launch_k(embed_kernel, dim3(row_grid(n)), dim3(kRowWarps * 32), 0, st, tok, n, E, V, d, x, err);
}

int rows_targets(const int* tok, int n, const int* next, int V, int* tgt, int* err, cudaStream_t st) {
  return (int)launch_k(targets_kernel, dim3((n + 255) / 256), dim3(256), 0, st, tok, n, next, V, tgt, err);
}

// Row kernels of the norm: 4 warps (4 rows) per block, per-lane register chunks
// of 8 columns; d % 8 == 0 and d <= 256 * kNormMaxChunks.
constexpr int kNormWarps = 4;
constexpr int kNormMaxChunks = 16;

template <int NCH>
int norm_fwd_n(const float* x, const float* g, float eps, int n, int d, bf16* yh, bf16* yl, float* rstd,
               float* x_copy, cudaStream_t st) {
  if constexpr (NCH > kNormMaxChunks) {
    return (int)cudaErrorInvalidValue;
  } else {
    if ((d + 255) / 256 > NCH) return norm_fwd_n<NCH + 1>(x, g, eps, n, d, yh, yl, rstd, x_copy, st);
    return (int)launch_k(rmsnorm_kernel<NCH>, dim3((n + kNormWarps - 1) / kNormWarps), dim3(kNormWarps * 32), 0, st,
                         x, g, eps, n, d, yh, yl, rstd, x_copy);
  }
}

template <int NCH>
int norm_bwd_n(const float* dy, const float* x, const float* g, const float* rstd, const float* resid, int n, int d,
               float* out, bf16* oh, bf16* ol, float* clear_dy, cudaStream_t st) {
  if constexpr (NCH > kNormMaxChunks) {
    return (int)cudaErrorInvalidValue;
  } else {
    if ((d + 255) / 256 > NCH) return norm_bwd_n<NCH + 1>(dy, x, g, rstd, resid, n, d, out, oh, ol, clear_dy, st);
    return (int)launch_k(rmsnorm_bwd_kernel<NCH>, dim3((n + kNormWarps - 1) / kNormWarps), dim3(kNormWarps * 32), 0,
                         st, dy, x, g, rstd, resid, n, d, out, oh, ol, clear_dy);
  }
}

int rows_rmsnorm(const float* x, const float* g, float eps, int n, int d, bf16* yh, bf16* yl, float* rstd,
                 cudaStream_t st, float* x_copy) {
  if (n <= 0) return 0;
  if (d % 8 || x_copy == x) return (int)cudaErrorInvalidValue;
  return norm_fwd_n<1>(x, g, eps, n, d, yh, yl, rstd, x_copy, st);
}

int rows_rmsnorm_bwd(const float* dy, const float* x, const float* g, const float* rstd, const float* resid, int n,
                     int d, float* out, bf16* oh, bf16* ol, cudaStream_t st, bool clear_dy) {
  if (n <= 0) return 0;
  if (d % 8) return (int)cudaErrorInvalidValue;
  // clearing dy must not touch a buffer the kernel reads or writes elsewhere
  if (clear_dy && (dy == x || dy == resid || dy == out)) return (int)cudaErrorInvalidValue;
  return norm_bwd_n<1>(dy, x, g, rstd, resid, n, d, out, oh, ol, clear_dy ? const_cast<float*>(dy) : nullptr, st);
}

int rows_rope_table(long pos0, int n, int dh, const double* inv_freq, float* cs, float* sn, cudaStream_t st) {
  const int half = dh / 2, tot = n * half;
  return (int)launch_k(rope_table_kernel, dim3((tot + 255) / 256), dim3(256), 0, st, pos0, n, half, inv_freq, cs, sn);
}

int rows_rope_qkv(const float* qkv, const float* cs, const float* sn, int n, int H, int dh, bf16* qh, bf16* ql,
                  bf16* kh, bf16* kl, bf16* vh, bf16* vl, cudaStream_t st) {
  const long tot = (long)n * H * (dh / 8);
  return (int)launch_k(rope_qkv_kernel, dim3((unsigned)((tot + 255) / 256)), dim3(256), 0, st, qkv, cs, sn, n, H, dh, qh, ql, kh, kl, vh, vl);
}

int rows_commit(const bf16* own, bf16* ring, long own_layer_stride, long ring_layer_stride, int n_layers, long pos0,
                int n, int window, int d, cudaStream_t st) {
  if (n <= 0 || n_layers <= 0) return 0;
  dim3 grid(n, n_layers);
  return (int)launch_k(commit_kernel, dim3(grid), dim3(128), 0, st, own, ring, own_layer_stride, ring_layer_stride, pos0, n, window, d);
}

int rows_ce_combine(const float2* part, const float* zt, const int* tgt, int n, int ntiles, float* lse,
                    float* loss_row, cudaStream_t st) {
  return (int)launch_k(ce_combine_kernel, dim3(row_grid(n)), dim3(kRowWarps * 32), 0, st, part, zt, tgt, n, ntiles, lse,
                       loss_row);
}

int rows_loss_mean(const float* loss_row, const int* tgt, int n, float* out, float* inv_count, cudaStream_t st) {
  return (int)launch_k(loss_mean_kernel, dim3(1), dim3(1024), 0, st, loss_row, tgt, n, out, inv_count);
}

int rows_convert(const float* src, long rows, int cols, long src_ld, bf16* dh, bf16* dl, long dst_ld,
                 cudaStream_t st) {
  const long tot = rows * cols;
  if (tot <= 0) return 0;
  return (int)launch_k(convert_kernel, dim3((unsigned)((tot + 255) / 256)), dim3(256), 0, st, src, rows, cols, src_ld, dh, dl, dst_ld);
}

int rows_attn_rowdot(const bf16* doh, const bf16* dol, const bf16* oh, const bf16* ol, int n, int H, int dh, float* D,
                     cudaStream_t st) {
  const int warps = n * H;
  return (int)launch_k(attn_rowdot_kernel, dim3((warps + kRowWarps - 1) / kRowWarps), dim3(kRowWarps * 32), 0, st, doh, dol, oh, ol, n, H, dh, D);
}

}  // namespace ttt

// Row-wise kernels of the P-EAGLE step: everything between the dense
// contractions. Each consumer first sums the K-slice partial slabs the
// tensor-core GEMM wrote, then applies the row operation in fp32.
#include <math.h>

#include <algorithm>

#include "rows.cuh"

namespace pe {

constexpr int kQkvThreads = 256, kQkvEpt = 8;
constexpr int kQkvChunk = kQkvThreads * kQkvEpt;   // per-row elements one qkv_finish block handles

__device__ __forceinline__ float sum_parts(const GemmOut& g, size_t idx) {
  float v = 0.f;
  for (int s = 0; s < g.splits; ++s) v += g.out[(size_t)s * g.split_stride + idx];
  return v;
}

// -------------------------------------------------------------------------
// Rotary table: cos/sin of p * theta^(-2j/hd) for every position p <
// max_position ("feat(speculative) ... #2376", RoPE fix commit: the cache is
// sized to the highest position and gathered by position value). Angles in
// double, so large positions keep their phase.
// -------------------------------------------------------------------------
__global__ void rope_table_kernel(float* cosb, float* sinb, int max_pos, int half, int hd, double theta) {
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)max_pos * half;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(e / half), j = (int)(e % half);
    const double a = (double)p * pow(theta, -2.0 * j / hd);
    double s, c;
    sincos(a, &s, &c);
    cosb[e] = (float)c;
    sinb[e] = (float)s;
  }
}

// -------------------------------------------------------------------------
// fc_norm and the layer-0 input rows ("P-EAGLE" user guide, Architecture;
// #2376 Changelog: mask_hidden is projected through the same fc/fc_norm).
// Row r: u = sum of partials; h = RMSNorm_fc(u);
//   x0[r] = [RMSNorm_in(E[tok]) , RMSNorm_hidden(h)]   (2H wide)
//   resid[r] = RMSNorm_hidden(h) if norm_before_residual else h.
// One block per row, EPT columns per thread held in registers: the gains are
// read before waiting on the producer, u and the token in one round, the
// embedding row in a second, and the three sums of squares in one block
// reduction (sum h^2 = inv_fc^2 * sum (u g_fc)^2).
// -------------------------------------------------------------------------
// Sums three per-thread values over the block; every thread gets the totals.
__device__ __forceinline__ void block_sum3(float& x, float& y, float& z, float (*red)[32]) {
  x = warp_sum(x);
  y = warp_sum(y);
  z = warp_sum(z);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  if (lane == 0) {
    red[0][w] = x;
    red[1][w] = y;
    red[2][w] = z;
  }
  __syncthreads();
  x = warp_sum(lane < nw ? red[0][lane] : 0.f);
  y = warp_sum(lane < nw ? red[1][lane] : 0.f);
  z = warp_sum(lane < nw ? red[2][lane] : 0.f);
}

template <typename T, int EPT>
__global__ void fc_finish_kernel(FcFinishArgs a) {
  pdl_trigger();
  __shared__ float red[3][32];
  const int r = blockIdx.x, H = a.H, bd = blockDim.x, tid = threadIdx.x;
  const T* g_fc = static_cast<const T*>(a.g_fc);
  const T* g_in = static_cast<const T*>(a.g_in);
  const T* g_h = static_cast<const T*>(a.g_h);
  float gf[EPT], gi[EPT], gh[EPT], u[EPT], ev[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int j = tid + i * bd;
    gf[i] = j < H ? to_f(g_fc[j]) : 0.f;
    gi[i] = j < H ? to_f(g_in[j]) : 0.f;
    gh[i] = j < H ? to_f(g_h[j]) : 0.f;
  }
  pdl_wait();
  int t = a.tok ? a.tok[r] : a.tok_const;
  const float* ur = a.u.out + (size_t)r * a.u.ldo;
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int j = tid + i * bd;
    u[i] = j < H ? ur[j] : 0.f;
  }
  for (int q = 1; q < a.u.splits; ++q) {
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const int j = tid + i * bd;
      if (j < H) u[i] += ur[(size_t)q * a.u.split_stride + j];
    }
  }
  if (t < 0 || t >= a.Vt) {
    if (tid == 0) set_status(a.status, PEAGLE_DEV_BOUNDS);
    t = 0;
  }
  const T* e = static_cast<const T*>(a.embed) + (size_t)t * H;
  float s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int j = tid + i * bd;
    ev[i] = j < H ? to_f(e[j]) : 0.f;
    const float ug = u[i] * gf[i];
    s1 += u[i] * u[i];
    s2 += ug * ug;
    s3 += ev[i] * ev[i];
  }
  block_sum3(s1, s2, s3, red);
  const float inv = rsqrtf(s1 / H + a.eps);
  const float inv2 = rsqrtf(inv * inv * s2 / H + a.eps);
  const float inv3 = rsqrtf(s3 / H + a.eps);
  T* x0 = static_cast<T*>(a.x0) + (size_t)r * 2 * H;
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int j = tid + i * bd;
    if (j < H) {
      const float h = u[i] * inv * gf[i];
      const float hn = h * inv2 * gh[i];
      x0[j] = from_f<T>(ev[i] * inv3 * gi[i]);
      x0[H + j] = from_f<T>(hn);
      if (a.resid) a.resid[(size_t)r * H + j] = a.nbr ? hn : h;
      if (a.hid) a.hid[(size_t)r * H + j] = h;
    }
  }
}

// -------------------------------------------------------------------------
// q/k/v rows with rotary phases gathered by position value (#2376, RoPE fix
// commit). Source of row r:
//   mode 0  the GEMM row r (layers >= 1);
//   mode 1  decode layer 0: row r = (b, d) takes GEMM row b if d == 0,
//           otherwise the precomputed masked q/k/v (every masked row of layer
//           0 has the same input: ptd embedding + projected mask_hidden);
//   mode 2  all rows masked (training layer 0, depths >= 1).
// Decode rows follow DecodeRows: row j of request b is new row j (its own
// position; GEMM row new_off[b] + j in layer 0) for j < n_b, else masked
// depth d = j - n_b + 1 at the anchor's position + d. Training: pos =
// row_pos[r]. Layer 0 also seeds the residual stream h with the row's layer-0
// residual. Decode can append the new rows' K/V to their cache slots
// kv_off[b] + kv_len[b] + j.
// -------------------------------------------------------------------------
template <typename T, int HD>
__global__ void __launch_bounds__(kQkvThreads) qkv_finish_kernel(QkvArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int HALF = HD / 2;
  const int r = blockIdx.x + a.row0;
  int src = -1, pos = 0, b = 0, j = 0, nb = 1;
  const bool decode = !a.row_pos;
  if (!decode) {
    src = a.mode == 0 ? r - a.src0 : -1;
    pos = a.row_pos[r];
  } else {
    b = dr_request(a.rows, r, &j);
    if (!dr_valid(a.rows, b) || j < 0 || j >= dr_new(a.rows, b) + a.K - 1) {
      if (threadIdx.x == 0 && blockIdx.y == 0) set_status(a.status, PEAGLE_DEV_BOUNDS);
      return;
    }
    nb = dr_new(a.rows, b);
    const int first = a.rows.new_off ? a.rows.new_off[b] : b;   // new-row index of (b, 0)
    if (a.mode == 0) src = r - a.src0;
    else src = j < nb ? first + j : -1;
    pos = j < nb ? a.anchor_pos[first + j] : a.anchor_pos[first + nb - 1] + (j - nb + 1);
  }
  if (pos < 0 || pos >= a.max_pos) {
    if (threadIdx.x == 0) set_status(a.status, PEAGLE_DEV_BOUNDS);
    pos = pos < 0 ? 0 : a.max_pos - 1;
  }
  T* Q = static_cast<T*>(a.Q) + (size_t)r * a.nq * HD;
  T* Ko = static_cast<T*>(a.Kout) + (size_t)r * a.nkv * HD;
  T* Vo = static_cast<T*>(a.Vout) + (size_t)r * a.nkv * HD;
  const float* cs = a.rcos + (size_t)pos * HALF;
  const float* sn = a.rsin + (size_t)pos * HALF;
  const float* in = src >= 0 ? a.in.out + (size_t)src * a.in.ldo : a.mask_qkv;
  const float* hin = !a.h ? nullptr : (src >= 0 ? a.resid0 + (size_t)src * a.H : a.mask_resid);

  bool append = false;
  size_t cache_row = 0;
  if (a.kcache && decode && j < nb) {   // a decode new row, every layer
    const long long row = a.kv_off[b] + (long long)a.kv_len[b] + j;
    if (a.kv_len[b] >= 0 && row < a.kv_off[b + 1] && row < a.kv_cap && a.kv_off[b] >= 0) {
      append = true;
      cache_row = (size_t)row;
    } else if (threadIdx.x == 0 && blockIdx.y == 0) {
      set_status(a.status, PEAGLE_DEV_BOUNDS);
    }
  }
  // this block's slice of the row: rotary pairs of q/k heads, then v
  // elements, then (layer 0) the residual seed; every operand of the
  // thread's elements is loaded before the first store
  const int pairs = (a.nq + a.nkv) * HALF;
  const int vcount = a.nkv * HD;
  const int total = pairs + vcount + (a.h ? a.H : 0);
  const int v0 = (a.nq + a.nkv) * HD;
  const int e0 = blockIdx.y * kQkvChunk + threadIdx.x;
  float x[kQkvEpt], y[kQkvEpt], c[kQkvEpt], sv[kQkvEpt];
#pragma unroll
  for (int i = 0; i < kQkvEpt; ++i) {
    const int e = e0 + i * kQkvThreads;
    x[i] = y[i] = c[i] = sv[i] = 0.f;
    if (e < pairs) {
      const int lo = (e / HALF) * HD + e % HALF;
      x[i] = in[lo];
      y[i] = in[lo + HALF];
      c[i] = cs[e % HALF];
      sv[i] = sn[e % HALF];
    } else if (e < pairs + vcount) {
      x[i] = in[v0 + e - pairs];
    } else if (e < total) {
      x[i] = hin[e - pairs - vcount];
    }
  }
#pragma unroll
  for (int i = 0; i < kQkvEpt; ++i) {
    const int e = e0 + i * kQkvThreads;
    if (e < pairs) {
      const int head = e / HALF, j = e % HALF;
      const float ol = x[i] * c[i] - y[i] * sv[i], oh = y[i] * c[i] + x[i] * sv[i];
      if (head < a.nq) {
        Q[head * HD + j] = from_f<T>(ol);
        Q[head * HD + j + HALF] = from_f<T>(oh);
      } else {
        const int kh = head - a.nq;
        Ko[kh * HD + j] = from_f<T>(ol);
        Ko[kh * HD + j + HALF] = from_f<T>(oh);
        if (append) {
          T* kc = static_cast<T*>(a.kcache) + cache_row * a.nkv * HD;
          kc[kh * HD + j] = from_f<T>(ol);
          kc[kh * HD + j + HALF] = from_f<T>(oh);
        }
      }
    } else if (e < pairs + vcount) {
      const int ev = e - pairs;
      Vo[ev] = from_f<T>(x[i]);
      if (append) static_cast<T*>(a.vcache)[cache_row * a.nkv * HD + ev] = from_f<T>(x[i]);
    } else if (e < total) {
      a.h[(size_t)r * a.H + e - pairs - vcount] = x[i];
    }
  }
}

// -------------------------------------------------------------------------
// Residual add + RMSNorm: h[r] += sum of partials; y[r] = RMSNorm_gain(h[r]).
// (Llama layer: after O-proj with the post-attention gain; after the MLP
// down-proj with the next layer's input gain or the final gain.)
// -------------------------------------------------------------------------
template <typename T, int EPT>
__global__ void resid_norm_kernel(ResidNormArgs a) {
  pdl_trigger();
  __shared__ float red[3][32];
  const int rl = blockIdx.x;           // row within the chunk
  const int r = a.row0 + rl;           // global row
  const int H = a.H, bd = blockDim.x, tid = threadIdx.x;
  const T* g = static_cast<const T*>(a.gain);
  float gv[EPT], v[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int j = tid + i * bd;
    gv[i] = j < H ? to_f(g[j]) : 0.f;
  }
  pdl_wait();
  float* h = a.h + (size_t)r * H;
  const float* ur = a.in.out + (size_t)rl * a.in.ldo;
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int j = tid + i * bd;
    v[i] = j < H ? h[j] + ur[j] : 0.f;
  }
  for (int q = 1; q < a.in.splits; ++q) {
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const int j = tid + i * bd;
      if (j < H) v[i] += ur[(size_t)q * a.in.split_stride + j];
    }
  }
  float ss = 0.f, d1 = 0.f, d2 = 0.f;
#pragma unroll
  for (int i = 0; i < EPT; ++i) ss += v[i] * v[i];
  block_sum3(ss, d1, d2, red);
  const float inv = rsqrtf(ss / H + a.eps);
  // the final norm of a decode step keeps only each request's depth rows
  // (the anchor and the masked rows), packed as row b * K + depth
  long long yrow = r;
  if (a.compact) {
    int jj;
    const int b = dr_request(a.crows, r, &jj);
    const int d = jj - (dr_new(a.crows, b) - 1);
    yrow = (dr_valid(a.crows, b) && d >= 0 && d < a.crows.K) ? (long long)b * a.crows.K + d : -1;
  }
  T* y = static_cast<T*>(a.y) + (yrow >= 0 ? (size_t)yrow * H : 0);
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int j = tid + i * bd;
    if (j < H) {
      h[j] = v[i];
      if (yrow >= 0) y[j] = from_f<T>(v[i] * inv * gv[i]);
    }
  }
}

// -------------------------------------------------------------------------
// SwiGLU: act[r, j] = silu(gate) * up, gate/up = columns j and I + j.
// -------------------------------------------------------------------------
template <typename T>
__global__ void swiglu_kernel(GemmOut in, int rows, int I, void* act_) {
  pdl_trigger();
  pdl_wait();
  T* act = static_cast<T*>(act_);
  // rows over blocks, columns over threads: coalesced, no index division
  for (int r = blockIdx.x; r < rows; r += gridDim.x)
    for (int j = threadIdx.x; j < I; j += blockDim.x) {
      const float gt = sum_parts(in, (size_t)r * in.ldo + j);
      const float up = sum_parts(in, (size_t)r * in.ldo + I + j);
      act[(size_t)r * I + j] = from_f<T>(gt / (1.f + expf(-gt)) * up);
    }
}

// -------------------------------------------------------------------------
// Draft-vocab argmax, two stages: per (row, vocab chunk) best pair, then per
// row over chunks, mapped through d2t. Lowest index wins ties.
// -------------------------------------------------------------------------
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (am_better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

__global__ void lm_argmax_partial_kernel(GemmOut in, int V, int chunk, float* logits, float* pval,
                                         int* pidx) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sv[32];
  __shared__ int si[32];
  const int r = blockIdx.y, c = blockIdx.x, nchunks = gridDim.x;
  const int v0 = c * chunk, v1 = min(V, v0 + chunk);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
#pragma unroll 8
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    const float x = sum_parts(in, (size_t)r * in.ldo + v);
    if (logits) logits[(size_t)r * V + v] = x;
    if (am_better(x, v, bv, bi)) {
      bv = x;
      bi = v;
    }
  }
  warp_argmax(bv, bi);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) {
    sv[w] = bv;
    si[w] = bi;
  }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    bv = lane < nw ? sv[lane] : -INFINITY;
    bi = lane < nw ? si[lane] : 0x7fffffff;
    warp_argmax(bv, bi);
    if (lane == 0) {
      pval[(size_t)r * nchunks + c] = bv;
      pidx[(size_t)r * nchunks + c] = bi;
    }
  }
}

__global__ void lm_argmax_final_kernel(int rows, int nchunks, const float* pval, const int* pidx,
                                       const int* d2t, int* tokens) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = lane; c < nchunks; c += 32) {
    const float v = pval[(size_t)r * nchunks + c];
    const int i = pidx[(size_t)r * nchunks + c];
    if (am_better(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
  warp_argmax(bv, bi);
  if (lane == 0) tokens[r] = d2t ? d2t[bi] : bi;
}

// -------------------------------------------------------------------------
// Per-row cross-entropy over the draft vocab (#2376: CE per depth, shared
// with EAGLE-3), one pass with an online max / sum of exponentials.
// row_ce = logsumexp - logit[label], NaN for rows without a label.
// -------------------------------------------------------------------------
__global__ void ce_rows_kernel(GemmOut in, int V, int row0, const int* row_label, float* logits_out,
                               float* row_ce, int* row_am) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm[32], ss[32], sv[32];
  __shared__ int si[32];
  const int rl = blockIdx.x, r = row0 + rl;
  float m = -INFINITY, s = 0.f, bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = sum_parts(in, (size_t)rl * in.ldo + v);
    if (logits_out) logits_out[(size_t)r * V + v] = x;
    if (am_better(x, v, bv, bi)) {
      bv = x;
      bi = v;
    }
    if (x > m) {
      s = s * expf(m - x) + 1.f;
      m = x;
    } else {
      s += expf(x - m);
    }
  }
  // combine (m, s) across the warp
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    const float nm = fmaxf(m, om);
    s = (m == -INFINITY ? 0.f : s * expf(m - nm)) + (om == -INFINITY ? 0.f : os * expf(om - nm));
    m = nm;
  }
  warp_argmax(bv, bi);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) {
    sm[w] = m;
    ss[w] = s;
    sv[w] = bv;
    si[w] = bi;
  }
  __syncthreads();
  if (w == 0) {
    m = lane < nw ? sm[lane] : -INFINITY;
    s = lane < nw ? ss[lane] : 0.f;
    bv = lane < nw ? sv[lane] : -INFINITY;
    bi = lane < nw ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, o);
      const float os = __shfl_xor_sync(0xffffffffu, s, o);
      const float nm = fmaxf(m, om);
      s = (m == -INFINITY ? 0.f : s * expf(m - nm)) + (om == -INFINITY ? 0.f : os * expf(om - nm));
      m = nm;
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      const int lab = row_label[r];
      float ce = __int_as_float(0x7fc00000);
      if (lab >= 0) ce = (m + logf(s)) - sum_parts(in, (size_t)rl * in.ldo + lab);
      row_ce[r] = ce;
      row_am[r] = bi;
    }
  }
}

// Row cross-entropy and argmax from the fused head epilogue's per-tile
// partials: logsumexp = M + log(sum_t s_t exp(m_t - M)); the label's logit
// comes from the one tile that holds it. A warp per row.
__global__ void ce_merge_kernel(int rows, int part_ld, int row0, const float* p_max, const float* p_sum,
                                const float* p_lab, const int* p_idx, const int* row_label, float* row_ce,
                                int* row_am) {
  pdl_trigger();
  pdl_wait();
  const int rl = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rl >= rows) return;
  const size_t base = (size_t)rl * part_ld;
  float M = -INFINITY, ll = -INFINITY, bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int t = lane; t < part_ld; t += 32) {
    const float mt = p_max[base + t];
    M = fmaxf(M, mt);
    ll = fmaxf(ll, p_lab[base + t]);
    if (am_better(mt, p_idx[base + t], bv, bi)) {
      bv = mt;
      bi = p_idx[base + t];
    }
  }
  M = warp_max(M);
  ll = warp_max(ll);
  warp_argmax(bv, bi);
  float sum = 0.f;
  for (int t = lane; t < part_ld; t += 32) {
    const float mt = p_max[base + t];
    if (mt != -INFINITY) sum += p_sum[base + t] * expf(mt - M);
  }
  sum = warp_sum(sum);
  if (lane == 0) {
    const int r = row0 + rl;
    const int lab = row_label[r];
    row_ce[r] = lab >= 0 ? (M + logf(sum)) - ll : __int_as_float(0x7fc00000);
    row_am[r] = bi;
  }
}

// Per-depth means and the decay-weighted total (#2376, Changelog: 0.8**d
// weighted-mean schedule). One block; fixed summation order.
__global__ void ce_reduce_kernel(CeReduceArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ double red_d[32];
  __shared__ int red_i[32], red_j[32];
  __shared__ double loss_acc;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) loss_acc = 0.0;
  for (int d = 0; d < a.K; ++d) {
    double sum = 0.0;
    int cnt = 0, cor = 0;
    for (int r = a.off[d] + threadIdx.x; r < a.off[d + 1]; r += blockDim.x) {
      const int lab = a.row_label[r];
      if (lab >= 0) {
        sum += (double)a.row_ce[r];
        cnt += 1;
        cor += (a.row_am[r] == lab) ? 1 : 0;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      cor += __shfl_xor_sync(0xffffffffu, cor, o);
    }
    __syncthreads();
    if (lane == 0) {
      red_d[w] = sum;
      red_i[w] = cnt;
      red_j[w] = cor;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      double S = 0.0;
      int C = 0, R = 0;
      for (int i = 0; i < nw; ++i) {
        S += red_d[i];
        C += red_i[i];
        R += red_j[i];
      }
      const double ld = C ? S / C : 0.0;
      a.loss_d[d] = (float)ld;
      a.acc_d[d] = C ? (float)((double)R / C) : 0.f;
      a.valid_d[d] = C;
      loss_acc += pow(a.decay, (double)d) * ld;
      if (a.sums) {   // this sequence's share of a batch (one stream: no race)
        a.sums[d] += S;
        a.sums[a.K + d] += (double)R;
        a.sums[2 * a.K + d] += (double)C;
      }
    }
  }
  if (threadIdx.x == 0) a.loss[0] = (float)loss_acc;
}

// Per-depth mean CE, accuracy and label count, and the loss
// sum_d decay^d * mean_d, from depth sums added over several packed
// sequences (and ranks): the same arithmetic as the single-sequence reduction.
__global__ void depth_sums_combine_kernel(int K, double decay, const double* sums, float* loss_d, float* acc_d,
                                          int* valid_d, float* loss) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x != 0) return;
  double acc = 0.0;
  for (int d = 0; d < K; ++d) {
    const double S = sums[d], R = sums[K + d], C = sums[2 * K + d];
    const double ld = C > 0 ? S / C : 0.0;
    loss_d[d] = (float)ld;
    acc_d[d] = C > 0 ? (float)(R / C) : 0.f;
    valid_d[d] = (int)C;
    acc += pow(decay, (double)d) * ld;
  }
  loss[0] = (float)acc;
}

// -------------------------------------------------------------------------
// Training rows: depth, anchor, rotary position, conversation start and
// label of every row (#2376, PR description; "P_Eagle" README: cu_seqlens
// isolation). Row r of depth d has anchor i = indices[r]; its label is
// labels[i + d] when i + d is inside i's conversation, unmasked and mapped
// into the draft vocab, else -1.
// -------------------------------------------------------------------------
__global__ void train_meta_kernel(TrainMetaArgs a) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    bool ok = a.cu[0] == 0 && a.cu[a.S] == a.n;
    for (int c = 0; c < a.S; ++c) ok = ok && a.cu[c] <= a.cu[c + 1];
    if (!ok) set_status(a.status, PEAGLE_DEV_BOUNDS);
  }
  if (r >= a.R) return;
  int d = 0;
  while (d + 1 < a.K && r >= a.off[d + 1]) ++d;
  int i = a.indices[r];
  if (i < 0 || i >= a.n) {
    set_status(a.status, PEAGLE_DEV_BOUNDS);
    i = 0;
  }
  int lo = 0, hi = a.S - 1;  // conversation c with cu[c] <= i < cu[c+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (a.cu[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const int s = a.cu[lo], e = a.cu[lo + 1];
  int pos = a.position_ids[i] + d;
  if (pos < 0 || pos >= a.max_pos) {
    set_status(a.status, PEAGLE_DEV_BOUNDS);
    pos = pos < 0 ? 0 : a.max_pos - 1;
  }
  int lab = -1;
  const int p = i + d;
  if (p < e && (!a.loss_mask || a.loss_mask[p])) {
    const int t = a.labels[p];
    if (t < 0 || t >= a.Vt) {
      set_status(a.status, PEAGLE_DEV_BOUNDS);
    } else {
      const int dl = a.t2d ? a.t2d[t] : t;
      if (dl >= a.Vd) set_status(a.status, PEAGLE_DEV_BOUNDS);
      else lab = dl;
    }
  }
  a.row_anchor[r] = i;
  a.row_depth[r] = d;
  a.row_pos[r] = pos;
  a.row_start[r] = s;
  a.row_label[r] = lab;
  if (a.row_end) a.row_end[r] = e;
}

// -------------------------------------------------------------------------
// Greedy verification ("P-EAGLE" user guide, Inference Process): accept the
// longest prefix of drafts equal to the target's tokens; next = target at
// the first mismatch (or the bonus column).
// -------------------------------------------------------------------------
__global__ void verify_kernel(int B, int K, const int* draft, const int* target, int* acc, int* next) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int* d = draft + (size_t)b * K;
  const int* t = target + (size_t)b * (K + 1);
  int a = 0;
  while (a < K && d[a] == t[a]) ++a;
  acc[b] = a;
  next[b] = t[a];
}

// -------------------------------------------------------------------------
// COD selection ("P-EAGLE" user guide, COD Sampling). Keys are SplitMix64
// outputs (Steele, Lea, Flood, OOPSLA 2014), distinct for distinct i.
// S_d = positions whose key is at most the counts[d]-th smallest key. One
// block: an 8-pass radix select finds every depth's threshold key at once,
// then a block scan writes each S_d in ascending order.
// -------------------------------------------------------------------------
__device__ __forceinline__ uint64_t splitmix64_out(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void __launch_bounds__(1024) cod_select_kernel(CodArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned hist[16][256];
  __shared__ uint64_t prefix[16], maskv[16], thr[16];
  __shared__ int rank_left[16], wsum[32], base[16];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int n = a.n, K = a.K;
  if (tid < 16) {
    prefix[tid] = 0;
    maskv[tid] = 0;
    rank_left[tid] = (tid < K) ? a.counts[tid] : 0;
    base[tid] = 0;
  }
  __syncthreads();
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int e = tid; e < 16 * 256; e += blockDim.x) hist[e >> 8][e & 255] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
      const uint64_t key = splitmix64_out(a.seed, (uint64_t)i);
      const unsigned dig = (unsigned)(key >> shift) & 255u;
      for (int d = 1; d < K; ++d)
        if (rank_left[d] > 0 && a.counts[d] < n && (key & maskv[d]) == prefix[d]) atomicAdd(&hist[d][dig], 1u);
    }
    __syncthreads();
    if (tid >= 1 && tid < K && rank_left[tid] > 0 && a.counts[tid] < n) {
      int left = rank_left[tid];
      unsigned bsel = 255;
      for (unsigned b = 0; b < 256; ++b) {
        const int c = (int)hist[tid][b];
        if (left <= c) {
          bsel = b;
          break;
        }
        left -= c;
      }
      rank_left[tid] = left;
      prefix[tid] |= (uint64_t)bsel << shift;
      maskv[tid] |= (uint64_t)255 << shift;
    }
    __syncthreads();
  }
  if (tid < 16) {
    if (tid == 0 || (tid < K && a.counts[tid] >= n)) thr[tid] = ~0ull;   // keep everything
    else if (tid < K && a.counts[tid] > 0) thr[tid] = prefix[tid];
    else thr[tid] = 0;                                                    // keep nothing
  }
  __syncthreads();
  // ascending compaction, tile by tile
  for (int t0 = 0; t0 < n; t0 += blockDim.x) {
    const int i = t0 + tid;
    const bool live = i < n;
    uint64_t key = live ? splitmix64_out(a.seed, (uint64_t)i) : 0;
    if (live) {
      a.indices[i] = i;
      if (a.row_of) a.row_of[i] = i;
    }
    for (int d = 1; d < K; ++d) {
      const bool keep = live && a.counts[d] > 0 && key <= thr[d];
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (lane == 0) wsum[w] = __popc(bal);
      __syncthreads();
      if (w == 0) {
        const int nw = blockDim.x >> 5;
        int v = lane < nw ? wsum[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane < nw) wsum[lane] = incl - v;   // exclusive warp offsets
        if (lane == 31) rank_left[0] = incl;    // tile total (scratch slot)
      }
      __syncthreads();
      const int pos = base[d] + wsum[w] + __popc(bal & ((1u << lane) - 1u));
      const bool fits = keep && pos < a.counts[d];   // always true for distinct keys
      if (fits) a.indices[a.off[d] + pos] = i;
      if (live && a.row_of) a.row_of[(size_t)d * n + i] = fits ? a.off[d] + pos : -1;
      __syncthreads();
      if (tid == 0) base[d] += rank_left[0];
      __syncthreads();
    }
  }
}

// D = sum of the partial slabs (the plain GEMM entry point).
__global__ void sum_splits_kernel(GemmOut in, int M, int N, float* D) {
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)M * N;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(e / N), n = (int)(e % N);
    D[e] = sum_parts(in, (size_t)m * in.ldo + n);
  }
}

// ------------------------------------------------------ host staging
// Copies between mapped page-locked host memory and device memory run as
// kernels so they stay in the stream's chain of dependent launches. The
// copy to the device loads its first batch (host memory, which no kernel
// of the chain writes) before waiting for the previous kernel; only its
// stores wait. 16-byte vectors, R per thread in flight.
constexpr int kStageR = 4;
__global__ void __launch_bounds__(256) copy_to_device_kernel(uint4* __restrict__ dst, const uint4* src,
                                                             long long n16) {
  pdl_trigger();
  const long long stride = (long long)gridDim.x * blockDim.x * kStageR;
  long long base = (long long)blockIdx.x * blockDim.x * kStageR + threadIdx.x;
  uint4 v[kStageR];
#pragma unroll
  for (int r = 0; r < kStageR; ++r) {
    const long long i = base + (long long)r * blockDim.x;
    if (i < n16) v[r] = src[i];
  }
  pdl_wait();
  for (;;) {
#pragma unroll
    for (int r = 0; r < kStageR; ++r) {
      const long long i = base + (long long)r * blockDim.x;
      if (i < n16) dst[i] = v[r];
    }
    base += stride;
    if (base >= n16) break;
#pragma unroll
    for (int r = 0; r < kStageR; ++r) {
      const long long i = base + (long long)r * blockDim.x;
      if (i < n16) v[r] = src[i];
    }
  }
}

// The copy to the host reads device memory an earlier kernel may write, so
// it waits first.
__global__ void __launch_bounds__(256) copy_to_host_kernel(uint4* dst, const uint4* __restrict__ src,
                                                           long long n16) {
  pdl_trigger();
  pdl_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// Byte copies for sizes or addresses off the 16-byte grid (either direction).
__global__ void __launch_bounds__(256) copy_bytes_kernel(uint8_t* dst, const uint8_t* src, long long n) {
  pdl_trigger();
  pdl_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// =========================================================================
// launchers
// =========================================================================
static int grid_for(long long total, int threads) {
  long long g = (total + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 8;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

// Block shape of a one-row-per-block kernel: EPT columns per thread in
// registers (4, 8 or 16, the fewest that cover the row with at most 1024
// threads), so each thread keeps all its loads in flight at once.
static int row_threads(int /*rows*/, int H, int* ept) {
  const int t0 = 1024;
  int e = 4;
  while (e < 16 && e * t0 < H) e *= 2;
  *ept = e;
  const int t = ((H + e - 1) / e + 31) / 32 * 32;
  return std::max(32, std::min(1024, t));
}

#define PE_LAUNCH_END() \
  do {                  \
    note_launch();      \
    return cudaGetLastError(); \
  } while (0)

cudaError_t launch_rope_table(float* c, float* s, int max_pos, int hd, double theta, cudaStream_t st) {
  const long long total = (long long)max_pos * (hd / 2);
  launch_pdl(rope_table_kernel, grid_for(total, 256), 256, 0, st, c, s, max_pos, hd / 2, hd, theta);
  PE_LAUNCH_END();
}

template <typename T>
static void fc_finish_dispatch(int rows, int threads, int ept, const FcFinishArgs& a, cudaStream_t st) {
  if (ept == 4) launch_pdl(fc_finish_kernel<T, 4>, rows, threads, 0, st, a);
  else if (ept == 8) launch_pdl(fc_finish_kernel<T, 8>, rows, threads, 0, st, a);
  else launch_pdl(fc_finish_kernel<T, 16>, rows, threads, 0, st, a);
}

cudaError_t launch_fc_finish(int dtype, int rows, const FcFinishArgs& a, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  int ept;
  const int threads = row_threads(rows, a.H, &ept);
  if (dtype == PEAGLE_BF16) fc_finish_dispatch<bf16>(rows, threads, ept, a, st);
  else fc_finish_dispatch<float>(rows, threads, ept, a, st);
  PE_LAUNCH_END();
}

cudaError_t launch_qkv_finish(int dtype, int rows, const QkvArgs& a, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int total = (a.nq + a.nkv) * (a.hd / 2) + a.nkv * a.hd + (a.h ? a.H : 0);
  if (a.in.splits != 1) {
    set_error("qkv_finish expects one partial slab");
    return cudaErrorInvalidValue;
  }
  const dim3 grid(rows, (total + kQkvChunk - 1) / kQkvChunk);
  if (dtype == PEAGLE_BF16) {
    if (a.hd == 128) launch_pdl(qkv_finish_kernel<bf16, 128>, grid, kQkvThreads, 0, st, a);
    else launch_pdl(qkv_finish_kernel<bf16, 64>, grid, kQkvThreads, 0, st, a);
  } else {
    if (a.hd == 128) launch_pdl(qkv_finish_kernel<float, 128>, grid, kQkvThreads, 0, st, a);
    else launch_pdl(qkv_finish_kernel<float, 64>, grid, kQkvThreads, 0, st, a);
  }
  PE_LAUNCH_END();
}

template <typename T>
static void resid_norm_dispatch(int rows, int threads, int ept, const ResidNormArgs& a, cudaStream_t st) {
  if (ept == 4) launch_pdl(resid_norm_kernel<T, 4>, rows, threads, 0, st, a);
  else if (ept == 8) launch_pdl(resid_norm_kernel<T, 8>, rows, threads, 0, st, a);
  else launch_pdl(resid_norm_kernel<T, 16>, rows, threads, 0, st, a);
}

cudaError_t launch_resid_norm(int dtype, int rows, const ResidNormArgs& a, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  int ept;
  const int threads = row_threads(rows, a.H, &ept);
  if (dtype == PEAGLE_BF16) resid_norm_dispatch<bf16>(rows, threads, ept, a, st);
  else resid_norm_dispatch<float>(rows, threads, ept, a, st);
  PE_LAUNCH_END();
}

cudaError_t launch_swiglu(int dtype, const GemmOut& in, int rows, int I, void* act, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int grid = std::min(rows, num_sms() * 8);
  if (dtype == PEAGLE_BF16) launch_pdl(swiglu_kernel<bf16>, grid, 256, 0, st, in, rows, I, act);
  else launch_pdl(swiglu_kernel<float>, grid, 256, 0, st, in, rows, I, act);
  PE_LAUNCH_END();
}

int lm_argmax_chunks(int V) { return (V + 2047) / 2048; }

cudaError_t launch_lm_argmax(const GemmOut& in, int rows, int V, float* logits, float* pval, int* pidx,
                             const int* d2t, int* tokens, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int nch = lm_argmax_chunks(V);
  launch_pdl(lm_argmax_partial_kernel, dim3(nch, rows), 256, 0, st, in, V, 2048, logits, pval, pidx);
  note_launch();
  launch_pdl(lm_argmax_final_kernel, (rows + 7) / 8, 256, 0, st, rows, nch, pval, pidx, d2t, tokens);
  PE_LAUNCH_END();
}

cudaError_t launch_ce_rows(const GemmOut& in, int rows, int V, int row0, const int* row_label,
                           float* logits_out, float* row_ce, int* row_am, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  launch_pdl(ce_rows_kernel, rows, 256, 0, st, in, V, row0, row_label, logits_out, row_ce, row_am);
  PE_LAUNCH_END();
}

cudaError_t launch_ce_merge(int rows, int part_ld, int row0, const float* p_max, const float* p_sum,
                            const float* p_lab, const int* p_idx, const int* row_label, float* row_ce, int* row_am,
                            cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  launch_pdl(ce_merge_kernel, (rows + 7) / 8, 256, 0, st, rows, part_ld, row0, p_max, p_sum, p_lab, p_idx, row_label, row_ce,
                                                  row_am);
  PE_LAUNCH_END();
}

cudaError_t launch_lm_argmax_final(int rows, int nchunks, const float* pval, const int* pidx, const int* d2t,
                                   int* tokens, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  launch_pdl(lm_argmax_final_kernel, (rows + 7) / 8, 256, 0, st, rows, nchunks, pval, pidx, d2t, tokens);
  PE_LAUNCH_END();
}

cudaError_t launch_ce_reduce(const CeReduceArgs& a, cudaStream_t st) {
  launch_pdl(ce_reduce_kernel, 1, 1024, 0, st, a);
  PE_LAUNCH_END();
}

// -------------------------------------------------------------------------
// The next draft step's new rows after verification ("P-EAGLE" user guide,
// Inference Process: the accepted drafts are kept, the target supplies the
// next token, and the next round continues from there). Request b: the
// current step's n_b rows become context (kv_lens[b] += n_b); the next step
// brings a_b + 1 rows -- drafts 0..a_b-1 and the next token -- at the
// positions after the current anchor. One CTA: a block scan of the counts.
// -------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) next_context_kernel(NextContextArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int b0 = 0; b0 < a.B; b0 += 1024) {
    const int b = b0 + tid;
    int n = 0, acc = 0, cur_lo = 0, cur_hi = 0;
    if (b < a.B) {
      cur_lo = a.cur_off[b];
      cur_hi = a.cur_off[b + 1];
      acc = a.accept[b];
      if (acc < 0 || acc > a.K || cur_hi <= cur_lo) {
        set_status(a.status, PEAGLE_DEV_BOUNDS);
        acc = acc < 0 ? 0 : (acc > a.K ? a.K : acc);
      }
      n = acc + 1;
    }
    int incl = n;   // inclusive scan of n over the block
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[w] = incl;
    __syncthreads();
    int before = s_carry;
    for (int i = 0; i < w; ++i) before += s_warp[i];
    const int off = before + incl - n;
    if (b < a.B) {
      a.next_off[b] = off;
      if (cur_hi > cur_lo) a.kv_lens[b] += cur_hi - cur_lo;
      const int p = cur_hi > cur_lo ? a.cur_pos[cur_hi - 1] : 0;   // the current anchor's position
      for (int j = 0; j < n; ++j) {
        a.next_tok[off + j] = j < acc ? a.drafts[(size_t)b * a.K + j] : a.next[b];
        a.next_pos[off + j] = p + 1 + j;
      }
    }
    __syncthreads();
    if (tid == 1023) s_carry = off + n;
    __syncthreads();
  }
  if (tid == 0) a.next_off[a.B] = s_carry;
}

cudaError_t launch_next_context(const NextContextArgs& a, cudaStream_t st) {
  launch_pdl(next_context_kernel, 1, 1024, 0, st, a);
  PE_LAUNCH_END();
}

cudaError_t launch_depth_sums_combine(int K, double decay, const double* sums, float* loss_d, float* acc_d,
                                      int* valid_d, float* loss, cudaStream_t st) {
  launch_pdl(depth_sums_combine_kernel, 1, 32, 0, st, K, decay, sums, loss_d, acc_d, valid_d, loss);
  PE_LAUNCH_END();
}

cudaError_t launch_train_meta(const TrainMetaArgs& a, cudaStream_t st) {
  if (a.R <= 0) return cudaSuccess;
  launch_pdl(train_meta_kernel, (a.R + 255) / 256, 256, 0, st, a);
  PE_LAUNCH_END();
}

cudaError_t launch_verify(int B, int K, const int* d, const int* t, int* acc, int* next, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  launch_pdl(verify_kernel, (B + 127) / 128, 128, 0, st, B, K, d, t, acc, next);
  PE_LAUNCH_END();
}

cudaError_t launch_cod_select(const CodArgs& a, cudaStream_t st) {
  if (a.n <= 0) return cudaSuccess;
  launch_pdl(cod_select_kernel, 1, 1024, 0, st, a);
  PE_LAUNCH_END();
}

cudaError_t launch_sum_splits(const GemmOut& in, int M, int N, float* D, cudaStream_t st) {
  const long long total = (long long)M * N;
  if (total <= 0) return cudaSuccess;
  launch_pdl(sum_splits_kernel, grid_for(total, 256), 256, 0, st, in, M, N, D);
  PE_LAUNCH_END();
}

cudaError_t launch_stage_copy(void* dst, const void* src, long long bytes, bool to_device, cudaStream_t st) {
  if (bytes <= 0) return cudaSuccess;
  const bool vec = (bytes & 15) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(src) & 15) == 0;
  if (!vec) {
    launch_pdl(copy_bytes_kernel, grid_for(bytes, 256), 256, 0, st, static_cast<uint8_t*>(dst),
               static_cast<const uint8_t*>(src), bytes);
    PE_LAUNCH_END();
  }
  const long long n16 = bytes / 16;
  if (to_device) {
    const long long per_block = 256LL * kStageR;
    const long long want = (n16 + per_block - 1) / per_block;
    const int grid = (int)std::min<long long>(want, (long long)num_sms() * 8);
    launch_pdl(copy_to_device_kernel, std::max(grid, 1), 256, 0, st, static_cast<uint4*>(dst),
               static_cast<const uint4*>(src), n16);
  } else {
    launch_pdl(copy_to_host_kernel, grid_for(n16, 256), 256, 0, st, static_cast<uint4*>(dst),
               static_cast<const uint4*>(src), n16);
  }
  PE_LAUNCH_END();
}

}  // namespace pe

// Kernels of the backward pass of the training-shaped forward ("feat(
// speculative): add P-EAGLE parallel-drafting training for EAGLE-3 drafts -
// #2376", PR description and Changelog: the trainer runs the parallel
// masked-depth loss). The contractions of the backward are the library's
// GEMM on transposed copies; the pieces between them live here:
//   the cross-entropy gradient, RMSNorm and its gain, SwiGLU, RoPE (rotation
//   by minus the angle), and the depth-masked attention (a query-major pass
//   for dQ, a key-major pass for dK and dV over the rows that see each key).
#include <math.h>

#include "rows.cuh"

namespace pe {

namespace {

template <typename T>
__device__ __forceinline__ float ld_f(const T* p) { return to_f(*p); }

// ---------------------------------------------------------------- layout
template <typename T>
__global__ void __launch_bounds__(256) transpose_kernel(const T* __restrict__ src, int rows, int cols, int lds,
                                                        T* __restrict__ dst, int ldd, int rows_pad) {
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[32][33];
  const int r0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    const int r = r0 + ty + k, c = c0 + tx;
    tile[ty + k][tx] = (r < rows && c < cols) ? to_f(src[(size_t)r * lds + c]) : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    const int c = c0 + ty + k, r = r0 + tx;
    if (c < cols && r < rows_pad) dst[(size_t)c * ldd + r] = from_f<T>(tile[tx][ty + k]);
  }
}

// bf16 with even widths and strides: 64 x 64 tiles moved as bf16 pairs, so
// every warp access is one 128-byte row
__global__ void __launch_bounds__(256) transpose_bf16x2_kernel(const bf16* __restrict__ src, int rows, int cols,
                                                               int lds, bf16* __restrict__ dst, int ldd, int rows_pad) {
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[64][65];
  const int r0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < 64; k += 8) {
    const int r = r0 + ty + k, c = c0 + 2 * tx;
    float2 v = make_float2(0.f, 0.f);
    if (r < rows && c < cols) v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + (size_t)r * lds + c));
    tile[ty + k][2 * tx] = v.x;
    tile[ty + k][2 * tx + 1] = v.y;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 64; k += 8) {
    const int c = c0 + ty + k, r = r0 + 2 * tx;
    if (c < cols && r < rows_pad)
      *reinterpret_cast<__nv_bfloat162*>(dst + (size_t)c * ldd + r) =
          __floats2bfloat162_rn(tile[2 * tx][ty + k], tile[2 * tx + 1][ty + k]);
  }
}

template <typename T>
__global__ void cast_kernel(const float* __restrict__ src, T* __restrict__ dst, long long count) {
  pdl_trigger();
  pdl_wait();
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < count; e += (long long)gridDim.x * blockDim.x)
    dst[e] = from_f<T>(src[e]);
}

// rows r < n copy source row r, rows r >= n copy source row n (the shared
// masked row)
template <typename T>
__global__ void gather_masked_kernel(const T* __restrict__ src, int n, int rows, int cols, T* __restrict__ dst) {
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)rows * cols;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(e / cols), c = (int)(e % cols);
    dst[e] = src[(size_t)(r < n ? r : n) * cols + c];
  }
}

// out[r][c] = a[r][c] + b[r][c]
__global__ void add_rows_kernel(const float* __restrict__ a, int lda, const float* __restrict__ b, int ldb,
                                float* __restrict__ out, int ldo, int rows, int cols) {
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)rows * cols;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(e / cols), c = (int)(e % cols);
    out[(size_t)r * ldo + c] = a[(size_t)r * lda + c] + b[(size_t)r * ldb + c];
  }
}

// dst[c] = sum of src[r][c] over rows [r0, r1)
__global__ void colsum_kernel(const float* __restrict__ src, int ld, int r0, int r1, int cols, float* __restrict__ dst) {
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  float s = 0.f;
  for (int r = r0; r < r1; ++r) s += src[(size_t)r * ld + c];
  dst[c] = s;
}

// -------------------------------------------------------- cross-entropy
// Gradient of sum_d decay^d * mean_d CE with respect to the logits of row r:
// w_r * (softmax(logits_r) - onehot(label_r)), w_r = decay^depth / (labelled
// rows of that depth); rows without a label get zeros. The forward's row CE
// gives the log-sum-exp (CE + the label's logit), so the row is read once.
template <typename T>
__global__ void __launch_bounds__(256) ce_bwd_kernel(const float* __restrict__ logits, int V, const int* row_label,
                                                     const int* row_depth, const int* valid_d, const float* row_ce,
                                                     double decay, T* __restrict__ dlogits, int ldd) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const float* x = logits + (size_t)r * V;
  T* out = dlogits + (size_t)r * ldd;
  const int lab = row_label[r];
  const int cnt = lab >= 0 ? valid_d[row_depth[r]] : 0;
  const bool vec = (V & 3) == 0 && (ldd & 3) == 0;
  if (lab < 0 || cnt <= 0) {
    for (int v = threadIdx.x; v < V; v += blockDim.x) out[v] = from_f<T>(0.f);
    return;
  }
  const float w = (float)(pow(decay, (double)row_depth[r]) / cnt);
  const float lse = row_ce[r] + x[lab];
  if (vec) {
    for (int v = threadIdx.x * 4; v < V; v += blockDim.x * 4) {
      const float4 xv = *reinterpret_cast<const float4*>(x + v);
      float g[4] = {w * __expf(xv.x - lse), w * __expf(xv.y - lse), w * __expf(xv.z - lse), w * __expf(xv.w - lse)};
#pragma unroll
      for (int e = 0; e < 4; ++e) out[v + e] = from_f<T>(v + e == lab ? g[e] - w : g[e]);
    }
  } else {
    for (int v = threadIdx.x; v < V; v += blockDim.x) out[v] = from_f<T>(w * (__expf(x[v] - lse) - (v == lab ? 1.f : 0.f)));
  }
}

// ---------------------------------------------------------------- RMSNorm
// y = g * x * r, r = rsqrt(mean(x^2) + eps). Given dy:
//   dx = r * g * dy - x * r^3 * sum(g * dy * x) / H   (+ add)
// r of every row goes to r_out for the gain gradient.
template <typename TX>
__global__ void __launch_bounds__(256) rms_bwd_kernel(const TX* __restrict__ x, int ldx, const void* gain, int gain_bf16,
                                                      const float* __restrict__ dy, int ldy, const float* add, int ld_add,
                                                      float* dx, int ldd, float* r_out, int H, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[33];
  const int row = blockIdx.x;
  const TX* xr = x + (size_t)row * ldx;
  const float* dyr = dy + (size_t)row * ldy;
  float ss = 0.f, sg = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float xv = to_f(xr[c]);
    const float g = gain_bf16 ? __bfloat162float(static_cast<const bf16*>(gain)[c]) : static_cast<const float*>(gain)[c];
    ss += xv * xv;
    sg += g * dyr[c] * xv;
  }
  ss = block_sum(ss, red);
  __syncthreads();
  sg = block_sum(sg, red);
  const float r = rsqrtf(ss / H + eps);
  const float k = r * r * r * sg / H;
  if (r_out && threadIdx.x == 0) r_out[row] = r;
  if (!dx) return;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float g = gain_bf16 ? __bfloat162float(static_cast<const bf16*>(gain)[c]) : static_cast<const float*>(gain)[c];
    float v = r * g * dyr[c] - to_f(xr[c]) * k;
    if (add) v += add[(size_t)row * ld_add + c];
    dx[(size_t)row * ldd + c] = v;
  }
}

// dg[c] = sum over rows of dy[row][c] * x[xrow][c] * r[row], with xrow =
// map[row] when a map is given (embedding rows by token), else row.
template <typename TX>
__global__ void __launch_bounds__(256) gain_grad_kernel(const TX* __restrict__ x, int ldx, const int* map, int map_mod,
                                                        int map_const, const float* __restrict__ dy, int ldy,
                                                        const float* __restrict__ r, int rows, int H, float* dg) {
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  const int r0 = blockIdx.y * 64, r1 = min(rows, r0 + 64);
  float s = 0.f;
  for (int row = r0; row < r1; ++row) {
    int xr = row;
    if (map) xr = row < map_mod ? map[row] : map_const;
    s += dy[(size_t)row * ldy + c] * to_f(x[(size_t)xr * ldx + c]) * r[row];
  }
  atomicAdd(dg + c, s);
}

// r of rows of x (gathered through map like gain_grad_kernel)
template <typename TX>
__global__ void __launch_bounds__(256) rms_of_rows_kernel(const TX* __restrict__ x, int ldx, const int* map, int map_mod,
                                                          int map_const, int H, float eps, float* r_out) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[33];
  const int row = blockIdx.x;
  const int xr = map ? (row < map_mod ? map[row] : map_const) : row;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float v = to_f(x[(size_t)xr * ldx + c]);
    ss += v * v;
  }
  ss = block_sum(ss, red);
  if (threadIdx.x == 0) r_out[row] = rsqrtf(ss / H + eps);
}

// ---------------------------------------------------------------- SwiGLU
// a = silu(g) * u: dg = da * u * s * (1 + g * (1 - s)), du = da * silu(g),
// s = sigmoid(g)
template <typename T>
__global__ void swiglu_bwd_kernel(const float* __restrict__ gu, const float* __restrict__ dact, int rows, int I,
                                  T* __restrict__ dgu) {
  pdl_trigger();
  pdl_wait();
  // rows over blocks, columns over threads: coalesced, no index division
  for (int r = blockIdx.x; r < rows; r += gridDim.x)
    for (int j = threadIdx.x; j < I; j += blockDim.x) {
      const float g = gu[(size_t)r * 2 * I + j], u = gu[(size_t)r * 2 * I + I + j], da = dact[(size_t)r * I + j];
      const float s = 1.f / (1.f + __expf(-g));
      dgu[(size_t)r * 2 * I + j] = from_f<T>(da * u * s * (1.f + g * (1.f - s)));
      dgu[(size_t)r * 2 * I + I + j] = from_f<T>(da * g * s);
    }
}

// ------------------------------------------------------------------ RoPE
// The rotation by angle a transposed (by -a) on dq and dk; dv copied; all
// into the row's [q; k; v] gradient.
template <typename T, int HD>
__global__ void rope_bwd_kernel(const float* __restrict__ dq, const float* __restrict__ dk, const float* __restrict__ dv,
                                const int* __restrict__ row_pos, const float* rcos, const float* rsin, int max_pos,
                                int nq, int nkv, T* __restrict__ dqkv) {
  pdl_trigger();
  pdl_wait();
  constexpr int HALF = HD / 2;
  const int r = blockIdx.x;
  int pos = row_pos[r];
  pos = pos < 0 ? 0 : (pos >= max_pos ? max_pos - 1 : pos);
  const float* cs = rcos + (size_t)pos * HALF;
  const float* sn = rsin + (size_t)pos * HALF;
  const int QKV = (nq + 2 * nkv) * HD;
  T* out = dqkv + (size_t)r * QKV;
  const int pairs = (nq + nkv) * HALF;
  for (int e = threadIdx.x; e < pairs; e += blockDim.x) {
    const int head = e / HALF, j = e % HALF;
    const float* src = head < nq ? dq + ((size_t)r * nq + head) * HD : dk + ((size_t)r * nkv + head - nq) * HD;
    const float a = src[j], b = src[j + HALF], c = cs[j], s = sn[j];
    out[head * HD + j] = from_f<T>(a * c + b * s);
    out[head * HD + j + HALF] = from_f<T>(b * c - a * s);
  }
  for (int e = threadIdx.x; e < nkv * HD; e += blockDim.x)
    out[(nq + nkv) * HD + e] = from_f<T>(dv[(size_t)r * nkv * HD + e]);
}

// ------------------------------------------------------------- attention
// Keys of row (i, d): depth-0 rows start(i)..i, then the chain rows (i, 1..d).
template <typename T, int E>
__device__ __forceinline__ void ld_vec(const T* p, float (&x)[E]) {
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = to_f(p[e]);
}
__device__ __forceinline__ int key_row(const AttnBwdArgs& a, int i, int s0, int t) {
  return (t <= i - s0) ? s0 + t : a.row_of[(size_t)(t - (i - s0)) * a.n + i];
}

// one warp per (row, query head): LSE and D = dO . O, then
// dq = scale * sum_j p_j (dO . v_j - D) k_j
template <typename T, int E>
__global__ void __launch_bounds__(128) attn_bwd_q_kernel(AttnBwdArgs a) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int G = a.nq / a.nkv, hd = a.hd;
  const int i = a.row_anchor[r], d = a.row_depth[r], s0 = a.row_start[r];
  const T* Q = static_cast<const T*>(a.Q);
  const T* Kr = static_cast<const T*>(a.Kr);
  const T* Vr = static_cast<const T*>(a.Vr);
  const T* O = static_cast<const T*>(a.O);
  const T* dO = static_cast<const T*>(a.dO);
  for (int h = blockIdx.y * nw + w; h < a.nq; h += gridDim.y * nw) {
    const int g = h / G;
    float q[E], o[E], dov[E], dq[E];
    ld_vec<T, E>(Q + ((size_t)r * a.nq + h) * hd + lane * E, q);
    ld_vec<T, E>(O + ((size_t)r * a.nq + h) * hd + lane * E, o);
    ld_vec<T, E>(dO + ((size_t)r * a.nq + h) * hd + lane * E, dov);
    float D = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      D = fmaf(dov[e], o[e], D);
      dq[e] = 0.f;
    }
    D = warp_sum(D);
    const int nkeys = (i - s0 + 1) + d;
    float m = -INFINITY, l = 0.f;
    for (int t = 0; t < nkeys; ++t) {
      const int kr = key_row(a, i, s0, t);
      if (kr < 0 || kr >= a.R) continue;
      float k[E];
      ld_vec<T, E>(Kr + ((size_t)kr * a.nkv + g) * hd + lane * E, k);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) s = fmaf(q[e], k[e], s);
      s = warp_sum(s) * a.scale;
      const float mn = fmaxf(m, s);
      l = l * __expf(m - mn) + __expf(s - mn);
      m = mn;
    }
    const float lse = m + __logf(l);
    for (int t = 0; t < nkeys; ++t) {
      const int kr = key_row(a, i, s0, t);
      if (kr < 0 || kr >= a.R) continue;
      float k[E], v[E];
      ld_vec<T, E>(Kr + ((size_t)kr * a.nkv + g) * hd + lane * E, k);
      ld_vec<T, E>(Vr + ((size_t)kr * a.nkv + g) * hd + lane * E, v);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        s = fmaf(q[e], k[e], s);
        dp = fmaf(dov[e], v[e], dp);
      }
      s = warp_sum(s) * a.scale;
      dp = warp_sum(dp);
      const float ds = __expf(s - lse) * (dp - D) * a.scale;
#pragma unroll
      for (int e = 0; e < E; ++e) dq[e] = fmaf(ds, k[e], dq[e]);
    }
    float* out = a.dQ + ((size_t)r * a.nq + h) * hd + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = dq[e];
    if (lane == 0) {
      a.lse[(size_t)r * a.nq + h] = lse;
      a.Dv[(size_t)r * a.nq + h] = D;
    }
  }
}

// First row of depth d whose anchor is >= x (depth-d anchors ascend).
__device__ __forceinline__ int lower_row(const AttnBwdArgs& a, int d, int x) {
  int lo = a.off[d], hi = a.off[d + 1];
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a.row_anchor[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// one warp per (key row j, KV head g): the rows that see key j -- for a
// depth-0 key (anchor a) every row of every depth whose anchor lies in
// [a, end of a's conversation); for a chain key (a, dj) the rows (a, d),
// d >= dj -- and the G query heads of g:
//   dv_j = sum p dO,  dk_j = scale * sum p (dO . v_j - D) q
template <typename T, int E>
__global__ void __launch_bounds__(128) attn_bwd_kv_kernel(AttnBwdArgs a) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int G = a.nq / a.nkv, hd = a.hd;
  const int aj = a.row_anchor[j], dj = a.row_depth[j];
  const T* Q = static_cast<const T*>(a.Q);
  const T* Kr = static_cast<const T*>(a.Kr);
  const T* Vr = static_cast<const T*>(a.Vr);
  const T* dO = static_cast<const T*>(a.dO);
  for (int g = blockIdx.y * nw + w; g < a.nkv; g += gridDim.y * nw) {
    float k[E], v[E], dk[E], dv[E];
    ld_vec<T, E>(Kr + ((size_t)j * a.nkv + g) * hd + lane * E, k);
    ld_vec<T, E>(Vr + ((size_t)j * a.nkv + g) * hd + lane * E, v);
#pragma unroll
    for (int e = 0; e < E; ++e) dk[e] = dv[e] = 0.f;
    auto visit = [&](int qr) {
      for (int hh = 0; hh < G; ++hh) {
        const int h = g * G + hh;
        float q[E], dov[E];
        ld_vec<T, E>(Q + ((size_t)qr * a.nq + h) * hd + lane * E, q);
        ld_vec<T, E>(dO + ((size_t)qr * a.nq + h) * hd + lane * E, dov);
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          s = fmaf(q[e], k[e], s);
          dp = fmaf(dov[e], v[e], dp);
        }
        s = warp_sum(s) * a.scale;
        dp = warp_sum(dp);
        const float p = __expf(s - a.lse[(size_t)qr * a.nq + h]);
        const float ds = p * (dp - a.Dv[(size_t)qr * a.nq + h]) * a.scale;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          dv[e] = fmaf(p, dov[e], dv[e]);
          dk[e] = fmaf(ds, q[e], dk[e]);
        }
      }
    };
    if (dj == 0) {
      const int end = a.row_end[j];
      for (int d = 0; d < a.K; ++d)
        for (int qr = lower_row(a, d, aj); qr < a.off[d + 1] && a.row_anchor[qr] < end; ++qr) visit(qr);
    } else {
      for (int d = dj; d < a.K; ++d) {
        const int qr = a.row_of[(size_t)d * a.n + aj];
        if (qr >= 0 && qr < a.R) visit(qr);
      }
    }
    float* odk = a.dK + ((size_t)j * a.nkv + g) * hd + lane * E;
    float* odv = a.dV + ((size_t)j * a.nkv + g) * hd + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      odk[e] = dk[e];
      odv[e] = dv[e];
    }
  }
}

int grid1(long long total, int threads) {
  long long b = (total + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 8;
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

#define BW_END() \
  do {           \
    note_launch(); \
    return cudaGetLastError(); \
  } while (0)

cudaError_t launch_transpose(int dtype, const void* src, int rows, int cols, int lds, void* dst, int ldd, int rows_pad,
                             cudaStream_t st) {
  if (rows_pad <= 0 || cols <= 0) return cudaSuccess;
  if (dtype == PEAGLE_BF16 && (cols & 1) == 0 && (lds & 1) == 0 && (ldd & 1) == 0 && (rows_pad & 1) == 0 &&
      (reinterpret_cast<uintptr_t>(src) & 3) == 0 && (reinterpret_cast<uintptr_t>(dst) & 3) == 0) {
    launch_pdl(transpose_bf16x2_kernel, dim3((rows_pad + 63) / 64, (cols + 63) / 64), 256, 0, st,
               static_cast<const bf16*>(src), rows, cols, lds, static_cast<bf16*>(dst), ldd, rows_pad);
    BW_END();
  }
  const dim3 grid((rows_pad + 31) / 32, (cols + 31) / 32);
  if (dtype == PEAGLE_BF16)
    launch_pdl(transpose_kernel<bf16>, grid, 256, 0, st, static_cast<const bf16*>(src), rows, cols, lds,
               static_cast<bf16*>(dst), ldd, rows_pad);
  else
    launch_pdl(transpose_kernel<float>, grid, 256, 0, st, static_cast<const float*>(src), rows, cols, lds,
               static_cast<float*>(dst), ldd, rows_pad);
  BW_END();
}

cudaError_t launch_cast(int dtype, const float* src, void* dst, long long count, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  if (dtype == PEAGLE_BF16) launch_pdl(cast_kernel<bf16>, grid1(count, 256), 256, 0, st, src, static_cast<bf16*>(dst), count);
  else launch_pdl(cast_kernel<float>, grid1(count, 256), 256, 0, st, src, static_cast<float*>(dst), count);
  BW_END();
}

cudaError_t launch_gather_masked(int es, const void* src, int n, int rows, int cols, void* dst, cudaStream_t st) {
  const long long total = (long long)rows * cols;
  if (total <= 0) return cudaSuccess;
  if (es == 2)
    launch_pdl(gather_masked_kernel<bf16>, grid1(total, 256), 256, 0, st, static_cast<const bf16*>(src), n, rows, cols,
               static_cast<bf16*>(dst));
  else
    launch_pdl(gather_masked_kernel<float>, grid1(total, 256), 256, 0, st, static_cast<const float*>(src), n, rows, cols,
               static_cast<float*>(dst));
  BW_END();
}

cudaError_t launch_colsum(const float* src, int ld, int r0, int r1, int cols, float* dst, cudaStream_t st) {
  launch_pdl(colsum_kernel, (cols + 255) / 256, 256, 0, st, src, ld, r0, r1, cols, dst);
  BW_END();
}

cudaError_t launch_ce_bwd(int dtype, const float* logits, int rows, int V, const int* row_label, const int* row_depth,
                          const int* valid_d, const float* row_ce, double decay, void* dlogits, int ldd,
                          cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (dtype == PEAGLE_BF16)
    launch_pdl(ce_bwd_kernel<bf16>, rows, 256, 0, st, logits, V, row_label, row_depth, valid_d, row_ce, decay,
               static_cast<bf16*>(dlogits), ldd);
  else
    launch_pdl(ce_bwd_kernel<float>, rows, 256, 0, st, logits, V, row_label, row_depth, valid_d, row_ce, decay,
               static_cast<float*>(dlogits), ldd);
  BW_END();
}

cudaError_t launch_add_rows(const float* a, int lda, const float* b, int ldb, float* out, int ldo, int rows, int cols,
                            cudaStream_t st) {
  const long long total = (long long)rows * cols;
  if (total <= 0) return cudaSuccess;
  launch_pdl(add_rows_kernel, grid1(total, 256), 256, 0, st, a, lda, b, ldb, out, ldo, rows, cols);
  BW_END();
}

cudaError_t launch_rms_bwd(int x_es, const void* x, int ldx, const void* gain, int gain_bf16, const float* dy, int ldy,
                           const float* add, int ld_add, float* dx, int ldd, float* r_out, int rows, int H, float eps,
                           cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (x_es == 2)
    launch_pdl(rms_bwd_kernel<bf16>, rows, 256, 0, st, static_cast<const bf16*>(x), ldx, gain, gain_bf16, dy, ldy, add,
               ld_add, dx, ldd, r_out, H, eps);
  else
    launch_pdl(rms_bwd_kernel<float>, rows, 256, 0, st, static_cast<const float*>(x), ldx, gain, gain_bf16, dy, ldy, add,
               ld_add, dx, ldd, r_out, H, eps);
  BW_END();
}

cudaError_t launch_gain_grad(int x_es, const void* x, int ldx, const int* map, int map_mod, int map_const, const float* dy,
                             int ldy, const float* r, int rows, int H, float* dg, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((H + 255) / 256, (rows + 63) / 64);
  if (x_es == 2)
    launch_pdl(gain_grad_kernel<bf16>, grid, 256, 0, st, static_cast<const bf16*>(x), ldx, map, map_mod, map_const, dy,
               ldy, r, rows, H, dg);
  else
    launch_pdl(gain_grad_kernel<float>, grid, 256, 0, st, static_cast<const float*>(x), ldx, map, map_mod, map_const, dy,
               ldy, r, rows, H, dg);
  BW_END();
}

cudaError_t launch_rms_of_rows(int x_es, const void* x, int ldx, const int* map, int map_mod, int map_const, int rows, int H,
                               float eps, float* r_out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (x_es == 2)
    launch_pdl(rms_of_rows_kernel<bf16>, rows, 256, 0, st, static_cast<const bf16*>(x), ldx, map, map_mod, map_const, H,
               eps, r_out);
  else
    launch_pdl(rms_of_rows_kernel<float>, rows, 256, 0, st, static_cast<const float*>(x), ldx, map, map_mod, map_const, H,
               eps, r_out);
  BW_END();
}

cudaError_t launch_swiglu_bwd(int dtype, const float* gu, const float* dact, int rows, int I, void* dgu, cudaStream_t st) {
  if (rows <= 0 || I <= 0) return cudaSuccess;
  const int grid = std::min(rows, num_sms() * 8);
  if (dtype == PEAGLE_BF16)
    launch_pdl(swiglu_bwd_kernel<bf16>, grid, 256, 0, st, gu, dact, rows, I, static_cast<bf16*>(dgu));
  else
    launch_pdl(swiglu_bwd_kernel<float>, grid, 256, 0, st, gu, dact, rows, I, static_cast<float*>(dgu));
  BW_END();
}

cudaError_t launch_rope_bwd(int dtype, int hd, const float* dq, const float* dk, const float* dv, const int* row_pos,
                            const float* rcos, const float* rsin, int max_pos, int rows, int nq, int nkv, void* dqkv,
                            cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (dtype == PEAGLE_BF16) {
    if (hd == 128)
      launch_pdl(rope_bwd_kernel<bf16, 128>, rows, 256, 0, st, dq, dk, dv, row_pos, rcos, rsin, max_pos, nq, nkv,
                 static_cast<bf16*>(dqkv));
    else
      launch_pdl(rope_bwd_kernel<bf16, 64>, rows, 256, 0, st, dq, dk, dv, row_pos, rcos, rsin, max_pos, nq, nkv,
                 static_cast<bf16*>(dqkv));
  } else {
    if (hd == 128)
      launch_pdl(rope_bwd_kernel<float, 128>, rows, 256, 0, st, dq, dk, dv, row_pos, rcos, rsin, max_pos, nq, nkv,
                 static_cast<float*>(dqkv));
    else
      launch_pdl(rope_bwd_kernel<float, 64>, rows, 256, 0, st, dq, dk, dv, row_pos, rcos, rsin, max_pos, nq, nkv,
                 static_cast<float*>(dqkv));
  }
  BW_END();
}

cudaError_t launch_attn_bwd(int dtype, const AttnBwdArgs& a, cudaStream_t st) {
  if (a.R <= 0) return cudaSuccess;
  if (attn_bwd_mma_supported(dtype, a)) return launch_attn_bwd_mma(a, st);
  const dim3 gq(a.R, (a.nq + 3) / 4), gkv(a.R, (a.nkv + 3) / 4);
  if (dtype == PEAGLE_BF16) {
    if (a.hd == 128) {
      launch_pdl(attn_bwd_q_kernel<bf16, 4>, gq, 128, 0, st, a);
      note_launch();
      launch_pdl(attn_bwd_kv_kernel<bf16, 4>, gkv, 128, 0, st, a);
    } else {
      launch_pdl(attn_bwd_q_kernel<bf16, 2>, gq, 128, 0, st, a);
      note_launch();
      launch_pdl(attn_bwd_kv_kernel<bf16, 2>, gkv, 128, 0, st, a);
    }
  } else {
    if (a.hd == 128) {
      launch_pdl(attn_bwd_q_kernel<float, 4>, gq, 128, 0, st, a);
      note_launch();
      launch_pdl(attn_bwd_kv_kernel<float, 4>, gkv, 128, 0, st, a);
    } else {
      launch_pdl(attn_bwd_q_kernel<float, 2>, gq, 128, 0, st, a);
      note_launch();
      launch_pdl(attn_bwd_kv_kernel<float, 2>, gkv, 128, 0, st, a);
    }
  }
  BW_END();
}

}  // namespace pe

// Depth-masked attention of the P-EAGLE step ("feat(speculative) ... #2376":
// the EAGLE-3 cache_hidden diagonal-extension attention, equal to vLLM's
// flat [context, mask_1..mask_{K-1}] layout; "P_Eagle" README: packed
// conversations isolated by cu_seqlens).
//
// Decode, row (b, d), query head h, KV head g = h / (nq/nkv):
//   keys = context rows kv_off[b] .. kv_off[b]+kv_len[b]-1 of the cache,
//          then chain rows (b, 0..d) of this pass.
// The context is split into chunks; one CTA per (chunk, g, b) streams that
// chunk once for all K*G query rows that read head g, keeping an online
// softmax (max m, sum l, unnormalised o) per row. A combine kernel merges
// the chunks' (m, l, o) and adds the chain keys.
//
// Training, row (i, d): keys = depth-0 rows start(i)..i, then chain rows
// (i, 1..d).
#include <math.h>

#include "rows.cuh"

namespace pe {

template <typename T, int E>
__device__ __forceinline__ void load_vec(const T* p, float (&x)[E]) {
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = to_f(p[e]);
}

// Online-softmax update with one more key of score s and value row v.
template <int E>
__device__ __forceinline__ void online_add(float s, const float (&v)[E], float& m, float& l, float (&o)[E]) {
  const float mn = fmaxf(m, s);
  const float corr = (m == -INFINITY) ? 0.f : __expf(m - mn);
  const float p = __expf(s - mn);
  l = l * corr + p;
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = o[e] * corr + p * v[e];
  m = mn;
}

// ---------------------------------------------------------------- decode
template <typename T, int E>
__global__ void __launch_bounds__(256) decode_split_simt(DecodeAttnArgs a) {
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.nq / a.nkv, KG = a.K * G, hd = a.hd;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const long long off = a.kv_off[b];
  int L = a.kv_len[b];
  bool ok = L >= 0 && L <= a.max_kv_len && off >= 0 && off + L <= a.kv_off[b + 1] && off + L <= a.kv_cap;
  if (!ok) {
    if (threadIdx.x == 0 && split == 0 && g == 0) set_status(a.status, PEAGLE_DEV_BOUNDS);
    L = 0;
  }
  const int k0 = split * a.chunk, k1 = min(L, k0 + a.chunk);
  const size_t prow = ((size_t)(b * a.nkv + g) * a.nsplit + split) * KG;
  const T* kc = static_cast<const T*>(a.kcache);
  const T* vc = static_cast<const T*>(a.vcache);
  const T* Q = static_cast<const T*>(a.Q);
  for (int qi = w; qi < KG; qi += nw) {
    const int d = qi / G, h = g * G + qi % G;
    const int r = b * a.K + d;
    float q[E], o[E];
    load_vec<T, E>(Q + ((size_t)r * a.nq + h) * hd + lane * E, q);
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int t = k0; t < k1; ++t) {
      const size_t base = ((size_t)(off + t) * a.nkv + g) * hd + lane * E;
      float k[E], v[E];
      load_vec<T, E>(kc + base, k);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot = fmaf(q[e], k[e], dot);
      dot = warp_sum(dot) * a.scale;
      load_vec<T, E>(vc + base, v);
      online_add<E>(dot, v, m, l, o);
    }
    float* po = a.part_o + (prow + qi) * hd + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) po[e] = o[e];
    if (lane == 0) {
      a.part_ml[(prow + qi) * 2 + 0] = m;
      a.part_ml[(prow + qi) * 2 + 1] = l;
    }
  }
}

template <typename T, int E>
__global__ void decode_combine(DecodeAttnArgs a) {
  const int r = blockIdx.x;
  const int b = r / a.K, d = r % a.K;
  const int G = a.nq / a.nkv, KG = a.K * G, hd = a.hd;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const T* Q = static_cast<const T*>(a.Q);
  const T* Kc = static_cast<const T*>(a.Kc);
  const T* Vc = static_cast<const T*>(a.Vc);
  T* O = static_cast<T*>(a.O);
  for (int h = w; h < a.nq; h += nw) {
    const int g = h / G, qi = d * G + h % G;
    float M = -INFINITY;
    const size_t prow = (size_t)(b * a.nkv + g) * a.nsplit * KG;
    for (int s = 0; s < a.nsplit; ++s) M = fmaxf(M, a.part_ml[(prow + (size_t)s * KG + qi) * 2]);
    float o[E], l = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < a.nsplit; ++s) {
        const size_t pr = prow + (size_t)s * KG + qi;
        const float ms = a.part_ml[pr * 2], ls = a.part_ml[pr * 2 + 1];
        if (ms == -INFINITY) continue;
        const float c = __expf(ms - M);
        l += ls * c;
        const float* po = a.part_o + pr * hd + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] += po[e] * c;
      }
    }
    float m = M;
    float q[E];
    load_vec<T, E>(Q + ((size_t)r * a.nq + h) * hd + lane * E, q);
    for (int j = 0; j <= d; ++j) {  // chain rows (b, 0..d)
      const size_t base = ((size_t)(b * a.K + j) * a.nkv + g) * hd + lane * E;
      float k[E], v[E];
      load_vec<T, E>(Kc + base, k);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot = fmaf(q[e], k[e], dot);
      dot = warp_sum(dot) * a.scale;
      load_vec<T, E>(Vc + base, v);
      online_add<E>(dot, v, m, l, o);
    }
    const float inv = 1.f / l;
    T* out = O + ((size_t)r * a.nq + h) * hd + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = from_f<T>(o[e] * inv);
  }
}

void decode_attn_plan(int B, int nkv, int max_kv_len, int* chunk, int* nsplit) {
  const long long work = (long long)B * nkv * (max_kv_len > 0 ? max_kv_len : 1);
  long long c = work / (2LL * num_sms());
  int ch = 32;
  while (ch < c && ch < 512) ch *= 2;
  *chunk = ch;
  *nsplit = max_kv_len > 0 ? (max_kv_len + ch - 1) / ch : 1;
}

template <typename T, int E>
static cudaError_t decode_attn_t(const DecodeAttnArgs& a, int probe_op, cudaStream_t st) {
  dim3 grid(a.nsplit, a.nkv, a.B);
  probe_start(probe_op, st);
  decode_split_simt<T, E><<<grid, 256, 0, st>>>(a);
  note_launch();
  probe_stop(probe_op, st);
  const int threads = 32 * (a.nq < 32 ? a.nq : 32);
  decode_combine<T, E><<<a.B * a.K, threads, 0, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_decode_attn(int dtype, const DecodeAttnArgs& a, int probe_op, cudaStream_t st) {
  if (a.B <= 0) return cudaSuccess;
  if (dtype == PEAGLE_BF16) {
    return a.hd == 128 ? decode_attn_t<bf16, 4>(a, probe_op, st) : decode_attn_t<bf16, 2>(a, probe_op, st);
  }
  return a.hd == 128 ? decode_attn_t<float, 4>(a, probe_op, st) : decode_attn_t<float, 2>(a, probe_op, st);
}

// ---------------------------------------------------------------- training
template <typename T, int E>
__global__ void __launch_bounds__(128) train_attn_simt(TrainAttnArgs a) {
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int G = a.nq / a.nkv, hd = a.hd;
  const int i = a.row_anchor[r], d = a.row_depth[r], s0 = a.row_start[r];
  const T* Q = static_cast<const T*>(a.Q);
  const T* Kr = static_cast<const T*>(a.Kr);
  const T* Vr = static_cast<const T*>(a.Vr);
  T* O = static_cast<T*>(a.O);
  for (int h = blockIdx.y * nw + w; h < a.nq; h += gridDim.y * nw) {
    const int g = h / G;
    float q[E], o[E];
    load_vec<T, E>(Q + ((size_t)r * a.nq + h) * hd + lane * E, q);
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int nkeys = (i - s0 + 1) + d;
    for (int t = 0; t < nkeys; ++t) {
      // depth-0 rows s0..i have row index = anchor; then chain rows (i, 1..d)
      const int kr = (t <= i - s0) ? s0 + t : a.row_of[(size_t)(t - (i - s0)) * a.n + i];
      if (kr < 0 || kr >= a.R) continue;   // nested COD sets always provide the chain row
      const size_t base = ((size_t)kr * a.nkv + g) * hd + lane * E;
      float k[E], v[E];
      load_vec<T, E>(Kr + base, k);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot = fmaf(q[e], k[e], dot);
      dot = warp_sum(dot) * a.scale;
      load_vec<T, E>(Vr + base, v);
      online_add<E>(dot, v, m, l, o);
    }
    const float inv = 1.f / l;
    T* out = O + ((size_t)r * a.nq + h) * hd + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = from_f<T>(o[e] * inv);
  }
}

template <typename T, int E>
static cudaError_t train_attn_t(const TrainAttnArgs& a, int probe_op, cudaStream_t st) {
  dim3 grid(a.R, (a.nq + 3) / 4);
  probe_start(probe_op, st);
  train_attn_simt<T, E><<<grid, 128, 0, st>>>(a);
  note_launch();
  probe_stop(probe_op, st);
  return cudaGetLastError();
}

cudaError_t launch_train_attn(int dtype, const TrainAttnArgs& a, int probe_op, cudaStream_t st) {
  if (a.R <= 0) return cudaSuccess;
  if (dtype == PEAGLE_BF16)
    return a.hd == 128 ? train_attn_t<bf16, 4>(a, probe_op, st) : train_attn_t<bf16, 2>(a, probe_op, st);
  return a.hd == 128 ? train_attn_t<float, 4>(a, probe_op, st) : train_attn_t<float, 2>(a, probe_op, st);
}

}  // namespace pe

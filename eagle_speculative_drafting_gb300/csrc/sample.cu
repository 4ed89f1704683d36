// Stochastic verification of a draft step ("P_Eagle" README, How Speculative
// Decoding Works, row 6: accepted tokens are used, rejected ones resampled;
// the output is distributed as the target's). The rule is the published
// speculative-sampling one (Leviathan, Kalman, Matias, ICML 2023; Chen et
// al., 2023), with the random numbers passed in:
//   depth i keeps draft x iff fl32(u[b,i] * q_i(x)) < p_i(x);
//   at the first rejection a the next token is drawn from max(0, p_a - q_a),
//   after K kept drafts from p_K (the bonus token);
//   the draw is exact integer inverse-CDF: W_j = floor(w_j * 2^40) with w_j
//   clamped to [0, 1] (NaN as 0), S = sum W_j, T = (draw * S) >> 32, token =
//   the smallest j whose inclusive prefix sum exceeds T; S = 0 gives the
//   lowest-index argmax of p_a.
// One CTA per request. Thread t owns vocabulary ids [t*C, (t+1)*C): it sums
// their integer weights, a block scan of the 256 sums locates the one thread
// whose range holds T, and that thread walks its range to the token.
#include "rows.cuh"

namespace pe {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ long long sample_weight(float w) {
  w = fminf(fmaxf(w, 0.f), 1.f);               // NaN -> 0: fmaxf returns the number
  return (long long)(w * 1099511627776.0f);    // w * 2^40 is exact; the cast floors it
}

__device__ __forceinline__ long long weight_at(const float* pr, const float* qr, int j) {
  return sample_weight(qr ? __fsub_rn(pr[j], qr[j]) : pr[j]);
}

__global__ void __launch_bounds__(kThreads) verify_sample_kernel(SampleArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_acc;
  __shared__ long long s_sum[kThreads / 32];
  __shared__ float s_bv[kThreads / 32];
  __shared__ int s_bi[kThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, V = a.V;

  // ---- acceptance: lane i tests depth i (32 depths per round)
  if (warp == 0) {
    int first = K;
    for (int i0 = 0; i0 < K; i0 += 32) {
      const int i = i0 + lane;
      bool rej = false;
      if (i < K) {
        const int x = a.drafts[(size_t)b * K + i];
        if (x < 0 || x >= V) {
          rej = true;
          set_status(a.status, PEAGLE_DEV_BOUNDS);
        } else {
          const float qx = a.q[((size_t)b * K + i) * V + x];
          const float px = a.p[((size_t)b * (K + 1) + i) * V + x];
          rej = !(__fmul_rn(a.u[(size_t)b * K + i], qx) < px);
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, rej);
      if (m) {
        first = i0 + __ffs(m) - 1;
        break;
      }
    }
    if (lane == 0) s_acc = first;
  }
  __syncthreads();
  const int acc = s_acc;
  const float* pr = a.p + ((size_t)b * (K + 1) + acc) * V;
  const float* qr = acc < K ? a.q + ((size_t)b * K + acc) * V : nullptr;

  // ---- this thread's range and the sum of its integer weights
  const int C = (V + kThreads - 1) / kThreads;
  const int j0 = min(V, tid * C), j1 = min(V, j0 + C);
  long long mine = 0;
#pragma unroll 8
  for (int j = j0; j < j1; ++j) mine += weight_at(pr, qr, j);
  // inclusive block scan of the 256 range sums
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_sum[warp] = incl;
  __syncthreads();
  long long before = 0, S = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    before += (w < warp) ? s_sum[w] : 0;
    S += s_sum[w];
  }
  const long long lo = before + incl - mine;   // exclusive prefix of this range

  if (S == 0) {
    // no weight anywhere: the lowest-index argmax of p_acc
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int j = j0; j < j1; ++j)
      if (am_better(pr[j], j, bv, bi)) {
        bv = pr[j];
        bi = j;
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (am_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      s_bv[warp] = bv;
      s_bi[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kThreads / 32; ++w)
        if (am_better(s_bv[w], s_bi[w], bv, bi)) {
          bv = s_bv[w];
          bi = s_bi[w];
        }
      a.accept[b] = acc;
      a.next[b] = (bi >= 0 && bi < V) ? bi : 0;
    }
    return;
  }
  // T = floor(draw * S / 2^32), from the exact 96-bit product
  const unsigned long long us = (unsigned long long)S, dr = a.draws[b];
  const unsigned long long T = (__umul64hi(us, dr) << 32) | ((us * dr) >> 32);
  if ((unsigned long long)lo <= T && T < (unsigned long long)(lo + mine)) {
    long long run = lo;
    int tok = j1 - 1;
    for (int j = j0; j < j1; ++j) {
      run += weight_at(pr, qr, j);
      if ((unsigned long long)run > T) {
        tok = j;
        break;
      }
    }
    a.accept[b] = acc;
    a.next[b] = tok;
  }
}

}  // namespace

cudaError_t launch_verify_sample(const SampleArgs& a, cudaStream_t st) {
  if (a.B <= 0) return cudaSuccess;
  launch_pdl(verify_sample_kernel, dim3(a.B), dim3(kThreads), 0, st, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pe

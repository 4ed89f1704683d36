// Depth-masked attention of the P-EAGLE step ("feat(speculative) ... #2376":
// the EAGLE-3 cache_hidden diagonal-extension attention, equal to vLLM's
// flat [context, mask_1..mask_{K-1}] layout; "P_Eagle" README: packed
// conversations isolated by cu_seqlens).
//
// Decode, row j of request b (DecodeRows: its new rows, the last of them the
// anchor, then its masked depths), query head h, KV head g = h / (nq/nkv):
//   keys = context rows kv_off[b] .. kv_off[b]+kv_len[b]-1 of the cache,
//          then the request's rows 0..j of this pass (causal in the flat
//          [context, new rows, mask_1..mask_{K-1}] layout).
// The context is split into chunks; one CTA per (chunk, g, b) streams that
// chunk once for all the request's query rows that read head g, keeping an
// online softmax (max m, sum l, unnormalised o) per row. A combine kernel
// merges the chunks' (m, l, o) and adds the in-request keys.
//
// Training, row (i, d): keys = depth-0 rows start(i)..i, then chain rows
// (i, 1..d).
#include <math.h>

#include "mma.cuh"
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
  pdl_trigger();
  pdl_wait();
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.nq / a.nkv, hd = a.hd;
  const int KGmax = a.rows_max * G;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const long long off = a.kv_off[b];
  int L = a.kv_len[b];
  bool ok = L >= 0 && L <= a.max_kv_len && off >= 0 && off + L <= a.kv_off[b + 1] && off + L <= a.kv_cap;
  if (!ok) {
    if (threadIdx.x == 0 && split == 0 && g == 0) set_status(a.status, PEAGLE_DEV_BOUNDS);
    L = 0;
  }
  if (!dr_valid(a.rows, b)) return;   // flagged by the q/k/v kernel
  const int KG = (dr_new(a.rows, b) + a.K - 1) * G, rb = dr_base(a.rows, b);
  const int k0 = split * a.chunk, k1 = min(L, k0 + a.chunk);
  const size_t prow = ((size_t)(b * a.nkv + g) * a.nsplit + split) * KGmax;
  const T* kc = static_cast<const T*>(a.kcache);
  const T* vc = static_cast<const T*>(a.vcache);
  const T* Q = static_cast<const T*>(a.Q);
  for (int qi = w; qi < KG; qi += nw) {
    const int d = qi / G, h = g * G + qi % G;
    const int r = rb + d;
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

// Output row r (row d of request b), head h, from the chunks' (m, l, o)
// plus the request's rows 0..d; one warp, lane owns dims [lane*E, lane*E + E). The query,
// the chunk statistics, the first chunk outputs and the first chain keys /
// values are all loaded before any of them is used, so the row costs about
// two memory round trips.
template <typename T, int E>
__device__ void combine_row(const DecodeAttnArgs& a, int r, int h, int lane) {
  constexpr int SB = 8, CB = 4;   // chunk outputs / chain rows per load round
  int d;
  const int b = dr_request(a.rows, r, &d);
  if (!dr_valid(a.rows, b) || d < 0 || d >= dr_new(a.rows, b) + a.K - 1) return;   // flagged by the q/k/v kernel
  const int rb = dr_base(a.rows, b);
  const int G = a.nq / a.nkv, KG = a.rows_max * G, hd = a.hd;
  const int g = h / G, qi = d * G + h % G;
  // only the chunks that hold context keys of request b carry partials
  const long long off = a.kv_off[b];
  int L = a.kv_len[b];
  if (!(L >= 0 && L <= a.max_kv_len && off >= 0 && off + L <= a.kv_off[b + 1] && off + L <= a.kv_cap)) L = 0;
  const int ns = min(a.nsplit, (L + a.chunk - 1) / a.chunk);
  const T* Q = static_cast<const T*>(a.Q);
  const T* Kc = static_cast<const T*>(a.Kc);
  const T* Vc = static_cast<const T*>(a.Vc);
  const size_t prow = (size_t)(b * a.nkv + g) * a.nsplit * KG;
  auto ml = [&](int s) { return a.part_ml + (prow + (size_t)s * KG + qi) * 2; };
  auto po_at = [&](int s) { return a.part_o + (prow + (size_t)s * KG + qi) * hd + lane * E; };
  auto kv_at = [&](int j) { return ((size_t)(rb + j) * a.nkv + g) * hd + lane * E; };

  float q[E];
  load_vec<T, E>(Q + ((size_t)r * a.nq + h) * hd + lane * E, q);
  float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;   // chunks lane, lane + 32
  if (lane < ns) {
    m0 = ml(lane)[0];
    l0 = ml(lane)[1];
  }
  if (lane + 32 < ns) {
    m1 = ml(lane + 32)[0];
    l1 = ml(lane + 32)[1];
  }
  float po[SB][E], kk[CB][E], vv[CB][E];
#pragma unroll
  for (int i = 0; i < SB; ++i) {
#pragma unroll
    for (int e = 0; e < E; ++e) po[i][e] = i < ns ? po_at(i)[e] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < CB; ++i) {
    if (i <= d) {
      load_vec<T, E>(Kc + kv_at(i), kk[i]);
      load_vec<T, E>(Vc + kv_at(i), vv[i]);
    }
  }
  // merged statistics of the chunks
  float M = fmaxf(m0, m1);
  for (int s = lane + 64; s < ns; s += 32) M = fmaxf(M, ml(s)[0]);
  M = warp_max(M);
  float l = (m0 == -INFINITY ? 0.f : l0 * __expf(m0 - M)) + (m1 == -INFINITY ? 0.f : l1 * __expf(m1 - M));
  for (int s = lane + 64; s < ns; s += 32) {
    const float ms = ml(s)[0];
    if (ms != -INFINITY) l += ml(s)[1] * __expf(ms - M);
  }
  l = warp_sum(l);
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < ns; s0 += SB) {
      if (s0 > 0) {
#pragma unroll
        for (int i = 0; i < SB; ++i) {
#pragma unroll
          for (int e = 0; e < E; ++e) po[i][e] = s0 + i < ns ? po_at(s0 + i)[e] : 0.f;
        }
      }
#pragma unroll
      for (int i = 0; i < SB; ++i) {
        const int s = s0 + i;
        if (s >= ns) break;
        const float ms = s < 64 ? __shfl_sync(0xffffffffu, s < 32 ? m0 : m1, s & 31) : ml(s)[0];
        const float c = (ms == -INFINITY) ? 0.f : __expf(ms - M);
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] += po[i][e] * c;
      }
    }
  }
  // chain rows (b, 0..d), CB at a time
  float m = M;
  for (int j0 = 0; j0 <= d; j0 += CB) {
    if (j0 > 0) {
#pragma unroll
      for (int i = 0; i < CB; ++i) {
        if (j0 + i <= d) {
          load_vec<T, E>(Kc + kv_at(j0 + i), kk[i]);
          load_vec<T, E>(Vc + kv_at(j0 + i), vv[i]);
        }
      }
    }
    float dot[CB];
#pragma unroll
    for (int i = 0; i < CB; ++i) {
      dot[i] = 0.f;
      if (j0 + i <= d) {
#pragma unroll
        for (int e = 0; e < E; ++e) dot[i] = fmaf(q[e], kk[i][e], dot[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < CB; ++i) dot[i] = warp_sum(dot[i]) * a.scale;
#pragma unroll
    for (int i = 0; i < CB; ++i)
      if (j0 + i <= d) online_add<E>(dot[i], vv[i], m, l, o);
  }
  const float inv = 1.f / l;
  T* out = static_cast<T*>(a.O) + ((size_t)r * a.nq + h) * hd + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = from_f<T>(o[e] * inv);
}

template <typename T, int E>
__global__ void decode_combine(DecodeAttnArgs a) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int h = blockIdx.y * nw + w; h < a.nq; h += gridDim.y * nw) combine_row<T, E>(a, r, h, lane);
}

// ------------------------------------------------- decode, bf16 tensor cores
// Same split as above, but the chunk's K/V stream through shared memory in
// 64-key tiles (cp.async, double-buffered) and both products run on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate):
//   S = Q K^T   warp w scores keys 16w..16w+15 of the tile for all rows;
//   softmax     row maxima/sums meet in shared memory, P goes to smem (bf16);
//   O += P V    warp w owns head dims [w*hd/4, (w+1)*hd/4).
// Rows are the K*G queries reading this KV head, padded to 16*MT.

// NW warps: warp w scores keys [w*KW, (w+1)*KW) of each 64-key tile for
// every row and owns head dims [w*DW, (w+1)*DW) of the P V product. This
// block-synchronous form (three barriers per tile) serves 64 or 128 query
// rows per KV head (multi-row steps), where every K/V tile is shared by
// many rows; up to 32 rows use the warp-independent kernel below.
// K and V tiles rotate through NS stages; their rows are unpadded with the
// 16-byte chunks of row r XOR-swizzled by r & 7 (conflict-free ldmatrix).
template <int MT, int HD, int NW, int NS>
struct MmaAttnCfg {
  static constexpr int THREADS = 32 * NW;
  static constexpr int QR = 16 * MT, TK = 64, KW = TK / NW, NK8 = KW / 8, DW = HD / NW, NP = DW / 16;
  static constexpr int LDS = HD + 8, LDP = TK + 8;
  static constexpr int SMEM = (QR * LDS + 2 * NS * TK * HD + QR * LDP) * 2 + 2 * NW * QR * 4;
};
// element offset of (row, 16-byte chunk c8) in a swizzled K/V tile
template <int HD>
__device__ __forceinline__ int kv_sw(int row, int c8) {
  return row * HD + ((c8 ^ (row & 7)) << 3);
}

template <int MT, int HD, int NW, int NS>
__global__ void __launch_bounds__(MmaAttnCfg<MT, HD, NW, NS>::THREADS) decode_split_mma(DecodeAttnArgs a) {
  pdl_trigger();
  pdl_wait();
  using C = MmaAttnCfg<MT, HD, NW, NS>;
  constexpr int QR = C::QR, TK = C::TK, LDS = C::LDS, LDP = C::LDP, KW = C::KW, NK8 = C::NK8, DW = C::DW;
  constexpr int NP = C::NP, NT = C::THREADS;
  static_assert((NK8 == 1 || NK8 == 2) && NP >= 1 && DW == 16 * NP, "8 or 16 keys and 16k dims per warp");
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
  bf16* sK = sQ + QR * LDS;           // [NS][TK][HD] swizzled
  bf16* sV = sK + NS * TK * HD;       // [NS][TK][HD] swizzled
  bf16* sP = sV + NS * TK * HD;       // [QR][LDP]
  float* sMax = reinterpret_cast<float*>(sP + QR * LDP);  // [NW][QR]
  float* sSum = sMax + NW * QR;                            // [NW][QR]

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.nq / a.nkv;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const long long off = a.kv_off[b];
  int L = a.kv_len[b];
  const bool ok = L >= 0 && L <= a.max_kv_len && off >= 0 && off + L <= a.kv_off[b + 1] && off + L <= a.kv_cap;
  if (!ok) {
    if (tid == 0 && split == 0 && g == 0) set_status(a.status, PEAGLE_DEV_BOUNDS);
    L = 0;
  }
  const int k0 = split * a.chunk, k1 = min(L, k0 + a.chunk);
  const int ntiles = k1 > k0 ? (k1 - k0 + TK - 1) / TK : 0;
  if (ntiles == 0) return;   // a chunk past the context end: the merge skips it
  if (!dr_valid(a.rows, b)) return;   // flagged by the q/k/v kernel
  // this request's query rows of KV head g: row qi = d*G + (h % G) for its
  // rows d = 0 .. n_b + K - 2; the partials are laid out for rows_max rows
  const int KG = (dr_new(a.rows, b) + a.K - 1) * G, KGmax = a.rows_max * G, rb = dr_base(a.rows, b);
  const bf16* kc = static_cast<const bf16*>(a.kcache);
  const bf16* vc = static_cast<const bf16*>(a.vcache);
  const bf16* Q = static_cast<const bf16*>(a.Q);

  auto load_tile = [&](int t, int buf) {
    const int base = k0 + t * TK;
    for (int e = tid; e < TK * (HD / 8); e += NT) {
      const int kr = e / (HD / 8), c8 = e % (HD / 8);
      const int key = base + kr;
      const bool in = key < k1;
      const size_t src = ((size_t)(off + (in ? key : k0)) * a.nkv + g) * HD + c8 * 8;
      mm::cp16(mm::sa(sK + buf * TK * HD + kv_sw<HD>(kr, c8)), kc + src, in ? 16 : 0);
      mm::cp16(mm::sa(sV + buf * TK * HD + kv_sw<HD>(kr, c8)), vc + src, in ? 16 : 0);
    }
  };
  // the first tiles' keys stream while the queries are staged (one commit
  // group per stage, empty groups included, so the waits below count tiles)
#pragma unroll
  for (int q = 0; q < NS - 1; ++q) {
    if (q < ntiles) load_tile(q, q);
    mm::cp_commit();
  }
  // queries of this KV head: row qi = d*G + (h % G)
  for (int e = tid; e < QR * (HD / 8); e += NT) {
    const int qi = e / (HD / 8), c8 = e % (HD / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (qi < KG) {
      const int r = rb + qi / G, h = g * G + qi % G;
      v = *reinterpret_cast<const uint4*>(Q + ((size_t)r * a.nq + h) * HD + c8 * 8);
    }
    *reinterpret_cast<uint4*>(sQ + qi * LDS + c8 * 8) = v;
  }
  // up to two row blocks keep their query fragments in registers
  constexpr bool QREG = MT <= 2;
  uint32_t qf[QREG ? MT : 1][HD / 16][4];
  if constexpr (QREG) {
    __syncthreads();
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks)
        mm::ldsm4(qf[mt][ks], mm::sa(sQ + (mt * 16 + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8));
  }
  auto qfrag = [&](int mt, int ks, uint32_t(&aq)[4]) {
    if constexpr (QREG) {
#pragma unroll
      for (int i = 0; i < 4; ++i) aq[i] = qf[mt][ks][i];
    } else {
      mm::ldsm4(aq, mm::sa(sQ + (mt * 16 + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8));
    }
  };

  const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units
  float m_run[MT][2], l_run[MT][2];
  float O[MT][2 * NP][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    m_run[mt][0] = m_run[mt][1] = -INFINITY;
    l_run[mt][0] = l_run[mt][1] = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2 * NP; ++nt) O[mt][nt][0] = O[mt][nt][1] = O[mt][nt][2] = O[mt][nt][3] = 0.f;
  }

  for (int t = 0; t < ntiles; ++t) {
    const int buf = t % NS;
    // tile t + NS - 1 goes to the stage tile t - 1 used (free since the
    // barrier that ended the previous iteration)
    if (t + NS - 1 < ntiles) load_tile(t + NS - 1, (t + NS - 1) % NS);
    mm::cp_commit();
    mm::cp_wait<NS - 1>();
    __syncthreads();
    const bf16* tK = sK + buf * TK * HD;
    const bf16* tV = sV + buf * TK * HD;
    // ---- S = Q K^T for keys w*KW .. w*KW + KW - 1; with up to two row
    // blocks, even and odd 16-dim steps accumulate separately (twice the
    // independent MMA chains)
    constexpr bool SPLIT = MT <= 2;
    float S[MT][NK8][4], S2[MT][NK8][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NK8; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) S[mt][nt][i] = S2[mt][nt][i] = 0.f;
    if constexpr (NK8 == 2) {
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        uint32_t bk[4];   // keys (2 x 8) x 16 dims
        mm::ldsm4(bk, mm::sa(tK + kv_sw<HD>(KW * w + (lane >> 4) * 8 + (lane & 7), ks * 2 + ((lane >> 3) & 1))));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t aq[4];
          qfrag(mt, ks, aq);
          float(&acc)[NK8][4] = (SPLIT && (ks & 1)) ? S2[mt] : S[mt];
          mm::mma16816(acc[0], aq, bk[0], bk[1]);
          mm::mma16816(acc[NK8 - 1], aq, bk[2], bk[3]);
        }
      }
    } else {
#pragma unroll
      for (int kp = 0; kp < HD / 32; ++kp) {
        uint32_t bk[4];   // 8 keys x (2 x 16) dims
        mm::ldsm4(bk, mm::sa(tK + kv_sw<HD>(KW * w + (lane & 7), kp * 4 + (lane >> 3))));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            uint32_t aq[4];
            qfrag(mt, kp * 2 + h2, aq);
            float(&acc)[NK8][4] = (SPLIT && h2) ? S2[mt] : S[mt];
            mm::mma16816(acc[0], aq, bk[2 * h2], bk[2 * h2 + 1]);
          }
        }
      }
    }
    if constexpr (SPLIT) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NK8; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) S[mt][nt][i] += S2[mt][nt][i];
    }
    // ---- scale, mask the tail, per-row maxima of this warp's keys
    const int kbase = k0 + t * TK + KW * w + (lane & 3) * 2;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NK8; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int key = kbase + nt * 8 + c;
            float v = S[mt][nt][hf * 2 + c] * sl2;
            v = key < k1 ? v : -INFINITY;
            S[mt][nt][hf * 2 + c] = v;
            mx = fmaxf(mx, v);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if ((lane & 3) == 0) sMax[w * QR + mt * 16 + hf * 8 + (lane >> 2)] = mx;
      }
    }
    __syncthreads();
    // ---- new running max, probabilities to smem, row sums
    float corr[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int row = mt * 16 + hf * 8 + (lane >> 2);
        float tmax = sMax[row];
#pragma unroll
        for (int q = 1; q < NW; ++q) tmax = fmaxf(tmax, sMax[q * QR + row]);
        const float mn = fmaxf(m_run[mt][hf], tmax);
        corr[mt][hf] = (mn == -INFINITY) ? 1.f : exp2f(m_run[mt][hf] - mn);
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < NK8; ++nt) {
          float p0 = (mn == -INFINITY) ? 0.f : exp2f(S[mt][nt][hf * 2] - mn);
          float p1 = (mn == -INFINITY) ? 0.f : exp2f(S[mt][nt][hf * 2 + 1] - mn);
          const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
          *reinterpret_cast<__nv_bfloat162*>(sP + row * LDP + KW * w + nt * 8 + (lane & 3) * 2) = pp;
          sum += __low2float(pp) + __high2float(pp);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if ((lane & 3) == 0) sSum[w * QR + row] = sum;
        m_run[mt][hf] = mn;
      }
    }
    __syncthreads();
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int row = mt * 16 + hf * 8 + (lane >> 2);
        float ts = 0.f;
#pragma unroll
        for (int q = 0; q < NW; ++q) ts += sSum[q * QR + row];
        l_run[mt][hf] = l_run[mt][hf] * corr[mt][hf] + ts;
#pragma unroll
        for (int nt = 0; nt < 2 * NP; ++nt) {
          O[mt][nt][hf * 2] *= corr[mt][hf];
          O[mt][nt][hf * 2 + 1] *= corr[mt][hf];
        }
      }
    // ---- O += P V over this warp's head dims
#pragma unroll
    for (int ks = 0; ks < TK / 16; ++ks) {
      uint32_t ap[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        mm::ldsm4(ap[mt], mm::sa(sP + (mt * 16 + (lane & 15)) * LDP + ks * 16 + (lane >> 4) * 8));
#pragma unroll
      for (int np = 0; np < NP; ++np) {
        uint32_t bv[4];
        mm::ldsm4t(bv, mm::sa(tV + kv_sw<HD>(ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8,
                                             (w * DW + np * 16) / 8 + (lane >> 4))));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mm::mma16816(O[mt][2 * np], ap[mt], bv[0], bv[1]);
          mm::mma16816(O[mt][2 * np + 1], ap[mt], bv[2], bv[3]);
        }
      }
    }
    __syncthreads();
  }
  // ---- partial (unnormalised O, m in natural-log units, l)
  const size_t prow = ((size_t)(b * a.nkv + g) * a.nsplit + split) * KGmax;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int row = mt * 16 + hf * 8 + (lane >> 2);
      if (row >= KG) continue;
      float* po = a.part_o + (prow + row) * HD + w * DW + (lane & 3) * 2;
#pragma unroll
      for (int nt = 0; nt < 2 * NP; ++nt)
        *reinterpret_cast<float2*>(po + nt * 8) = make_float2(O[mt][nt][hf * 2], O[mt][nt][hf * 2 + 1]);
      if (w == 0 && (lane & 3) == 0) {
        a.part_ml[(prow + row) * 2 + 0] = m_run[mt][hf] * 0.6931471805599453f;
        a.part_ml[(prow + row) * 2 + 1] = l_run[mt][hf];
      }
    }
}

// ------------------------------------ decode, bf16, warp-independent split
// The same (chunk, KV head, request) CTAs, but no block barrier in the main
// loop: warp w streams its own 16-key tiles t = w, w + NW, ... of the chunk
// through its own NS-stage cp.async ring and keeps a private online softmax
// over them for all 16*MT query rows and all HD dims:
//   S = Q K^T   (rows x 16 keys; Q fragments from shared memory);
//   row maxima within the quad of lanes that holds a row (two shuffles);
//   the row's reference maximum moves only when a tile exceeds it by more
//   than 2^8, so O is rescaled rarely; probabilities relative to it stay
//   below 256 and are rounded to bf16;
//   O += P V   (P straight from the score registers; V by ldmatrix.trans).
// At the end the NW warps' (m, l, O) meet once in shared memory and the CTA
// writes the chunk's partial as the block-synchronous kernel does, so the
// combine is shared.
// RG = 2 (multi-row steps, up to 32*MT*2 rows): warp w keeps the online
// softmax of row group w % RG over key stream w / RG. The RG warps of a
// stream share its ring: each issues 1/RG of a tile's copies, and once per
// tile they meet on a named barrier (after each has waited for its own
// copies, before either refills the stage the previous tile used). Each K/V
// tile still leaves HBM once, and a warp holds O for 16*MT rows only.
template <int MT, int HD, int NW, int NS, int RG = 1>
struct WarpAttnCfg {
  static constexpr int THREADS = 32 * NW;
  static constexpr int NTS = NW / RG;                            // key streams
  static constexpr int QR = 16 * MT, QT = RG * QR, TK = 16, LDS = HD + 8;
  static constexpr int STAGE = 2 * TK * HD * 2;                  // K and V of one 16-key tile, bytes
  static constexpr int RING = NTS * NS * STAGE;
  static constexpr int MERGE = NW * QR * (HD + 2) * 4;           // per-warp O, m, l at the end
  static constexpr int SMEM = QT * LDS * 2 + (RING > MERGE ? RING : MERGE);
  static_assert(NW % RG == 0 && NTS <= 8, "warps per key stream");
};

template <int MT, int HD, int NW, int NS, int RG = 1>
__global__ void __launch_bounds__(WarpAttnCfg<MT, HD, NW, NS, RG>::THREADS) decode_warp_mma(DecodeAttnArgs a) {
  pdl_trigger();
  pdl_wait();
  using C = WarpAttnCfg<MT, HD, NW, NS, RG>;
  constexpr int QR = C::QR, QT = C::QT, TK = C::TK, LDS = C::LDS, NT = HD / 8, NTS = C::NTS;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
  uint8_t* ring = smem_raw + QT * LDS * 2;

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.nq / a.nkv;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int rg = w % RG, ts = w / RG;   // row group, key stream
  const long long off = a.kv_off[b];
  int L = a.kv_len[b];
  const bool ok = L >= 0 && L <= a.max_kv_len && off >= 0 && off + L <= a.kv_off[b + 1] && off + L <= a.kv_cap;
  if (!ok) {
    if (tid == 0 && split == 0 && g == 0) set_status(a.status, PEAGLE_DEV_BOUNDS);
    L = 0;
  }
  const int k0 = split * a.chunk, k1 = min(L, k0 + a.chunk);
  const int ntiles = k1 > k0 ? (k1 - k0 + TK - 1) / TK : 0;
  if (ntiles == 0) return;   // a chunk past the context end: the merge skips it
  if (!dr_valid(a.rows, b)) return;   // flagged by the q/k/v kernel
  const int KG = (dr_new(a.rows, b) + a.K - 1) * G, KGmax = a.rows_max * G, rb = dr_base(a.rows, b);
  const bf16* kc = static_cast<const bf16*>(a.kcache);
  const bf16* vc = static_cast<const bf16*>(a.vcache);
  const bf16* Q = static_cast<const bf16*>(a.Q);

  // this stream's tiles: i-th = chunk tile ts + i * NTS
  const int my_tiles = ntiles > ts ? (ntiles - ts + NTS - 1) / NTS : 0;
  uint8_t* wring = ring + (size_t)ts * NS * C::STAGE;
  auto load_tile = [&](int i) {
    const int t = ts + i * NTS;
    bf16* sk = reinterpret_cast<bf16*>(wring + (i % NS) * C::STAGE);
    bf16* sv = sk + TK * HD;
    const int base = k0 + t * TK;
#pragma unroll
    for (int e = lane + 32 * rg; e < TK * (HD / 8); e += 32 * RG) {
      const int kr = e / (HD / 8), c8 = e % (HD / 8);
      const int key = base + kr;
      const bool in = key < k1;
      const size_t src = ((size_t)(off + (in ? key : k0)) * a.nkv + g) * HD + c8 * 8;
      mm::cp16(mm::sa(sk + kv_sw<HD>(kr, c8)), kc + src, in ? 16 : 0);
      mm::cp16(mm::sa(sv + kv_sw<HD>(kr, c8)), vc + src, in ? 16 : 0);
    }
  };
  // the first tiles stream while the queries are staged
#pragma unroll
  for (int i = 0; i < NS - 1; ++i) {
    if (i < my_tiles) load_tile(i);
    mm::cp_commit();
  }
  for (int e = tid; e < QT * (HD / 8); e += C::THREADS) {
    const int qi = e / (HD / 8), c8 = e % (HD / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (qi < KG) {
      const int r = rb + qi / G, h = g * G + qi % G;
      v = *reinterpret_cast<const uint4*>(Q + ((size_t)r * a.nq + h) * HD + c8 * 8);
    }
    *reinterpret_cast<uint4*>(sQ + qi * LDS + c8 * 8) = v;
  }
  __syncthreads();

  const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units
  constexpr float kRaise = 8.f;                        // log2 headroom of the reference maximum
  float m_ref[MT][2], l_part[MT][2];
  float O[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    m_ref[mt][0] = m_ref[mt][1] = -INFINITY;
    l_part[mt][0] = l_part[mt][1] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) O[mt][nt][0] = O[mt][nt][1] = O[mt][nt][2] = O[mt][nt][3] = 0.f;
  }

  // a row group past the request's rows only helps stream the tiles
  const bool live = RG == 1 || rg * QR < KG;
  for (int i = 0; i < my_tiles; ++i) {
    if constexpr (RG == 1) {
      if (i + NS - 1 < my_tiles) load_tile(i + NS - 1);
      mm::cp_commit();
      mm::cp_wait<NS - 1>();
      __syncwarp();
    } else {
      // this warp's share of tile i has landed; after the barrier so has the
      // partner's, and both are done with tile i - 1, whose stage is refilled
      mm::cp_wait<NS - 2>();
      asm volatile("bar.sync %0, %1;" ::"r"(1 + ts), "r"(32 * RG) : "memory");
      if (i + NS - 1 < my_tiles) load_tile(i + NS - 1);
      mm::cp_commit();
    }
    if (!live) continue;
    const bf16* tK = reinterpret_cast<const bf16*>(wring + (i % NS) * C::STAGE);
    const bf16* tV = tK + TK * HD;
    // ---- S = Q K^T over this tile's 16 keys
    float S[MT][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) S[mt][nt][0] = S[mt][nt][1] = S[mt][nt][2] = S[mt][nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      uint32_t bk[4];   // keys (2 x 8) x 16 dims
      mm::ldsm4(bk, mm::sa(tK + kv_sw<HD>((lane >> 4) * 8 + (lane & 7), ks * 2 + ((lane >> 3) & 1))));
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t aq[4];
        mm::ldsm4(aq, mm::sa(sQ + (rg * QR + mt * 16 + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8));
        mm::mma16816(S[mt][0], aq, bk[0], bk[1]);
        mm::mma16816(S[mt][1], aq, bk[2], bk[3]);
      }
    }
    // ---- mask the tail, tile maxima per row (the quad of lanes holding it)
    const int kbase = k0 + (ts + i * NTS) * TK + (lane & 3) * 2;
    bool raise_any = false;
    float tmax[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float v = S[mt][nt][hf * 2 + c] * sl2;
            v = (kbase + nt * 8 + c < k1) ? v : -INFINITY;
            S[mt][nt][hf * 2 + c] = v;
            mx = fmaxf(mx, v);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        tmax[mt][hf] = mx;
        raise_any |= mx > m_ref[mt][hf] + kRaise;
      }
    // ---- raise a row's reference maximum (and rescale its O) only when
    // the tile exceeds it by more than 2^8; a warp-uniform branch
    if (__any_sync(0xffffffffu, raise_any)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const bool up = tmax[mt][hf] > m_ref[mt][hf] + kRaise;
          const float corr = !up ? 1.f : (m_ref[mt][hf] == -INFINITY ? 0.f : exp2f(m_ref[mt][hf] - tmax[mt][hf]));
          if (up) m_ref[mt][hf] = tmax[mt][hf];
          l_part[mt][hf] *= corr;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            O[mt][nt][hf * 2] *= corr;
            O[mt][nt][hf * 2 + 1] *= corr;
          }
        }
    }
    // ---- probabilities (bf16 A fragments straight from the scores)
    uint32_t ap[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      float p[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float mr = m_ref[mt][c >> 1];
          p[nt][c] = (mr == -INFINITY) ? 0.f : exp2f(S[mt][nt][c] - mr);
        }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        l_part[mt][hf] += (p[0][hf * 2] + p[0][hf * 2 + 1]) + (p[1][hf * 2] + p[1][hf * 2 + 1]);
      ap[mt][0] = pack_bf16(p[0][0], p[0][1]);
      ap[mt][1] = pack_bf16(p[0][2], p[0][3]);
      ap[mt][2] = pack_bf16(p[1][0], p[1][1]);
      ap[mt][3] = pack_bf16(p[1][2], p[1][3]);
    }
    // ---- O += P V
#pragma unroll
    for (int np = 0; np < HD / 16; ++np) {
      uint32_t bv[4];
      mm::ldsm4t(bv, mm::sa(tV + kv_sw<HD>((lane & 7) + ((lane >> 3) & 1) * 8, np * 2 + (lane >> 4))));
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mm::mma16816(O[mt][2 * np], ap[mt], bv[0], bv[1]);
        mm::mma16816(O[mt][2 * np + 1], ap[mt], bv[2], bv[3]);
      }
    }
    __syncwarp();
  }
  mm::cp_wait<0>();
  // ---- the warps meet once: (m, l, O) of each warp, merged per row
  __syncthreads();   // every warp is done with its ring, which now holds the merge
  float* sO = reinterpret_cast<float*>(ring);                 // [NW][QR][HD]
  float* sM = sO + (size_t)NW * QR * HD;                      // [NW][QR]
  float* sL = sM + NW * QR;                                   // [NW][QR]
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int row = mt * 16 + hf * 8 + (lane >> 2);
      float l = l_part[mt][hf];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      float* orow = sO + ((size_t)w * QR + row) * HD + (lane & 3) * 2;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float2*>(orow + nt * 8) = make_float2(O[mt][nt][hf * 2], O[mt][nt][hf * 2 + 1]);
      if ((lane & 3) == 0) {
        sM[w * QR + row] = m_ref[mt][hf];
        sL[w * QR + row] = l;
      }
    }
  __syncthreads();
  const size_t prow = ((size_t)(b * a.nkv + g) * a.nsplit + split) * KGmax;
  for (int e = tid; e < KG * (HD / 4); e += C::THREADS) {
    const int row = e / (HD / 4), c4 = (e % (HD / 4)) * 4;
    const int rgr = RG == 1 ? 0 : row / QR, lr = RG == 1 ? row : row % QR;   // its row group, row there
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < NTS; ++q) M = fmaxf(M, sM[(q * RG + rgr) * QR + lr]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
#pragma unroll
    for (int q = 0; q < NTS; ++q) {
      const int wq = q * RG + rgr;
      const float mq = sM[wq * QR + lr];
      const float f = (mq == -INFINITY) ? 0.f : exp2f(mq - M);
      const float4 o = *reinterpret_cast<const float4*>(sO + ((size_t)wq * QR + lr) * HD + c4);
      acc.x += o.x * f;
      acc.y += o.y * f;
      acc.z += o.z * f;
      acc.w += o.w * f;
      l += sL[wq * QR + lr] * f;
    }
    *reinterpret_cast<float4*>(a.part_o + (prow + row) * HD + c4) = acc;
    if (c4 == 0) {
      a.part_ml[(prow + row) * 2 + 0] = M * 0.6931471805599453f;
      a.part_ml[(prow + row) * 2 + 1] = l;
    }
  }
}

template <int MT, int HD, int NW, int NS, int RG = 1>
static cudaError_t launch_warp_mma(const DecodeAttnArgs& a, cudaStream_t st) {
  using C = WarpAttnCfg<MT, HD, NW, NS, RG>;
  static std::atomic<unsigned long long> attr{0};
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(decode_warp_mma<MT, HD, NW, NS, RG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SMEM);
  });
  if (e != cudaSuccess) return e;
  launch_pdl(decode_warp_mma<MT, HD, NW, NS, RG>, dim3(a.nsplit, a.nkv, a.B), C::THREADS, C::SMEM, st, a);
  return cudaGetLastError();
}

template <int MT, int HD, int NW = 4, int NS = 2>
static cudaError_t launch_split_mma(const DecodeAttnArgs& a, cudaStream_t st) {
  using C = MmaAttnCfg<MT, HD, NW, NS>;
  static std::atomic<unsigned long long> attr{0};
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(decode_split_mma<MT, HD, NW, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SMEM);
  });
  if (e != cudaSuccess) return e;
  launch_pdl(decode_split_mma<MT, HD, NW, NS>, dim3(a.nsplit, a.nkv, a.B), C::THREADS, C::SMEM, st, a);
  return cudaGetLastError();
}

template <int HD>
static cudaError_t split_mma_hd(const DecodeAttnArgs& a, cudaStream_t st) {
  const int KG = a.rows_max * (a.nq / a.nkv);
  // up to 32 query rows per KV head: warp-independent key slices; up to 64
  // (multi-row steps): two row groups whose warp pairs share each key tile;
  // more rows share each K/V tile across the block
  if (KG <= 16) return launch_warp_mma<1, HD, 4, 3>(a, st);
  if (KG <= 32) return launch_warp_mma<2, HD, 4, 3>(a, st);
  if (KG <= 64) return launch_warp_mma<2, HD, 8, 3, 2>(a, st);
  return launch_split_mma<8, HD>(a, st);
}

void decode_attn_plan(int B, int nkv, int max_kv_len, int* chunk, int* nsplit) {
  // about one chunk per SM: each chunk streams its keys once, and fewer
  // chunks keep the combine short
  const long long work = (long long)B * nkv * (max_kv_len > 0 ? max_kv_len : 1);
  long long c = work / num_sms();
  int ch = 64;
  while (ch < c && ch < 2048) ch *= 2;
  *chunk = ch;
  *nsplit = max_kv_len > 0 ? (max_kv_len + ch - 1) / ch : 1;
}

template <typename T, int E>
static cudaError_t decode_attn_t(const DecodeAttnArgs& a_in, int probe_op, cudaStream_t st) {
  const DecodeAttnArgs& a = a_in;
  dim3 grid(a.nsplit, a.nkv, a.B);
  probe_start(probe_op, st);
  if (sizeof(T) == 2 && a.rows_max * (a.nq / a.nkv) <= 128) {
    cudaError_t e = (E == 4) ? split_mma_hd<128>(a, st) : split_mma_hd<64>(a, st);
    if (e != cudaSuccess) return e;
  } else {
    launch_pdl(decode_split_simt<T, E>, grid, 256, 0, st, a);
  }
  note_launch();
  probe_stop(probe_op, st);
  launch_pdl(decode_combine<T, E>, dim3(a.R, (a.nq + 3) / 4), 128, 0, st, a);
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
  pdl_trigger();
  pdl_wait();
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

// ---------------------------------------------- training, bf16 tensor cores
// One CTA = 64 consecutive rows of one depth (anchors ascending) x one query
// head; warp w owns rows 16w..16w+15. Keys stream through shared memory in
// 64-row tiles (cp.async double buffer):
//   depth-0 tiles  rows j in [min start, max anchor]; row (i, d) keeps key j
//                  when start(i) <= j <= i (its own conversation, causal);
//   chain tiles    for c = 1..d the tile holds rows (a_t, c) of this tile's
//                  anchors a_t, gathered through row_of; row t keeps only
//                  key t (its own chain).
// S = Q K^T and O += P V run on mma.sync m16n8k16; P stays in registers
// (the accumulator layout of two 8-key tiles is the A layout of a 16-key
// step). Online softmax in exp2 units.
template <int HD>
struct TrainMmaCfg {
  static constexpr int TQ = 64, TK = 64, LDS = HD + 8;
  static constexpr int SMEM = (TQ * LDS + 4 * TK * LDS) * 2 + 2 * TK * 4;
};


template <int HD>
__global__ void __launch_bounds__(128) train_attn_mma(TrainAttnArgs a, TrainTileArgs tt) {
  pdl_trigger();
  pdl_wait();
  using C = TrainMmaCfg<HD>;
  constexpr int TQ = C::TQ, TK = C::TK, LDS = C::LDS, NTO = HD / 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
  bf16* sK = sQ + TQ * LDS;             // [2][TK][LDS]
  bf16* sV = sK + 2 * TK * LDS;         // [2][TK][LDS]
  int* sKey = reinterpret_cast<int*>(sV + 2 * TK * LDS);  // [2][TK] key row ids (-1 = none)

  const int tile = blockIdx.x, h = blockIdx.y;
  int d = 0;
  while (d + 1 < tt.K && tile >= tt.tile_off[d + 1]) ++d;
  const int row0 = tt.row_off[d] + (tile - tt.tile_off[d]) * TQ;
  const int nrows = min(TQ, tt.row_off[d + 1] - row0);
  const int G = a.nq / a.nkv, g = h / G;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const bf16* Q = static_cast<const bf16*>(a.Q);
  const bf16* Kr = static_cast<const bf16*>(a.Kr);
  const bf16* Vr = static_cast<const bf16*>(a.Vr);

  for (int e = tid; e < TQ * (HD / 8); e += 128) {
    const int q = e / (HD / 8), c8 = e % (HD / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (q < nrows) v = *reinterpret_cast<const uint4*>(Q + ((size_t)(row0 + q) * a.nq + h) * HD + c8 * 8);
    *reinterpret_cast<uint4*>(sQ + q * LDS + c8 * 8) = v;
  }
  // this thread's two rows (r, r + 8 within the warp's 16)
  int anc[2], st[2];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int q = 16 * w + hf * 8 + (lane >> 2);
    const bool live = q < nrows;
    anc[hf] = live ? a.row_anchor[row0 + q] : -1;
    st[hf] = live ? a.row_start[row0 + q] : 0x7fffffff;
  }
  // key range of the depth-0 part
  const int last = row0 + nrows - 1;
  const int kend = a.row_anchor[last];
  int kbeg = a.row_start[row0];
  // conversation starts are non-decreasing in the anchor, so row0's start is the minimum
  const int n0 = (kend - kbeg + 1 + TK - 1) / TK;    // depth-0 key tiles
  const int ntiles = n0 + d;                         // + one chain tile per depth 1..d

  auto load_tile = [&](int t, int buf) {
    for (int e = tid; e < TK; e += 128) {
      int kr;
      if (t < n0) {
        const int j = kbeg + t * TK + e;
        kr = j <= kend ? j : -1;
      } else {
        const int c = t - n0 + 1;
        kr = e < nrows ? a.row_of[(size_t)c * a.n + a.row_anchor[row0 + e]] : -1;
        if (kr >= a.R) kr = -1;
      }
      sKey[buf * TK + e] = kr;
    }
    __syncthreads();
    for (int e = tid; e < TK * (HD / 8); e += 128) {
      const int kk = e / (HD / 8), c8 = e % (HD / 8);
      const int kr = sKey[buf * TK + kk];
      const size_t src = ((size_t)(kr >= 0 ? kr : 0) * a.nkv + g) * HD + c8 * 8;
      mm::cp16(mm::sa(sK + (buf * TK + kk) * LDS + c8 * 8), Kr + src, kr >= 0 ? 16 : 0);
      mm::cp16(mm::sa(sV + (buf * TK + kk) * LDS + c8 * 8), Vr + src, kr >= 0 ? 16 : 0);
    }
  };

  const float sl2 = a.scale * 1.4426950408889634f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float O[NTO][4];
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;

  if (ntiles > 0) load_tile(0, 0);
  mm::cp_commit();
  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < ntiles) {
      load_tile(t + 1, buf ^ 1);
      mm::cp_commit();
      mm::cp_wait<1>();
    } else {
      mm::cp_wait<0>();
    }
    __syncthreads();
    const bf16* tK = sK + buf * TK * LDS;
    const bf16* tV = sV + buf * TK * LDS;
    const int* keys = sKey + buf * TK;
    const bool chain = t >= n0;
    // S = Q_w K^T : 16 rows x 64 keys
    float S[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      uint32_t aq[4];
      mm::ldsm4(aq, mm::sa(sQ + (16 * w + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8));
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bk[4];
        mm::ldsm4(bk, mm::sa(tK + (np * 16 + (lane >> 4) * 8 + (lane & 7)) * LDS + ks * 16 + ((lane >> 3) & 1) * 8));
        mm::mma16816(S[2 * np], aq, bk[0], bk[1]);
        mm::mma16816(S[2 * np + 1], aq, bk[2], bk[3]);
      }
    }
    // mask + online softmax (rows owned by this quad)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int qrow = 16 * w + hf * 8 + (lane >> 2);
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int kk = nt * 8 + (lane & 3) * 2 + c;
          const int kr = keys[kk];
          bool ok;
          if (!chain) ok = kr >= 0 && kr >= st[hf] && kr <= anc[hf];
          else ok = kr >= 0 && kk == qrow;
          const float v = ok ? S[nt][hf * 2 + c] * sl2 : -INFINITY;
          S[nt][hf * 2 + c] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m_run[hf], mx);
      const float corr = (mn == -INFINITY) ? 1.f : exp2f(m_run[hf] - mn);
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float p = (mn == -INFINITY) ? 0.f : exp2f(S[nt][hf * 2 + c] - mn);
          S[nt][hf * 2 + c] = p;
          sum += p;
        }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      l_run[hf] = l_run[hf] * corr + sum;
      m_run[hf] = mn;
#pragma unroll
      for (int nt = 0; nt < NTO; ++nt) {
        O[nt][hf * 2] *= corr;
        O[nt][hf * 2 + 1] *= corr;
      }
    }
    // O += P V, P from registers
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t ap[4];
      ap[0] = pack_bf16(S[2 * kc][0], S[2 * kc][1]);
      ap[1] = pack_bf16(S[2 * kc][2], S[2 * kc][3]);
      ap[2] = pack_bf16(S[2 * kc + 1][0], S[2 * kc + 1][1]);
      ap[3] = pack_bf16(S[2 * kc + 1][2], S[2 * kc + 1][3]);
#pragma unroll
      for (int np = 0; np < NTO / 2; ++np) {
        uint32_t bv[4];
        mm::ldsm4t(bv, mm::sa(tV + (kc * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDS + np * 16 + (lane >> 4) * 8));
        mm::mma16816(O[2 * np], ap, bv[0], bv[1]);
        mm::mma16816(O[2 * np + 1], ap, bv[2], bv[3]);
      }
    }
    __syncthreads();
  }
  bf16* Og = static_cast<bf16*>(a.O);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int q = 16 * w + hf * 8 + (lane >> 2);
    if (q >= nrows) continue;
    if (a.lse2 && (lane & 3) == 0) a.lse2[(size_t)(row0 + q) * a.nq + h] = m_run[hf] + log2f(l_run[hf]);
    const float inv = l_run[hf] > 0.f ? 1.f / l_run[hf] : 0.f;
    bf16* dst = Og + ((size_t)(row0 + q) * a.nq + h) * HD + (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt)
      *reinterpret_cast<__nv_bfloat162*>(dst + nt * 8) = __floats2bfloat162_rn(O[nt][hf * 2] * inv, O[nt][hf * 2 + 1] * inv);
  }
}

template <int HD>
static cudaError_t launch_train_mma(const TrainAttnArgs& a, const TrainTileArgs& tt_in, int probe_op, cudaStream_t st) {
  using C = TrainMmaCfg<HD>;
  TrainTileArgs tt = tt_in;
  tt.tile_off[0] = 0;
  for (int d = 0; d < tt.K; ++d)
    tt.tile_off[d + 1] = tt.tile_off[d] + (tt.row_off[d + 1] - tt.row_off[d] + C::TQ - 1) / C::TQ;
  static std::atomic<unsigned long long> attr{0};
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(train_attn_mma<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (e != cudaSuccess) return e;
  probe_start(probe_op, st);
  launch_pdl(train_attn_mma<HD>, dim3(tt.tile_off[tt.K], a.nq), 128, C::SMEM, st, a, tt);
  note_launch();
  probe_stop(probe_op, st);
  return cudaGetLastError();
}

template <typename T, int E>
static cudaError_t train_attn_t(const TrainAttnArgs& a, int probe_op, cudaStream_t st) {
  dim3 grid(a.R, (a.nq + 3) / 4);
  probe_start(probe_op, st);
  launch_pdl(train_attn_simt<T, E>, grid, 128, 0, st, a);
  note_launch();
  probe_stop(probe_op, st);
  return cudaGetLastError();
}

cudaError_t launch_train_attn(int dtype, const TrainAttnArgs& a, const TrainTileArgs& tt, int probe_op,
                              cudaStream_t st) {
  if (a.R <= 0) return cudaSuccess;
  if (train_attn_tc_supported(dtype, a)) {
    probe_start(probe_op, st);
    cudaError_t e = launch_train_attn_tc(a, tt, st);
    probe_stop(probe_op, st);
    return e;
  }
  if (dtype == PEAGLE_BF16)
    return a.hd == 128 ? launch_train_mma<128>(a, tt, probe_op, st) : launch_train_mma<64>(a, tt, probe_op, st);
  return a.hd == 128 ? train_attn_t<float, 4>(a, probe_op, st) : train_attn_t<float, 2>(a, probe_op, st);
}

}  // namespace pe

// Backward of the depth-masked training attention on the bf16 tensor cores
// (mma.sync m16n8k16, fp32 accumulation) -- the attention of "feat(
// speculative): add P-EAGLE parallel-drafting training for EAGLE-3 drafts -
// #2376" (PR description and Changelog: row (i, d) sees the depth-0 rows
// start(i)..i of its own conversation, then its chain rows (i, 1..d)).
//
// With P = softmax(scale * Q K^T) over each row's keys, dP = dO V^T and
// D = rowsum(dO * O):
//   dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO.
// P is rebuilt from the forward's base-2 log-sum-exp, so no softmax state
// is kept between the kernels. Every output element is written by one CTA
// or warp (no atomics, deterministic):
//   attn_bwd_dq_mma  query-major: 64 rows of one depth x one query head over
//                    their depth-0 keys in 64-key tiles; D first;
//   attn_bwd_kv_mma  key-major: 64 depth-0 keys x one KV head over every row
//                    (any depth, any of the G query heads of that KV head)
//                    that sees one of them, in 32-row steps;
//   attn_bwd_chain   one warp per (anchor with chain rows, KV head): the
//                    lower-triangular block of the anchor's chain rows
//                    (i, 1..D) -- a chain key (i, c) is seen only by the rows
//                    (i, d >= c) -- adds their part of dQ and writes dK, dV of
//                    the chain rows.
#include "mma.cuh"
#include "rows.cuh"

namespace pe {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int HD>
struct BwdMmaCfg {
  static constexpr int LDS = HD + 8;   // padded rows: conflict-free ldmatrix
  static constexpr int TQ = 64, TK = 64, NQ = 32;
  // dq: Q and dO of 64 rows, two stages of 64-key K and V tiles, D and lse2 of the rows
  static constexpr int DQ_SMEM = (2 * TQ * LDS + 4 * TK * LDS) * 2 + 2 * TQ * 4;
  // kv: K and V of 64 keys, two stages of 32-row Q and dO tiles and their
  // row data (lse2, D, anchor, start), the row range of every depth
  static constexpr int KV_SMEM = (2 * TK * LDS + 4 * NQ * LDS) * 2 + 2 * 4 * NQ * 4 + 2 * 17 * 4;
};

// First row of depth d whose anchor is >= x (depth-d anchors ascend).
__device__ __forceinline__ int first_row_at(const AttnBwdArgs& a, int d, int x) {
  int lo = a.off[d], hi = a.off[d + 1];
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a.row_anchor[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void pack_a(uint32_t (&ap)[4], const float (&c0)[4], const float (&c1)[4]) {
  ap[0] = pack_bf16(c0[0], c0[1]);
  ap[1] = pack_bf16(c0[2], c0[3]);
  ap[2] = pack_bf16(c1[0], c1[1]);
  ap[3] = pack_bf16(c1[2], c1[3]);
}

// ------------------------------------------------------------------- dQ
template <int HD>
__global__ void __launch_bounds__(128) attn_bwd_dq_mma(AttnBwdArgs a, TrainTileArgs tt) {
  pdl_trigger();
  pdl_wait();
  using C = BwdMmaCfg<HD>;
  constexpr int TQ = C::TQ, TK = C::TK, LDS = C::LDS, NTO = HD / 8, C8 = HD / 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* sQ = reinterpret_cast<bf16*>(smem_raw);   // [TQ][LDS]
  bf16* sO = sQ + TQ * LDS;                       // [TQ][LDS] dO
  bf16* sK = sO + TQ * LDS;                       // [2][TK][LDS]
  bf16* sV = sK + 2 * TK * LDS;                   // [2][TK][LDS]
  float* sD = reinterpret_cast<float*>(sV + 2 * TK * LDS);   // [TQ]
  float* sL = sD + TQ;                                       // [TQ]

  const int tile = blockIdx.x, h = blockIdx.y;
  int d = 0;
  while (d + 1 < tt.K && tile >= tt.tile_off[d + 1]) ++d;
  const int row0 = tt.row_off[d] + (tile - tt.tile_off[d]) * TQ;
  const int nrows = min(TQ, tt.row_off[d + 1] - row0);
  const int G = a.nq / a.nkv, g = h / G;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const bf16* Q = static_cast<const bf16*>(a.Q);
  const bf16* dO = static_cast<const bf16*>(a.dO);
  const bf16* Og = static_cast<const bf16*>(a.O);
  const bf16* Kr = static_cast<const bf16*>(a.Kr);
  const bf16* Vr = static_cast<const bf16*>(a.Vr);

  for (int e = tid; e < TQ * C8; e += 128) {
    const int q = e / C8, c8 = e % C8;
    const bool live = q < nrows;
    const size_t src = ((size_t)(row0 + (live ? q : 0)) * a.nq + h) * HD + c8 * 8;
    mm::cp16(mm::sa(sQ + q * LDS + c8 * 8), Q + src, live ? 16 : 0);
    mm::cp16(mm::sa(sO + q * LDS + c8 * 8), dO + src, live ? 16 : 0);
  }
  mm::cp_commit();
  // the depth-0 keys of the tile: conversation starts are non-decreasing in
  // the anchor, so row0 has the smallest start and the last row the largest
  // anchor; every row sees at least its anchor, so there is one tile or more
  const int kend = a.row_anchor[row0 + nrows - 1];
  const int kbeg = a.row_start[row0];
  const int n0 = (kend - kbeg + 1 + TK - 1) / TK;
  auto load_tile = [&](int t, int buf) {
    for (int e = tid; e < TK * C8; e += 128) {
      const int kk = e / C8, c8 = e % C8;
      const int j = kbeg + t * TK + kk;
      const bool ok = j <= kend;
      const size_t src = ((size_t)(ok ? j : kbeg) * a.nkv + g) * HD + c8 * 8;
      mm::cp16(mm::sa(sK + (buf * TK + kk) * LDS + c8 * 8), Kr + src, ok ? 16 : 0);
      mm::cp16(mm::sa(sV + (buf * TK + kk) * LDS + c8 * 8), Vr + src, ok ? 16 : 0);
    }
  };
  load_tile(0, 0);
  mm::cp_commit();
  mm::cp_wait<1>();   // Q and dO have landed
  __syncthreads();
  {
    // D = dO . O (O from the forward) and the base-2 log-sum-exp; two
    // threads per row
    const int q = tid >> 1, half = tid & 1;
    const bool live = q < nrows;
    float s = 0.f;
    if (live) {
      const uint4* op = reinterpret_cast<const uint4*>(Og + ((size_t)(row0 + q) * a.nq + h) * HD) + half * (C8 / 2);
#pragma unroll
      for (int c = 0; c < C8 / 2; ++c) {
        const uint4 ov = op[c];
        const uint4 dv = *reinterpret_cast<const uint4*>(sO + q * LDS + (half * (C8 / 2) + c) * 8);
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
        const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
        for (int z = 0; z < 4; ++z) {
          const float2 of = __bfloat1622float2(o2[z]), df = __bfloat1622float2(d2[z]);
          s = fmaf(of.x, df.x, s);
          s = fmaf(of.y, df.y, s);
        }
      }
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    if (half == 0) {
      sD[q] = s;
      sL[q] = live ? a.lse2[(size_t)(row0 + q) * a.nq + h] : 0.f;
      if (live) a.Dv[(size_t)(row0 + q) * a.nq + h] = s;
    }
  }
  __syncthreads();
  // this thread's two rows (r, r + 8 within the warp's 16)
  int anc[2], st[2];
  float lse[2], Dr[2];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int q = 16 * w + hf * 8 + (lane >> 2);
    const bool live = q < nrows;
    anc[hf] = live ? a.row_anchor[row0 + q] : -1;
    st[hf] = live ? a.row_start[row0 + q] : 0x7fffffff;
    lse[hf] = sL[q];
    Dr[hf] = sD[q];
  }
  const float sl2 = a.scale * kLog2e;
  float dq[NTO][4];
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) dq[nt][0] = dq[nt][1] = dq[nt][2] = dq[nt][3] = 0.f;

  for (int t = 0; t < n0; ++t) {
    const int buf = t & 1;
    if (t + 1 < n0) {
      load_tile(t + 1, buf ^ 1);
      mm::cp_commit();
      mm::cp_wait<1>();
    } else {
      mm::cp_wait<0>();
    }
    __syncthreads();
    const bf16* tK = sK + buf * TK * LDS;
    const bf16* tV = sV + buf * TK * LDS;
    // S = Q K^T and dP = dO V^T: 16 rows x 64 keys each
    float S[8][4], P[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[nt][c] = P[nt][c] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      uint32_t aq[4], ao[4];
      const int aoff = (16 * w + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8;
      mm::ldsm4(aq, mm::sa(sQ + aoff));
      mm::ldsm4(ao, mm::sa(sO + aoff));
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bk[4], bv[4];
        const int boff = (np * 16 + (lane >> 4) * 8 + (lane & 7)) * LDS + ks * 16 + ((lane >> 3) & 1) * 8;
        mm::ldsm4(bk, mm::sa(tK + boff));
        mm::ldsm4(bv, mm::sa(tV + boff));
        mm::mma16816(S[2 * np], aq, bk[0], bk[1]);
        mm::mma16816(S[2 * np + 1], aq, bk[2], bk[3]);
        mm::mma16816(P[2 * np], ao, bv[0], bv[1]);
        mm::mma16816(P[2 * np + 1], ao, bv[2], bv[3]);
      }
    }
    // dS = P * (dP - D), P from the log-sum-exp and the row's visible keys
    const int kt0 = kbeg + t * TK;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int j = kt0 + nt * 8 + (lane & 3) * 2 + c;
          const bool vis = j >= st[hf] && j <= anc[hf];
          const float p = vis ? exp2f(fmaf(S[nt][hf * 2 + c], sl2, -lse[hf])) : 0.f;
          P[nt][hf * 2 + c] = p * (P[nt][hf * 2 + c] - Dr[hf]);
        }
    // dQ += dS K
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t ap[4];
      pack_a(ap, P[2 * kc], P[2 * kc + 1]);
#pragma unroll
      for (int np = 0; np < NTO / 2; ++np) {
        uint32_t bk[4];
        mm::ldsm4t(bk, mm::sa(tK + (kc * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDS + np * 16 + (lane >> 4) * 8));
        mm::mma16816(dq[2 * np], ap, bk[0], bk[1]);
        mm::mma16816(dq[2 * np + 1], ap, bk[2], bk[3]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int q = 16 * w + hf * 8 + (lane >> 2);
    if (q >= nrows) continue;
    float* dst = a.dQ + ((size_t)(row0 + q) * a.nq + h) * HD + (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt)
      *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(dq[nt][hf * 2] * a.scale, dq[nt][hf * 2 + 1] * a.scale);
  }
}

// -------------------------------------------------------------- dK, dV
template <int HD>
__global__ void __launch_bounds__(128) attn_bwd_kv_mma(AttnBwdArgs a) {
  pdl_trigger();
  pdl_wait();
  using C = BwdMmaCfg<HD>;
  constexpr int TK = C::TK, NQ = C::NQ, LDS = C::LDS, NTO = HD / 8, C8 = HD / 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* sK = reinterpret_cast<bf16*>(smem_raw);   // [TK][LDS]
  bf16* sV = sK + TK * LDS;                       // [TK][LDS]
  bf16* sQ = sV + TK * LDS;                       // [2][NQ][LDS]
  bf16* sO = sQ + 2 * NQ * LDS;                   // [2][NQ][LDS] dO
  float* sL = reinterpret_cast<float*>(sO + 2 * NQ * LDS);   // [2][NQ] base-2 log-sum-exp
  float* sD = sL + 2 * NQ;                                   // [2][NQ] D
  int* sA = reinterpret_cast<int*>(sD + 2 * NQ);             // [2][NQ] anchor (-1: no row)
  int* sS = sA + 2 * NQ;                                     // [2][NQ] conversation start
  int* sLo = sS + 2 * NQ;                                    // [17] first row of each depth
  int* sHi = sLo + 17;                                       // [17] end of each depth's rows

  const int j0 = blockIdx.x * TK, g = blockIdx.y;
  const int jn = min(TK, a.n - j0);
  const int G = a.nq / a.nkv;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const bf16* Q = static_cast<const bf16*>(a.Q);
  const bf16* dO = static_cast<const bf16*>(a.dO);
  const bf16* Kr = static_cast<const bf16*>(a.Kr);
  const bf16* Vr = static_cast<const bf16*>(a.Vr);

  for (int e = tid; e < TK * C8; e += 128) {
    const int kk = e / C8, c8 = e % C8;
    const bool ok = kk < jn;
    const size_t src = ((size_t)(j0 + (ok ? kk : 0)) * a.nkv + g) * HD + c8 * 8;
    mm::cp16(mm::sa(sK + kk * LDS + c8 * 8), Kr + src, ok ? 16 : 0);
    mm::cp16(mm::sa(sV + kk * LDS + c8 * 8), Vr + src, ok ? 16 : 0);
  }
  mm::cp_commit();
  // the rows that see a key of the tile have anchors in [j0, end of the last
  // key's conversation); per depth they are one contiguous range
  const int qend = a.row_end[j0 + jn - 1];
  if (tid < a.K) {
    sLo[tid] = first_row_at(a, tid, j0);
    sHi[tid] = first_row_at(a, tid, qend);
  }
  __syncthreads();
  int total = 0;   // steps: per depth, 32-row blocks, each for the G query heads
  for (int dd = 0; dd < a.K; ++dd) total += (sHi[dd] - sLo[dd] + NQ - 1) / NQ * G;

  int cd = 0, cb = 0, ch = 0;   // depth, row block and head of the next step to load
  auto skip_empty = [&]() {
    while (cd < a.K && sLo[cd] + cb * NQ >= sHi[cd]) {
      ++cd;
      cb = 0;
    }
  };
  skip_empty();
  auto load_step = [&](int buf) {
    const int r0 = sLo[cd] + cb * NQ, h = g * G + ch;
    const int nr = min(NQ, sHi[cd] - r0);
    for (int e = tid; e < NQ * C8; e += 128) {
      const int q = e / C8, c8 = e % C8;
      const bool live = q < nr;
      const size_t src = ((size_t)(r0 + (live ? q : 0)) * a.nq + h) * HD + c8 * 8;
      mm::cp16(mm::sa(sQ + (buf * NQ + q) * LDS + c8 * 8), Q + src, live ? 16 : 0);
      mm::cp16(mm::sa(sO + (buf * NQ + q) * LDS + c8 * 8), dO + src, live ? 16 : 0);
    }
    if (tid < NQ) {
      const bool live = tid < nr;
      const size_t ri = (size_t)(r0 + tid) * a.nq + h;
      sL[buf * NQ + tid] = live ? a.lse2[ri] : 0.f;
      sD[buf * NQ + tid] = live ? a.Dv[ri] : 0.f;
      sA[buf * NQ + tid] = live ? a.row_anchor[r0 + tid] : -1;
      sS[buf * NQ + tid] = live ? a.row_start[r0 + tid] : 0x7fffffff;
    }
    if (++ch == G) {
      ch = 0;
      ++cb;
      skip_empty();
    }
  };

  const float sl2 = a.scale * kLog2e;
  const int jk = j0 + 16 * w + (lane >> 2);   // this thread's keys: jk and jk + 8
  float dk[NTO][4], dv[NTO][4];
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) dk[nt][c] = dv[nt][c] = 0.f;

  if (total > 0) load_step(0);
  mm::cp_commit();
  for (int s = 0; s < total; ++s) {
    const int buf = s & 1;
    if (s + 1 < total) {
      load_step(buf ^ 1);
      mm::cp_commit();
      mm::cp_wait<1>();
    } else {
      mm::cp_wait<0>();
    }
    __syncthreads();
    const bf16* tQ = sQ + buf * NQ * LDS;
    const bf16* tO = sO + buf * NQ * LDS;
    const float* tL = sL + buf * NQ;
    const float* tD = sD + buf * NQ;
    const int* tA = sA + buf * NQ;
    const int* tS = sS + buf * NQ;
    // S^T = K Q^T and dP^T = V dO^T: 16 keys x 32 rows each
    float S[4][4], P[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[nt][c] = P[nt][c] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      uint32_t ak[4], av[4];
      const int aoff = (16 * w + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8;
      mm::ldsm4(ak, mm::sa(sK + aoff));
      mm::ldsm4(av, mm::sa(sV + aoff));
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t bq[4], bo[4];
        const int boff = (np * 16 + (lane >> 4) * 8 + (lane & 7)) * LDS + ks * 16 + ((lane >> 3) & 1) * 8;
        mm::ldsm4(bq, mm::sa(tQ + boff));
        mm::ldsm4(bo, mm::sa(tO + boff));
        mm::mma16816(S[2 * np], ak, bq[0], bq[1]);
        mm::mma16816(S[2 * np + 1], ak, bq[2], bq[3]);
        mm::mma16816(P[2 * np], av, bo[0], bo[1]);
        mm::mma16816(P[2 * np + 1], av, bo[2], bo[3]);
      }
    }
    // P^T (into S) and dS^T (into P); key j is visible to row q when
    // start(q) <= j <= anchor(q)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int q = nt * 8 + (lane & 3) * 2 + c;
        const int qa = tA[q], qs = tS[q];
        const float ql = tL[q], qd = tD[q];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int j = jk + hf * 8;
          const bool vis = j >= qs && j <= qa;
          const float p = vis ? exp2f(fmaf(S[nt][hf * 2 + c], sl2, -ql)) : 0.f;
          S[nt][hf * 2 + c] = p;
          P[nt][hf * 2 + c] = p * (P[nt][hf * 2 + c] - qd);
        }
      }
    // dV += P^T dO and dK += dS^T Q over the 32 rows
#pragma unroll
    for (int kc = 0; kc < 2; ++kc) {
      uint32_t ap[4], ad[4];
      pack_a(ap, S[2 * kc], S[2 * kc + 1]);
      pack_a(ad, P[2 * kc], P[2 * kc + 1]);
#pragma unroll
      for (int np = 0; np < NTO / 2; ++np) {
        const int off = (kc * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDS + np * 16 + (lane >> 4) * 8;
        uint32_t bo[4], bq[4];
        mm::ldsm4t(bo, mm::sa(tO + off));
        mm::ldsm4t(bq, mm::sa(tQ + off));
        mm::mma16816(dv[2 * np], ap, bo[0], bo[1]);
        mm::mma16816(dv[2 * np + 1], ap, bo[2], bo[3]);
        mm::mma16816(dk[2 * np], ad, bq[0], bq[1]);
        mm::mma16816(dk[2 * np + 1], ad, bq[2], bq[3]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int kk = 16 * w + hf * 8 + (lane >> 2);
    if (kk >= jn) continue;
    const size_t base = ((size_t)(j0 + kk) * a.nkv + g) * HD + (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) {
      *reinterpret_cast<float2*>(a.dK + base + nt * 8) =
          make_float2(dk[nt][hf * 2] * a.scale, dk[nt][hf * 2 + 1] * a.scale);
      *reinterpret_cast<float2*>(a.dV + base + nt * 8) = make_float2(dv[nt][hf * 2], dv[nt][hf * 2 + 1]);
    }
  }
}

// ---------------------------------------------------------------- chain
template <int E>
__device__ __forceinline__ void ld_row(const bf16* p, float (&x)[E]) {
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = __bfloat162float(p[e]);
}

// one warp per (depth-1 row, KV head g): the chain rows (i, 1..D) of the
// row's anchor i; lane l holds head dims [l*E, (l+1)*E)
template <int E>
__global__ void __launch_bounds__(128) attn_bwd_chain(AttnBwdArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int HD = 32 * E;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int r1 = a.off[1] + blockIdx.x * 4 + w;
  if (r1 >= a.off[2]) return;
  const int g = blockIdx.y, G = a.nq / a.nkv;
  const int an = a.row_anchor[r1];
  // nested COD sets: the anchor's chain rows are depths 1..D, no gap
  auto chain_row = [&](int c) { return a.row_of[(size_t)c * a.n + an]; };
  int D = 0;
  while (D + 1 < a.K) {
    const int kr = chain_row(D + 1);
    if (kr < 0 || kr >= a.R) break;
    ++D;
  }
  const bf16* Q = static_cast<const bf16*>(a.Q);
  const bf16* dO = static_cast<const bf16*>(a.dO);
  const bf16* Kr = static_cast<const bf16*>(a.Kr);
  const bf16* Vr = static_cast<const bf16*>(a.Vr);
  const float sl2 = a.scale * kLog2e;
  // ds and p of query row qr (head h) against chain key kr
  auto score = [&](const float (&q)[E], const float (&o)[E], float l2, float Dq, const float (&k)[E],
                   const float (&v)[E], float& p) {
    float s = 0.f, dp = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      s = fmaf(q[e], k[e], s);
      dp = fmaf(o[e], v[e], dp);
    }
    s = warp_sum(s);
    dp = warp_sum(dp);
    p = exp2f(fmaf(s, sl2, -l2));
    return p * (dp - Dq);
  };
  // dQ of each chain row (i, d) and head: + scale * sum_{c <= d} ds_c k_c
  for (int dd = 1; dd <= D; ++dd) {
    const int qr = chain_row(dd);
    for (int hh = 0; hh < G; ++hh) {
      const int h = g * G + hh;
      const size_t ri = (size_t)qr * a.nq + h;
      float q[E], o[E], dq[E];
      ld_row<E>(Q + ri * HD + lane * E, q);
      ld_row<E>(dO + ri * HD + lane * E, o);
      const float l2 = a.lse2[ri], Dq = a.Dv[ri];
#pragma unroll
      for (int e = 0; e < E; ++e) dq[e] = 0.f;
      for (int c = 1; c <= dd; ++c) {
        const size_t kb = ((size_t)chain_row(c) * a.nkv + g) * HD + lane * E;
        float k[E], v[E], p;
        ld_row<E>(Kr + kb, k);
        ld_row<E>(Vr + kb, v);
        const float ds = score(q, o, l2, Dq, k, v, p);
#pragma unroll
        for (int e = 0; e < E; ++e) dq[e] = fmaf(ds, k[e], dq[e]);
      }
      float* out = a.dQ + ri * HD + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) out[e] += dq[e] * a.scale;
    }
  }
  // dK, dV of each chain row (i, c): the rows (i, d >= c), every head of g
  for (int c = 1; c <= D; ++c) {
    const int kr = chain_row(c);
    const size_t kb = ((size_t)kr * a.nkv + g) * HD + lane * E;
    float k[E], v[E], dk[E], dv[E];
    ld_row<E>(Kr + kb, k);
    ld_row<E>(Vr + kb, v);
#pragma unroll
    for (int e = 0; e < E; ++e) dk[e] = dv[e] = 0.f;
    for (int dd = c; dd <= D; ++dd) {
      const int qr = chain_row(dd);
      for (int hh = 0; hh < G; ++hh) {
        const size_t ri = (size_t)qr * a.nq + g * G + hh;
        float q[E], o[E], p;
        ld_row<E>(Q + ri * HD + lane * E, q);
        ld_row<E>(dO + ri * HD + lane * E, o);
        const float ds = score(q, o, a.lse2[ri], a.Dv[ri], k, v, p);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          dk[e] = fmaf(ds, q[e], dk[e]);
          dv[e] = fmaf(p, o[e], dv[e]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      a.dK[kb + e] = dk[e] * a.scale;
      a.dV[kb + e] = dv[e];
    }
  }
}

template <int HD>
cudaError_t attn_bwd_mma_hd(const AttnBwdArgs& a, cudaStream_t st) {
  using C = BwdMmaCfg<HD>;
  static std::atomic<unsigned long long> attr_q{0}, attr_kv{0};
  cudaError_t e = once_per_device(attr_q, [] {
    return cudaFuncSetAttribute(attn_bwd_dq_mma<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DQ_SMEM);
  });
  if (e == cudaSuccess)
    e = once_per_device(attr_kv, [] {
      return cudaFuncSetAttribute(attn_bwd_kv_mma<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::KV_SMEM);
    });
  if (e != cudaSuccess) return e;
  TrainTileArgs tt{};
  tt.K = a.K;
  for (int d = 0; d <= a.K; ++d) tt.row_off[d] = a.off[d];
  tt.tile_off[0] = 0;
  for (int d = 0; d < a.K; ++d) tt.tile_off[d + 1] = tt.tile_off[d] + (a.off[d + 1] - a.off[d] + C::TQ - 1) / C::TQ;
  launch_pdl(attn_bwd_dq_mma<HD>, dim3(tt.tile_off[a.K], a.nq), 128, C::DQ_SMEM, st, a, tt);
  note_launch();
  launch_pdl(attn_bwd_kv_mma<HD>, dim3((a.n + C::TK - 1) / C::TK, a.nkv), 128, C::KV_SMEM, st, a);
  note_launch();
  if (a.K >= 2 && a.off[2] > a.off[1]) {
    launch_pdl(attn_bwd_chain<HD / 32>, dim3((a.off[2] - a.off[1] + 3) / 4, a.nkv), 128, 0, st, a);
    note_launch();
  }
  return cudaGetLastError();
}

}  // namespace

bool attn_bwd_mma_supported(int dtype, const AttnBwdArgs& a) {
  return dtype == PEAGLE_BF16 && a.lse2 != nullptr && (a.hd == 64 || a.hd == 128) && a.nkv > 0 &&
         a.nq % a.nkv == 0 && a.K >= 1 && a.K <= 16 && a.n >= 1;
}

cudaError_t launch_attn_bwd_mma(const AttnBwdArgs& a, cudaStream_t st) {
  if (a.R <= 0) return cudaSuccess;
  return a.hd == 128 ? attn_bwd_mma_hd<128>(a, st) : attn_bwd_mma_hd<64>(a, st);
}

}  // namespace pe

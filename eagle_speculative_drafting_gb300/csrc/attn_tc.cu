// Training attention of the P-EAGLE parallel forward on the 5th-generation
// tensor cores ("feat(speculative) ... #2376": depth-0 rows see their own
// conversation causally, a depth-d row sees the depth-0 rows of its
// conversation up to its anchor plus its own chain rows (anchor, 1..d);
// "P_Eagle" README: packed conversations isolated by cu_seqlens).
//
// One CTA = 128 consecutive rows of one depth (anchors ascending) x one query
// head, 480 threads:
//   warp 0     one thread loads Q once and streams 128-key tiles of K with
//              TMA into a 3-stage ring released by the score product;
//   warp 14    one thread streams the tiles of V transposed (V^T, so both
//              products take K-major operands) into a 2-stage ring
//              released by P V (two producers: a K load never waits for a
//              V slot);
//   warp 1     one thread issues tcgen05.mma: S = Q K^T (M = 128 rows,
//              N = 128 keys, K = hd) into one of two TMEM buffers, and
//              O += P V (N = hd, K = 128 keys) into a TMEM accumulator with
//              P read from TMEM;
//   warps 2-9  two threads per row (64 columns each): read the scores from
//              TMEM, mask (start(i) <= key <= anchor(i)), online softmax in
//              exp2 units (the two halves of a row meet in shared memory
//              behind a named barrier of their two warps), write P (bf16,
//              two per 32-bit column) back over the first 32 of the thread's
//              own 64 score columns; the buffer is free again once P V has
//              read it;
//   warps 10-13 meanwhile, one thread per row: the <= d chain keys of the
//              row on the CUDA cores (their maximum, sum and weighted value
//              sum, the latter in spare TMEM columns), merged at the end.
// The reference maximum of a row is only raised when the tile maximum
// exceeds it by more than 2^8 (then O is rescaled in TMEM, after the
// previous P V has landed); in between, probabilities relative to the older
// maximum stay below 256. With lse2 given, each row's base-2 log-sum-exp of
// its scaled scores is written too.
// Every mbarrier wait is bounded (1 s); on expiry the kernel sets
// PEAGLE_DEV_TIMEOUT and stops, after waiting (again bounded) for the TMA
// copies and tensor-core products it has already issued.
#include "rows.cuh"
#include "tc.cuh"

namespace pe {

namespace ta {
constexpr int TQ = 128, TK = 128, HD = 128, NK = 3, NV = 2, THREADS = 480;
constexpr int QB = TQ * HD * 2;    // Q tile (two 64-column boxes)
constexpr int KB = TK * HD * 2;    // K tile
constexpr int VB = HD * TK * 2;    // V^T tile
constexpr int BOX = 128 * 128;     // one 64-column x 128-row box
constexpr int SMEM = 1024 + QB + NK * KB + NV * VB + 8 * TQ * 4 + 256;
constexpr float kRescale = 8.f;    // log2 headroom before the reference max moves
constexpr int kWarpV = 14;         // the V producer
}  // namespace ta

// named barrier of the two softmax warps that hold rows quad*32 .. +31
__device__ __forceinline__ void pair_sync(int quad) {
  asm volatile("bar.sync %0, 64;" ::"r"(2 + quad) : "memory");
}

__global__ void __launch_bounds__(ta::THREADS, 1)
    train_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, TrainAttnArgs a, TrainTileArgs tt) {
  using namespace ta;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + QB;              // [NK][KB]
  uint8_t* sV = sK + NK * KB;         // [NV][VB]
  float* sX = reinterpret_cast<float*>(sV + NV * VB);   // [2 tiles][2 halves][TQ] partial row maxima
  float* sCm = sX + 4 * TQ;                            // [TQ] chain maximum per row
  float* sCl = sCm + TQ;                               // [TQ] chain sum per row
  float* sL = sCl + TQ;                                // [2 halves][TQ] partial row sums
  uint64_t* qfull = reinterpret_cast<uint64_t*>(sL + 2 * TQ);
  uint64_t* kfull = qfull + 1;        // [NK]
  uint64_t* kempty = kfull + NK;      // [NK]
  uint64_t* vfull = kempty + NK;      // [NV]
  uint64_t* vempty = vfull + NV;      // [NV]
  uint64_t* sfull = vempty + NV;      // [2] scores of a tile are in TMEM buffer b
  uint64_t* sfree = sfull + 2;        // [2] buffer b's P has been read by P V
  uint64_t* pfull = sfree + 2;        // P of a tile is in TMEM and O is rescaled (both halves)
  uint64_t* pfree = pfull + 1;        // one completion per P V product
  uint64_t* chfull = pfree + 1;       // chain results of every row
  uint64_t* drain = chfull + 1;       // completion of every product issued, on abort
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* v_issued_s = abort_flag + 1;   // V^T tiles whose copies the V producer issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(qfull, 1);
    for (int s = 0; s < NK; ++s) {
      tc::mbar_init(&kfull[s], 1);
      tc::mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      tc::mbar_init(&vfull[s], 1);
      tc::mbar_init(&vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&sfull[b], 1);
      tc::mbar_init(&sfree[b], 1);
    }
    tc::mbar_init(pfull, 256);
    tc::mbar_init(pfree, 1);
    tc::mbar_init(chfull, 128);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    *v_issued_s = 0;
    tc::fence_mbar_init();
    tc::prefetch_map(&tmQ);
    tc::prefetch_map(&tmK);
    tc::prefetch_map(&tmV);
  }
  if (warp == 1) tc::tmem_alloc(tslot, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();
  pdl_wait();   // Q, K, V^T and the row metadata come from earlier kernels

  // this CTA's rows and key range
  const int tile = blockIdx.x, h = blockIdx.y;
  int d = 0;
  while (d + 1 < tt.K && tile >= tt.tile_off[d + 1]) ++d;
  const int row0 = tt.row_off[d] + (tile - tt.tile_off[d]) * TQ;
  const int nrows = min(TQ, tt.row_off[d + 1] - row0);
  const int G = a.nq / a.nkv, g = h / G;
  // conversation starts are non-decreasing in the anchor: row0 has the
  // smallest start, the last row the largest anchor. Tiles begin on a
  // 64-key boundary so every TMA column coordinate is 16-byte aligned.
  const int kend = a.row_anchor[row0 + nrows - 1];
  const int kbeg = a.row_start[row0] & ~63;
  const int ntiles = (kend - kbeg) / TK + 1;
  const float sl2 = a.scale * 1.4426950408889634f;
  constexpr uint32_t idesc = tc::idesc_bf16(128, 128);
  int k_issued = 0;   // K tiles whose copies warp 0 issued

  if (warp == 0) {
    if (lane == 0) {
      tc::mbar_expect_tx(qfull, QB);
      tc::tma_load_2d(sQ, &tmQ, h * HD, row0, qfull);
      tc::tma_load_2d(sQ + BOX, &tmQ, h * HD + 64, row0, qfull);
      for (int t = 0; t < ntiles && !*abort_flag; ++t) {
        const int sk = t % NK;
        const int key0 = kbeg + t * TK;
        if (!tc::mbar_wait(&kempty[sk], ((t / NK) & 1) ^ 1)) {
          *abort_flag = 1;
          set_status(a.status, PEAGLE_DEV_TIMEOUT);
          break;
        }
        tc::mbar_expect_tx(&kfull[sk], KB);
        tc::tma_load_2d(sK + sk * KB, &tmK, g * HD, key0, &kfull[sk]);
        tc::tma_load_2d(sK + sk * KB + BOX, &tmK, g * HD + 64, key0, &kfull[sk]);
        k_issued = t + 1;
      }
    }
  } else if (warp == kWarpV) {
    if (lane == 0) {
      int v_issued = 0;
      for (int t = 0; t < ntiles && !*abort_flag; ++t) {
        const int sv = t % NV;
        const int key0 = kbeg + t * TK;
        if (!tc::mbar_wait(&vempty[sv], ((t / NV) & 1) ^ 1)) {
          *abort_flag = 1;
          set_status(a.status, PEAGLE_DEV_TIMEOUT);
          break;
        }
        tc::mbar_expect_tx(&vfull[sv], VB);
        tc::tma_load_2d(sV + sv * VB, &tmV, key0, g * HD, &vfull[sv]);
        tc::tma_load_2d(sV + sv * VB + BOX, &tmV, key0 + 64, g * HD, &vfull[sv]);
        v_issued = t + 1;
      }
      *v_issued_s = v_issued;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t tO = tbase + 256;
      // O += P_u V_u, P_u from TMEM buffer u & 1 (keys 64i .. 64i+63 in
      // columns 64i .. 64i+31); then release the V^T stage, the buffer and O
      auto pv = [&](int u) -> bool {
        const int su = u % NV, b = u & 1;
        // every softmax thread has written its P and rescaled its O columns
        // (each product of the tile adds into all of O)
        if (!tc::mbar_wait(&vfull[su], (u / NV) & 1) || !tc::mbar_wait(pfull, u & 1)) return false;
        tc::fence_after();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t b0 = tc::smem_u32(sV + su * VB + i * BOX);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_tmem_a(tO, tbase + b * 128 + i * 64 + kk * 8, tc::sw128_desc(b0 + kk * 32), idesc,
                                (u > 0 || i > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(pfree);
        tc::mma_commit(&vempty[su]);
        tc::mma_commit(&sfree[b]);
        return true;
      };
      bool ok = tc::mbar_wait(qfull, 0);
      for (int t = 0; ok && t < ntiles && !*abort_flag; ++t) {
        const int s = t % NK, b = t & 1;
        ok = tc::mbar_wait(&kfull[s], (t / NK) & 1) && tc::mbar_wait(&sfree[b], ((t >> 1) & 1) ^ 1);
        if (!ok) break;
        tc::fence_after();
        const uint32_t tS = tbase + b * 128;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t a0 = tc::smem_u32(sQ + i * BOX), b0 = tc::smem_u32(sK + s * KB + i * BOX);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16(tS, tc::sw128_desc(a0 + kk * 32), tc::sw128_desc(b0 + kk * 32), idesc,
                         (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sfull[b]);
        tc::mma_commit(&kempty[s]);
        if (t >= 1) ok = pv(t - 1);
      }
      if (ok && !*abort_flag) ok = pv(ntiles - 1);
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, PEAGLE_DEV_TIMEOUT);
      }
    }
  } else if (warp < 10) {
    // ---- softmax: warp w holds row quad*32 + lane (TMEM lane quadrant =
    // warp % 4) and columns [hf*64, hf*64 + 64) of every score tile and of O
    const int quad = warp & 3, hf = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const bool live = row < nrows;
    const int anc = live ? a.row_anchor[row0 + row] : -1;
    const int st = live ? a.row_start[row0 + row] : 0x7fffffff;
    const uint32_t tl = (uint32_t)(quad * 32) << 16;
    const uint32_t tO = tbase + 256 + tl + hf * 64;
    constexpr int HC = TK / 2;   // columns per thread
    float m_ref = -INFINITY, l = 0.f;
    // every wait is skipped once the kernel has aborted, so a timeout never
    // leaves the other threads waiting on this one; the loop itself (and
    // its pair barriers) always runs to the end
    auto wait = [&](uint64_t* bar, uint32_t par) -> bool {
      bool ok = !*abort_flag && tc::mbar_wait(bar, par);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0 && !*abort_flag) {
        *abort_flag = 1;
        set_status(a.status, PEAGLE_DEV_TIMEOUT);
      }
      return ok;
    };
    // P V completions are observed strictly in order (one pfree phase at a
    // time): a parity wait is only unambiguous while the barrier is at most
    // one phase ahead of the phase waited for. The warp catches up on
    // product t-1 before it signals P of tile t: product t cannot start
    // before that signal, so the barrier is never two phases ahead.
    int pv_seen = 0;
    auto wait_pv = [&](int u) -> bool {   // until product u has completed
      bool ok = true;
      while (pv_seen <= u) {
        ok = wait(pfree, pv_seen & 1) && ok;
        ++pv_seen;
      }
      return ok;
    };
    for (int t = 0; t < ntiles; ++t) {
      const int b = t & 1;
      const bool have = wait(&sfull[b], (t >> 1) & 1);
      tc::fence_after();
      float sv[HC];
      if (have) {
        uint32_t r[HC / 16][16];
#pragma unroll
        for (int c = 0; c < HC / 16; ++c) tc::tmem_ld16_nowait(tbase + tl + b * 128 + hf * HC + c * 16, r[c]);
#pragma unroll
        for (int c = 0; c < HC / 16; ++c) tc::tmem_ld_wait16(r[c]);
#pragma unroll
        for (int c = 0; c < HC / 16; ++c)
#pragma unroll
          for (int k = 0; k < 16; ++k) sv[c * 16 + k] = __uint_as_float(r[c][k]);
      } else {
#pragma unroll
        for (int c = 0; c < HC; ++c) sv[c] = -INFINITY;
      }
      // mask to the row's visible columns [lo, hi] of this half tile and take
      // the row maximum of the raw scores (the scale is positive, so it is
      // applied to the maximum and folded into the exponent below); eight
      // independent partial maxima keep the reduction off one dependency chain
      const int key0 = kbeg + t * TK + hf * HC;
      const int lo = max(st - key0, 0), hi = min(anc - key0, HC - 1);
      float pm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = -INFINITY;
      if (lo == 0 && hi == HC - 1) {   // the whole half tile is visible to this row
#pragma unroll
        for (int c = 0; c < HC; ++c) pm[c & 7] = fmaxf(pm[c & 7], sv[c]);
      } else {
        // hi < lo (nothing visible) leaves span negative: no column passes
        const int span = hi - lo;
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          const bool vis = (unsigned)(c - lo) <= (unsigned)span && span >= 0;
          sv[c] = vis ? sv[c] : -INFINITY;
          pm[c & 7] = fmaxf(pm[c & 7], sv[c]);
        }
      }
      // the row maximum from both halves (slots alternate by tile parity, so
      // a slot is rewritten only after the partner has passed the next
      // tile's barrier, i.e. read this one)
      float* xs = sX + b * 2 * TQ;
      xs[hf * TQ + row] = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      pair_sync(quad);
      const float mraw = fmaxf(xs[row], xs[TQ + row]);
      const float mx = mraw == -INFINITY ? -INFINITY : mraw * sl2;
      // a row raises its reference maximum when the tile exceeds it by more
      // than 2^8 (both halves decide alike); O holds earlier tiles' products
      // only from tile 1 on, and a row whose reference was still -inf
      // contributed zeros, so only the others rescale, after the previous
      // P V product has landed (TMEM accesses are warp-wide)
      const bool raise = mx > m_ref + kRescale;
      const float corr = !raise ? 1.f : (m_ref == -INFINITY ? 0.f : tc::ex2_approx(m_ref - mx));
      const bool rescale = raise && t >= 1 && m_ref != -INFINITY;
      if (__any_sync(0xffffffffu, rescale) && wait_pv(t - 1)) {
        tc::fence_after();
#pragma unroll 1
        for (int c = 0; c < HC / 16; ++c) {
          uint32_t r[16];
          tc::tmem_ld16(tO + c * 16, r);
          if (rescale) {
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * corr);
          }
          tc::tmem_st16(tO + c * 16, r);
        }
      }
      if (raise) {
        l *= corr;
        m_ref = mx;
      }
      // probabilities, two bf16 per 32-bit column, over the first 32 of this
      // thread's 64 score columns (written 16 columns at a time, one wait);
      // eight partial sums; a quarter of the exponentials run on the FMA pipe
      float ps[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ps[k] = 0.f;
      const float nref = m_ref == -INFINITY ? -INFINITY : -m_ref;   // -inf rows: every p = 0
      const uint32_t tP = tbase + tl + b * 128 + hf * HC;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        uint32_t w[16];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int q = hc * 4 + qq;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = q * 8 + e * 2;
            const float x0 = fmaf(sv[c], sl2, nref), x1 = fmaf(sv[c + 1], sl2, nref);
            const bool poly = (q & 3) == 3;
            const float p0 = poly ? tc::ex2_poly(x0) : tc::ex2_approx(x0);
            const float p1 = poly ? tc::ex2_poly(x1) : tc::ex2_approx(x1);
            ps[q] += p0 + p1;
            const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
            w[qq * 4 + e] = *reinterpret_cast<const uint32_t*>(&pp);
          }
        }
        if (have) tc::tmem_st16_nowait(tP + hc * 16, w);
      }
      tc::tmem_st_wait();
      l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      if (t >= 1) wait_pv(t - 1);   // issued a tile ago, long done: keeps the count in step
      tc::fence_before();
      tc::mbar_arrive(pfull);
    }
    // ---- the row sum from both halves, the chain keys, then the output
    const bool done = wait_pv(ntiles - 1);
    tc::fence_after();
    sL[hf * TQ + row] = l;
    pair_sync(quad);
    const bool summed = wait(chfull, 0);
    if (done && summed) {
      const float lt = sL[row] + sL[TQ + row];
      const float m_c = sCm[row], l_c = sCl[row];
      const float m_f = fmaxf(m_ref, m_c);
      const float so = (m_ref == -INFINITY) ? 0.f : tc::ex2_approx(m_ref - m_f);
      const float sc = (m_c == -INFINITY) ? 0.f : tc::ex2_approx(m_c - m_f);
      const float lf = lt * so + l_c * sc;
      const float inv = lf > 0.f ? 1.f / lf : 0.f;
      // the base-2 log-sum-exp of the row's scaled scores (all its keys), for the backward
      if (a.lse2 && live && hf == 0) a.lse2[(size_t)(row0 + row) * a.nq + h] = m_f + __log2f(lf);
      const uint32_t tA = tbase + 384 + tl + hf * 64;
      uint4* Og = reinterpret_cast<uint4*>(static_cast<bf16*>(a.O) + ((size_t)(row0 + row) * a.nq + h) * HD + hf * 64);
      uint32_t ro[4][16], ra[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld16_nowait(tO + c * 16, ro[c]);
      if (d > 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld16_nowait(tA + c * 16, ra[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld_wait16(ra[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 16; ++k) ra[c][k] = 0u;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld_wait16(ro[c]);
      if (live) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t wo[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float x0 = (__uint_as_float(ro[c][2 * k]) * so + __uint_as_float(ra[c][2 * k]) * sc) * inv;
            const float x1 =
                (__uint_as_float(ro[c][2 * k + 1]) * so + __uint_as_float(ra[c][2 * k + 1]) * sc) * inv;
            const __nv_bfloat162 pp = __floats2bfloat162_rn(x0, x1);
            wo[k] = *reinterpret_cast<const uint32_t*>(&pp);
          }
          Og[c * 2] = make_uint4(wo[0], wo[1], wo[2], wo[3]);
          Og[c * 2 + 1] = make_uint4(wo[4], wo[5], wo[6], wo[7]);
        }
      }
    }
  } else if (warp < kWarpV) {
    // ---- chain keys (anchor, 1..d) of row quad*32 + lane, while the tiles
    // run: their maximum m_c, sum l_c and value sum relative to m_c (in TMEM
    // columns 384..511 of the row's lane)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const bool live = row < nrows;
    const uint32_t tA = tbase + 384 + ((uint32_t)(quad * 32) << 16);
    float m_c = -INFINITY, l_c = 0.f;
    bool ok = true;
    if (d > 0) {
      const int anc = live ? a.row_anchor[row0 + row] : -1;
      const bf16* Kg = static_cast<const bf16*>(a.Kr);
      const bf16* Vg = static_cast<const bf16*>(a.Vr);
      int kc[16];
      float sc[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        kc[c] = -1;
        if (live && c < d) {
          const int kr = a.row_of[(size_t)(c + 1) * a.n + anc];
          kc[c] = (kr >= 0 && kr < a.R) ? kr : -1;   // nested COD sets always provide it
        }
      }
      ok = __all_sync(0xffffffffu, tc::mbar_wait(qfull, 0));   // q is read from the Q tile
      if (ok) {
#pragma unroll 1
        for (int c = 0; c < d; ++c) {
          sc[c] = -INFINITY;
          if (kc[c] < 0) continue;
          const uint4* kp = reinterpret_cast<const uint4*>(Kg + ((size_t)kc[c] * a.nkv + g) * HD);
          uint4 kv[HD / 8];
#pragma unroll
          for (int e = 0; e < HD / 8; ++e) kv[e] = kp[e];
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < HD / 8; ++e) {
            // 16-byte chunk e of the row in the swizzled Q tile
            const uint4 qa = *reinterpret_cast<const uint4*>(sQ + (e / 8) * BOX + row * 128 +
                                                             (((e & 7) ^ (row & 7)) << 4));
            const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qa);
            const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kv[e]);
#pragma unroll
            for (int z = 0; z < 4; ++z) {
              const float2 qf = __bfloat1622float2(q2[z]), kf = __bfloat1622float2(k2[z]);
              dot = fmaf(qf.x, kf.x, dot);
              dot = fmaf(qf.y, kf.y, dot);
            }
          }
          sc[c] = dot * sl2;
          m_c = fmaxf(m_c, sc[c]);
        }
        // value sum: the chain loop is uniform over the warp (d is the
        // tile's depth), so every lane takes part in the TMEM accesses
#pragma unroll 1
        for (int c = 0; c < d; ++c) {
          const bool has = kc[c] >= 0 && m_c != -INFINITY;
          const float w = has ? tc::ex2_approx(sc[c] - m_c) : 0.f;
          l_c += w;
          uint4 vv[HD / 8];
          if (has) {
            const uint4* vp = reinterpret_cast<const uint4*>(Vg + ((size_t)kc[c] * a.nkv + g) * HD);
#pragma unroll
            for (int e = 0; e < HD / 8; ++e) vv[e] = vp[e];
          } else {
#pragma unroll
            for (int e = 0; e < HD / 8; ++e) vv[e] = make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int cc = 0; cc < HD / 16; ++cc) {
            uint32_t r[16];
            if (c > 0) tc::tmem_ld16(tA + cc * 16, r);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&vv[cc * 2 + e]);
#pragma unroll
              for (int z = 0; z < 4; ++z) {
                const float2 vf = __bfloat1622float2(v2[z]);
                const int k0 = e * 8 + 2 * z;
                r[k0] = __float_as_uint((c > 0 ? __uint_as_float(r[k0]) : 0.f) + w * vf.x);
                r[k0 + 1] = __float_as_uint((c > 0 ? __uint_as_float(r[k0 + 1]) : 0.f) + w * vf.y);
              }
            }
            tc::tmem_st16(tA + cc * 16, r);
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) {
        *abort_flag = 1;
        set_status(a.status, PEAGLE_DEV_TIMEOUT);
      }
    }
    sCm[row] = m_c;
    sCl[row] = l_c;
    tc::fence_before();
    tc::mbar_arrive(chfull);
  }
  tc::fence_before();
  __syncthreads();   // every role has stopped issuing
  if (*abort_flag) {
    // an aborted CTA drains what it issued before its shared memory and TMEM
    // go: Q, the last phase of every K and V^T stage, then every product
    if (warp == 0 && lane == 0) {
      const int v_issued = *v_issued_s;
      tc::mbar_wait(qfull, 0);
      for (int t = max(0, k_issued - NK); t < k_issued; ++t) tc::mbar_wait(&kfull[t % NK], (t / NK) & 1);
      for (int t = max(0, v_issued - NV); t < v_issued; ++t) tc::mbar_wait(&vfull[t % NV], (t / NV) & 1);
    } else if (warp == 1 && lane == 0) {
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0);
    }
    tc::fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tbase, 512);
  }
}

// V [R, nkv*hd] -> V^T [nkv*hd, Rp] (bf16), 32 x 32 tiles through shared memory
__global__ void __launch_bounds__(256) transpose_v_kernel(const bf16* __restrict__ V, int R, int C, bf16* __restrict__ Vt,
                                                          int Rp) {
  pdl_trigger();
  pdl_wait();
  __shared__ bf16 tileb[32][34];
  const int r0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 8 rows per pass
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    const int r = r0 + ty + k, c = c0 + tx;
    tileb[ty + k][tx] = (r < R && c < C) ? V[(size_t)r * C + c] : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    const int c = c0 + ty + k, r = r0 + tx;
    if (c < C && r < Rp) Vt[(size_t)c * Rp + r] = tileb[tx][ty + k];
  }
}

bool train_attn_tc_supported(int dtype, const TrainAttnArgs& a) {
  return dtype == PEAGLE_BF16 && a.hd == 128 && a.Vt != nullptr && a.Rp >= a.R && a.Rp % 64 == 0 &&
         a.nq % a.nkv == 0;
}

cudaError_t launch_train_attn_tc(const TrainAttnArgs& a, const TrainTileArgs& tt_in, cudaStream_t st) {
  using namespace ta;
  TrainTileArgs tt = tt_in;
  tt.tile_off[0] = 0;
  for (int d = 0; d < tt.K; ++d) tt.tile_off[d + 1] = tt.tile_off[d] + (tt.row_off[d + 1] - tt.row_off[d] + TQ - 1) / TQ;
  const int C = a.nkv * HD;
  launch_pdl(transpose_v_kernel, dim3((a.Rp + 31) / 32, (C + 31) / 32), 256, 0, st,
             static_cast<const bf16*>(a.Vr), a.R, C, static_cast<bf16*>(a.Vt), a.Rp);
  note_launch();
  CUtensorMap mq, mk, mv;
  if (!make_tma_2d(&mq, a.Q, a.R, a.nq * HD, a.nq * HD, 128) ||
      !make_tma_2d(&mk, a.Kr, a.R, C, C, 128) || !make_tma_2d(&mv, a.Vt, C, a.R, a.Rp, 128)) {
    set_error("train attention: cuTensorMapEncodeTiled failed");
    return cudaErrorInvalidValue;
  }
  static std::atomic<unsigned long long> attr{0};
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(train_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  });
  if (e != cudaSuccess) return e;
  if (tt.tile_off[tt.K] > 0) {
    launch_pdl(train_attn_tc, dim3(tt.tile_off[tt.K], a.nq), THREADS, SMEM, st, mq, mk, mv, a, tt);
    note_launch();
  }
  return cudaGetLastError();
}

}  // namespace pe

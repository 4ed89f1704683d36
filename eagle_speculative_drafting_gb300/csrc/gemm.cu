// Dense contractions D = X W^T of the draft model (fc, QKV, O, gate/up, down,
// lm_head; "P-EAGLE" user guide, Architecture: the projected hidden states
// pass through Llama-style decoder layers and a draft-vocab head).
//
// bf16: a persistent, warp-specialized tcgen05 kernel for sm_103a.
//   warp 0  one thread issues TMA tile loads (128B-swizzled, K-major) into a
//           STAGES-deep shared-memory ring, completing on mbarriers;
//   warp 1  one thread issues tcgen05.mma (kind::f16, fp32 accumulate) into
//           one of two TMEM accumulators and commits to mbarriers;
//   warps 2-5 drain a finished accumulator with tcgen05.ld and store fp32
//           partial sums while the next work item accumulates in the other.
// The 128-row operand ("A role") is the activation tile, or -- for a few
// activation rows (M <= 128) -- the weight tile ("swap": weights stream
// through the 128-lane side, activations sit in the narrow N side). Work
// items are (output tile, K slice); the K slices of a tile land in separate
// partial slabs that the consumer kernel sums, so no item waits on another.
// Every mbarrier wait is bounded (1 s by default, TcArgs::wait_ns); on
// expiry the kernel sets PEAGLE_DEV_TIMEOUT and stops issuing. Before it
// frees its TMEM and returns it waits (again bounded) for the TMA copies and
// tensor-core products it has already issued, so nothing lands in shared
// memory or TMEM after the CTA has gone.
//
// fp32: a tiled CUDA-core kernel (FFMA), exact fp32 accumulation.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc.cuh"

namespace pe {


// =========================================================================
// The tcgen05 kernel
// =========================================================================
enum { EPI_STORE = 0, EPI_ARGMAX = 1, EPI_CE = 2, EPI_SWIGLU = 3, EPI_QKV = 4 };

struct TcArgs {
  int rowsA, rowsB, K;     // A role has rowsA rows, B role rowsB rows, both K wide
  int splits;              // K slices per output tile (split mode)
  int streamk;             // 1: stream-K schedule (see Sched)
  int coop;                // 1: every split item runs in the first round (see the epilogue)
  float* out;              // fp32 partial slabs
  int ldo;                 // row stride of a slab (elements)
  size_t split_stride;     // elements between slabs
  int M, N;                // D is M x N
  int* sem;                // per-tile arrival counters (zero between launches)
  int* status;
  unsigned long long wait_ns;  // bound of every wait of the roles (0: one try)
  int w_early;             // W is not written by the kernels just before: its first
                           // tiles may load before the dependency wait
  // fused head epilogue (op != EPI_STORE): one partial per (row, column tile)
  int op;
  int part_ld;             // column tiles per row
  float* logits;           // optional fp32 copy of D, row stride logits_ld
  int logits_ld;
  float *p_max, *p_sum, *p_lab;
  int* p_idx;
  const int* labels;       // EPI_CE: draft-vocab label per GEMM row, -1 = none
  // EPI_SWIGLU: each weight tile pairs gate rows with the matching up rows
  // (rows gate_off + ...); the epilogue writes silu(gate) * up as bf16
  int gate_off;
  void* act;
  int act_ld;
  float* gu;               // optional fp32 gate / up values [M, gu_ld] (unsplit wide tiles)
  int gu_ld;
  // EPI_QKV: rotate q/k by position, write q/k/v as bf16 (head dim 128)
  int nq, nkv, max_pos, row_base;
  const float *rcos, *rsin;
  const int* row_pos;
  void *q_out, *k_out, *v_out;
};

// Running head statistics of one row over some columns: argmax (lowest
// index on ties), and for cross-entropy the online max / sum of exp and the
// logit of the label.
struct HeadAcc {
  float bv, mx, se, ll;
  int bi;
  __device__ __forceinline__ void init() {
    bv = -INFINITY;
    bi = 0x7fffffff;
    mx = -INFINITY;
    se = 0.f;
    ll = -INFINITY;
  }
  __device__ __forceinline__ void add(float v, int n, int lab, bool ce) {
    if (am_better(v, n, bv, bi)) {
      bv = v;
      bi = n;
    }
    if (ce) {
      if (v > mx) {
        se = se * __expf(mx - v) + 1.f;
        mx = v;
      } else {
        se += __expf(v - mx);
      }
      if (n == lab) ll = v;
    }
  }
  // 32 consecutive columns at once: independent max / exp / compare steps
  // instead of a dependent chain per element (NaN falls back to add()).
  __device__ __forceinline__ void add_chunk(const float (&v)[32], int n0, int nvalid, int lab, bool ce) {
    bool nan = false;
    float cm = -INFINITY;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float x = c < nvalid ? v[c] : -INFINITY;
      nan |= (x != x);
      cm = fmaxf(cm, x);
    }
    if (nan) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid) add(v[c], n0 + c, lab, ce);
      return;
    }
    int ci = 0x7fffffff;
#pragma unroll
    for (int c = 31; c >= 0; --c)
      if (c < nvalid && v[c] == cm) ci = n0 + c;
    if (am_better(cm, ci, bv, bi)) {
      bv = cm;
      bi = ci;
    }
    if (ce && cm != -INFINITY) {
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) sum += (c < nvalid) ? __expf(v[c] - cm) : 0.f;
      const float nm = fmaxf(mx, cm);
      se = (mx == -INFINITY ? 0.f : se * __expf(mx - nm)) + sum * __expf(cm - nm);
      mx = nm;
      const int off = lab - n0;
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c == off && c < nvalid) ll = v[c];
    }
  }
  __device__ __forceinline__ void warp_merge(bool ce) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (am_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
      if (ce) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const float os = __shfl_xor_sync(0xffffffffu, se, o);
        const float nm = fmaxf(mx, om);
        se = (mx == -INFINITY ? 0.f : se * __expf(mx - nm)) + (om == -INFINITY ? 0.f : os * __expf(om - nm));
        mx = nm;
        ll = fmaxf(ll, __shfl_xor_sync(0xffffffffu, ll, o));
      }
    }
  }
  __device__ __forceinline__ void write(const struct TcArgs& g, int m, int ct) const;
};

__device__ __forceinline__ void HeadAcc::write(const TcArgs& g, int m, int ct) const {
  const size_t idx = (size_t)m * g.part_ld + ct;
  g.p_idx[idx] = bi;
  g.p_max[idx] = bv;
  if (g.op == EPI_CE) {
    g.p_sum[idx] = se;
    g.p_lab[idx] = ll;
  }
}

// Head statistics of finished rows read back from slab 0: a warp per row,
// lanes across the tile's columns.
__device__ void head_finish_rows(const TcArgs& g, int m_begin, int m_end, int m_step, int n0, int ncols,
                                 int ct, int lane) {
  const bool ce = g.op == EPI_CE;
  for (int m = m_begin; m < m_end; m += m_step) {
    const int lab = (ce && g.labels) ? g.labels[m] : -1;
    HeadAcc a;
    a.init();
    for (int c = lane; c < ncols; c += 32) {
      const int n = n0 + c;
      const float v = __ldcg(g.out + (size_t)m * g.ldo + n);
      if (g.logits) g.logits[(size_t)m * g.logits_ld + n] = v;
      a.add(v, n, lab, ce);
    }
    a.warp_merge(ce);
    if (lane == 0) a.write(g, m, ct);
  }
}

// Work of one persistent CTA, as segments (tile, k-tiles [kb, ke)).
//   stream-K: with at least as many tiles as CTAs, every CTA ends with
//     tiles/gridDim whole tiles of its own (no cross-CTA sum, so the
//     kernel's last epilogues are local), and the leftover tiles come
//     first: their (tile, k-tile) units are cut into gridDim equal
//     contiguous ranges, so every CTA streams the same number of k-tiles
//     (+-1). The CTAs sharing a tile each write one partial slab:
//     slab = CTA - first CTA of the tile.
//   split: items (tile, slice) are dealt round-robin; slice s writes slab s.
struct Seg {
  int tile, kb, ke, slab, nslab;
};

struct Sched {
  long long U, u, ue;   // stream-K units of the leftover tiles, this CTA's range
  int tiles, ktiles, splits, streamk, grid, cta, w;
  int skt, dpt, dp;     // leftover tiles, whole tiles per CTA, whole tiles taken

  __host__ __device__ static long long begin(long long U, int G, long long c) { return c * U / G; }
  __host__ __device__ static int owner(long long u, long long U, int G) {
    long long c = u * G / U;
    while (c + 1 < G && begin(U, G, c + 1) <= u) ++c;
    while (c > 0 && begin(U, G, c) > u) --c;
    return (int)c;
  }
  __host__ __device__ void init(int tiles_, int ktiles_, int splits_, int streamk_, int grid_, int cta_) {
    tiles = tiles_;
    ktiles = ktiles_;
    splits = splits_;
    streamk = streamk_;
    grid = grid_;
    cta = cta_;
    dpt = (streamk && tiles >= grid) ? tiles / grid : 0;
    skt = tiles - dpt * grid;
    // a stream-K share needs at least one unit per CTA (an empty range
    // would count as a partial slab of its tile)
    if (dpt > 0 && skt > 0 && (long long)skt * ktiles < grid) {
      --dpt;
      skt += grid;
    }
    dp = 0;
    U = (long long)skt * ktiles;
    u = begin(U, grid, cta);
    ue = begin(U, grid, cta + 1);
    w = cta;
  }
  __host__ __device__ bool next(Seg& s) {
    if (streamk) {
      if (u >= ue) {
        if (dp >= dpt) return false;
        s.tile = skt + cta * dpt + dp;
        s.kb = 0;
        s.ke = ktiles;
        s.slab = 0;
        s.nslab = 1;
        ++dp;
        return true;
      }
      s.tile = (int)(u / ktiles);
      s.kb = (int)(u % ktiles);
      s.ke = (int)((long long)s.kb + (ue - u) < ktiles ? s.kb + (ue - u) : ktiles);
      const int first = owner((long long)s.tile * ktiles, U, grid);
      const int last = owner((long long)s.tile * ktiles + ktiles - 1, U, grid);
      s.slab = cta - first;
      s.nslab = last - first + 1;
      u += s.ke - s.kb;
      return true;
    }
    if (w >= tiles * splits) return false;
    s.tile = w / splits;
    const int sp = w % splits;
    s.kb = (int)((long long)sp * ktiles / splits);
    s.ke = (int)((long long)(sp + 1) * ktiles / splits);
    s.slab = sp;
    s.nslab = splits;
    w += grid;
    return true;
  }
};

constexpr int TC_THREADS = 192;
constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per block

constexpr int pow2_at_least(int v, int p = 32) { return p >= v ? p : pow2_at_least(v, 2 * p); }

// MA = 2: the A role tile is two 128-row blocks that share every weight
// stage (two M = 128 products per K step into two accumulators): 256-row
// items, fewer of them, for contractions whose 128-row items would leave
// the last round of CTAs mostly empty. (Per byte received it does 1.3-1.5x
// the tensor work of a 128 x 256 tile, but only three of its stages fit,
// and with the ring latency-bound a K step then takes about as long per
// flop as with four 128 x 256 stages.)
template <int BN, bool SWAP, int MA = 1>
struct TcCfg {
  // Narrow (swapped) tiles read several 64-wide boxes per stage, so each
  // weight row is fetched in 256-512 byte runs rather than 128-byte pieces.
  static constexpr int SUB = (SWAP && BN == 16) ? 4 : ((SWAP && BN <= 64) ? 2 : 1);
  static constexpr int A_SUB = 128 * 128;               // 128 rows x 64 bf16
  static constexpr int B_SUB = BN * 128;                // BN rows x 64 bf16
  static constexpr int A_BYTES = MA * SUB * A_SUB;
  static constexpr int B_BYTES = SUB * B_SUB;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int KT = 64 * SUB;                   // K elements per stage
  // wide tiles stage each epilogue warp's 32 x 32 fp32 block in shared
  // memory so the stores leave as whole 128-byte lines
  static constexpr int STG_LD = 33;
  static constexpr int STAGING = SWAP ? 0 : 4 * 32 * STG_LD * 4;
  static constexpr int STAGES = std::min(12, (kSmemLimit - 1024 - 256 - STAGING) / STAGE);
  static constexpr int SMEM = 1024 + STAGES * STAGE + 256 + STAGING;
  // TMEM columns of one work item's accumulators; two sets (the next item
  // accumulates while the last drains) when both fit in the 512 columns
  static constexpr int ACC = MA * BN;
  static constexpr int NBUF = 2 * ACC <= 512 ? 2 : 1;
  static constexpr int TMEM_COLS = pow2_at_least(NBUF * ACC);
  static_assert(MA == 1 || (!SWAP && SUB == 1), "two row blocks only on wide tiles");
  static_assert(ACC <= 512 && BN % 16 == 0 && BN <= 256, "tile does not fit one CTA's TMEM");
  static_assert(STAGES >= 2, "ring too shallow");
};

// silu(gate) * up of finished rows read back from slab 0, where a tile's
// columns [src0, src0 + half) are gate and [src0 + half, src0 + 2 half) up.
__device__ void swiglu_finish_rows(const TcArgs& g, int m_begin, int m_end, int m_step, int src0, int half,
                                   int dst0, int lane) {
  bf16* act = static_cast<bf16*>(g.act);
  constexpr int U = 4;   // columns per lane whose loads issue before their stores
  for (int m = m_begin; m < m_end; m += m_step) {
    for (int j0 = 0; j0 < half; j0 += 32 * U) {
      float gt[U], up[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * 32 + lane;
        gt[u] = j < half ? __ldcg(g.out + (size_t)m * g.ldo + src0 + j) : 0.f;
        up[u] = j < half ? __ldcg(g.out + (size_t)m * g.ldo + src0 + half + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * 32 + lane;
        if (j < half) act[(size_t)m * g.act_ld + dst0 + j] = __float2bfloat16_rn(gt[u] / (1.f + __expf(-gt[u])) * up[u]);
      }
    }
  }
}

// Waits (bounded by limit_ns) until a global counter reaches target; the
// load is an acquire, so the writes released before the increments that
// brought it there are visible afterwards.
__device__ __forceinline__ bool wait_count(const int* ctr, int target, unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
    __nanosleep(100);
  }
}

// Sum of a split tile's slabs for rows [mlo, mhi) and columns [n0, n0 + BN)
// into slab 0, in slab order: warp ew of the four epilogue warps takes rows
// in blocks of four, lanes take float4 columns (lane * 4 + 128 j). All loads
// of two slabs x four rows are in flight before their sums.
template <int BN>
__device__ void coop_sum_rows(const TcArgs& g, int mlo, int mhi, int n0, int nslab, int ew, int lane) {
  const int ncol = min(g.N, n0 + BN);
  const bool al4 = (g.N & 3) == 0 && (g.ldo & 3) == 0 && (g.split_stride & 3) == 0 &&
                   (reinterpret_cast<uintptr_t>(g.out) & 15) == 0;
  if (al4) {
    constexpr int NV = (BN + 127) / 128;
    constexpr int RB = 4;
    for (int mb = mlo + ew * RB; mb < mhi; mb += 4 * RB) {
      float4 acc[RB][NV];
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int jv = 0; jv < NV; ++jv) acc[i][jv] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q0 = 0; q0 < nslab; q0 += 2) {
        float4 t[2][RB][NV];
#pragma unroll
        for (int qi = 0; qi < 2; ++qi)
#pragma unroll
          for (int i = 0; i < RB; ++i)
#pragma unroll
            for (int jv = 0; jv < NV; ++jv) {
              const int m = mb + i, n = n0 + jv * 128 + lane * 4;
              t[qi][i][jv] = (q0 + qi < nslab && m < mhi && n < ncol)
                                 ? __ldcg(reinterpret_cast<const float4*>(g.out + (size_t)(q0 + qi) * g.split_stride +
                                                                          (size_t)m * g.ldo + n))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int qi = 0; qi < 2; ++qi)
#pragma unroll
          for (int i = 0; i < RB; ++i)
#pragma unroll
            for (int jv = 0; jv < NV; ++jv)
              if (q0 + qi < nslab) {
                acc[i][jv].x += t[qi][i][jv].x;
                acc[i][jv].y += t[qi][i][jv].y;
                acc[i][jv].z += t[qi][i][jv].z;
                acc[i][jv].w += t[qi][i][jv].w;
              }
      }
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int jv = 0; jv < NV; ++jv) {
          const int m = mb + i, n = n0 + jv * 128 + lane * 4;
          if (m < mhi && n < ncol) *reinterpret_cast<float4*>(g.out + (size_t)m * g.ldo + n) = acc[i][jv];
        }
    }
  } else {
    constexpr int NC = BN >= 32 ? BN / 32 : 1;
    for (int m = mlo + ew; m < mhi; m += 4) {
      const size_t base = (size_t)m * g.ldo + n0 + lane;
      float acc[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] = 0.f;
      for (int q0 = 0; q0 < nslab; q0 += 4) {
        float t[4][NC];
#pragma unroll
        for (int qi = 0; qi < 4; ++qi)
#pragma unroll
          for (int c = 0; c < NC; ++c)
            t[qi][c] = (q0 + qi < nslab && n0 + c * 32 + lane < ncol)
                           ? __ldcg(g.out + (size_t)(q0 + qi) * g.split_stride + base + c * 32)
                           : 0.f;
#pragma unroll
        for (int qi = 0; qi < 4; ++qi)
#pragma unroll
          for (int c = 0; c < NC; ++c)
            if (q0 + qi < nslab) acc[c] += t[qi][c];
      }
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (n0 + c * 32 + lane < ncol) g.out[base + c * 32] = acc[c];
    }
  }
}

// CM = 2: two CTAs of a cluster take the two A tiles (row blocks 2p, 2p+1) of
// the same weight tile; each loads its half of the weight rows and
// multicasts it into both CTAs' ring stage, so every SM fetches half the
// weight bytes per product. A stage is free again once both CTAs' products
// have read it (each commit arrives on both CTAs' empty barrier).
// MA = 2: a work item covers 256 activation rows (row blocks 2t, 2t+1) in
// one CTA; both 128-row blocks and the weight tile share a ring stage.
template <int BN, bool SWAP, int CM, int MA>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   TcArgs g) {
  static_assert(CM == 1 || (CM == 2 && !SWAP), "clusters pair wide (unswapped) tiles only");
  static_assert(MA == 1 || CM == 1, "one pairing at a time");
  using C = TcCfg<BN, SWAP, MA>;
  constexpr uint16_t kPeers = (uint16_t)((1u << CM) - 1);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;   // completion of every product issued, on abort
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* s_last = abort_flag + 1;
  float* staging = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], CM);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 4);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_map(&tmA);
    tc::prefetch_map(&tmB);
  }
  if (warp == 1) tc::tmem_alloc(tslot, C::TMEM_COLS);
  tc::fence_before();
  if constexpr (CM > 1) tc::cluster_sync();   // the peer's barriers exist before any multicast
  else __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();   // the next kernel may launch now and wait for this one

  const int tilesA = (g.rowsA + 128 * MA - 1) / (128 * MA);
  const int tilesB = (g.rowsB + BN - 1) / BN;
  const int ktiles = (g.K + C::KT - 1) / C::KT;
  // work items are cluster tiles: CM consecutive A tiles of one weight tile
  // (the host pairs tiles only when tilesA is a multiple of CM)
  const int cr = CM > 1 ? (int)tc::cluster_ctarank() : 0;
  const int tilesAg = tilesA / CM;
  auto tile_of = [&](int t, int& ta, int& tb) {
    ta = (t % tilesAg) * CM + cr;
    tb = t / tilesAg;
  };
  // k-tile j of a work item: wide tiles start their K walk at an offset
  // that depends on the weight tile, so the CTAs running at once read
  // different column ranges of the weights (a lockstep walk sends every
  // request to the same column slice of thousands of rows)
  auto k_at = [&](int tb, int kb, int ke, int j) {
    if (SWAP) return kb + j;
    const int n = ke - kb;
    int q = j + (int)(((long long)tb * n) / tilesB);
    if (q >= n) q -= n;
    return kb + q;
  };
  Sched sc;
  sc.init(tilesAg * tilesB, ktiles, g.splits, g.streamk, gridDim.x / CM, blockIdx.x / CM);
  Seg sg;
  int p_issued = 0;   // ring iterations whose TMA copies the producer issued
  // boxes of 64 K-columns that exist in k-tile k (the last one may be short)
  auto nsub = [&](int k) { return min(C::SUB, (g.K - k * C::KT + 63) / 64); };

  if (warp == 0) {
    if (lane == 0) {
      // weight rows of tile t (row block of the weight operand) into one
      // sub-box; a gated tile takes its first half from the gate rows and its
      // second half from the matching up rows
      auto load_w = [&](uint8_t* dst, int x, int t, uint64_t* bar) {
        if (SWAP) {
          if (g.gate_off) {
            tc::tma_load_2d(dst, &tmA, x, t * 64, bar);
            tc::tma_load_2d(dst + 64 * 128, &tmA, x, g.gate_off + t * 64, bar);
          } else {
            tc::tma_load_2d(dst, &tmA, x, t * 128, bar);
          }
        } else {
          if constexpr (CM > 1) {
            // this CTA's half: the gate rows (rank 0) or the up rows (rank 1)
            // of a gated tile, else rows [cr * BN/2, (cr + 1) * BN/2)
            const int y = g.gate_off ? (cr == 0 ? t * (BN / 2) : g.gate_off + t * (BN / 2)) : t * BN + cr * (BN / 2);
            tc::tma_load_2d_mc(dst + cr * (BN / 2) * 128, &tmB, x, y, bar, kPeers);
          } else if (g.gate_off) {
            tc::tma_load_2d(dst, &tmB, x, t * (BN / 2), bar);
            tc::tma_load_2d(dst + (BN / 2) * 128, &tmB, x, g.gate_off + t * (BN / 2), bar);
          } else {
            tc::tma_load_2d(dst, &tmB, x, t * BN, bar);
          }
        }
      };
      int it = 0, pre = 0;
      bool waited = false;
      while (!*abort_flag && sc.next(sg)) {
        int ta, tb;
        tile_of(sg.tile, ta, tb);
        const int kb = sg.kb, ke = sg.ke;
        if (!waited) {
          // the weight tiles of the first stages depend on no earlier kernel:
          // start streaming them before waiting for the activations
          pre = g.w_early ? min(ke - kb, C::STAGES) : 0;
          for (int q = 0; q < pre; ++q) {
            const int k = k_at(tb, kb, ke, q), nv = nsub(k);
            tc::mbar_expect_tx(&full[q], nv * (MA * C::A_SUB + C::B_SUB));
            for (int i = 0; i < nv; ++i) {
              if (SWAP) load_w(sA + q * C::A_BYTES + i * C::A_SUB, k * C::KT + i * 64, ta, &full[q]);
              else load_w(sB + q * C::B_BYTES + i * C::B_SUB, k * C::KT + i * 64, tb, &full[q]);
            }
          }
          pdl_wait();
          waited = true;
        }
        for (int j = 0; j < ke - kb; ++j, ++it) {
          const int k = k_at(tb, kb, ke, j);
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          const int nv = nsub(k);
          if (it < pre) {   // weight half already in flight
            for (int i = 0; i < nv; ++i) {
              if (SWAP) tc::tma_load_2d(sB + s * C::B_BYTES + i * C::B_SUB, &tmB, k * C::KT + i * 64, tb * BN, &full[s]);
              else
                for (int h = 0; h < MA; ++h)
                  tc::tma_load_2d(sA + s * C::A_BYTES + (h + i) * C::A_SUB, &tmA, k * C::KT + i * 64,
                                  (ta * MA + h) * 128, &full[s]);
            }
            continue;
          }
          if (!tc::mbar_wait_for(&empty[s], ph ^ 1, g.wait_ns)) {
            *abort_flag = 1;
            set_status(g.status, PEAGLE_DEV_TIMEOUT);
            break;
          }
          tc::mbar_expect_tx(&full[s], nv * (MA * C::A_SUB + C::B_SUB));
          for (int i = 0; i < nv; ++i) {
            if (SWAP) {
              load_w(sA + s * C::A_BYTES + i * C::A_SUB, k * C::KT + i * 64, ta, &full[s]);
              tc::tma_load_2d(sB + s * C::B_BYTES + i * C::B_SUB, &tmB, k * C::KT + i * 64, tb * BN, &full[s]);
            } else {
              // (wide tiles have one box per stage: i = 0, block h at h * A_SUB)
              for (int h = 0; h < MA; ++h)
                tc::tma_load_2d(sA + s * C::A_BYTES + (h + i) * C::A_SUB, &tmA, k * C::KT + i * 64,
                                (ta * MA + h) * 128, &full[s]);
              load_w(sB + s * C::B_BYTES + i * C::B_SUB, k * C::KT + i * 64, tb, &full[s]);
            }
          }
        }
      }
      if (!waited) pdl_wait();
      p_issued = max(it, pre);
      if constexpr (CM > 1) {
        // the peer's products arrive on this CTA's empty barriers: wait for
        // the release of the last stages before the CTA may go
        for (int q = max(0, it - C::STAGES); q < it && !*abort_flag; ++q) {
          if (!tc::mbar_wait_for(&empty[q % C::STAGES], (q / C::STAGES) & 1, g.wait_ns)) {
            *abort_flag = 1;
            set_status(g.status, PEAGLE_DEV_TIMEOUT);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(128, BN);
      int it = 0, j = 0;
      for (; !*abort_flag && sc.next(sg); ++j) {
        const int kb = sg.kb, ke = sg.ke;
        int ta, tb;
        tile_of(sg.tile, ta, tb);
        const int buf = j % C::NBUF;
        const uint32_t use = j / C::NBUF;
        if (!tc::mbar_wait_for(&tempty[buf], (use & 1) ^ 1, g.wait_ns)) {
          *abort_flag = 1;
          set_status(g.status, PEAGLE_DEV_TIMEOUT);
          break;
        }
        tc::fence_after();
        const uint32_t dcol = tbase + buf * C::ACC;
        bool ok = true;
        for (int jk = 0; jk < ke - kb; ++jk, ++it) {
          const int k = k_at(tb, kb, ke, jk);
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!tc::mbar_wait_for(&full[s], ph, g.wait_ns)) {
            ok = false;
            break;
          }
          tc::fence_after();
          const int nv = nsub(k);
          for (int i = 0; i < nv; ++i) {
            const uint32_t a0 = tc::smem_u32(sA + s * C::A_BYTES + i * C::A_SUB);
            const uint32_t b0 = tc::smem_u32(sB + s * C::B_BYTES + i * C::B_SUB);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
              for (int h = 0; h < MA; ++h)
                tc::mma_bf16(dcol + h * BN, tc::sw128_desc(a0 + h * C::A_SUB + kk * 32), tc::sw128_desc(b0 + kk * 32),
                             idesc, (jk > 0 || i > 0 || kk > 0) ? 1u : 0u);
            }
          }
          if constexpr (CM > 1) tc::mma_commit_mc(&empty[s], kPeers);
          else tc::mma_commit(&empty[s]);
        }
        if (!ok) {
          *abort_flag = 1;
          set_status(g.status, PEAGLE_DEV_TIMEOUT);
          break;
        }
        tc::mma_commit(&tfull[buf]);
      }
    }
  } else {
    // epilogue: warps 2..5 cover TMEM lane quadrants (warp % 4); the output
    // slabs may still be read by the previous kernel until it completes
    pdl_wait();
    const int quad = warp & 3;
    int j = 0;
    for (; sc.next(sg); ++j) {
      int ta, tb;
      tile_of(sg.tile, ta, tb);
      const int tile = tb * tilesA + ta, sp = sg.slab;
      const int buf = j % C::NBUF;
      const uint32_t use = j / C::NBUF;
      // Whether to go on is decided by the four epilogue warps together (an
      // OR over the named barrier they share): a warp that left alone would
      // leave the others waiting at the barriers of the tile's finish.
      const bool ready = !*abort_flag && tc::mbar_wait_for(&tfull[buf], use & 1, g.wait_ns);
      if (!ready && !*abort_flag) {
        *abort_flag = 1;
        set_status(g.status, PEAGLE_DEV_TIMEOUT);
      }
      if (tc::bar_or_epilogue(!ready)) break;
      tc::fence_after();
      float* slab = g.out + (size_t)sp * g.split_stride;
      const int arow = ta * 128 + quad * 32 + lane;
      if (SWAP) {
        // lane = weight row n, column = activation row m: each store of the
        // warp covers 32 consecutive n
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t r[16];
          tc::tmem_ld16(tbase + ((uint32_t)(quad * 32) << 16) + buf * BN + c0, r);
          const int n = arow;
          if (n < g.N) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int m = tb * BN + c0 + c;
              if (m < g.M) slab[(size_t)m * g.ldo + n] = __uint_as_float(r[c]);
            }
          }
        }
      } else {
#pragma unroll 1
       for (int h = 0; h < MA; ++h) {
        const int tr = ta * MA + h;                          // 128-row block of the item
        const uint32_t tcol = (uint32_t)((buf * MA + h) * BN);   // its accumulator
        // lane = row m: transpose 32 x 32 blocks through shared memory, then
        // each warp store writes 4 rows x 128 contiguous bytes. A fused head
        // epilogue on an unsplit tile reduces the row straight from TMEM and
        // stores fp32 only if the caller asked for logits.
        float* stg = staging + (warp - 2) * 32 * C::STG_LD;
        const int m0 = tr * 128 + quad * 32;
        const bool head = g.op == EPI_ARGMAX || g.op == EPI_CE;
        if (g.op == EPI_QKV) {
          // columns [q heads | k heads | v heads] of 128: q and k rotated by
          // the row's position (pairs j, j + 64), all three written as bf16
          // (the host only asks for this on unsplit tiles)
          const int my_m = m0 + lane;
          int pos = 0;
          if (my_m < g.M) {
            pos = g.row_pos[g.row_base + my_m];
            if (pos < 0 || pos >= g.max_pos) {
              set_status(g.status, PEAGLE_DEV_BOUNDS);
              pos = pos < 0 ? 0 : g.max_pos - 1;
            }
          }
          const float4* cs = reinterpret_cast<const float4*>(g.rcos + (size_t)pos * 64);
          const float4* sn = reinterpret_cast<const float4*>(g.rsin + (size_t)pos * 64);
          const int qcols = g.nq * 128, kcols = g.nkv * 128;
#pragma unroll 1
          for (int hh = 0; hh < BN / 128; ++hh) {
            const int nh = tb * BN + hh * 128;   // the head's first column
            if (nh >= g.N) break;
            const bool rot = nh < qcols + kcols;
            bf16* dst;
            int ld;
            if (nh < qcols) {
              dst = static_cast<bf16*>(g.q_out) + nh;
              ld = qcols;
            } else if (nh < qcols + kcols) {
              dst = static_cast<bf16*>(g.k_out) + (nh - qcols);
              ld = kcols;
            } else {
              dst = static_cast<bf16*>(g.v_out) + (nh - qcols - kcols);
              ld = kcols;
            }
#pragma unroll 1
            for (int j0 = 0; j0 < 64; j0 += 16) {
              uint32_t rl[16], rh[16];
              tc::tmem_ld16(tbase + ((uint32_t)(quad * 32) << 16) + tcol + hh * 128 + j0, rl);
              tc::tmem_ld16(tbase + ((uint32_t)(quad * 32) << 16) + tcol + hh * 128 + 64 + j0, rh);
              float c[16], sv[16];
              if (rot) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const float4 cv = cs[j0 / 4 + q4], s4 = sn[j0 / 4 + q4];
                  c[q4 * 4] = cv.x, c[q4 * 4 + 1] = cv.y, c[q4 * 4 + 2] = cv.z, c[q4 * 4 + 3] = cv.w;
                  sv[q4 * 4] = s4.x, sv[q4 * 4 + 1] = s4.y, sv[q4 * 4 + 2] = s4.z, sv[q4 * 4 + 3] = s4.w;
                }
              }
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const float x = __uint_as_float(rl[k]), y = __uint_as_float(rh[k]);
                stg[lane * C::STG_LD + k] = rot ? x * c[k] - y * sv[k] : x;
                stg[lane * C::STG_LD + 16 + k] = rot ? y * c[k] + x * sv[k] : y;
              }
              __syncwarp();
              // 32 rows x (16 + 16) bf16: lane & 7 takes two columns of a row,
              // four rows per pass
              const int cc = (lane & 7) * 2;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int rr = i * 4 + (lane >> 3);
                const int m = m0 + rr;
                if (m < g.M) {
                  const float* srow = stg + rr * C::STG_LD;
                  bf16* drow = dst + (size_t)(g.row_base + m) * ld;
                  *reinterpret_cast<__nv_bfloat162*>(drow + j0 + cc) = __floats2bfloat162_rn(srow[cc], srow[cc + 1]);
                  *reinterpret_cast<__nv_bfloat162*>(drow + 64 + j0 + cc) =
                      __floats2bfloat162_rn(srow[16 + cc], srow[16 + cc + 1]);
                }
              }
              __syncwarp();
            }
          }
        } else if (g.op == EPI_SWIGLU && sg.nslab == 1) {
          // columns c and BN/2 + c are gate and up of output column
          // tb * BN/2 + c: write silu(gate) * up as bf16, coalesced
          constexpr int HALF = BN / 2;
          bf16* act = static_cast<bf16*>(g.act);
          const int I = g.N / 2;
          // the warp's staged 32 rows x 32 fp32 columns to gu from column col0
          // (4 rows x 128 bytes per store); this half of gu ends at column lim
          auto store_gu = [&](int col0, int lim) {
            __syncwarp();
            const int cc = (lane & 7) * 4;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = i * 4 + (lane >> 3);
              const int m = m0 + rr;
              const int n = col0 + cc;
              if (m < g.M && n < lim) {
                const float* srow = stg + rr * C::STG_LD + cc;
                float* dst = g.gu + (size_t)m * g.gu_ld + n;
                if (n + 4 <= lim) {
                  *reinterpret_cast<float4*>(dst) = make_float4(srow[0], srow[1], srow[2], srow[3]);
                } else {
#pragma unroll
                  for (int c = 0; c < 4; ++c)
                    if (n + c < lim) dst[c] = srow[c];
                }
              }
            }
            __syncwarp();
          };
#pragma unroll 1
          for (int c0 = 0; c0 < HALF; c0 += 32) {
            uint32_t rg[2][16], ru[2][16];   // gate / up columns c0 .. c0 + 31
            const uint32_t tl = tbase + ((uint32_t)(quad * 32) << 16) + tcol;
            tc::tmem_ld16(tl + c0, rg[0]);
            tc::tmem_ld16(tl + c0 + 16, rg[1]);
            tc::tmem_ld16(tl + HALF + c0, ru[0]);
            tc::tmem_ld16(tl + HALF + c0 + 16, ru[1]);
            if (g.gu) {
              // the gate and up values themselves, kept for the SwiGLU backward
#pragma unroll
              for (int c = 0; c < 32; ++c) stg[lane * C::STG_LD + c] = __uint_as_float(rg[c >> 4][c & 15]);
              store_gu(tb * HALF + c0, I);
#pragma unroll
              for (int c = 0; c < 32; ++c) stg[lane * C::STG_LD + c] = __uint_as_float(ru[c >> 4][c & 15]);
              store_gu(I + tb * HALF + c0, 2 * I);
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float gt = __uint_as_float(rg[c >> 4][c & 15]);
              stg[lane * C::STG_LD + c] = gt / (1.f + __expf(-gt)) * __uint_as_float(ru[c >> 4][c & 15]);
            }
            __syncwarp();
            const int cc = (lane & 7) * 4;
            const int n = tb * HALF + c0 + cc;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = i * 4 + (lane >> 3);
              const int m = m0 + rr;
              if (m < g.M) {
                const float* srow = stg + rr * C::STG_LD + cc;
                bf16* dst = act + (size_t)m * g.act_ld + n;
                if (n + 4 <= I && ((reinterpret_cast<uintptr_t>(dst) & 7) == 0)) {
                  __nv_bfloat162 lo = __floats2bfloat162_rn(srow[0], srow[1]);
                  __nv_bfloat162 hi = __floats2bfloat162_rn(srow[2], srow[3]);
                  uint2 pk;
                  pk.x = *reinterpret_cast<uint32_t*>(&lo);
                  pk.y = *reinterpret_cast<uint32_t*>(&hi);
                  *reinterpret_cast<uint2*>(dst) = pk;
                } else {
#pragma unroll
                  for (int c = 0; c < 4; ++c)
                    if (n + c < I) dst[c] = __float2bfloat16_rn(srow[c]);
                }
              }
            }
            __syncwarp();
          }
        } else {
        const bool fuse = head && sg.nslab == 1;
        float* tgt = fuse ? g.logits : slab;
        const int ldt = fuse ? g.logits_ld : g.ldo;
        const bool ce = g.op == EPI_CE;
        const int my_m = m0 + lane;
        const int lab = (fuse && ce && g.labels && my_m < g.M) ? g.labels[my_m] : -1;
        HeadAcc acc;
        acc.init();
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[16];
          float v[32];
          tc::tmem_ld16(tbase + ((uint32_t)(quad * 32) << 16) + tcol + c0, r);
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] = __uint_as_float(r[c]);
          tc::tmem_ld16(tbase + ((uint32_t)(quad * 32) << 16) + tcol + c0 + 16, r);
#pragma unroll
          for (int c = 0; c < 16; ++c) v[16 + c] = __uint_as_float(r[c]);
          if (fuse) acc.add_chunk(v, tb * BN + c0, min(32, g.N - (tb * BN + c0)), lab, ce);
          if (tgt) {
#pragma unroll
            for (int c = 0; c < 32; ++c) stg[lane * C::STG_LD + c] = v[c];
          }
          __syncwarp();
          if (tgt) {
            const int cc = (lane & 7) * 4;
            const int n = tb * BN + c0 + cc;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = i * 4 + (lane >> 3);
              const int m = m0 + rr;
              if (m < g.M) {
                const float* srow = stg + rr * C::STG_LD + cc;
                float* dst = tgt + (size_t)m * ldt + n;
                if (n + 4 <= g.N && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
                  *reinterpret_cast<float4*>(dst) = make_float4(srow[0], srow[1], srow[2], srow[3]);
                } else {
#pragma unroll
                  for (int c = 0; c < 4; ++c)
                    if (n + c < g.N) dst[c] = srow[c];
                }
              }
            }
          }
          __syncwarp();
        }
        if (fuse && my_m < g.M) acc.write(g, my_m, tb);
        }
       }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[buf]);
      const bool coop = !SWAP && g.coop && sg.nslab > 1;
      if (coop) {
        // every K slice of every tile runs at once (one round of items): the
        // tile's CTAs wait for all of its partial slabs, then each sums its
        // own share of the tile's rows into slab 0 (in slab order) and runs
        // the fused head / SwiGLU step on those rows. The counter goes to
        // nslab (slabs written), then to 2 nslab (shares done); the last
        // CTA re-arms it for the next launch.
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 2 && lane == 0) {
          atomicAdd(&g.sem[tile], 1);
          const bool all_in = wait_count(&g.sem[tile], sg.nslab, g.wait_ns);
          if (!all_in) set_status(g.status, PEAGLE_DEV_TIMEOUT);
          *s_last = all_in ? 1 : 0;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (*s_last) {
          __threadfence();
          const int ew = warp - 2;
          const int RT = 128 * MA;
          const int mlo = ta * RT + RT * sp / sg.nslab;
          const int mhi = min(g.M, ta * RT + RT * (sp + 1) / sg.nslab);
          coop_sum_rows<BN>(g, mlo, mhi, tb * BN, sg.nslab, ew, lane);
          if (g.op == EPI_SWIGLU || g.op == EPI_ARGMAX || g.op == EPI_CE) {
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (g.op == EPI_SWIGLU)
              swiglu_finish_rows(g, mlo + ew, mhi, 4, tb * BN, BN / 2, tb * (BN / 2), lane);
            else
              head_finish_rows(g, mlo + ew, mhi, 4, tb * BN, min(BN, g.N - tb * BN), tb, lane);
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 2 && lane == 0) {
          __threadfence();
          if (atomicAdd(&g.sem[tile], 1) == 2 * sg.nslab - 1) g.sem[tile] = 0;
        }
      }
      if (sg.nslab > 1 && !coop) {
        // the last of the tile's CTAs to arrive sums every slab of the tile
        // into slab 0, in slab order (deterministic), and re-arms the tile's
        // counter for the next launch
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 2 && lane == 0) *s_last = (atomicAdd(&g.sem[tile], 1) == sg.nslab - 1) ? 1 : 0;
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (*s_last) {
          __threadfence();
          const bool al4 = (g.N & 3) == 0 && (g.ldo & 3) == 0 && (g.split_stride & 3) == 0 &&
                           (reinterpret_cast<uintptr_t>(g.out) & 15) == 0;
          if (SWAP && al4) {
            // warp w of the epilogue sums rows w, w + 4, ... of the tile;
            // lanes take 4 consecutive columns each (float4). Up to eight
            // rows of four slabs are in flight per thread before any of their
            // sums is stored (slab 0 is read and rewritten by the same
            // thread): the finishing CTA's sum is the kernel's tail.
            const int m0 = tb * BN, mc = min(BN, g.M - m0);
            const int et = threadIdx.x - 64, rg = et >> 5;
            const int n0 = ta * 128 + (et & 31) * 4;
            if (n0 < g.N) {
              constexpr int RB = BN / 4 < 8 ? BN / 4 : 8;
              for (int r0 = rg; r0 < mc; r0 += 4 * RB) {
                float4 acc[RB];
#pragma unroll
                for (int i = 0; i < RB; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q0 = 0; q0 < sg.nslab; q0 += 4) {
                  float4 t[4][RB];
#pragma unroll
                  for (int qi = 0; qi < 4; ++qi)
#pragma unroll
                    for (int i = 0; i < RB; ++i) {
                      const int m = r0 + 4 * i;
                      t[qi][i] = (q0 + qi < sg.nslab && m < mc)
                                     ? __ldcg(reinterpret_cast<const float4*>(
                                           g.out + (size_t)(q0 + qi) * g.split_stride + (size_t)(m0 + m) * g.ldo + n0))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                  for (int qi = 0; qi < 4; ++qi)
#pragma unroll
                    for (int i = 0; i < RB; ++i)
                      if (q0 + qi < sg.nslab) {
                        acc[i].x += t[qi][i].x;
                        acc[i].y += t[qi][i].y;
                        acc[i].z += t[qi][i].z;
                        acc[i].w += t[qi][i].w;
                      }
                }
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                  const int m = r0 + 4 * i;
                  if (m < mc) *reinterpret_cast<float4*>(g.out + (size_t)(m0 + m) * g.ldo + n0) = acc[i];
                }
              }
            }
          } else if (SWAP) {
            const int n = arow, m0 = tb * BN, mc = min(BN, g.M - m0);
            if (n < g.N) {
              for (int c0 = 0; c0 < mc; c0 += 8) {
                float acc[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[c] = 0.f;
                const float* src = g.out + (size_t)(m0 + c0) * g.ldo + n;
#pragma unroll 4
                for (int q = 0; q < sg.nslab; ++q) {
#pragma unroll
                  for (int c = 0; c < 8; ++c)
                    if (c0 + c < mc) acc[c] += __ldcg(src + (size_t)q * g.split_stride + (size_t)c * g.ldo);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  if (c0 + c < mc) g.out[(size_t)(m0 + c0 + c) * g.ldo + n] = acc[c];
              }
            }
          } else if (!SWAP && al4) {
            // warp sums its 32 rows, four at a time; lanes take float4
            // columns lane*4 + 128j. Four rows of two slabs are in flight
            // per thread before any of their sums is stored.
            constexpr int NV = (BN + 127) / 128;
            constexpr int RB = 4;
            const int n0 = tb * BN;
            const int ncol = min(g.N, n0 + BN);   // this tile's columns end here
            for (int r0 = 0; r0 < 32 * MA; r0 += RB) {
              const int mb = (ta * MA + r0 / 32) * 128 + quad * 32 + r0 % 32;
              if (mb >= g.M) break;
              float4 acc[RB][NV];
#pragma unroll
              for (int i = 0; i < RB; ++i)
#pragma unroll
                for (int jv = 0; jv < NV; ++jv) acc[i][jv] = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int q0 = 0; q0 < sg.nslab; q0 += 2) {
                float4 t[2][RB][NV];
#pragma unroll
                for (int qi = 0; qi < 2; ++qi)
#pragma unroll
                  for (int i = 0; i < RB; ++i)
#pragma unroll
                    for (int jv = 0; jv < NV; ++jv) {
                      const int m = mb + i, n = n0 + jv * 128 + lane * 4;
                      t[qi][i][jv] = (q0 + qi < sg.nslab && m < g.M && n < ncol)
                                         ? __ldcg(reinterpret_cast<const float4*>(
                                               g.out + (size_t)(q0 + qi) * g.split_stride + (size_t)m * g.ldo + n))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                for (int qi = 0; qi < 2; ++qi)
#pragma unroll
                  for (int i = 0; i < RB; ++i)
#pragma unroll
                    for (int jv = 0; jv < NV; ++jv)
                      if (q0 + qi < sg.nslab) {
                        acc[i][jv].x += t[qi][i][jv].x;
                        acc[i][jv].y += t[qi][i][jv].y;
                        acc[i][jv].z += t[qi][i][jv].z;
                        acc[i][jv].w += t[qi][i][jv].w;
                      }
              }
#pragma unroll
              for (int i = 0; i < RB; ++i)
#pragma unroll
                for (int jv = 0; jv < NV; ++jv) {
                  const int m = mb + i, n = n0 + jv * 128 + lane * 4;
                  if (m < g.M && n < ncol) *reinterpret_cast<float4*>(g.out + (size_t)m * g.ldo + n) = acc[i][jv];
                }
            }
          } else {
            // warp sums its 32 rows; lanes walk 32 consecutive columns.
            // A row's loads (up to four slabs at a time) all issue before
            // its stores, which could alias them.
            constexpr int NC = BN >= 32 ? BN / 32 : 1;
            const int n0 = tb * BN;
            for (int rr = 0; rr < 32 * MA; ++rr) {
              const int m = (ta * MA + rr / 32) * 128 + quad * 32 + rr % 32;
              if (m >= g.M) break;
              const size_t base = (size_t)m * g.ldo + n0 + lane;
              float acc[NC];
#pragma unroll
              for (int c = 0; c < NC; ++c) acc[c] = 0.f;
              for (int q0 = 0; q0 < sg.nslab; q0 += 4) {
                float t[4][NC];
#pragma unroll
                for (int qi = 0; qi < 4; ++qi)
#pragma unroll
                  for (int c = 0; c < NC; ++c)
                    t[qi][c] = (q0 + qi < sg.nslab && n0 + c * 32 + lane < g.N)
                                   ? __ldcg(g.out + (size_t)(q0 + qi) * g.split_stride + base + c * 32)
                                   : 0.f;
#pragma unroll
                for (int qi = 0; qi < 4; ++qi)
#pragma unroll
                  for (int c = 0; c < NC; ++c)
                    if (q0 + qi < sg.nslab) acc[c] += t[qi][c];
              }
#pragma unroll
              for (int c = 0; c < NC; ++c)
                if (n0 + c * 32 + lane < g.N) g.out[base + c * 32] = acc[c];
            }
          }
          if (warp == 2 && lane == 0) g.sem[tile] = 0;
        }
      }
      if (g.op == EPI_SWIGLU && (SWAP || sg.nslab > 1) && !coop) {
        // silu(gate) * up of a finished tile, from slab 0
        const bool fin = (sg.nslab == 1) || *s_last;
        if (fin) {
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (SWAP)
            swiglu_finish_rows(g, warp - 2, g.M, 4, ta * 128, 64, ta * 64, lane);
          else
            for (int h = 0; h < MA; ++h) {
              const int r0 = (ta * MA + h) * 128 + quad * 32;
              swiglu_finish_rows(g, r0, min(g.M, r0 + 32), 1, tb * BN, BN / 2, tb * (BN / 2), lane);
            }
        }
      }
      if ((g.op == EPI_ARGMAX || g.op == EPI_CE) && (SWAP || sg.nslab > 1) && !coop) {
        // head statistics of a finished tile, from slab 0: by the only CTA
        // of an unsplit tile, or by the CTA that summed the slabs
        const bool fin = (sg.nslab == 1) || *s_last;
        if (fin) {
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (SWAP)
            head_finish_rows(g, warp - 2, g.M, 4, ta * 128, min(128, g.N - ta * 128), ta, lane);
          else
            for (int h = 0; h < MA; ++h) {
              const int r0 = (ta * MA + h) * 128 + quad * 32;
              head_finish_rows(g, r0, min(g.M, r0 + 32), 1, tb * BN, min(BN, g.N - tb * BN), tb, lane);
            }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();   // every role has stopped issuing
  if (*abort_flag) {
    // an aborted CTA drains what it issued before its shared memory and TMEM
    // go: the last TMA phase of every ring stage, then (one commit tracks
    // all of them) every tensor-core product
    if (warp == 0 && lane == 0) {
      for (int q = max(0, p_issued - C::STAGES); q < p_issued; ++q)
        tc::mbar_wait(&full[q % C::STAGES], (q / C::STAGES) & 1);
    } else if (warp == 1 && lane == 0) {
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0);
    }
    tc::fence_before();
    __syncthreads();
  }
  if constexpr (CM > 1) tc::cluster_sync();   // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

// =========================================================================
// fp32 CUDA-core kernel: 64x64 output tile, 256 threads x (4x4) outputs
// =========================================================================
template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ X, int ldx,
                                                        const T* __restrict__ W, int M, int N, int K,
                                                        float* __restrict__ out, int ldo) {
  __shared__ float sx[16][64 + 4];
  __shared__ float sw[16][64 + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int e = threadIdx.x; e < 64 * 16; e += 256) {
      const int r = e / 16, c = e % 16;
      const int m = m0 + r, n = n0 + r, k = k0 + c;
      sx[c][r] = (m < M && k < K) ? to_f(X[(size_t)m * ldx + k]) : 0.f;
      sw[c][r] = (n < N && k < K) ? to_f(W[(size_t)n * K + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = sx[c][ty * 4 + i];
        b[i] = sw[c][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + jj;
      if (m < M && n < N) out[(size_t)m * ldo + n] = acc[i][jj];
    }
}

// =========================================================================
// Host side: tensor maps, planning, launch
// =========================================================================
static std::atomic<unsigned long long> g_wait_ns{tc::kWaitLimitNs};
void gemm_set_wait_limit(unsigned long long ns) { g_wait_ns.store(ns, std::memory_order_relaxed); }

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 map over a [rows, K] matrix (row stride ld elements); box = 64 x box_rows.
static bool make_map(CUtensorMap* map, const void* base, int rows, int K, int ld, int box_rows) {
  if (!get_encoder()) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tma_2d(CUtensorMap* map, const void* base, int rows, int cols, int ld, int box_rows) {
  return make_map(map, base, rows, cols, ld, box_rows);
}

static int swap_bn(int M) {
  int bn = 16;
  while (bn < M) bn *= 2;
  return bn;
}

struct Plan {
  bool swap;
  int bn;
  int cm;       // CTAs per cluster sharing a weight tile (1 or 2)
  int ma;       // 128-row blocks per work item (1 or 2)
  int splits;   // partial slabs per tile (the most any tile needs)
  int tiles;
  int ktiles;
  int streamk;
  int grid;
};

static int sub_boxes(int bn) { return bn == 16 ? 4 : (bn <= 64 ? 2 : 1); }
static int cluster_slots(int bn);

// A few hundred rows (128 < M <= 1024, a batched decode step): the plan with
// the least estimated time among 128-row items 128 or 256 wide (whole, or in
// up to four K slices when every slice of every tile runs in the first round,
// so the tile's CTAs share its sum) and, for M a multiple of 256, whole
// 256-row items 224 or 256 wide. An item's K step costs what was measured on
// GB300 for that shape with the whole GPU busy (the ring is latency-bound
// there: 0.33 / 0.47 us per 128-row step 128 / 256 wide, 0.81 / 0.88 us per
// 256-row step 224 / 256 wide); a sliced tile adds about 3 us for its sum.
// Gated (SwiGLU) tiles keep 128-row items.
static void plan_few_hundred_rows(Plan& p, int M, int N, int K, bool gated) {
  const int sms = num_sms();
  const int ktiles = (K + 63) / 64;
  struct Shape {
    int ma, bn, step_ns;
  };
  const Shape shapes[] = {{1, 128, 330}, {1, 256, 470}, {2, 224, 810}, {2, 256, 880}};
  long long best = -1;
  for (const Shape& sh : shapes) {
    if (sh.ma == 2 && (gated || M % 256 != 0)) continue;
    const int tiles = ((M + 128 * sh.ma - 1) / (128 * sh.ma)) * ((N + sh.bn - 1) / sh.bn);
    const int smax = sh.ma == 2 ? 1 : std::min(4, ktiles);
    for (int sp = 1; sp <= smax; ++sp) {
      if (sp > 1 && ((long long)tiles * sp > sms || tiles > kGemmSemCount)) break;
      const long long rounds = ((long long)tiles * sp + sms - 1) / sms;
      const long long cost = rounds * (long long)((ktiles + sp - 1) / sp) * sh.step_ns + (sp > 1 ? 3000 : 0);
      if (best < 0 || cost < best) {
        best = cost;
        p.ma = sh.ma;
        p.bn = sh.bn;
        p.splits = sp;
        p.tiles = tiles;
      }
    }
  }
  p.swap = false;
  p.cm = 1;
  p.streamk = 0;
  p.ktiles = ktiles;
  p.grid = (int)std::min<long long>((long long)p.tiles * p.splits, sms);
}

// Few activation rows (swap): stream-K over all (tile, k-tile) units, one
// persistent CTA per SM. Wide tiles: items (tile, K slice), choosing the
// slice count that best fills whole rounds of CTAs (fewer on ties).
static Plan plan_gemm(int M, int N, int K, bool gated = false) {
  Plan p;
  p.ma = 1;
  // up to 128 rows the weights stream through the 128-lane side; from 129
  // rows the wide plans below measured faster (205 rows x 4096 x 4096: 48 ->
  // 29 us; x 12288 K: 59 -> 45 us)
  p.swap = M <= 128;
  if (!p.swap && M <= 1024) {
    plan_few_hundred_rows(p, M, N, K, gated);
    return p;
  }
  p.bn = p.swap ? swap_bn(M) : 256;
  if (!p.swap && N <= 128 * 6) p.bn = 128;
  // too few 256-wide tiles to give every SM work: halve the tile width
  // before cutting K into slices, which need a cross-CTA sum -- unless K is
  // long: there 128-wide tiles re-read the operands from L2 twice as often
  // per flop and the contraction stalls on the L2 stream (the down
  // projection of a 512-row batched decode step, K = 14336: 85 us at 128
  // wide, about 18 us less at 256 wide in two K slices)
  if (!p.swap && p.bn == 256 && K < 8192 && 2LL * ((M + 127) / 128) * ((N + 255) / 256) < num_sms()) p.bn = 128;
  const int tilesA = p.swap ? (N + 127) / 128 : (M + 127) / 128;
  const int tilesB = p.swap ? (M + p.bn - 1) / p.bn : (N + p.bn - 1) / p.bn;
  p.tiles = tilesA * tilesB;
  // wide tiles in pairs of A tiles that share each weight tile (multicast):
  // measured to pay on long row counts (training) and to cost a little on
  // the 512-row batched decode contractions (gate/up +1.5 us, head +2.4 us)
  p.cm = (!p.swap && tilesA % 2 == 0 && tilesA >= 8) ? 2 : 1;
  const int kt_elems = 64 * (p.swap ? sub_boxes(p.bn) : 1);
  p.ktiles = (K + kt_elems - 1) / kt_elems;
  const int sms = num_sms();
  if (p.swap && p.tiles <= kGemmSemCount) {
    p.cm = 1;
    p.streamk = 1;
    const long long U = (long long)p.tiles * p.ktiles;
    p.grid = (int)std::min<long long>(U, sms);
    // the tiles stream-K cuts (all of them when there are fewer tiles than
    // CTAs; see Sched)
    Sched ref;
    ref.init(p.tiles, p.ktiles, 1, 1, p.grid, 0);
    const int skt = ref.skt;
    const long long Usk = ref.U;
    int most = 1;
    for (int t = 0; t < skt; ++t) {
      const int first = Sched::owner((long long)t * p.ktiles, Usk, p.grid);
      const int last = Sched::owner((long long)t * p.ktiles + p.ktiles - 1, Usk, p.grid);
      most = std::max(most, last - first + 1);
    }
    p.splits = most;
    return p;
  }
  p.streamk = 0;
  p.cm = p.cm > 1 && cluster_slots(p.bn) > 0 ? p.cm : 1;
  // items and CTA slots counted in clusters
  const int slots = p.cm > 1 ? cluster_slots(p.bn) : sms;
  const int tiles = p.tiles / p.cm;
  const int smax = (2 * tiles >= slots) ? 1 : std::max(1, std::min(4, p.ktiles / 2));
  double best = -1.0;
  p.splits = 1;
  for (int s = 1; s <= smax && (s == 1 || p.tiles <= kGemmSemCount); ++s) {
    const long long items = (long long)tiles * s;
    const long long rounds = (items + slots - 1) / slots;
    const double eff = (double)items / (double)(rounds * slots);
    if (eff > best + 0.02) {
      best = eff;
      p.splits = s;
    }
  }
  p.grid = (int)std::min<long long>((long long)tiles * p.splits, slots) * p.cm;
  return p;
}

int gemm_splits(int M, int N, int K) { return plan_gemm(M, N, K).splits; }

bool gemm_swiglu_keeps_gu(int dtype, int M, int N, int K) {
  if (dtype != PEAGLE_BF16 || M <= 0 || N % 256 != 0) return false;
  const Plan p = plan_gemm(M, N, K, true);
  return !p.swap && p.splits == 1;
}

bool gemm_qkv_fusable(int dtype, int M, int N, int K) {
  if (dtype != PEAGLE_BF16 || M <= 0 || N % 128 != 0) return false;
  const Plan p = plan_gemm(M, N, K);
  return !p.swap && p.splits == 1 && p.bn % 128 == 0;
}

size_t gemm_out_floats(int dtype, int M, int N, int K) {
  if (dtype != PEAGLE_BF16) return (size_t)M * N;
  // a gated (SwiGLU) contraction may plan other K slices than a plain one
  const int sp = std::max(plan_gemm(M, N, K).splits, plan_gemm(M, N, K, true).splits);
  return (size_t)sp * M * N;
}

template <int BN, bool SWAP, int CM, int MA = 1>
static cudaError_t set_smem_attr() {
  using C = TcCfg<BN, SWAP, MA>;
  static std::atomic<unsigned long long> attr_done{0};
  return once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(gemm_tc_kernel<BN, SWAP, CM, MA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SMEM);
  });
}

template <int BN, bool SWAP, int CM, int MA = 1>
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b, const TcArgs& args, int grid,
                             cudaStream_t s) {
  using C = TcCfg<BN, SWAP, MA>;
  cudaError_t e0 = set_smem_attr<BN, SWAP, CM, MA>();
  if (e0 != cudaSuccess) return e0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CM;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CM > 1 ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, SWAP, CM, MA>, a, b, args);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Clusters of two wide-tile CTAs that fit on the current device at once (one
// CTA per SM; a pair needs two SMs of one GPC), or 0 if none.
template <int BN>
static int cluster_slots_bn() {
  static std::atomic<int> slots[kMaxDevices];
  static std::atomic<unsigned long long> done{0};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 0;
  // the shared-memory limit first: set-up calls do not nest (one lock)
  if (set_smem_attr<BN, false, 2>() != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaError_t e = once_per_device(done, [dev] {
    int n = 0;
    {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(TC_THREADS);
      cfg.dynamicSmemBytes = TcCfg<BN, false>::SMEM;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, false, 2, 1>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();   // a refused query leaves no sticky error
    slots[dev].store(n);
    return cudaSuccess;
  });
  if (e != cudaSuccess) return 0;
  return slots[dev].load();
}

static int cluster_slots(int bn) { return bn == 128 ? cluster_slots_bn<128>() : cluster_slots_bn<256>(); }

int gemm_col_tiles(int M, int N, int K) {
  const Plan p = plan_gemm(M, N, K);
  return p.swap ? (N + 127) / 128 : (N + p.bn - 1) / p.bn;
}

cudaError_t gemm_launch(int dtype, const void* X, int ldx, const void* W, int M, int N, int K, float* out,
                        GemmOut* o, int* sem, int* dev_status, int probe_op, cudaStream_t s, bool w_early) {
  return gemm_launch_epi(dtype, X, ldx, W, M, N, K, out, o, sem, dev_status, probe_op, nullptr, s, w_early);
}

cudaError_t gemm_launch_epi(int dtype, const void* X, int ldx, const void* W, int M, int N, int K, float* out,
                            GemmOut* o, int* sem, int* dev_status, int probe_op, const GemmEpi* epi,
                            cudaStream_t s, bool w_early) {
  if (M <= 0 || N <= 0) {
    if (o) *o = GemmOut{out, N, 1, 0};
    return cudaSuccess;
  }
  if (dtype != PEAGLE_BF16) {
    if (o) *o = GemmOut{out, N, 1, 0};
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    probe_start(probe_op, s);
    gemm_simt_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(X), ldx,
                                                  static_cast<const float*>(W), M, N, K, out, N);
    note_launch();
    probe_stop(probe_op, s);
    return cudaGetLastError();
  }
  const bool gated = epi && epi->op == GEMM_EPI_SWIGLU;
  const Plan p = plan_gemm(M, N, K, gated);
  TcArgs args;
  args.K = K;
  args.splits = p.splits;
  args.streamk = p.streamk;
  // every split item in the first round (the tile's CTAs then share its sum)
  args.coop = (!p.swap && p.splits > 1 && (long long)(p.tiles / p.cm) * p.splits <= p.grid / p.cm) ? 1 : 0;
  args.out = out;
  args.ldo = N;
  args.split_stride = (size_t)M * N;
  args.M = M;
  args.N = N;
  args.sem = sem;
  args.status = dev_status;
  args.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  args.w_early = w_early ? 1 : 0;
  args.op = EPI_STORE;
  args.gate_off = 0;
  args.gu = nullptr;
  args.gu_ld = 0;
  if (epi && epi->op == GEMM_EPI_QKV) {
    if (p.swap || p.splits != 1 || N % 128 != 0 || p.bn % 128 != 0) {
      set_error("q/k/v epilogue needs wide unsplit tiles (M=%d N=%d K=%d)", M, N, K);
      return cudaErrorInvalidValue;
    }
    args.op = EPI_QKV;
    args.nq = epi->nq;
    args.nkv = epi->nkv;
    args.max_pos = epi->max_pos;
    args.row_base = epi->row_base;
    args.rcos = epi->rcos;
    args.rsin = epi->rsin;
    args.row_pos = epi->row_pos;
    args.q_out = epi->q;
    args.k_out = epi->k;
    args.v_out = epi->v;
  } else if (epi && epi->op == GEMM_EPI_SWIGLU) {
    if (N % 256 != 0) {
      set_error("fused SwiGLU needs the gate/up width %d to be a multiple of 256", N);
      return cudaErrorInvalidValue;
    }
    if (epi->gu && (p.swap || p.splits != 1)) {
      set_error("keeping the gate/up values needs wide unsplit tiles (M=%d N=%d K=%d)", M, N, K);
      return cudaErrorInvalidValue;
    }
    args.op = EPI_SWIGLU;
    args.gate_off = N / 2;
    args.act = epi->act;
    args.act_ld = epi->act_ld;
    args.gu = epi->gu;
    args.gu_ld = epi->gu_ld;
  } else if (epi) {
    args.op = epi->op;
    args.part_ld = p.swap ? (N + 127) / 128 : (N + p.bn - 1) / p.bn;
    args.logits = epi->logits;
    args.logits_ld = epi->logits_ld;
    args.p_max = epi->p_max;
    args.p_sum = epi->p_sum;
    args.p_lab = epi->p_lab;
    args.p_idx = epi->p_idx;
    args.labels = epi->labels;
  }
  CUtensorMap ma, mb;
  bool ok;
  // a gated weight tile is loaded as two half-height boxes
  const int wdiv = args.gate_off ? 2 : 1;
  if (p.swap) {
    args.rowsA = N;
    args.rowsB = M;
    ok = make_map(&ma, W, N, K, K, 128 / wdiv) && make_map(&mb, X, M, K, ldx, p.bn);
  } else {
    args.rowsA = M;
    args.rowsB = N;
    // a paired CTA loads half of each weight tile (one half-height box)
    ok = make_map(&ma, X, M, K, ldx, 128) && make_map(&mb, W, N, K, K, p.bn / (p.cm > 1 ? 2 : wdiv));
  }
  if (!ok) {
    set_error("cuTensorMapEncodeTiled failed (M=%d N=%d K=%d)", M, N, K);
    return cudaErrorInvalidValue;
  }
  // the kernel folds the K slices into slab 0
  if (o) *o = GemmOut{out, N, 1, 0};
  const int items = p.grid;
  cudaError_t e;
  probe_start(probe_op, s);
  if (p.swap) {
    switch (p.bn) {
      case 16: e = launch_tc<16, true, 1>(ma, mb, args, items, s); break;
      case 32: e = launch_tc<32, true, 1>(ma, mb, args, items, s); break;
      case 64: e = launch_tc<64, true, 1>(ma, mb, args, items, s); break;
      default: e = launch_tc<128, true, 1>(ma, mb, args, items, s); break;
    }
  } else if (p.ma == 2) {
    e = (p.bn == 224) ? launch_tc<224, false, 1, 2>(ma, mb, args, items, s)
                      : launch_tc<256, false, 1, 2>(ma, mb, args, items, s);
  } else if (p.cm == 2) {
    e = (p.bn == 128) ? launch_tc<128, false, 2>(ma, mb, args, items, s)
                      : launch_tc<256, false, 2>(ma, mb, args, items, s);
  } else {
    e = (p.bn == 128) ? launch_tc<128, false, 1>(ma, mb, args, items, s)
                      : launch_tc<256, false, 1>(ma, mb, args, items, s);
  }
  probe_stop(probe_op, s);
  return e;
}

}  // namespace pe

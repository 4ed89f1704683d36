// Shared internals of the P-EAGLE GB300 library: element types, reductions,
// the device status word, launch bookkeeping and the launchers each .cu file
// exports to the host API (api.cu).
#pragma once
#include <cuda.h>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/peagle.h"

namespace pe {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- elements
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Block-wide sum; every thread gets the result. `red` holds >= 33 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

// Argmax pair order: larger value wins, NaN above every number, then the
// lower index wins among equal values (and among NaNs).
__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) {
  const bool vn = v != v, bn = bv != bv;
  if (vn != bn) return vn;
  if (!vn && v != bv) return v > bv;
  return i < bi;
}

// ---------------------------------------------------------------- status
__device__ __forceinline__ void set_status(int* st, int bits) {
  if (st) atomicOr(st, bits);
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: every kernel of the library is launched
// with programmatic stream serialization, lets its dependents launch as soon
// as it starts (pdl_trigger), and waits for its predecessor to complete and
// flush (pdl_wait) before it reads or writes anything the predecessor
// touches. Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- host side
// Launch with programmatic stream serialization: the kernel may start while
// its predecessor finishes, and waits (pdl_wait) before touching its data.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

void note_launch();                       // counts one kernel launch
void set_error(const char* fmt, ...);     // records peagle_last_error()
void probe_start(int op, cudaStream_t s); // timing probe around main kernels
void probe_stop(int op, cudaStream_t s);
int num_sms();                            // SMs of the current device

// Devices the per-device set-up below tracks (device ordinals 0..63).
constexpr int kMaxDevices = 64;
int current_device();                     // cudaGetDevice, or -1 on failure
std::mutex& setup_mutex();
// Device address of the current device's status word for calls that take
// no model handle (PEAGLE_DEV_* bits, sticky).
cudaError_t library_status_word(int** out);

// Runs fn() on the current device once: `done` holds one bit per device,
// set after fn() succeeded there. Launch attributes such as the dynamic
// shared-memory limit apply to the device current when they are set, so
// every device a kernel runs on needs its own set-up. Safe across threads;
// fn() must not call once_per_device itself (the set-up lock is not
// recursive).
template <typename F>
inline cudaError_t once_per_device(std::atomic<unsigned long long>& done, F&& fn) {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  std::lock_guard<std::mutex> lk(setup_mutex());
  if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
  const cudaError_t e = fn();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// ---------------------------------------------------------------- GEMM
// Partial-sum output of a contraction D = X W^T: `splits` slabs of
// [M][ldo] floats, `split_stride` floats apart; the consumer sums them.
struct GemmOut {
  float* out;
  int ldo;
  int splits;
  size_t split_stride;
};
// Choose the split count for an M x N x K contraction (bf16 tensor-core path).
int gemm_splits(int M, int N, int K);
// Workspace floats the partial output of gemm_launch needs.
size_t gemm_out_floats(int dtype, int M, int N, int K);
// Per-tile arrival counters a contraction needs when it splits K (ints).
// They must be zero before the first launch that uses them; every launch
// leaves them zero again.
constexpr int kGemmSemCount = 4096;
// Runs D = X W^T into out (planning the split itself; fills *o). The K
// slices are summed inside the kernel, so *o always describes one slab.
// X [M, K] with row stride ldx elements, W [N, K] contiguous. With w_early
// the first tiles of W load before the kernel waits for its predecessor
// (programmatic dependent launch): only for W that no kernel of the chain
// writes, such as model weights; pass false when W was just produced.
cudaError_t gemm_launch(int dtype, const void* X, int ldx, const void* W, int M, int N, int K,
                        float* out, GemmOut* o, int* sem, int* dev_status, int probe_op, cudaStream_t s,
                        bool w_early = true);

// Fused head epilogue of a bf16 contraction: instead of (or besides) the
// fp32 result, per (row, column tile) partials of the row's argmax (value,
// lowest index) and, for cross-entropy, the max, the sum of exp(x - max) and
// the label's logit (-inf when the label is in another tile).
// GEMM_EPI_SWIGLU: W is a [2I, K] gate/up weight (gate rows first); the
// result silu(gate) * up [M, I] is written as bf16 to act (row stride
// act_ld). Needs 2I % 256 == 0. With gu set (wide unsplit tiles only, see
// gemm_swiglu_keeps_gu), the fp32 gate and up values are written too, at
// their own columns of gu [M, gu_ld] (gate j at j, up j at I + j).
// GEMM_EPI_QKV: D's columns are [q heads | k heads | v heads], head dim
// 128; q and k are rotated by the position of their row (pairs j, j + 64,
// cos/sin tables [max_pos][64]) and q, k, v are written as bf16 to
// q [rows, nq*128] and k, v [rows, nkv*128] at row row_base + GEMM row.
// Only where gemm_qkv_fusable() holds (one partial slab, wide tiles).
enum { GEMM_EPI_ARGMAX = 1, GEMM_EPI_CE = 2, GEMM_EPI_SWIGLU = 3, GEMM_EPI_QKV = 4 };
struct GemmEpi {
  int op;
  void* act;
  int act_ld;
  float* gu;            // GEMM_EPI_SWIGLU: optional fp32 gate / up values
  int gu_ld;
  float* logits;        // optional fp32 copy of D [M, logits_ld]
  int logits_ld;
  float *p_max, *p_sum, *p_lab;   // [M, gemm_col_tiles]
  int* p_idx;
  const int* labels;    // GEMM_EPI_CE: label per row, -1 = none
  // GEMM_EPI_QKV
  int nq, nkv, max_pos, row_base;
  const float *rcos, *rsin;
  const int* row_pos;
  void *q, *k, *v;
};
// Whether D = X W^T [M, N] (bf16) can take the q/k/v epilogue: unswapped
// tiles, one partial slab, whole 128-column heads.
bool gemm_qkv_fusable(int dtype, int M, int N, int K);
// Whether the gated contraction (N = 2I) can also keep its fp32 gate / up
// values in the SwiGLU epilogue: unswapped tiles, one partial slab.
bool gemm_swiglu_keeps_gu(int dtype, int M, int N, int K);
// 2-D bf16 tensor map over a [rows, cols] matrix (row stride ld elements),
// box = 64 columns x box_rows rows, 128-byte swizzle. False if the driver
// rejects it.
bool make_tma_2d(CUtensorMap* map, const void* base, int rows, int cols, int ld, int box_rows);
// Bound of every in-kernel wait of the tensor-core contractions launched
// from now on (default 1 s; 0 = a single try). A test hook.
void gemm_set_wait_limit(unsigned long long ns);
// Column tiles (partials per row) of the fused head epilogue.
int gemm_col_tiles(int M, int N, int K);
cudaError_t gemm_launch_epi(int dtype, const void* X, int ldx, const void* W, int M, int N, int K,
                            float* out, GemmOut* o, int* sem, int* dev_status, int probe_op,
                            const GemmEpi* epi, cudaStream_t s, bool w_early = true);

}  // namespace pe

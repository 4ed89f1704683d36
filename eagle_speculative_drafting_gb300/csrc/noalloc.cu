// peagle_gemm_noalloc: the library's dense contraction for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc, or have no spare device memory to
// hand this library:
//   - serving engines whose allocator reserved the whole device heap up
//     front;
//   - plugins that their host framework forbids to allocate;
//   - latency-critical loops where cudaMalloc's implicit device
//     synchronisation is not acceptable.
// For them, this variant keeps the split-K partial slabs and per-tile
// counters of the tcgen05 GEMM in one file-scope device array of fixed size.
// Every GPU that loads the library holds that array until the process exits.
//
// The array's name is a host-side stand-in in host code, not a device
// address. The device address is fetched with cudaGetSymbolAddress once per
// device, with that device current, on the first call made on that device;
// make that first call before any stream capture. The caller still passes
// the inputs and the output.
//
// The cached address does not survive a device reset (cudaDeviceReset):
// after one, restart the process before calling this entry point again.
//
// A bounded wait that runs out inside the contraction sets PEAGLE_DEV_TIMEOUT
// in the library status word (peagle_get_library_status), which also needs
// no allocation: it is a device variable of the library.
//
// All calls share the array, and it keeps the last call's contents. The
// per-tile counters must start at zero, so every call clears them first.
// The slabs need no clearing: every element a call reads was written by the
// same call. Calls that overlap on the GPU race on the array; serialise them,
// for example on one stream.
#include <mutex>

#include "rows.cuh"

namespace {

constexpr size_t kSlabFloats = (size_t)2 << 20;    // 8 MiB of partial sums
constexpr size_t kSlabBytes = kSlabFloats * sizeof(float);
constexpr size_t kScratchBytes = kSlabBytes + pe::kGemmSemCount * sizeof(int);
using pe::kMaxDevices;

static __device__ __align__(256) unsigned char g_gemm_scratch[kScratchBytes];

std::mutex g_mu;
void* g_dev_scratch[kMaxDevices] = {};

// Device address of g_gemm_scratch on the current device (set up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev_scratch[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gemm_scratch);
    if (e != cudaSuccess) return e;
    g_dev_scratch[dev] = p;
  }
  *out = g_dev_scratch[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" peagle_status peagle_gemm_noalloc(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* X,
                                             const void* W, float* D, void* stream) {
  using namespace pe;
  if (M < 0 || N < 0 || K < 1 || (dtype != PEAGLE_F32 && dtype != PEAGLE_BF16)) {
    set_error("gemm_noalloc: M=%d N=%d K=%d dtype=%d", M, N, K, dtype);
    return PEAGLE_ERR_INVALID_ARG;
  }
  if (M == 0 || N == 0) return PEAGLE_OK;
  if (!X || !W || !D) {
    set_error("gemm_noalloc: NULL operand");
    return PEAGLE_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == PEAGLE_F32) {  // the CUDA-core kernel writes D directly and needs no scratch
    cudaError_t e = gemm_launch(dtype, X, K, W, M, N, K, D, nullptr, nullptr, nullptr, -1, s);
    if (e != cudaSuccess) {
      set_error("gemm_noalloc: %s", cudaGetErrorString(e));
      return PEAGLE_ERR_CUDA;
    }
    return PEAGLE_OK;
  }
  if (K % 8 || (reinterpret_cast<uintptr_t>(X) & 15) || (reinterpret_cast<uintptr_t>(W) & 15)) {
    set_error("gemm_noalloc: bf16 needs K %% 8 == 0 and 16-byte aligned operands");
    return PEAGLE_ERR_INVALID_ARG;
  }
  const size_t need = gemm_out_floats(dtype, M, N, K);
  if (need > kSlabFloats) {
    set_error("gemm_noalloc: M=%d N=%d K=%d needs %zu partial floats, more than the fixed %zu "
              "(use peagle_gemm with a caller workspace)", M, N, K, need, kSlabFloats);
    return PEAGLE_ERR_UNSUPPORTED;
  }
  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) {
    set_error("gemm_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    return PEAGLE_ERR_CUDA;
  }
  float* slabs = static_cast<float*>(base);
  int* sem = reinterpret_cast<int*>(static_cast<char*>(base) + kSlabBytes);
  int* lib_status = nullptr;
  if ((e = library_status_word(&lib_status)) != cudaSuccess) {
    set_error("gemm_noalloc: cudaGetSymbolAddress (status word): %s", cudaGetErrorString(e));
    return PEAGLE_ERR_CUDA;
  }
  GemmOut go;
  if ((e = cudaMemsetAsync(sem, 0, kGemmSemCount * sizeof(int), s)) != cudaSuccess ||
      (e = gemm_launch(dtype, X, K, W, M, N, K, slabs, &go, sem, lib_status, -1, s)) != cudaSuccess ||
      (e = launch_sum_splits(go, M, N, D, s)) != cudaSuccess) {
    set_error("gemm_noalloc: %s", cudaGetErrorString(e));
    return PEAGLE_ERR_CUDA;
  }
  return PEAGLE_OK;
}

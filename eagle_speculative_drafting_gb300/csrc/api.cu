// C ABI of the P-EAGLE library: argument validation, the model handle,
// workspace layout and the launch sequence of each entry point.
// The arithmetic lives in gemm.cu, rows.cu and attn.cu.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "rows.cuh"

using namespace pe;

// ===================================================================== state
static thread_local std::string g_err;
static std::atomic<unsigned long long> g_launches{0};

namespace pe {
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
}
int current_device() {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}
std::mutex& setup_mutex() {
  static std::mutex mu;
  return mu;
}
// SM count of the current device, looked up once per device
int num_sms() {
  static std::atomic<int> sms[kMaxDevices];
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 148;
  int v = sms[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    sms[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// ---- status word of the calls that take no model handle (peagle_gemm,
// peagle_gemm_noalloc): a device variable, so it exists on every device that
// loads the library without any allocation. Its device address is looked up
// once per device (cudaGetSymbolAddress with that device current) and
// cached; a cached address does not survive a device reset.
static __device__ int g_lib_status;
static void* g_lib_status_addr[kMaxDevices];

cudaError_t library_status_word(int** out) {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(setup_mutex());
  if (!g_lib_status_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_lib_status);
    if (e != cudaSuccess) return e;
    g_lib_status_addr[dev] = p;
  }
  *out = static_cast<int*>(g_lib_status_addr[dev]);
  return cudaSuccess;
}

// ---- timing probe: event pairs around the main kernel of one op class
static std::mutex g_probe_mu;
static int g_probe_op = -1, g_probe_cap = 0, g_probe_n = 0;
static bool g_probe_armed = false;
static std::vector<cudaEvent_t> g_ev0, g_ev1;

void probe_start(int op, cudaStream_t s) {
  if (op < 0 || op != g_probe_op || g_probe_n >= g_probe_cap) return;
  cudaEventRecord(g_ev0[g_probe_n], s);
  g_probe_armed = true;
}
void probe_stop(int op, cudaStream_t s) {
  if (!g_probe_armed || op != g_probe_op) return;
  cudaEventRecord(g_ev1[g_probe_n], s);
  ++g_probe_n;
  g_probe_armed = false;
}
}  // namespace pe

struct peagle_model {
  peagle_config cfg;
  peagle_weights w;
  std::vector<peagle_layer_weights> layers;
  float* rcos = nullptr;
  float* rsin = nullptr;
  float* mask_qkv0 = nullptr;   // [QKV] pre-rotary q/k/v of a masked layer-0 row
  float* mask_resid0 = nullptr; // [H] its layer-0 residual
  int* status = nullptr;
  int* sem = nullptr;           // [kGemmSemCount] draft-step arrival counters, zero between launches
};

#define FAIL(code, ...)      \
  do {                       \
    set_error(__VA_ARGS__);  \
    return code;             \
  } while (0)

#define CUDA_TRY(expr)                                                                 \
  do {                                                                                 \
    cudaError_t e_ = (expr);                                                           \
    if (e_ != cudaSuccess) FAIL(PEAGLE_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Bump allocator over the caller's workspace; a dry run (base == NULL)
// measures the size.
struct Bump {
  char* base;
  size_t off = 0;
  explicit Bump(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T) + 16;
    return p;
  }
  void* take_bytes(size_t bytes) { return take<char>(bytes); }
};

static size_t esize(const peagle_config& c) { return c.dtype == PEAGLE_BF16 ? 2 : 4; }
static int qkv_out(const peagle_config& c) { return (c.num_q_heads + 2 * c.num_kv_heads) * c.head_dim; }

// ================================================================== library
extern "C" {

const char* peagle_version(void) { return "peagle-gb300 0.1 (sm_103a)"; }

const char* peagle_status_string(peagle_status s) {
  switch (s) {
    case PEAGLE_OK: return "ok";
    case PEAGLE_ERR_INVALID_ARG: return "invalid argument";
    case PEAGLE_ERR_UNSUPPORTED: return "unsupported";
    case PEAGLE_ERR_CUDA: return "CUDA error";
    case PEAGLE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case PEAGLE_ERR_DEVICE: return "device status set";
  }
  return "unknown status";
}

const char* peagle_last_error(void) { return g_err.c_str(); }

uint64_t peagle_kernel_launches(void) { return g_launches.load(); }

const char* peagle_op_name(int32_t op) {
  static const char* names[] = {"fc", "qkv", "attn", "o_proj", "gate_up", "down", "lm_head",
                                "verify", "cod", "ce", "bwd_gemm"};
  return (op >= 0 && op < PEAGLE_OP_COUNT) ? names[op] : "unknown";
}

peagle_status peagle_probe_begin(int32_t op, int32_t capacity) {
  if (op < 0 || op >= PEAGLE_OP_COUNT || capacity <= 0 || capacity > (1 << 20))
    FAIL(PEAGLE_ERR_INVALID_ARG, "probe_begin: bad op %d or capacity %d", op, capacity);
  std::lock_guard<std::mutex> lk(g_probe_mu);
  for (auto e : g_ev0) cudaEventDestroy(e);
  for (auto e : g_ev1) cudaEventDestroy(e);
  g_ev0.assign(capacity, nullptr);
  g_ev1.assign(capacity, nullptr);
  for (int i = 0; i < capacity; ++i) {
    CUDA_TRY(cudaEventCreate(&g_ev0[i]));
    CUDA_TRY(cudaEventCreate(&g_ev1[i]));
  }
  g_probe_cap = capacity;
  g_probe_n = 0;
  g_probe_armed = false;
  g_probe_op = op;
  return PEAGLE_OK;
}

peagle_status peagle_probe_end(float* ms_out, int32_t capacity, int32_t* count) {
  std::lock_guard<std::mutex> lk(g_probe_mu);
  if (!count) FAIL(PEAGLE_ERR_INVALID_ARG, "probe_end: count is NULL");
  const int n = g_probe_n;
  for (int i = 0; i < n; ++i) {
    CUDA_TRY(cudaEventSynchronize(g_ev1[i]));
    float ms = 0.f;
    CUDA_TRY(cudaEventElapsedTime(&ms, g_ev0[i], g_ev1[i]));
    if (ms_out && i < capacity) ms_out[i] = ms;
  }
  *count = n;
  for (auto e : g_ev0) cudaEventDestroy(e);
  for (auto e : g_ev1) cudaEventDestroy(e);
  g_ev0.clear();
  g_ev1.clear();
  g_probe_op = -1;
  g_probe_cap = 0;
  g_probe_n = 0;
  return PEAGLE_OK;
}

// ==================================================================== model
static peagle_status validate_config(const peagle_config* c) {
  if (!c) FAIL(PEAGLE_ERR_INVALID_ARG, "config is NULL");
  if (c->dtype != PEAGLE_F32 && c->dtype != PEAGLE_BF16) FAIL(PEAGLE_ERR_INVALID_ARG, "dtype %d", c->dtype);
  if (c->hidden <= 0 || c->target_hidden <= 0 || c->num_aux <= 0 || c->num_layers <= 0 ||
      c->num_q_heads <= 0 || c->num_kv_heads <= 0 || c->intermediate <= 0 || c->target_vocab <= 0 ||
      c->draft_vocab <= 0 || c->max_position <= 0)
    FAIL(PEAGLE_ERR_INVALID_ARG, "config sizes must be positive");
  if (c->num_q_heads % c->num_kv_heads) FAIL(PEAGLE_ERR_INVALID_ARG, "num_q_heads %% num_kv_heads != 0");
  if (c->head_dim != 64 && c->head_dim != 128) FAIL(PEAGLE_ERR_UNSUPPORTED, "head_dim %d not in {64,128}", c->head_dim);
  if (c->ptd_token_id < 0 || c->ptd_token_id >= c->target_vocab)
    FAIL(PEAGLE_ERR_INVALID_ARG, "ptd_token_id %d outside [0, %d)", c->ptd_token_id, c->target_vocab);
  if (!(c->rms_eps > 0) || !(c->rope_theta > 0)) FAIL(PEAGLE_ERR_INVALID_ARG, "rms_eps and rope_theta must be > 0");
  if (c->norm_before_residual != 0 && c->norm_before_residual != 1)
    FAIL(PEAGLE_ERR_INVALID_ARG, "norm_before_residual must be 0 or 1");
  if (c->hidden > 12288) FAIL(PEAGLE_ERR_UNSUPPORTED, "hidden %d > 12288", c->hidden);
  if (c->num_layers > 64) FAIL(PEAGLE_ERR_UNSUPPORTED, "num_layers %d > 64", c->num_layers);
  if ((long long)c->max_position * c->head_dim > (1LL << 31)) FAIL(PEAGLE_ERR_UNSUPPORTED, "max_position too large");
  if (c->dtype == PEAGLE_BF16) {
    const long long ks[] = {(long long)c->num_aux * c->target_hidden, 2LL * c->hidden, c->hidden,
                            (long long)c->num_q_heads * c->head_dim, c->intermediate};
    for (long long k : ks)
      if (k % 8) FAIL(PEAGLE_ERR_UNSUPPORTED, "bf16 contraction width %lld not a multiple of 8", k);
  }
  return PEAGLE_OK;
}

peagle_status peagle_model_create(const peagle_config* cfg, const peagle_weights* w, void* stream,
                                  peagle_model** out) {
  if (!out) FAIL(PEAGLE_ERR_INVALID_ARG, "out is NULL");
  peagle_status st = validate_config(cfg);
  if (st) return st;
  if (!w || !w->embed || !w->fc_w || !w->fc_norm_w || !w->mask_hidden || !w->final_norm_w || !w->lm_head_w ||
      !w->layers)
    FAIL(PEAGLE_ERR_INVALID_ARG, "a required weight pointer is NULL");
  for (int l = 0; l < cfg->num_layers; ++l) {
    const peagle_layer_weights& L = w->layers[l];
    if (!L.in_norm_w || !L.qkv_w || !L.o_w || !L.post_norm_w || !L.gate_up_w || !L.down_w ||
        (l == 0 && !L.hidden_norm_w))
      FAIL(PEAGLE_ERR_INVALID_ARG, "layer %d: a required weight pointer is NULL", l);
    if (cfg->dtype == PEAGLE_BF16 &&
        !(aligned16(L.qkv_w) && aligned16(L.o_w) && aligned16(L.gate_up_w) && aligned16(L.down_w)))
      FAIL(PEAGLE_ERR_INVALID_ARG, "layer %d: bf16 weights must be 16-byte aligned", l);
  }
  if (cfg->dtype == PEAGLE_BF16 && !(aligned16(w->fc_w) && aligned16(w->lm_head_w) && aligned16(w->mask_hidden)))
    FAIL(PEAGLE_ERR_INVALID_ARG, "bf16 weights must be 16-byte aligned");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  peagle_model* m = new peagle_model();
  m->cfg = *cfg;
  m->w = *w;
  m->layers.assign(w->layers, w->layers + cfg->num_layers);
  m->w.layers = m->layers.data();
  const peagle_config& c = m->cfg;
  const int H = c.hidden, QKV = qkv_out(c), AHt = c.num_aux * c.target_hidden;
  const size_t half = c.head_dim / 2;
  void* tmp = nullptr;
  auto cleanup = [&](peagle_status code) {
    if (tmp) cudaFree(tmp);
    if (code != PEAGLE_OK) {
      cudaFree(m->rcos);
      cudaFree(m->rsin);
      cudaFree(m->mask_qkv0);
      cudaFree(m->mask_resid0);
      cudaFree(m->status);
      cudaFree(m->sem);
      delete m;
    }
    return code;
  };
#define CREATE_TRY(expr)                                                                    \
  do {                                                                                      \
    cudaError_t e_ = (expr);                                                                \
    if (e_ != cudaSuccess) {                                                                \
      set_error("model_create: %s: %s", #expr, cudaGetErrorString(e_));                     \
      return cleanup(PEAGLE_ERR_CUDA);                                                      \
    }                                                                                       \
  } while (0)
  CREATE_TRY(cudaMalloc(&m->rcos, (size_t)c.max_position * half * sizeof(float)));
  CREATE_TRY(cudaMalloc(&m->rsin, (size_t)c.max_position * half * sizeof(float)));
  CREATE_TRY(cudaMalloc(&m->mask_qkv0, (size_t)QKV * sizeof(float)));
  CREATE_TRY(cudaMalloc(&m->mask_resid0, (size_t)H * sizeof(float)));
  CREATE_TRY(cudaMalloc(&m->status, sizeof(int)));
  CREATE_TRY(cudaMemsetAsync(m->status, 0, sizeof(int), s));
  CREATE_TRY(cudaMalloc(&m->sem, kGemmSemCount * sizeof(int)));
  CREATE_TRY(cudaMemsetAsync(m->sem, 0, kGemmSemCount * sizeof(int), s));
  CREATE_TRY(launch_rope_table(m->rcos, m->rsin, c.max_position, c.head_dim, c.rope_theta, s));

  // masked-row constants: fc_norm(fc(mask_hidden)), the ptd embedding, and
  // the layer-0 pre-rotary q/k/v + residual every masked row shares
  const size_t part_f = std::max(gemm_out_floats(c.dtype, 1, H, AHt), gemm_out_floats(c.dtype, 1, QKV, 2 * H));
  const size_t x0_bytes = ((2 * (size_t)H * esize(c)) + 255) & ~size_t(255);
  const size_t part_bytes = ((part_f * sizeof(float)) + 255) & ~size_t(255);
  CREATE_TRY(cudaMalloc(&tmp, x0_bytes + part_bytes + kGemmSemCount * sizeof(int)));
  void* x0m = tmp;
  float* part = reinterpret_cast<float*>(static_cast<char*>(tmp) + x0_bytes);
  int* sem = reinterpret_cast<int*>(static_cast<char*>(tmp) + x0_bytes + part_bytes);
  CREATE_TRY(cudaMemsetAsync(sem, 0, kGemmSemCount * sizeof(int), s));
  GemmOut go;
  CREATE_TRY(gemm_launch(c.dtype, w->mask_hidden, AHt, w->fc_w, 1, H, AHt, part, &go, sem, m->status, -1, s));
  FcFinishArgs fa{};
  fa.u = go;
  fa.H = H;
  fa.Vt = c.target_vocab;
  fa.tok = nullptr;
  fa.tok_const = c.ptd_token_id;
  fa.embed = w->embed;
  fa.g_fc = w->fc_norm_w;
  fa.g_in = m->layers[0].in_norm_w;
  fa.g_h = m->layers[0].hidden_norm_w;
  fa.eps = (float)c.rms_eps;
  fa.nbr = c.norm_before_residual;
  fa.x0 = x0m;
  fa.resid = m->mask_resid0;
  fa.status = m->status;
  CREATE_TRY(launch_fc_finish(c.dtype, 1, fa, s));
  CREATE_TRY(gemm_launch(c.dtype, x0m, 2 * H, m->layers[0].qkv_w, 1, QKV, 2 * H, part, &go, sem, m->status, -1, s));
  CREATE_TRY(launch_sum_splits(go, 1, QKV, m->mask_qkv0, s));
  CREATE_TRY(cudaStreamSynchronize(s));
  int hs = 0;
  CREATE_TRY(cudaMemcpy(&hs, m->status, sizeof(int), cudaMemcpyDeviceToHost));
  if (hs) {
    set_error("model_create: device status 0x%x while precomputing masked-row constants", hs);
    return cleanup(PEAGLE_ERR_DEVICE);
  }
  cleanup(PEAGLE_OK);
  *out = m;
#undef CREATE_TRY
  return PEAGLE_OK;
}

peagle_status peagle_model_destroy(peagle_model* m) {
  if (!m) return PEAGLE_OK;
  cudaDeviceSynchronize();
  cudaFree(m->rcos);
  cudaFree(m->rsin);
  cudaFree(m->mask_qkv0);
  cudaFree(m->mask_resid0);
  cudaFree(m->status);
  cudaFree(m->sem);
  delete m;
  return PEAGLE_OK;
}

peagle_status peagle_get_device_status(const peagle_model* m, void* stream, int32_t* host_status) {
  if (!m || !host_status) FAIL(PEAGLE_ERR_INVALID_ARG, "get_device_status: NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaStreamSynchronize(s));
  int v = 0;
  CUDA_TRY(cudaMemcpy(&v, m->status, sizeof(int), cudaMemcpyDeviceToHost));
  *host_status = v;
  return PEAGLE_OK;
}

peagle_status peagle_clear_device_status(const peagle_model* m, void* stream) {
  if (!m) FAIL(PEAGLE_ERR_INVALID_ARG, "clear_device_status: NULL model");
  CUDA_TRY(cudaMemsetAsync(m->status, 0, sizeof(int), static_cast<cudaStream_t>(stream)));
  CUDA_TRY(cudaMemsetAsync(m->sem, 0, kGemmSemCount * sizeof(int), static_cast<cudaStream_t>(stream)));
  return PEAGLE_OK;
}

// gate/up projection and SwiGLU over rows of width K: bf16 with 2I % 256 == 0
// writes silu(gate) * up straight from the GEMM epilogue; otherwise the fp32
// result goes through the SwiGLU row kernel.
static cudaError_t gate_up_swiglu(int dt, const void* X, int K, const void* W, int rows, int I, float* part,
                                  void* act, int* sem, int* status, cudaStream_t s) {
  GemmOut go;
  if (dt == PEAGLE_BF16 && (2 * I) % 256 == 0) {
    GemmEpi ep{};
    ep.op = GEMM_EPI_SWIGLU;
    ep.act = act;
    ep.act_ld = I;
    return gemm_launch_epi(dt, X, K, W, rows, 2 * I, K, part, &go, sem, status, PEAGLE_OP_GATE_UP, &ep, s);
  }
  cudaError_t e = gemm_launch(dt, X, K, W, rows, 2 * I, K, part, &go, sem, status, PEAGLE_OP_GATE_UP, s);
  if (e != cudaSuccess) return e;
  return launch_swiglu(dt, go, rows, I, act, s);
}

// =============================================================== draft step
struct DraftWs {
  void *x0, *xin, *act, *q, *kc, *vc, *ao;
  float *h, *resid0, *part, *attn_o, *attn_ml, *am_val;
  int* am_idx;
  int chunk, nsplit;
};

// Workspace of a step with N new rows in all (at most max_new per request);
// rows = N + B*(K-1). The one-anchor step is N = B, max_new = 1.
static void draft_layout(const peagle_config& c, int B, int K, int N, int max_new, int max_kv_len, Bump& bp,
                         DraftWs& ws) {
  const size_t es = esize(c);
  const int H = c.hidden, I = c.intermediate, QKV = qkv_out(c), rows = N + B * (K - 1), heads = B * K;
  const int nq = c.num_q_heads, nkv = c.num_kv_heads, hd = c.head_dim, AHt = c.num_aux * c.target_hidden;
  ws.x0 = bp.take_bytes((size_t)N * 2 * H * es);
  ws.xin = bp.take_bytes((size_t)rows * H * es);
  ws.act = bp.take_bytes((size_t)rows * I * es);
  ws.q = bp.take_bytes((size_t)rows * nq * hd * es);
  ws.kc = bp.take_bytes((size_t)rows * nkv * hd * es);
  ws.vc = bp.take_bytes((size_t)rows * nkv * hd * es);
  ws.ao = bp.take_bytes((size_t)rows * nq * hd * es);
  ws.h = bp.take<float>((size_t)rows * H);
  ws.resid0 = bp.take<float>((size_t)N * H);
  size_t pf = gemm_out_floats(c.dtype, N, H, AHt);
  pf = std::max(pf, gemm_out_floats(c.dtype, N, QKV, 2 * H));
  pf = std::max(pf, gemm_out_floats(c.dtype, rows, QKV, H));
  pf = std::max(pf, gemm_out_floats(c.dtype, rows, H, nq * hd));
  pf = std::max(pf, gemm_out_floats(c.dtype, rows, 2 * I, H));
  pf = std::max(pf, gemm_out_floats(c.dtype, rows, H, I));
  pf = std::max(pf, gemm_out_floats(c.dtype, heads, c.draft_vocab, H));
  ws.part = bp.take<float>(pf);
  decode_attn_plan(B, nkv, max_kv_len, &ws.chunk, &ws.nsplit);
  const size_t prow = (size_t)B * nkv * ws.nsplit * (max_new + K - 1) * (nq / nkv);
  ws.attn_o = bp.take<float>(prow * hd);
  ws.attn_ml = bp.take<float>(prow * 2);
  const size_t nch = std::max<size_t>(lm_argmax_chunks(c.draft_vocab), (c.draft_vocab + 127) / 128);
  ws.am_val = bp.take<float>((size_t)heads * nch);
  ws.am_idx = bp.take<int>((size_t)heads * nch);
}

peagle_status peagle_draft_step_workspace_size(const peagle_model* m, int32_t B, int32_t K, int32_t max_kv_len,
                                               size_t* bytes) {
  if (!m || !bytes) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_workspace_size: NULL argument");
  if (B < 0 || K < 1 || K > 16 || max_kv_len < 0)
    FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_workspace_size: B=%d K=%d max_kv_len=%d", B, K, max_kv_len);
  Bump bp(nullptr);
  DraftWs ws;
  draft_layout(m->cfg, B, K, B, 1, max_kv_len, bp, ws);
  *bytes = bp.off;
  return PEAGLE_OK;
}

peagle_status peagle_draft_step_ctx_workspace_size(const peagle_model* m, int32_t B, int32_t K, int32_t total_new,
                                                   int32_t max_new, int32_t max_kv_len, size_t* bytes) {
  if (!m || !bytes) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_ctx_workspace_size: NULL argument");
  if (B < 0 || K < 1 || K > 16 || max_kv_len < 0 || max_new < 1 || max_new > 64 || total_new < B ||
      (long long)total_new > (long long)B * max_new)
    FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_ctx_workspace_size: B=%d K=%d total_new=%d max_new=%d max_kv_len=%d", B,
         K, total_new, max_new, max_kv_len);
  Bump bp(nullptr);
  DraftWs ws;
  draft_layout(m->cfg, B, K, total_new, max_new, max_kv_len, bp, ws);
  *bytes = bp.off;
  return PEAGLE_OK;
}

// One draft step over the rows `dr` describes: new rows (aux, tok, pos per
// new row; the last new row of a request is its anchor) and K-1 masked rows
// per request.
static peagle_status draft_step_impl(const peagle_model* m, const DecodeRows& dr, const void* aux, const int32_t* tok,
                                     const int32_t* pos, void* const* k_cache, void* const* v_cache,
                                     const int64_t* kv_offsets, const int32_t* kv_lens, int64_t kv_capacity,
                                     int32_t max_kv_len, int32_t append_kv, int32_t* draft_tokens, float* logits,
                                     void* workspace, cudaStream_t s) {
  const peagle_config& c = m->cfg;
  const int B = dr.B, K = dr.K, N = dr.total_new;
  Bump bp(workspace);
  DraftWs ws;
  draft_layout(c, B, K, N, dr.max_new, max_kv_len, bp, ws);
  const int H = c.hidden, I = c.intermediate, QKV = qkv_out(c), rows = N + B * (K - 1), L = c.num_layers;
  const int heads = B * K;
  const int nq = c.num_q_heads, nkv = c.num_kv_heads, hd = c.head_dim, AHt = c.num_aux * c.target_hidden;
  const int dt = c.dtype;
  const float eps = (float)c.rms_eps;
  GemmOut go;

  // fc + fc_norm over the new rows' aux states, then their layer-0 inputs
  FcFinishArgs fa{};
  fa.H = H;
  fa.Vt = c.target_vocab;
  fa.tok = tok;
  fa.embed = m->w.embed;
  fa.g_fc = m->w.fc_norm_w;
  fa.g_in = m->layers[0].in_norm_w;
  fa.g_h = m->layers[0].hidden_norm_w;
  fa.eps = eps;
  fa.nbr = c.norm_before_residual;
  fa.x0 = ws.x0;
  fa.resid = ws.resid0;
  fa.status = m->status;
  CUDA_TRY(gemm_launch(dt, aux, AHt, m->w.fc_w, N, H, AHt, ws.part, &go, m->sem, m->status, PEAGLE_OP_FC, s));
  fa.u = go;
  CUDA_TRY(launch_fc_finish(dt, N, fa, s));

  for (int l = 0; l < L; ++l) {
    const peagle_layer_weights& W = m->layers[l];
    QkvArgs qa{};
    if (l == 0) {
      CUDA_TRY(gemm_launch(dt, ws.x0, 2 * H, W.qkv_w, N, QKV, 2 * H, ws.part, &go, m->sem, m->status, PEAGLE_OP_QKV, s));
      qa.mode = 1;
      qa.resid0 = ws.resid0;
      qa.mask_resid = m->mask_resid0;
      qa.h = ws.h;
    } else {
      CUDA_TRY(gemm_launch(dt, ws.xin, H, W.qkv_w, rows, QKV, H, ws.part, &go, m->sem, m->status, PEAGLE_OP_QKV, s));
      qa.mode = 0;
    }
    qa.in = go;
    qa.nq = nq;
    qa.nkv = nkv;
    qa.hd = hd;
    qa.H = H;
    qa.K = K;
    qa.rows = dr;
    qa.mask_qkv = m->mask_qkv0;
    qa.rcos = m->rcos;
    qa.rsin = m->rsin;
    qa.max_pos = c.max_position;
    qa.anchor_pos = pos;
    qa.Q = ws.q;
    qa.Kout = ws.kc;
    qa.Vout = ws.vc;
    if (append_kv) {
      qa.kcache = k_cache[l];
      qa.vcache = v_cache[l];
    }
    qa.kv_off = kv_offsets;
    qa.kv_len = kv_lens;
    qa.kv_cap = kv_capacity;
    qa.status = m->status;
    CUDA_TRY(launch_qkv_finish(dt, rows, qa, s));

    DecodeAttnArgs da{};
    da.B = B;
    da.K = K;
    da.nq = nq;
    da.nkv = nkv;
    da.hd = hd;
    da.rows = dr;
    da.R = rows;
    da.rows_max = dr.max_new + K - 1;
    da.Q = ws.q;
    da.Kc = ws.kc;
    da.Vc = ws.vc;
    da.kcache = k_cache[l];
    da.vcache = v_cache[l];
    da.kv_off = kv_offsets;
    da.kv_len = kv_lens;
    da.kv_cap = kv_capacity;
    da.max_kv_len = max_kv_len;
    da.chunk = ws.chunk;
    da.nsplit = ws.nsplit;
    da.part_o = ws.attn_o;
    da.part_ml = ws.attn_ml;
    da.O = ws.ao;
    da.scale = 1.0f / sqrtf((float)hd);
    da.status = m->status;
    CUDA_TRY(launch_decode_attn(dt, da, PEAGLE_OP_ATTN, s));

    ResidNormArgs ra{};
    ra.H = H;
    ra.row0 = 0;
    ra.h = ws.h;
    ra.gain = W.post_norm_w;
    ra.eps = eps;
    ra.y = ws.xin;
    CUDA_TRY(gemm_launch(dt, ws.ao, nq * hd, W.o_w, rows, H, nq * hd, ws.part, &go, m->sem, m->status, PEAGLE_OP_O, s));
    ra.in = go;
    CUDA_TRY(launch_resid_norm(dt, rows, ra, s));

    CUDA_TRY(gate_up_swiglu(dt, ws.xin, H, W.gate_up_w, rows, I, ws.part, ws.act, m->sem, m->status, s));
    CUDA_TRY(gemm_launch(dt, ws.act, I, W.down_w, rows, H, I, ws.part, &go, m->sem, m->status, PEAGLE_OP_DOWN, s));
    ra.in = go;
    ra.gain = (l + 1 < L) ? m->layers[l + 1].in_norm_w : m->w.final_norm_w;
    if (l + 1 == L && dr.new_off) {   // only the depth rows go on to the head
      ra.compact = 1;
      ra.crows = dr;
    }
    CUDA_TRY(launch_resid_norm(dt, rows, ra, s));
  }
  // draft-vocab head and argmax per depth over the B*K depth rows: bf16
  // reduces each output tile inside the GEMM (warp argmax); fp32 stores the
  // logits and reduces them
  if (dt == PEAGLE_BF16) {
    GemmEpi ep{};
    ep.op = GEMM_EPI_ARGMAX;
    ep.logits = logits;
    ep.logits_ld = c.draft_vocab;
    ep.p_max = ws.am_val;
    ep.p_idx = ws.am_idx;
    CUDA_TRY(gemm_launch_epi(dt, ws.xin, H, m->w.lm_head_w, heads, c.draft_vocab, H, ws.part, &go, m->sem,
                             m->status, PEAGLE_OP_LM_HEAD, &ep, s));
    CUDA_TRY(launch_lm_argmax_final(heads, gemm_col_tiles(heads, c.draft_vocab, H), ws.am_val, ws.am_idx, m->w.d2t,
                                    draft_tokens, s));
  } else {
    CUDA_TRY(gemm_launch(dt, ws.xin, H, m->w.lm_head_w, heads, c.draft_vocab, H, ws.part, &go, m->sem, m->status,
                         PEAGLE_OP_LM_HEAD, s));
    CUDA_TRY(launch_lm_argmax(go, heads, c.draft_vocab, logits, ws.am_val, ws.am_idx, m->w.d2t, draft_tokens, s));
  }
  return PEAGLE_OK;
}

static peagle_status check_caches(const peagle_config& c, void* const* k_cache, void* const* v_cache) {
  for (int l = 0; l < c.num_layers; ++l) {
    if (!k_cache[l] || !v_cache[l]) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step: cache of layer %d is NULL", l);
    if (!aligned16(k_cache[l]) || !aligned16(v_cache[l]))
      FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step: cache of layer %d is not 16-byte aligned", l);
  }
  return PEAGLE_OK;
}

peagle_status peagle_draft_step(const peagle_model* m, int32_t B, int32_t K, const void* aux,
                                const int32_t* anchor_tokens, const int32_t* anchor_pos, void* const* k_cache,
                                void* const* v_cache, const int64_t* kv_offsets, const int32_t* kv_lens,
                                int64_t kv_capacity, int32_t max_kv_len, int32_t append_anchor_kv,
                                int32_t* draft_tokens, float* logits, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (!m) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step: model is NULL");
  const peagle_config& c = m->cfg;
  if (B < 0 || K < 1 || K > 16) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step: B=%d K=%d (K in [1,16])", B, K);
  if (max_kv_len < 0 || kv_capacity < 0) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step: negative KV bound");
  if (append_anchor_kv != 0 && append_anchor_kv != 1) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step: append_anchor_kv");
  if (B == 0) return PEAGLE_OK;
  if (!aux || !anchor_tokens || !anchor_pos || !k_cache || !v_cache || !kv_offsets || !kv_lens || !draft_tokens)
    FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step: a required pointer is NULL");
  peagle_status st = check_caches(c, k_cache, v_cache);
  if (st) return st;
  if (c.dtype == PEAGLE_BF16 && !aligned16(aux)) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step: aux not 16-byte aligned");
  size_t need = 0;
  peagle_draft_step_workspace_size(m, B, K, max_kv_len, &need);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    FAIL(PEAGLE_ERR_WORKSPACE, "draft_step: workspace %zu bytes at %p, need %zu (256-byte aligned)",
         workspace_bytes, workspace, need);
  DecodeRows dr{};
  dr.B = B;
  dr.K = K;
  dr.new_off = nullptr;   // one anchor row per request
  dr.total_new = B;
  dr.max_new = 1;
  return draft_step_impl(m, dr, aux, anchor_tokens, anchor_pos, k_cache, v_cache, kv_offsets, kv_lens, kv_capacity,
                         max_kv_len, append_anchor_kv, draft_tokens, logits, workspace, static_cast<cudaStream_t>(stream));
}

peagle_status peagle_draft_step_ctx(const peagle_model* m, int32_t B, int32_t K, int32_t total_new, int32_t max_new,
                                    const int32_t* new_offsets, const void* new_aux, const int32_t* new_tokens,
                                    const int32_t* new_pos, void* const* k_cache, void* const* v_cache,
                                    const int64_t* kv_offsets, const int32_t* kv_lens, int64_t kv_capacity,
                                    int32_t max_kv_len, int32_t append_new_kv, int32_t* draft_tokens, float* logits,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (!m) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_ctx: model is NULL");
  const peagle_config& c = m->cfg;
  size_t need = 0;
  peagle_status st = peagle_draft_step_ctx_workspace_size(m, B, K, total_new, max_new, max_kv_len, &need);
  if (st) return st;
  if (kv_capacity < 0) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_ctx: negative KV capacity");
  if (append_new_kv != 0 && append_new_kv != 1) FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_ctx: append_new_kv");
  if (B == 0) return PEAGLE_OK;
  if (!new_offsets || !new_aux || !new_tokens || !new_pos || !k_cache || !v_cache || !kv_offsets || !kv_lens ||
      !draft_tokens)
    FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_ctx: a required pointer is NULL");
  st = check_caches(c, k_cache, v_cache);
  if (st) return st;
  if (c.dtype == PEAGLE_BF16 && !aligned16(new_aux))
    FAIL(PEAGLE_ERR_INVALID_ARG, "draft_step_ctx: new_aux not 16-byte aligned");
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    FAIL(PEAGLE_ERR_WORKSPACE, "draft_step_ctx: workspace %zu bytes at %p, need %zu (256-byte aligned)",
         workspace_bytes, workspace, need);
  DecodeRows dr{};
  dr.B = B;
  dr.K = K;
  dr.new_off = new_offsets;
  dr.total_new = total_new;
  dr.max_new = max_new;
  return draft_step_impl(m, dr, new_aux, new_tokens, new_pos, k_cache, v_cache, kv_offsets, kv_lens, kv_capacity,
                         max_kv_len, append_new_kv, draft_tokens, logits, workspace, static_cast<cudaStream_t>(stream));
}

peagle_status peagle_next_context(int32_t B, int32_t K, const int32_t* draft_tokens, const int32_t* accept_len,
                                  const int32_t* next_token, const int32_t* cur_offsets, const int32_t* cur_pos,
                                  int32_t* kv_lens, int32_t* next_offsets, int32_t* next_tokens, int32_t* next_pos,
                                  void* stream) {
  if (B < 0 || B > 65536 || K < 1 || K > 16) FAIL(PEAGLE_ERR_INVALID_ARG, "next_context: B=%d K=%d", B, K);
  if (!next_offsets) FAIL(PEAGLE_ERR_INVALID_ARG, "next_context: next_offsets is NULL");
  if (B > 0 && (!draft_tokens || !accept_len || !next_token || !cur_offsets || !cur_pos || !kv_lens ||
                !next_tokens || !next_pos))
    FAIL(PEAGLE_ERR_INVALID_ARG, "next_context: a pointer is NULL");
  NextContextArgs na{};
  na.B = B;
  na.K = K;
  na.drafts = draft_tokens;
  na.accept = accept_len;
  na.next = next_token;
  na.cur_off = cur_offsets;
  na.cur_pos = cur_pos;
  na.kv_lens = kv_lens;
  na.next_off = next_offsets;
  na.next_tok = next_tokens;
  na.next_pos = next_pos;
  CUDA_TRY(library_status_word(&na.status));
  CUDA_TRY(launch_next_context(na, static_cast<cudaStream_t>(stream)));
  return PEAGLE_OK;
}

// ==================================================================== verify
peagle_status peagle_verify_accept(int32_t B, int32_t K, const int32_t* draft_tokens, const int32_t* target_tokens,
                                   int32_t* accept_len, int32_t* next_token, void* stream) {
  if (B < 0 || K < 1 || K > 64) FAIL(PEAGLE_ERR_INVALID_ARG, "verify_accept: B=%d K=%d (K in [1,64])", B, K);
  if (B == 0) return PEAGLE_OK;
  if (!draft_tokens || !target_tokens || !accept_len || !next_token)
    FAIL(PEAGLE_ERR_INVALID_ARG, "verify_accept: a pointer is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  probe_start(PEAGLE_OP_VERIFY, s);
  CUDA_TRY(launch_verify(B, K, draft_tokens, target_tokens, accept_len, next_token, s));
  probe_stop(PEAGLE_OP_VERIFY, s);
  return PEAGLE_OK;
}

peagle_status peagle_verify_sample(int32_t B, int32_t K, int32_t V, const int32_t* draft_tokens,
                                   const float* draft_probs, const float* target_probs, const float* accept_u,
                                   const uint32_t* draws, int32_t* accept_len, int32_t* next_token, void* stream) {
  if (B < 0 || K < 1 || K > 64 || V < 1 || V > (1 << 23))
    FAIL(PEAGLE_ERR_INVALID_ARG, "verify_sample: B=%d K=%d V=%d (K in [1,64], V in [1, 2^23])", B, K, V);
  if (B == 0) return PEAGLE_OK;
  if (!draft_tokens || !draft_probs || !target_probs || !accept_u || !draws || !accept_len || !next_token)
    FAIL(PEAGLE_ERR_INVALID_ARG, "verify_sample: a pointer is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SampleArgs sa{};
  sa.B = B;
  sa.K = K;
  sa.V = V;
  sa.drafts = draft_tokens;
  sa.q = draft_probs;
  sa.p = target_probs;
  sa.u = accept_u;
  sa.draws = draws;
  sa.accept = accept_len;
  sa.next = next_token;
  CUDA_TRY(library_status_word(&sa.status));
  probe_start(PEAGLE_OP_VERIFY, s);
  CUDA_TRY(launch_verify_sample(sa, s));
  probe_stop(PEAGLE_OP_VERIFY, s);
  return PEAGLE_OK;
}

// ======================================================================= COD
peagle_status peagle_cod_counts(int32_t n, int32_t K, double r, double r_min, int32_t* counts) {
  if (n < 0 || n > (1 << 24) || K < 1 || K > 16) FAIL(PEAGLE_ERR_INVALID_ARG, "cod_counts: n=%d K=%d", n, K);
  if (!(r_min > 0.0) || !(r_min <= r) || !(r <= 1.0))
    FAIL(PEAGLE_ERR_INVALID_ARG, "cod_counts: need 0 < r_min <= r <= 1 (r=%g r_min=%g)", r, r_min);
  if (!counts) FAIL(PEAGLE_ERR_INVALID_ARG, "cod_counts: counts is NULL");
  counts[0] = n;
  double rd = 1.0;
  const long long fmin = (long long)floor((double)n * r_min);
  for (int d = 1; d < K; ++d) {
    rd = rd * r;
    long long c = (long long)floor((double)n * rd);
    if (c < fmin) c = fmin;
    if (c > counts[d - 1]) c = counts[d - 1];
    counts[d] = (int32_t)c;
  }
  return PEAGLE_OK;
}

peagle_status peagle_cod_select_workspace_size(int32_t n, int32_t K, size_t* bytes) {
  if (!bytes || n < 0 || K < 1 || K > 16) FAIL(PEAGLE_ERR_INVALID_ARG, "cod_select_workspace_size: bad argument");
  *bytes = 0;  // keys are regenerated from the counter, nothing is staged
  return PEAGLE_OK;
}

static peagle_status cod_enqueue(int n, int K, uint64_t seed, const int32_t* counts, int32_t* indices,
                                 int32_t* row_of, cudaStream_t s) {
  CodArgs ca{};
  ca.n = n;
  ca.K = K;
  ca.seed = seed;
  ca.off[0] = 0;
  for (int d = 0; d < K; ++d) {
    ca.counts[d] = counts[d];
    ca.off[d + 1] = ca.off[d] + counts[d];
  }
  ca.indices = indices;
  ca.row_of = row_of;
  probe_start(PEAGLE_OP_COD, s);
  CUDA_TRY(launch_cod_select(ca, s));
  probe_stop(PEAGLE_OP_COD, s);
  return PEAGLE_OK;
}

peagle_status peagle_cod_select(int32_t n, int32_t K, double r, double r_min, uint64_t seed, int32_t* counts_host,
                                int32_t* indices, int32_t* row_of, void* workspace, size_t workspace_bytes,
                                void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  int32_t counts[16];
  peagle_status st = peagle_cod_counts(n, K, r, r_min, counts);
  if (st) return st;
  if (counts_host) memcpy(counts_host, counts, sizeof(int32_t) * K);
  if (n == 0) return PEAGLE_OK;
  if (!indices) FAIL(PEAGLE_ERR_INVALID_ARG, "cod_select: indices is NULL");
  return cod_enqueue(n, K, seed, counts, indices, row_of, static_cast<cudaStream_t>(stream));
}

// ============================================================= dense GEMM
peagle_status peagle_get_library_status(void* stream, int32_t* host_status) {
  if (!host_status) FAIL(PEAGLE_ERR_INVALID_ARG, "get_library_status: host_status is NULL");
  int* w = nullptr;
  CUDA_TRY(library_status_word(&w));
  CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int v = 0;
  CUDA_TRY(cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost));
  *host_status = v;
  return PEAGLE_OK;
}

peagle_status peagle_clear_library_status(void* stream) {
  int* w = nullptr;
  CUDA_TRY(library_status_word(&w));
  CUDA_TRY(cudaMemsetAsync(w, 0, sizeof(int), static_cast<cudaStream_t>(stream)));
  return PEAGLE_OK;
}

peagle_status peagle_set_wait_limit_ns(uint64_t ns) {
  gemm_set_wait_limit(ns);
  return PEAGLE_OK;
}

static size_t gemm_slab_bytes(int M, int N, int K) {
  return ((gemm_out_floats(PEAGLE_BF16, M, N, K) * sizeof(float)) + 255) & ~size_t(255);
}
static size_t gemm_ws_bytes(int M, int N, int K) {
  return gemm_slab_bytes(M, N, K) + kGemmSemCount * sizeof(int);
}

peagle_status peagle_gemm_workspace_size(int32_t dtype, int32_t M, int32_t N, int32_t K, size_t* bytes) {
  if (!bytes || M < 0 || N < 0 || K < 1 || (dtype != PEAGLE_F32 && dtype != PEAGLE_BF16))
    FAIL(PEAGLE_ERR_INVALID_ARG, "gemm_workspace_size: bad argument");
  *bytes = dtype == PEAGLE_BF16 ? gemm_ws_bytes(M, N, K) : 0;
  return PEAGLE_OK;
}

// The address through which the device reaches page-locked, mapped host
// memory `p`, or NULL when `p` is not such memory (pageable, device or
// unknown memory: the staging copies refuse it rather than launch).
static const void* mapped_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

peagle_status peagle_copy_to_device(void* dev, const void* host, size_t bytes, void* stream) {
  if (bytes == 0) return PEAGLE_OK;
  if (!dev || !host) FAIL(PEAGLE_ERR_INVALID_ARG, "copy_to_device: NULL pointer");
  const void* src = mapped_host(host);
  if (!src) FAIL(PEAGLE_ERR_INVALID_ARG, "copy_to_device: the host buffer is not mapped page-locked memory");
  CUDA_TRY(launch_stage_copy(dev, src, (long long)bytes, true, static_cast<cudaStream_t>(stream)));
  return PEAGLE_OK;
}

peagle_status peagle_copy_to_host(void* host, const void* dev, size_t bytes, void* stream) {
  if (bytes == 0) return PEAGLE_OK;
  if (!dev || !host) FAIL(PEAGLE_ERR_INVALID_ARG, "copy_to_host: NULL pointer");
  void* dst = const_cast<void*>(mapped_host(host));
  if (!dst) FAIL(PEAGLE_ERR_INVALID_ARG, "copy_to_host: the host buffer is not mapped page-locked memory");
  CUDA_TRY(launch_stage_copy(dst, dev, (long long)bytes, false, static_cast<cudaStream_t>(stream)));
  return PEAGLE_OK;
}

peagle_status peagle_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* X, const void* W, float* D,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 1 || (dtype != PEAGLE_F32 && dtype != PEAGLE_BF16))
    FAIL(PEAGLE_ERR_INVALID_ARG, "gemm: M=%d N=%d K=%d dtype=%d", M, N, K, dtype);
  if (M == 0 || N == 0) return PEAGLE_OK;
  if (!X || !W || !D) FAIL(PEAGLE_ERR_INVALID_ARG, "gemm: NULL operand");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == PEAGLE_F32) {
    CUDA_TRY(gemm_launch(dtype, X, K, W, M, N, K, D, nullptr, nullptr, nullptr, -1, s));
    return PEAGLE_OK;
  }
  if (K % 8 || !aligned16(X) || !aligned16(W)) FAIL(PEAGLE_ERR_INVALID_ARG, "gemm: bf16 needs K %% 8 == 0 and 16-byte aligned operands");
  size_t need = gemm_ws_bytes(M, N, K);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    FAIL(PEAGLE_ERR_WORKSPACE, "gemm: workspace %zu bytes, need %zu", workspace_bytes, need);
  GemmOut go;
  int* sem = reinterpret_cast<int*>(static_cast<char*>(workspace) + gemm_slab_bytes(M, N, K));
  int* lib_status = nullptr;
  CUDA_TRY(library_status_word(&lib_status));
  CUDA_TRY(cudaMemsetAsync(sem, 0, kGemmSemCount * sizeof(int), s));
  CUDA_TRY(gemm_launch(dtype, X, K, W, M, N, K, static_cast<float*>(workspace), &go, sem, lib_status, -1, s));
  CUDA_TRY(launch_sum_splits(go, M, N, D, s));
  return PEAGLE_OK;
}

}  // extern "C"


// ========================================================= parallel forward
struct TrainWs {
  int* sem;
  int *indices, *row_of, *anchor, *depth, *pos, *start, *label;
  void *x0, *xin, *act, *q, *kr, *vr, *ao;
  void* vt;  // V transposed [nkv*hd, rp] for the tensor-core attention, or NULL
  int rp;
  float *resid0, *h, *part, *row_ce;
  int* row_am;
  float *p_max, *p_sum, *p_lab;   // fused head partials of one chunk
  int* p_idx;
  int rc;  // rows per GEMM chunk
};

static const int kTrainChunk = 16384;

static size_t chunk_part_floats(int dt, int total, int rc, int N, int K) {
  if (total <= 0) return 0;
  size_t f = gemm_out_floats(dt, std::min(total, rc), N, K);
  const int last = total % rc;
  if (last) f = std::max(f, gemm_out_floats(dt, last, N, K));
  return f;
}

static void train_layout(const peagle_config& c, int n, int K, int R, Bump& bp, TrainWs& ws) {
  const size_t es = esize(c);
  const int H = c.hidden, I = c.intermediate, QKV = qkv_out(c), AHt = c.num_aux * c.target_hidden;
  const int nq = c.num_q_heads, nkv = c.num_kv_heads, hd = c.head_dim, dt = c.dtype;
  const int rc = std::max(1, std::min(R, kTrainChunk));
  ws.rc = rc;
  ws.sem = bp.take<int>(kGemmSemCount);
  ws.indices = bp.take<int>(R);
  ws.row_of = bp.take<int>((size_t)K * n);
  ws.anchor = bp.take<int>(R);
  ws.depth = bp.take<int>(R);
  ws.pos = bp.take<int>(R);
  ws.start = bp.take<int>(R);
  ws.label = bp.take<int>(R);
  ws.x0 = bp.take_bytes((size_t)n * 2 * H * es);
  ws.resid0 = bp.take<float>((size_t)n * H);
  ws.h = bp.take<float>((size_t)R * H);
  ws.xin = bp.take_bytes((size_t)R * H * es);
  ws.act = bp.take_bytes((size_t)rc * I * es);
  ws.q = bp.take_bytes((size_t)R * nq * hd * es);
  ws.kr = bp.take_bytes((size_t)R * nkv * hd * es);
  ws.vr = bp.take_bytes((size_t)R * nkv * hd * es);
  ws.ao = bp.take_bytes((size_t)R * nq * hd * es);
  ws.rp = (R + 63) / 64 * 64;
  ws.vt = (dt == PEAGLE_BF16 && hd == 128) ? bp.take_bytes((size_t)nkv * hd * ws.rp * es) : nullptr;
  size_t pf = chunk_part_floats(dt, n, rc, H, AHt);
  pf = std::max(pf, chunk_part_floats(dt, n, rc, QKV, 2 * H));
  pf = std::max(pf, chunk_part_floats(dt, R, rc, QKV, H));
  pf = std::max(pf, chunk_part_floats(dt, R, rc, H, nq * hd));
  pf = std::max(pf, chunk_part_floats(dt, R, rc, 2 * I, H));
  pf = std::max(pf, chunk_part_floats(dt, R, rc, H, I));
  pf = std::max(pf, chunk_part_floats(dt, R, rc, c.draft_vocab, H));
  ws.part = bp.take<float>(pf);
  ws.row_ce = bp.take<float>(R);
  ws.row_am = bp.take<int>(R);
  const size_t parts = (size_t)rc * ((c.draft_vocab + 127) / 128);
  ws.p_max = bp.take<float>(parts);
  ws.p_sum = bp.take<float>(parts);
  ws.p_lab = bp.take<float>(parts);
  ws.p_idx = bp.take<int>(parts);
}

extern "C" {

peagle_status peagle_parallel_forward_workspace_size(const peagle_model* m, int32_t n, int32_t K, double r,
                                                     double r_min, size_t* bytes) {
  if (!m || !bytes) FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_forward_workspace_size: NULL argument");
  int32_t counts[16];
  peagle_status st = peagle_cod_counts(n, K, r, r_min, counts);
  if (st) return st;
  int R = 0;
  for (int d = 0; d < K; ++d) R += counts[d];
  Bump bp(nullptr);
  TrainWs ws;
  train_layout(m->cfg, n, K, R, bp, ws);
  *bytes = bp.off;
  return PEAGLE_OK;
}

peagle_status peagle_parallel_forward(const peagle_model* m, int32_t n, const void* aux, const int32_t* input_ids,
                                      const int32_t* position_ids, const int32_t* cu_seqlens, int32_t num_seqs,
                                      const int32_t* labels, const uint8_t* loss_mask, int32_t K, double r,
                                      double r_min, uint64_t seed, double depth_decay, float* per_depth_loss,
                                      float* per_depth_acc, int32_t* per_depth_valid, float* loss,
                                      int32_t* row_argmax, float* row_ce, float* logits, double* depth_sums,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!m) FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_forward: model is NULL");
  const peagle_config& c = m->cfg;
  int32_t counts[16];
  peagle_status st = peagle_cod_counts(n, K, r, r_min, counts);
  if (st) return st;
  if (!isfinite(depth_decay)) FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_forward: depth_decay not finite");
  if (!per_depth_loss || !per_depth_acc || !per_depth_valid || !loss)
    FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_forward: a required output is NULL");
  if (n > 0 && (!aux || !input_ids || !position_ids || !cu_seqlens || !labels || num_seqs < 1 || num_seqs > n))
    FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_forward: a required input is NULL or num_seqs=%d out of [1, n]", num_seqs);
  if (c.dtype == PEAGLE_BF16 && n > 0 && !aligned16(aux)) FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_forward: aux not 16-byte aligned");
  int off[17];
  off[0] = 0;
  for (int d = 0; d < K; ++d) off[d + 1] = off[d] + counts[d];
  const int R = off[K];
  size_t need = 0;
  peagle_parallel_forward_workspace_size(m, n, K, r, r_min, &need);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    FAIL(PEAGLE_ERR_WORKSPACE, "parallel_forward: workspace %zu bytes at %p, need %zu (256-byte aligned)",
         workspace_bytes, workspace, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Bump bp(workspace);
  TrainWs ws;
  train_layout(c, n, K, R, bp, ws);
  const int H = c.hidden, I = c.intermediate, QKV = qkv_out(c), L = c.num_layers, V = c.draft_vocab;
  const int nq = c.num_q_heads, nkv = c.num_kv_heads, hd = c.head_dim, AHt = c.num_aux * c.target_hidden;
  const int dt = c.dtype, rc = ws.rc;
  const size_t es = esize(c);
  const float eps = (float)c.rms_eps;
  float* rce = row_ce ? row_ce : ws.row_ce;
  int* ram = row_argmax ? row_argmax : ws.row_am;
  auto at = [es](void* base, size_t elems) { return static_cast<char*>(base) + elems * es; };
  auto atc = [es](const void* base, size_t elems) { return static_cast<const char*>(base) + elems * es; };
  GemmOut go;

  if (n > 0) {
    CUDA_TRY(cudaMemsetAsync(ws.sem, 0, kGemmSemCount * sizeof(int), s));
    // COD rows and per-row metadata
    st = cod_enqueue(n, K, seed, counts, ws.indices, ws.row_of, s);
    if (st) return st;
    TrainMetaArgs ta{};
    ta.n = n;
    ta.R = R;
    ta.K = K;
    ta.S = num_seqs;
    ta.Vt = c.target_vocab;
    ta.Vd = V;
    ta.max_pos = c.max_position;
    memcpy(ta.off, off, sizeof off);
    ta.indices = ws.indices;
    ta.position_ids = position_ids;
    ta.cu = cu_seqlens;
    ta.labels = labels;
    ta.loss_mask = loss_mask;
    ta.t2d = m->w.t2d;
    ta.row_anchor = ws.anchor;
    ta.row_depth = ws.depth;
    ta.row_pos = ws.pos;
    ta.row_start = ws.start;
    ta.row_label = ws.label;
    ta.status = m->status;
    CUDA_TRY(launch_train_meta(ta, s));

    // fc + fc_norm + layer-0 inputs of the n depth-0 rows
    for (int c0 = 0; c0 < n; c0 += rc) {
      const int mr = std::min(rc, n - c0);
      CUDA_TRY(gemm_launch(dt, atc(aux, (size_t)c0 * AHt), AHt, m->w.fc_w, mr, H, AHt, ws.part, &go, ws.sem, m->status,
                           PEAGLE_OP_FC, s));
      FcFinishArgs fa{};
      fa.u = go;
      fa.H = H;
      fa.Vt = c.target_vocab;
      fa.tok = input_ids + c0;
      fa.embed = m->w.embed;
      fa.g_fc = m->w.fc_norm_w;
      fa.g_in = m->layers[0].in_norm_w;
      fa.g_h = m->layers[0].hidden_norm_w;
      fa.eps = eps;
      fa.nbr = c.norm_before_residual;
      fa.x0 = at(ws.x0, (size_t)c0 * 2 * H);
      fa.resid = ws.resid0 + (size_t)c0 * H;
      fa.status = m->status;
      CUDA_TRY(launch_fc_finish(dt, mr, fa, s));
    }

    for (int l = 0; l < L; ++l) {
      const peagle_layer_weights& W = m->layers[l];
      QkvArgs qa{};
      qa.nq = nq;
      qa.nkv = nkv;
      qa.hd = hd;
      qa.H = H;
      qa.K = K;
      qa.mask_qkv = m->mask_qkv0;
      qa.mask_resid = m->mask_resid0;
      qa.rcos = m->rcos;
      qa.rsin = m->rsin;
      qa.max_pos = c.max_position;
      qa.row_pos = ws.pos;
      qa.Q = ws.q;
      qa.Kout = ws.kr;
      qa.Vout = ws.vr;
      qa.status = m->status;
      const int src_rows = (l == 0) ? n : R;
      for (int c0 = 0; c0 < src_rows; c0 += rc) {
        const int mr = std::min(rc, src_rows - c0);
        const int kin = (l == 0) ? 2 * H : H;
        const void* X = (l == 0) ? atc(ws.x0, (size_t)c0 * 2 * H) : atc(ws.xin, (size_t)c0 * H);
        if (hd == 128 && gemm_qkv_fusable(dt, mr, QKV, kin)) {
          // rotary and the bf16 q/k/v in the contraction's epilogue; the
          // layer-0 residual seed is a copy
          GemmEpi ep{};
          ep.op = GEMM_EPI_QKV;
          ep.nq = nq;
          ep.nkv = nkv;
          ep.max_pos = c.max_position;
          ep.row_base = c0;
          ep.rcos = m->rcos;
          ep.rsin = m->rsin;
          ep.row_pos = ws.pos;
          ep.q = ws.q;
          ep.k = ws.kr;
          ep.v = ws.vr;
          CUDA_TRY(gemm_launch_epi(dt, X, kin, W.qkv_w, mr, QKV, kin, ws.part, &go, ws.sem, m->status, PEAGLE_OP_QKV,
                                   &ep, s));
          qa.in = go;   // (unread by the masked-row finish below, which takes mask_qkv)
          if (l == 0)
            CUDA_TRY(cudaMemcpyAsync(ws.h + (size_t)c0 * H, ws.resid0 + (size_t)c0 * H, (size_t)mr * H * 4,
                                     cudaMemcpyDeviceToDevice, s));
          continue;
        }
        CUDA_TRY(gemm_launch(dt, X, kin, W.qkv_w, mr, QKV, kin, ws.part, &go, ws.sem, m->status, PEAGLE_OP_QKV, s));
        qa.in = go;
        qa.mode = 0;
        qa.row0 = c0;
        qa.src0 = c0;
        qa.resid0 = (l == 0) ? ws.resid0 + (size_t)c0 * H : nullptr;
        qa.h = (l == 0) ? ws.h : nullptr;
        CUDA_TRY(launch_qkv_finish(dt, mr, qa, s));
      }
      if (l == 0 && R > n) {  // every masked row of layer 0 shares one pre-rotary q/k/v
        qa.mode = 2;
        qa.row0 = n;
        qa.src0 = n;
        qa.resid0 = nullptr;
        qa.h = ws.h;
        CUDA_TRY(launch_qkv_finish(dt, R - n, qa, s));
      }
      TrainAttnArgs aa{};
      aa.R = R;
      aa.n = n;
      aa.nq = nq;
      aa.nkv = nkv;
      aa.hd = hd;
      aa.Q = ws.q;
      aa.Kr = ws.kr;
      aa.Vr = ws.vr;
      aa.row_anchor = ws.anchor;
      aa.row_depth = ws.depth;
      aa.row_start = ws.start;
      aa.row_of = ws.row_of;
      aa.O = ws.ao;
      aa.scale = 1.0f / sqrtf((float)hd);
      aa.Vt = ws.vt;
      aa.Rp = ws.rp;
      aa.status = m->status;
      TrainTileArgs tt{};
      tt.K = K;
      for (int d = 0; d <= K; ++d) tt.row_off[d] = off[d];
      CUDA_TRY(launch_train_attn(dt, aa, tt, PEAGLE_OP_ATTN, s));

      for (int c0 = 0; c0 < R; c0 += rc) {
        const int mr = std::min(rc, R - c0);
        CUDA_TRY(gemm_launch(dt, atc(ws.ao, (size_t)c0 * nq * hd), nq * hd, W.o_w, mr, H, nq * hd, ws.part, &go,
                             ws.sem, m->status, PEAGLE_OP_O, s));
        ResidNormArgs ra{};
        ra.in = go;
        ra.H = H;
        ra.row0 = c0;
        ra.h = ws.h;
        ra.gain = W.post_norm_w;
        ra.eps = eps;
        ra.y = ws.xin;
        CUDA_TRY(launch_resid_norm(dt, mr, ra, s));
        CUDA_TRY(gate_up_swiglu(dt, atc(ws.xin, (size_t)c0 * H), H, W.gate_up_w, mr, I, ws.part, ws.act, ws.sem,
                                m->status, s));
        CUDA_TRY(gemm_launch(dt, ws.act, I, W.down_w, mr, H, I, ws.part, &go, ws.sem, m->status, PEAGLE_OP_DOWN, s));
        ra.in = go;
        ra.gain = (l + 1 < L) ? m->layers[l + 1].in_norm_w : m->w.final_norm_w;
        CUDA_TRY(launch_resid_norm(dt, mr, ra, s));
      }
    }
    // draft-vocab head + per-row CE, chunked so the logits never all exist
    for (int c0 = 0; c0 < R; c0 += rc) {
      const int mr = std::min(rc, R - c0);
      if (dt == PEAGLE_BF16) {  // cross-entropy partials reduced inside the GEMM
        GemmEpi ep{};
        ep.op = GEMM_EPI_CE;
        ep.logits = logits ? logits + (size_t)c0 * V : nullptr;
        ep.logits_ld = V;
        ep.p_max = ws.p_max;
        ep.p_sum = ws.p_sum;
        ep.p_lab = ws.p_lab;
        ep.p_idx = ws.p_idx;
        ep.labels = ws.label + c0;
        CUDA_TRY(gemm_launch_epi(dt, atc(ws.xin, (size_t)c0 * H), H, m->w.lm_head_w, mr, V, H, ws.part, &go, ws.sem,
                                 m->status, PEAGLE_OP_LM_HEAD, &ep, s));
        probe_start(PEAGLE_OP_CE, s);
        CUDA_TRY(launch_ce_merge(mr, gemm_col_tiles(mr, V, H), c0, ws.p_max, ws.p_sum, ws.p_lab, ws.p_idx, ws.label,
                                 rce, ram, s));
        probe_stop(PEAGLE_OP_CE, s);
      } else {
        CUDA_TRY(gemm_launch(dt, atc(ws.xin, (size_t)c0 * H), H, m->w.lm_head_w, mr, V, H, ws.part, &go, ws.sem,
                             m->status, PEAGLE_OP_LM_HEAD, s));
        probe_start(PEAGLE_OP_CE, s);
        CUDA_TRY(launch_ce_rows(go, mr, V, c0, ws.label, logits, rce, ram, s));
        probe_stop(PEAGLE_OP_CE, s);
      }
    }
  }
  CeReduceArgs cr{};
  cr.row_ce = rce;
  cr.row_am = ram;
  cr.row_label = ws.label;
  memcpy(cr.off, off, sizeof off);
  cr.K = K;
  cr.decay = depth_decay;
  cr.loss_d = per_depth_loss;
  cr.acc_d = per_depth_acc;
  cr.valid_d = per_depth_valid;
  cr.loss = loss;
  cr.sums = depth_sums;
  CUDA_TRY(launch_ce_reduce(cr, s));
  return PEAGLE_OK;
}

// ================================================================ backward
// Gradients of the training loss (sum_d decay^d * mean_d CE) with respect to
// every weight but the (frozen) embedding. The call runs the forward once
// more, keeping each layer's activations, then goes backward: cross-entropy
// -> head -> layers (MLP, post-norm, O, attention, RoPE, QKV, input norm) ->
// layer-0 inputs -> fc_norm / fc and mask_hidden. Contractions run on the
// library's GEMM over transposed copies: dX = dY W as dY (W^T)^T, dW = dY^T X
// as (dY^T)(X^T)^T with the rows padded to a multiple of 64.
struct BwdWs {
  int* sem;
  int *indices, *row_of, *anchor, *depth, *pos, *start, *end, *label;
  int Rp, np1p, Vp;
  void *x0src, *x0full, *z, *dlog, *ta, *tb, *gcast, *dgu, *dqkv, *auxm;
  void* vt;   // V transposed [nkv*hd, Rp] for the tensor-core forward attention, or NULL
  float *U, *Um, *hidsrc, *residsrc, *hidfull, *residfull, *hL, *logits, *part, *rce;
  int* ram;
  float *p_max, *p_sum, *p_lab;   // fused head partials [R, column tiles] (bf16 path)
  int* p_idx;
  float *loss_d, *acc_d;
  int* valid_d;
  float *dh, *dh2, *dhid, *dbig, *dQ, *dK, *dV, *lse, *Dv, *rrow, *rrow2, *du, *dmask;
  std::vector<void*> xin, q, k, v, o, y, act, wT_qkv, wT_o, wT_gu, wT_down;
  std::vector<float*> hin, hmid, gu, lse2;   // lse2: each layer's base-2 log-sum-exp (bf16 path)
  void *wT_lm, *wT_fc;
};

// a gradient buffer of the caller's peagle_weights (declared const there)
static float* gout(const void* p) { return const_cast<float*>(static_cast<const float*>(p)); }

static void bwd_layout(const peagle_config& c, int n, int K, int R, Bump& bp, BwdWs& ws) {
  const size_t es = esize(c);
  const int H = c.hidden, I = c.intermediate, QKV = qkv_out(c), AHt = c.num_aux * c.target_hidden;
  const int nqhd = c.num_q_heads * c.head_dim, nkvhd = c.num_kv_heads * c.head_dim, V = c.draft_vocab, L = c.num_layers;
  const int dt = c.dtype;
  ws.Rp = (R + 63) / 64 * 64;
  ws.np1p = (n + 1 + 63) / 64 * 64;
  ws.Vp = (V + 7) / 8 * 8;
  const int Rp = ws.Rp, Vp = ws.Vp;
  ws.sem = bp.take<int>(kGemmSemCount);
  ws.indices = bp.take<int>(R);
  ws.row_of = bp.take<int>((size_t)K * n);
  ws.anchor = bp.take<int>(R);
  ws.depth = bp.take<int>(R);
  ws.pos = bp.take<int>(R);
  ws.start = bp.take<int>(R);
  ws.end = bp.take<int>(R);
  ws.label = bp.take<int>(R);
  ws.U = bp.take<float>(gemm_out_floats(dt, std::max(n, 1), H, AHt));
  ws.Um = bp.take<float>(gemm_out_floats(dt, 1, H, AHt));
  ws.x0src = bp.take_bytes((size_t)(n + 1) * 2 * H * es);
  ws.hidsrc = bp.take<float>((size_t)(n + 1) * H);
  ws.residsrc = bp.take<float>((size_t)(n + 1) * H);
  ws.x0full = bp.take_bytes((size_t)R * 2 * H * es);
  ws.hidfull = bp.take<float>((size_t)R * H);
  ws.residfull = bp.take<float>((size_t)R * H);
  ws.xin.assign(L, nullptr);
  ws.q.assign(L, nullptr);
  ws.k.assign(L, nullptr);
  ws.v.assign(L, nullptr);
  ws.o.assign(L, nullptr);
  ws.y.assign(L, nullptr);
  ws.act.assign(L, nullptr);
  ws.wT_qkv.assign(L, nullptr);
  ws.wT_o.assign(L, nullptr);
  ws.wT_gu.assign(L, nullptr);
  ws.wT_down.assign(L, nullptr);
  ws.hin.assign(L, nullptr);
  ws.hmid.assign(L, nullptr);
  ws.gu.assign(L, nullptr);
  ws.lse2.assign(L, nullptr);
  for (int l = 0; l < L; ++l) {
    const int in = l == 0 ? 2 * H : H;
    ws.xin[l] = l == 0 ? ws.x0full : bp.take_bytes((size_t)R * H * es);
    ws.hin[l] = bp.take<float>((size_t)R * H);
    ws.q[l] = bp.take_bytes((size_t)R * nqhd * es);
    ws.k[l] = bp.take_bytes((size_t)R * nkvhd * es);
    ws.v[l] = bp.take_bytes((size_t)R * nkvhd * es);
    ws.o[l] = bp.take_bytes((size_t)R * nqhd * es);
    ws.hmid[l] = bp.take<float>((size_t)R * H);
    ws.y[l] = bp.take_bytes((size_t)R * H * es);
    ws.gu[l] = bp.take<float>((size_t)R * 2 * I);
    ws.act[l] = bp.take_bytes((size_t)R * I * es);
    ws.lse2[l] = bp.take<float>((size_t)R * c.num_q_heads);
    ws.wT_qkv[l] = bp.take_bytes((size_t)in * QKV * es);
    ws.wT_o[l] = bp.take_bytes((size_t)nqhd * H * es);
    ws.wT_gu[l] = bp.take_bytes((size_t)H * 2 * I * es);
    ws.wT_down[l] = bp.take_bytes((size_t)I * H * es);
  }
  ws.hL = bp.take<float>((size_t)R * H);
  ws.z = bp.take_bytes((size_t)R * H * es);
  ws.wT_lm = bp.take_bytes((size_t)H * Vp * es);
  ws.wT_fc = bp.take_bytes((size_t)AHt * H * es);
  ws.logits = bp.take<float>((size_t)R * V);
  ws.rce = bp.take<float>(R);
  ws.ram = bp.take<int>(R);
  {
    const size_t np = dt == PEAGLE_BF16 ? (size_t)R * gemm_col_tiles(R, V, H) : 0;
    ws.p_max = bp.take<float>(np);
    ws.p_sum = bp.take<float>(np);
    ws.p_lab = bp.take<float>(np);
    ws.p_idx = bp.take<int>(np);
  }
  ws.loss_d = bp.take<float>(K);
  ws.acc_d = bp.take<float>(K);
  ws.valid_d = bp.take<int>(K);
  ws.dlog = bp.take_bytes((size_t)R * Vp * es);
  // partial slabs of every contraction of the pass
  const int widths[] = {H, I, 2 * I, QKV, nqhd, 2 * H, V, Vp, AHt};
  size_t pf = 0;
  for (int N : widths)
    for (int Kd : widths) pf = std::max(pf, gemm_out_floats(dt, R, N, Kd));
  pf = std::max(pf, gemm_out_floats(dt, R, V, H));
  const int outs[] = {V, Vp, H, 2 * I, QKV, nqhd, I};
  const int ins[] = {H, I, 2 * H, nqhd, AHt};
  for (int M : outs)
    for (int N : ins) pf = std::max(pf, gemm_out_floats(dt, M, N, Rp));
  pf = std::max(pf, gemm_out_floats(dt, H, AHt, ws.np1p));
  pf = std::max(pf, gemm_out_floats(dt, 1, AHt, H));
  ws.part = bp.take<float>(pf);
  const int tw = std::max(std::max(std::max(Vp, 2 * I), std::max(QKV, 2 * H)), std::max(AHt, nqhd));
  const int tr = std::max(Rp, ws.np1p);
  ws.ta = bp.take_bytes((size_t)tw * tr * es);
  ws.tb = bp.take_bytes((size_t)tw * tr * es);
  const int gw = std::max(std::max(std::max(H, I), std::max(2 * I, QKV)), std::max(nqhd, 2 * H));
  ws.gcast = bp.take_bytes((size_t)R * gw * es);
  ws.dgu = bp.take_bytes((size_t)R * 2 * I * es);
  ws.dqkv = bp.take_bytes((size_t)R * QKV * es);
  ws.dh = bp.take<float>((size_t)R * H);
  ws.dh2 = bp.take<float>((size_t)R * H);
  // the n depth-0 rows and, in row n, the masked rows' summed gradient (with
  // K = 1 there are no masked rows and R = n)
  ws.dhid = bp.take<float>((size_t)std::max(R, n + 1) * H);
  ws.dbig = bp.take<float>((size_t)std::max(R, n + 1) * gw);
  ws.dQ = bp.take<float>((size_t)R * nqhd);
  ws.dK = bp.take<float>((size_t)R * nkvhd);
  ws.dV = bp.take<float>((size_t)R * nkvhd);
  ws.lse = bp.take<float>((size_t)R * c.num_q_heads);
  ws.Dv = bp.take<float>((size_t)R * c.num_q_heads);
  ws.rrow = bp.take<float>(std::max(R, n + 1));
  ws.rrow2 = bp.take<float>(std::max(R, n + 1));
  ws.du = bp.take<float>((size_t)(n + 1) * H);
  ws.dmask = bp.take<float>(H);
  ws.auxm = bp.take_bytes((size_t)(n + 1) * AHt * es);
  ws.vt = (dt == PEAGLE_BF16 && c.head_dim == 128) ? bp.take_bytes((size_t)c.num_kv_heads * c.head_dim * Rp * es)
                                                     : nullptr;
}

peagle_status peagle_parallel_backward_workspace_size(const peagle_model* m, int32_t n, int32_t K, double r, double r_min,
                                                      size_t* bytes) {
  if (!m || !bytes) FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_backward_workspace_size: NULL argument");
  int32_t counts[16];
  peagle_status st = peagle_cod_counts(n, K, r, r_min, counts);
  if (st) return st;
  int R = 0;
  for (int d = 0; d < K; ++d) R += counts[d];
  Bump bp(nullptr);
  BwdWs ws;
  bwd_layout(m->cfg, n, K, R, bp, ws);
  *bytes = bp.off;
  return PEAGLE_OK;
}

peagle_status peagle_parallel_backward(const peagle_model* m, int32_t n, const void* aux, const int32_t* input_ids,
                                       const int32_t* position_ids, const int32_t* cu_seqlens, int32_t num_seqs,
                                       const int32_t* labels, const uint8_t* loss_mask, int32_t K, double r,
                                       double r_min, uint64_t seed, double depth_decay, float* loss,
                                       const peagle_weights* grads, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  if (!m) FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_backward: model is NULL");
  const peagle_config& c = m->cfg;
  int32_t counts[16];
  peagle_status st = peagle_cod_counts(n, K, r, r_min, counts);
  if (st) return st;
  if (!isfinite(depth_decay)) FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_backward: depth_decay not finite");
  if (n < 1 || !aux || !input_ids || !position_ids || !cu_seqlens || !labels || num_seqs < 1 || num_seqs > n || !loss)
    FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_backward: a required input is NULL, n < 1 or num_seqs=%d out of [1, n]",
         num_seqs);
  if (!grads || !grads->fc_w || !grads->fc_norm_w || !grads->mask_hidden || !grads->final_norm_w || !grads->lm_head_w ||
      !grads->layers)
    FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_backward: a gradient buffer is NULL");
  for (int l = 0; l < c.num_layers; ++l) {
    const peagle_layer_weights& G = grads->layers[l];
    if (!G.in_norm_w || !G.qkv_w || !G.o_w || !G.post_norm_w || !G.gate_up_w || !G.down_w || (l == 0 && !G.hidden_norm_w))
      FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_backward: a gradient buffer of layer %d is NULL", l);
  }
  if (c.dtype == PEAGLE_BF16 && !aligned16(aux)) FAIL(PEAGLE_ERR_INVALID_ARG, "parallel_backward: aux not 16-byte aligned");
  int off[17];
  off[0] = 0;
  for (int d = 0; d < K; ++d) off[d + 1] = off[d] + counts[d];
  const int R = off[K];
  size_t need = 0;
  peagle_parallel_backward_workspace_size(m, n, K, r, r_min, &need);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    FAIL(PEAGLE_ERR_WORKSPACE, "parallel_backward: workspace %zu bytes at %p, need %zu (256-byte aligned)",
         workspace_bytes, workspace, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Bump bp(workspace);
  BwdWs ws;
  bwd_layout(c, n, K, R, bp, ws);
  const int H = c.hidden, I = c.intermediate, QKV = qkv_out(c), L = c.num_layers, V = c.draft_vocab;
  const int nq = c.num_q_heads, nkv = c.num_kv_heads, hd = c.head_dim, AHt = c.num_aux * c.target_hidden;
  const int nqhd = nq * hd;
  const int dt = c.dtype, es = (int)esize(c), gbf = dt == PEAGLE_BF16 ? 1 : 0;
  const int Rp = ws.Rp, Vp = ws.Vp;
  const float eps = (float)c.rms_eps;
  auto at = [es](const void* base, size_t elems) { return static_cast<char*>(const_cast<void*>(base)) + elems * es; };
  GemmOut go;
  // D = X W^T into the partial slabs; the result is ws.part (row stride N).
  // Only a model weight (w_early) may be read before the kernel waits for
  // its predecessor: the transposed copies of this pass are written by
  // kernels of the same launch chain.
  auto mm = [&](const void* X, int ldx, const void* W, int M, int N, int Kd, bool w_early = false) {
    return gemm_launch(dt, X, ldx, W, M, N, Kd, ws.part, &go, ws.sem, m->status, PEAGLE_OP_BWD_GEMM, s,
                       w_early);
  };
  auto copy_out = [&](int M, int N, float* dst) { return launch_sum_splits(go, M, N, dst, s); };
  // D = X W^T into dst [M, N]: straight there when the contraction needs one
  // slab (the kernel leaves the finished tile in slab 0), else through the
  // partial slabs and a copy
  auto mm_into = [&](float* dst, const void* X, int ldx, const void* W, int M, int N, int Kd,
                     bool w_early = false) -> cudaError_t {
    if (gemm_out_floats(dt, M, N, Kd) == (size_t)M * N)
      return gemm_launch(dt, X, ldx, W, M, N, Kd, dst, &go, ws.sem, m->status, PEAGLE_OP_BWD_GEMM, s,
                         w_early);
    cudaError_t e = mm(X, ldx, W, M, N, Kd, w_early);
    return e == cudaSuccess ? copy_out(M, N, dst) : e;
  };

  CUDA_TRY(cudaMemsetAsync(ws.sem, 0, kGemmSemCount * sizeof(int), s));
  // ---- rows and their metadata (the forward's)
  st = cod_enqueue(n, K, seed, counts, ws.indices, ws.row_of, s);
  if (st) return st;
  TrainMetaArgs ta{};
  ta.n = n;
  ta.R = R;
  ta.K = K;
  ta.S = num_seqs;
  ta.Vt = c.target_vocab;
  ta.Vd = V;
  ta.max_pos = c.max_position;
  memcpy(ta.off, off, sizeof off);
  ta.indices = ws.indices;
  ta.position_ids = position_ids;
  ta.cu = cu_seqlens;
  ta.labels = labels;
  ta.loss_mask = loss_mask;
  ta.t2d = m->w.t2d;
  ta.row_anchor = ws.anchor;
  ta.row_depth = ws.depth;
  ta.row_pos = ws.pos;
  ta.row_start = ws.start;
  ta.row_end = ws.end;
  ta.row_label = ws.label;
  ta.status = m->status;
  CUDA_TRY(launch_train_meta(ta, s));

  // ---- forward, keeping activations. fc over the n aux rows and the
  // mask_hidden row (source row n)
  CUDA_TRY(gemm_launch(dt, aux, AHt, m->w.fc_w, n, H, AHt, ws.U, &go, ws.sem, m->status, PEAGLE_OP_BWD_GEMM,
                       s));
  FcFinishArgs fa{};
  fa.u = go;
  fa.H = H;
  fa.Vt = c.target_vocab;
  fa.tok = input_ids;
  fa.embed = m->w.embed;
  fa.g_fc = m->w.fc_norm_w;
  fa.g_in = m->layers[0].in_norm_w;
  fa.g_h = m->layers[0].hidden_norm_w;
  fa.eps = eps;
  fa.nbr = c.norm_before_residual;
  fa.x0 = ws.x0src;
  fa.resid = ws.residsrc;
  fa.hid = ws.hidsrc;
  fa.status = m->status;
  CUDA_TRY(launch_fc_finish(dt, n, fa, s));
  CUDA_TRY(gemm_launch(dt, m->w.mask_hidden, AHt, m->w.fc_w, 1, H, AHt, ws.Um, &go, ws.sem, m->status,
                       PEAGLE_OP_BWD_GEMM, s));
  fa.u = go;
  fa.tok = nullptr;
  fa.tok_const = c.ptd_token_id;
  fa.x0 = at(ws.x0src, (size_t)n * 2 * H);
  fa.resid = ws.residsrc + (size_t)n * H;
  fa.hid = ws.hidsrc + (size_t)n * H;
  CUDA_TRY(launch_fc_finish(dt, 1, fa, s));
  CUDA_TRY(launch_gather_masked(es, ws.x0src, n, R, 2 * H, ws.x0full, s));
  CUDA_TRY(launch_gather_masked(4, ws.hidsrc, n, R, H, ws.hidfull, s));
  CUDA_TRY(launch_gather_masked(4, ws.residsrc, n, R, H, ws.residfull, s));

  for (int l = 0; l < L; ++l) {
    const peagle_layer_weights& W = m->layers[l];
    const int in = l == 0 ? 2 * H : H;
    float* hstream = ws.hmid[l];   // the residual stream while the layer runs
    const bool fuse_qkv = hd == 128 && gemm_qkv_fusable(dt, R, QKV, in);
    if (fuse_qkv) {   // rotary and the bf16 q/k/v in the contraction's epilogue
      GemmEpi ep{};
      ep.op = GEMM_EPI_QKV;
      ep.nq = nq;
      ep.nkv = nkv;
      ep.max_pos = c.max_position;
      ep.row_base = 0;
      ep.rcos = m->rcos;
      ep.rsin = m->rsin;
      ep.row_pos = ws.pos;
      ep.q = ws.q[l];
      ep.k = ws.k[l];
      ep.v = ws.v[l];
      CUDA_TRY(gemm_launch_epi(dt, ws.xin[l], in, W.qkv_w, R, QKV, in, ws.part, &go, ws.sem, m->status, PEAGLE_OP_BWD_GEMM, &ep, s,
                               true));
      if (l == 0)
        CUDA_TRY(cudaMemcpyAsync(hstream, ws.residfull, (size_t)R * H * 4, cudaMemcpyDeviceToDevice, s));
    } else {
      CUDA_TRY(mm(ws.xin[l], in, W.qkv_w, R, QKV, in, true));
    }
    QkvArgs qa{};
    qa.in = go;
    qa.nq = nq;
    qa.nkv = nkv;
    qa.hd = hd;
    qa.H = H;
    qa.K = K;
    qa.mode = 0;
    qa.row0 = 0;
    qa.src0 = 0;
    qa.rcos = m->rcos;
    qa.rsin = m->rsin;
    qa.max_pos = c.max_position;
    qa.row_pos = ws.pos;
    qa.Q = ws.q[l];
    qa.Kout = ws.k[l];
    qa.Vout = ws.v[l];
    qa.status = m->status;
    if (l == 0) {   // the layer-0 residual seeds the stream
      qa.resid0 = ws.residfull;
      qa.h = hstream;
    }
    if (!fuse_qkv) CUDA_TRY(launch_qkv_finish(dt, R, qa, s));
    if (l == 0) CUDA_TRY(cudaMemcpyAsync(ws.hin[0], hstream, (size_t)R * H * 4, cudaMemcpyDeviceToDevice, s));
    else CUDA_TRY(cudaMemcpyAsync(hstream, ws.hin[l], (size_t)R * H * 4, cudaMemcpyDeviceToDevice, s));
    TrainAttnArgs aa{};
    aa.R = R;
    aa.n = n;
    aa.nq = nq;
    aa.nkv = nkv;
    aa.hd = hd;
    aa.Q = ws.q[l];
    aa.Kr = ws.k[l];
    aa.Vr = ws.v[l];
    aa.row_anchor = ws.anchor;
    aa.row_depth = ws.depth;
    aa.row_start = ws.start;
    aa.row_of = ws.row_of;
    aa.O = ws.o[l];
    aa.scale = 1.0f / sqrtf((float)hd);
    aa.status = m->status;
    aa.Vt = ws.vt;   // bf16, hd 128: the tcgen05 kernel; else mma.sync / CUDA cores
    aa.Rp = Rp;
    aa.lse2 = dt == PEAGLE_BF16 ? ws.lse2[l] : nullptr;   // the tensor-core backward rebuilds P from it
    TrainTileArgs tt{};
    tt.K = K;
    for (int d = 0; d <= K; ++d) tt.row_off[d] = off[d];
    CUDA_TRY(launch_train_attn(dt, aa, tt, -1, s));
    CUDA_TRY(mm(ws.o[l], nqhd, W.o_w, R, H, nqhd, true));
    ResidNormArgs ra{};
    ra.in = go;
    ra.H = H;
    ra.row0 = 0;
    ra.h = hstream;
    ra.gain = W.post_norm_w;
    ra.eps = eps;
    ra.y = ws.y[l];
    CUDA_TRY(launch_resid_norm(dt, R, ra, s));   // hstream = h_mid
    if (gemm_swiglu_keeps_gu(dt, R, 2 * I, H)) {
      // one contraction: the activation for the down projection and the
      // fp32 gate / up values the SwiGLU backward needs
      GemmEpi ep{};
      ep.op = GEMM_EPI_SWIGLU;
      ep.act = ws.act[l];
      ep.act_ld = I;
      ep.gu = ws.gu[l];
      ep.gu_ld = 2 * I;
      CUDA_TRY(gemm_launch_epi(dt, ws.y[l], H, W.gate_up_w, R, 2 * I, H, ws.part, &go, ws.sem, m->status,
                               PEAGLE_OP_BWD_GEMM, &ep, s, true));
    } else {
      CUDA_TRY(mm_into(ws.gu[l], ws.y[l], H, W.gate_up_w, R, 2 * I, H, true));
      CUDA_TRY(launch_swiglu(dt, GemmOut{ws.gu[l], 2 * I, 1, 0}, R, I, ws.act[l], s));
    }
    CUDA_TRY(mm(ws.act[l], I, W.down_w, R, H, I, true));
    // h_out = h_mid + down: into the next layer's input stream (or hL)
    float* hnext = (l + 1 < L) ? ws.hin[l + 1] : ws.hL;
    CUDA_TRY(cudaMemcpyAsync(hnext, hstream, (size_t)R * H * 4, cudaMemcpyDeviceToDevice, s));
    ra.in = go;
    ra.h = hnext;
    ra.gain = (l + 1 < L) ? m->layers[l + 1].in_norm_w : m->w.final_norm_w;
    ra.y = (l + 1 < L) ? ws.xin[l + 1] : ws.z;
    CUDA_TRY(launch_resid_norm(dt, R, ra, s));
  }
  // head: logits, per-row CE, the loss and its per-depth counts
  if (dt == PEAGLE_BF16) {
    // the logits (kept for the cross-entropy gradient) and each row's CE
    // and argmax partials from the contraction's epilogue, merged per row
    GemmEpi ep{};
    ep.op = GEMM_EPI_CE;
    ep.logits = ws.logits;
    ep.logits_ld = V;
    ep.p_max = ws.p_max;
    ep.p_sum = ws.p_sum;
    ep.p_lab = ws.p_lab;
    ep.p_idx = ws.p_idx;
    ep.labels = ws.label;
    CUDA_TRY(gemm_launch_epi(dt, ws.z, H, m->w.lm_head_w, R, V, H, ws.part, &go, ws.sem, m->status,
                             PEAGLE_OP_BWD_GEMM, &ep, s, true));
    CUDA_TRY(launch_ce_merge(R, gemm_col_tiles(R, V, H), 0, ws.p_max, ws.p_sum, ws.p_lab, ws.p_idx, ws.label,
                             ws.rce, ws.ram, s));
  } else {
    CUDA_TRY(mm_into(ws.logits, ws.z, H, m->w.lm_head_w, R, V, H, true));
    CUDA_TRY(launch_ce_rows(GemmOut{ws.logits, V, 1, 0}, R, V, 0, ws.label, nullptr, ws.rce, ws.ram, s));
  }
  CeReduceArgs cr{};
  cr.row_ce = ws.rce;
  cr.row_am = ws.ram;
  cr.row_label = ws.label;
  memcpy(cr.off, off, sizeof off);
  cr.K = K;
  cr.decay = depth_decay;
  cr.loss_d = ws.loss_d;
  cr.acc_d = ws.acc_d;
  cr.valid_d = ws.valid_d;
  cr.loss = loss;
  CUDA_TRY(launch_ce_reduce(cr, s));

  // ---- backward. Weight transposes W^T [in, out] (lm_head padded to Vp)
  CUDA_TRY(launch_transpose(dt, m->w.lm_head_w, V, H, H, ws.wT_lm, Vp, Vp, s));
  CUDA_TRY(launch_transpose(dt, m->w.fc_w, H, AHt, AHt, ws.wT_fc, H, H, s));
  for (int l = 0; l < L; ++l) {
    const peagle_layer_weights& W = m->layers[l];
    const int in = l == 0 ? 2 * H : H;
    CUDA_TRY(launch_transpose(dt, W.qkv_w, QKV, in, in, ws.wT_qkv[l], QKV, QKV, s));
    CUDA_TRY(launch_transpose(dt, W.o_w, H, nqhd, nqhd, ws.wT_o[l], H, H, s));
    CUDA_TRY(launch_transpose(dt, W.gate_up_w, 2 * I, H, H, ws.wT_gu[l], 2 * I, 2 * I, s));
    CUDA_TRY(launch_transpose(dt, W.down_w, H, I, I, ws.wT_down[l], H, H, s));
  }
  // gain gradients accumulate
  CUDA_TRY(cudaMemsetAsync(gout(grads->fc_norm_w), 0, (size_t)H * 4, s));
  CUDA_TRY(cudaMemsetAsync(gout(grads->final_norm_w), 0, (size_t)H * 4, s));
  for (int l = 0; l < L; ++l) {
    CUDA_TRY(cudaMemsetAsync(gout(grads->layers[l].in_norm_w), 0, (size_t)H * 4, s));
    CUDA_TRY(cudaMemsetAsync(gout(grads->layers[l].post_norm_w), 0, (size_t)H * 4, s));
    if (l == 0) CUDA_TRY(cudaMemsetAsync(gout(grads->layers[0].hidden_norm_w), 0, (size_t)H * 4, s));
  }
  // dW = dY^T X: both transposed ([out, Rp], [in, Rp]) then contracted over Rp
  // (the first out_rows rows of the [out, in] result go to dW)
  auto dweight = [&](const void* dY_es, int out, const void* X_es, int in, int rows, int rows_pad, float* dW,
                     int out_rows) -> cudaError_t {
    cudaError_t e = launch_transpose(dt, dY_es, rows, out, out, ws.ta, rows_pad, rows_pad, s);
    if (e == cudaSuccess) e = launch_transpose(dt, X_es, rows, in, in, ws.tb, rows_pad, rows_pad, s);
    if (e == cudaSuccess) e = mm_into(dW, ws.ta, rows_pad, ws.tb, out_rows, in, rows_pad);
    return e;
  };
  // cross-entropy -> logits gradient (padded to Vp columns)
  CUDA_TRY(cudaMemsetAsync(ws.dlog, 0, (size_t)R * Vp * es, s));   // the Vp - V pad columns stay 0
  CUDA_TRY(launch_ce_bwd(dt, ws.logits, R, V, ws.label, ws.depth, ws.valid_d, ws.rce, depth_decay, ws.dlog, Vp, s));
  // lm_head: dW_lm = dlogits^T z; dz = dlogits W_lm
  CUDA_TRY(dweight(ws.dlog, Vp, ws.z, H, R, Rp, gout((grads->lm_head_w)), V));
  CUDA_TRY(mm_into(ws.dh2, ws.dlog, Vp, ws.wT_lm, R, H, Vp));
  // final norm: dh = RMSNorm'(hL) dz
  CUDA_TRY(launch_rms_bwd(4, ws.hL, H, m->w.final_norm_w, gbf, ws.dh2, H, nullptr, 0, ws.dh, H, ws.rrow, R, H, eps, s));
  CUDA_TRY(launch_gain_grad(4, ws.hL, H, nullptr, 0, 0, ws.dh2, H, ws.rrow, R, H, const_cast<float*>(
                            static_cast<const float*>(grads->final_norm_w)), s));

  for (int l = L - 1; l >= 0; --l) {
    const peagle_layer_weights& W = m->layers[l];
    const peagle_layer_weights& G = grads->layers[l];
    const int in = l == 0 ? 2 * H : H;
    // MLP: dact = dh W_down; dW_down = dh^T act
    CUDA_TRY(launch_cast(dt, ws.dh, ws.gcast, (long long)R * H, s));
    CUDA_TRY(dweight(ws.gcast, H, ws.act[l], I, R, Rp, gout((G.down_w)), H));
    CUDA_TRY(mm(ws.gcast, H, ws.wT_down[l], R, I, H));
    CUDA_TRY(launch_swiglu_bwd(dt, ws.gu[l], ws.part, R, I, ws.dgu, s));
    // dy = dgu W_gu; dW_gu = dgu^T y
    CUDA_TRY(dweight(ws.dgu, 2 * I, ws.y[l], H, R, Rp, gout((G.gate_up_w)), 2 * I));
    CUDA_TRY(mm_into(ws.dh2, ws.dgu, 2 * I, ws.wT_gu[l], R, H, 2 * I));
    // post-attention norm: dh_mid = dh + RMSNorm'(h_mid) dy
    CUDA_TRY(launch_rms_bwd(4, ws.hmid[l], H, W.post_norm_w, gbf, ws.dh2, H, ws.dh, H, ws.dh, H, ws.rrow, R, H, eps, s));
    CUDA_TRY(launch_gain_grad(4, ws.hmid[l], H, nullptr, 0, 0, ws.dh2, H, ws.rrow, R, H,
                              gout((G.post_norm_w)), s));
    // O projection: do = dh_mid W_o; dW_o = dh_mid^T o
    CUDA_TRY(launch_cast(dt, ws.dh, ws.gcast, (long long)R * H, s));
    CUDA_TRY(dweight(ws.gcast, H, ws.o[l], nqhd, R, Rp, gout((G.o_w)), H));
    CUDA_TRY(mm(ws.gcast, H, ws.wT_o[l], R, nqhd, H));
    CUDA_TRY(launch_cast(dt, ws.part, ws.gcast, (long long)R * nqhd, s));   // do, model dtype
    // attention and RoPE
    AttnBwdArgs ab{};
    ab.R = R;
    ab.n = n;
    ab.K = K;
    ab.nq = nq;
    ab.nkv = nkv;
    ab.hd = hd;
    ab.Q = ws.q[l];
    ab.Kr = ws.k[l];
    ab.Vr = ws.v[l];
    ab.O = ws.o[l];
    ab.dO = ws.gcast;
    ab.row_anchor = ws.anchor;
    ab.row_depth = ws.depth;
    ab.row_start = ws.start;
    ab.row_end = ws.end;
    ab.row_of = ws.row_of;
    memcpy(ab.off, off, sizeof off);
    ab.scale = 1.0f / sqrtf((float)hd);
    ab.dQ = ws.dQ;
    ab.dK = ws.dK;
    ab.dV = ws.dV;
    ab.lse = ws.lse;
    ab.Dv = ws.Dv;
    ab.lse2 = dt == PEAGLE_BF16 ? ws.lse2[l] : nullptr;
    CUDA_TRY(launch_attn_bwd(dt, ab, s));
    CUDA_TRY(launch_rope_bwd(dt, hd, ws.dQ, ws.dK, ws.dV, ws.pos, m->rcos, m->rsin, c.max_position, R, nq, nkv, ws.dqkv,
                             s));
    // QKV: dxin = dqkv W_qkv; dW_qkv = dqkv^T xin
    CUDA_TRY(dweight(ws.dqkv, QKV, ws.xin[l], in, R, Rp, gout((G.qkv_w)), QKV));
    CUDA_TRY(mm_into(ws.dbig, ws.dqkv, QKV, ws.wT_qkv[l], R, in, QKV));
    if (l > 0) {   // input norm: dh = dh_mid + RMSNorm'(h_in) dxin
      CUDA_TRY(launch_rms_bwd(4, ws.hin[l], H, W.in_norm_w, gbf, ws.dbig, H, ws.dh, H, ws.dh, H, ws.rrow, R, H, eps, s));
      CUDA_TRY(launch_gain_grad(4, ws.hin[l], H, nullptr, 0, 0, ws.dbig, H, ws.rrow, R, H,
                                gout((G.in_norm_w)), s));
    } else {
      // layer-0 input [RMSNorm_in(E[tok]) ; RMSNorm_h(hid)], residual = the
      // normed hidden (norm_before_residual) or hid itself
      CUDA_TRY(launch_rms_of_rows(es, m->w.embed, H, input_ids, n, c.ptd_token_id, R, H, eps, ws.rrow2, s));
      CUDA_TRY(launch_gain_grad(es, m->w.embed, H, input_ids, n, c.ptd_token_id, ws.dbig, 2 * H, ws.rrow2, R, H,
                                gout((G.in_norm_w)), s));
      const float* dhn = ws.dbig + H;   // row stride 2H
      if (c.norm_before_residual)   // d(hn) total = dxin's hidden half + the residual's gradient
        CUDA_TRY(launch_add_rows(dhn, 2 * H, ws.dh, H, ws.dh2, H, R, H, s));
      const float* dtot = c.norm_before_residual ? ws.dh2 : dhn;
      const int ldt = c.norm_before_residual ? H : 2 * H;
      CUDA_TRY(launch_rms_bwd(4, ws.hidfull, H, W.hidden_norm_w, gbf, dtot, ldt, c.norm_before_residual ? nullptr : ws.dh,
                              H, ws.dhid, H, ws.rrow, R, H, eps, s));
      CUDA_TRY(launch_gain_grad(4, ws.hidfull, H, nullptr, 0, 0, dtot, ldt, ws.rrow, R, H,
                                gout((G.hidden_norm_w)), s));
    }
  }
  // fc_norm and fc: depth-0 rows take u = aux W_fc^T; the masked rows share
  // u_mask = mask_hidden W_fc^T, so their hid gradients add up first
  CUDA_TRY(launch_colsum(ws.dhid, H, n, R, H, ws.dmask, s));
  CUDA_TRY(cudaMemcpyAsync(ws.dhid + (size_t)n * H, ws.dmask, (size_t)H * 4, cudaMemcpyDeviceToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(ws.dbig, ws.U, (size_t)n * H * 4, cudaMemcpyDeviceToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(ws.dbig + (size_t)n * H, ws.Um, (size_t)H * 4, cudaMemcpyDeviceToDevice, s));
  CUDA_TRY(launch_rms_bwd(4, ws.dbig, H, m->w.fc_norm_w, gbf, ws.dhid, H, nullptr, 0, ws.du, H, ws.rrow, n + 1, H, eps, s));
  CUDA_TRY(launch_gain_grad(4, ws.dbig, H, nullptr, 0, 0, ws.dhid, H, ws.rrow, n + 1, H,
                            gout((grads->fc_norm_w)), s));
  // dW_fc = [du; du_m]^T [aux; mask_hidden]; d mask_hidden = du_m W_fc
  CUDA_TRY(launch_cast(dt, ws.du, ws.gcast, (long long)(n + 1) * H, s));
  CUDA_TRY(cudaMemcpyAsync(ws.auxm, aux, (size_t)n * AHt * es, cudaMemcpyDeviceToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(at(ws.auxm, (size_t)n * AHt), m->w.mask_hidden, (size_t)AHt * es, cudaMemcpyDeviceToDevice, s));
  CUDA_TRY(dweight(ws.gcast, H, ws.auxm, AHt, n + 1, ws.np1p, gout((grads->fc_w)),
                   H));
  CUDA_TRY(mm_into(gout(grads->mask_hidden), at(ws.gcast, (size_t)n * H), H, ws.wT_fc, 1, AHt, H));
  return PEAGLE_OK;
}

peagle_status peagle_combine_depth_sums(int32_t K, double depth_decay, const double* depth_sums,
                                        float* per_depth_loss, float* per_depth_acc, int32_t* per_depth_valid,
                                        float* loss, void* stream) {
  if (K < 1 || K > 16 || !isfinite(depth_decay)) FAIL(PEAGLE_ERR_INVALID_ARG, "combine_depth_sums: K=%d", K);
  if (!depth_sums || !per_depth_loss || !per_depth_acc || !per_depth_valid || !loss)
    FAIL(PEAGLE_ERR_INVALID_ARG, "combine_depth_sums: a pointer is NULL");
  CUDA_TRY(launch_depth_sums_combine(K, depth_decay, depth_sums, per_depth_loss, per_depth_acc, per_depth_valid,
                                     loss, static_cast<cudaStream_t>(stream)));
  return PEAGLE_OK;
}

}  // extern "C"

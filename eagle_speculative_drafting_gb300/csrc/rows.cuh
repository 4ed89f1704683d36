// Argument blocks and launchers of the row-wise and attention kernels.
#pragma once
#include "common.cuh"

namespace pe {

// Rows of a decode step. Request b owns rows [base(b), base(b) + n_b + K - 1):
// its n_b new rows (context rows whose K/V are new; the last one is the
// anchor, depth 0), then its K - 1 masked rows (depths 1..K-1). In this flat
// layout ["feat(speculative) ... #2376", Equivalence to vLLM inference:
// context, then the new rows, then mask_1..mask_{K-1}] row j of request b
// attends to the cached context and to the request's rows 0..j.
// new_off == NULL is the one-anchor step: n_b = 1, base(b) = b * K.
struct DecodeRows {
  int B, K;
  const int* new_off;   // device [B+1], exclusive prefix sums of n_b, or NULL
  int total_new;        // new_off[B] (host copy)
  int max_new;          // host bound on n_b
};
__device__ __forceinline__ int dr_new(const DecodeRows& d, int b) {
  return d.new_off ? d.new_off[b + 1] - d.new_off[b] : 1;
}
__device__ __forceinline__ int dr_base(const DecodeRows& d, int b) {
  return d.new_off ? d.new_off[b] + b * (d.K - 1) : b * d.K;
}
// Whether request b's new-row range is well formed (1 <= n_b <= max_new,
// inside [0, total_new]).
__device__ __forceinline__ bool dr_valid(const DecodeRows& d, int b) {
  if (!d.new_off) return true;
  const int lo = d.new_off[b], hi = d.new_off[b + 1];
  return lo >= 0 && hi <= d.total_new && hi - lo >= 1 && hi - lo <= d.max_new;
}
// Request of row r (the largest b with base(b) <= r), and r's index within it.
__device__ __forceinline__ int dr_request(const DecodeRows& d, int r, int* j) {
  int b;
  if (!d.new_off) {
    b = r / d.K;
  } else {
    int lo = 0, hi = d.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (dr_base(d, mid) <= r) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
  }
  *j = r - dr_base(d, b);
  return b;
}

struct FcFinishArgs {
  GemmOut u;              // fc partials, row r at u.out + r * ldo
  int H, Vt;
  const int* tok;         // token per row, or NULL -> tok_const
  int tok_const;
  const void* embed;      // [Vt, H]
  const void *g_fc, *g_in, *g_h;
  float eps;
  int nbr;                // norm_before_residual
  void* x0;               // out [rows, 2H]
  float* resid;           // out [rows, H] or NULL
  float* hid;             // out [rows, H] fc_norm output, or NULL
  int* status;
};

struct QkvArgs {
  GemmOut in;             // QKV partials (rows = GEMM rows)
  int nq, nkv, hd, H;
  int mode;               // 0 GEMM row r - src0; 1 decode layer 0; 2 all masked
  int K;                  // decode depths (mode 1 and decode positions)
  int row0, src0;         // first output row of this launch; GEMM row of output row src0
  const float* mask_qkv;  // [QKV] pre-rotary q/k/v of a masked layer-0 row
  const float* resid0;    // layer-0 residual rows of GEMM rows (mode 1) or NULL
  const float* mask_resid;// layer-0 residual of a masked row
  float* h;               // residual stream to seed (layer 0) or NULL
  const float *rcos, *rsin;
  int max_pos;
  const int* anchor_pos;  // decode: position of each new row (one per request when rows.new_off is NULL)
  const int* row_pos;     // training positions per row
  DecodeRows rows;        // decode row layout (mode 1 and decode mode 0)
  void *Q, *Kout, *Vout;  // [rows, nq*hd], [rows, nkv*hd] x2
  void *kcache, *vcache;  // decode append target (layer's cache) or NULL
  const int64_t* kv_off;
  const int* kv_len;
  long long kv_cap;
  int* status;
};

struct ResidNormArgs {
  GemmOut in;             // partials, chunk-local rows
  int H;
  int row0;               // global row of chunk row 0
  float* h;               // residual stream [rows, H] (global rows)
  const void* gain;
  float eps;
  void* y;                // out normalised rows (global rows)
  int compact;            // decode final norm: write y only for each request's depth
                          // rows, at row b * K + depth (the anchor is depth 0)
  DecodeRows crows;       // the step's row layout when compact
};

struct CeReduceArgs {
  const float* row_ce;
  const int* row_am;
  const int* row_label;
  int off[17];            // depth d rows: [off[d], off[d+1])
  int K;
  double decay;
  float *loss_d, *acc_d, *loss;
  int* valid_d;
  double* sums;           // optional [3, K]: += sum CE, correct rows, labelled rows per depth
};

struct TrainMetaArgs {
  int n, R, K, S, Vt, Vd, max_pos;
  int off[17];
  const int* indices;
  const int* position_ids;
  const int* cu;
  const int* labels;
  const uint8_t* loss_mask;
  const int* t2d;
  int *row_anchor, *row_depth, *row_pos, *row_start, *row_label;
  int* row_end;           // optional: end of the row's conversation
  int* status;
};

struct CodArgs {
  int n, K;
  uint64_t seed;
  int counts[16];
  int off[17];
  int* indices;
  int* row_of;
};

// Depth-masked decode attention (split over the context) + combine.
struct DecodeAttnArgs {
  int B, K, nq, nkv, hd;
  DecodeRows rows;        // request b's rows: [base(b), base(b) + n_b + K - 1)
  int R;                  // rows of the step
  int rows_max;           // max_new + K - 1: query rows per request the partials are sized for
  const void* Q;          // [R, nq, hd]
  const void *Kc, *Vc;    // the step's rows [R, nkv, hd]
  const void *kcache, *vcache;  // [cap, nkv, hd]
  const int64_t* kv_off;
  const int* kv_len;
  long long kv_cap;
  int max_kv_len;
  int chunk, nsplit;      // context keys per split, splits per (b, kv head)
  float* part_o;          // [B, nkv, nsplit, rows_max*G, hd]
  float* part_ml;         // [B, nkv, nsplit, rows_max*G, 2]
  void* O;                // out [R, nq, hd]
  float scale;
  int* status;
};

struct TrainAttnArgs {
  int R, n, nq, nkv, hd;
  const void *Q, *Kr, *Vr;   // [R, nq|nkv, hd]
  const int *row_anchor, *row_depth, *row_start, *row_of;  // row_of [K, n]
  void* O;
  float scale;
  void* Vt;                  // bf16 scratch [nkv*hd, Rp] for V transposed (tensor-core path) or NULL
  int Rp;                    // row stride of Vt: R rounded up to 64
  int* status;
  float* lse2;               // fp32 [R, nq] or NULL: log2 of each row's softmax sum of 2^(s * scale * log2 e),
                             // i.e. the log-sum-exp in base-2 units of the scaled scores (the backward's input)
};

cudaError_t launch_rope_table(float* c, float* s, int max_pos, int hd, double theta, cudaStream_t st);
cudaError_t launch_fc_finish(int dtype, int rows, const FcFinishArgs& a, cudaStream_t st);
cudaError_t launch_qkv_finish(int dtype, int rows, const QkvArgs& a, cudaStream_t st);
cudaError_t launch_resid_norm(int dtype, int rows, const ResidNormArgs& a, cudaStream_t st);
cudaError_t launch_swiglu(int dtype, const GemmOut& in, int rows, int I, void* act, cudaStream_t st);
int lm_argmax_chunks(int V);
cudaError_t launch_lm_argmax(const GemmOut& in, int rows, int V, float* logits, float* pval, int* pidx,
                             const int* d2t, int* tokens, cudaStream_t st);
cudaError_t launch_ce_rows(const GemmOut& in, int rows, int V, int row0, const int* row_label,
                           float* logits_out, float* row_ce, int* row_am, cudaStream_t st);
cudaError_t launch_ce_reduce(const CeReduceArgs& a, cudaStream_t st);
// Per-depth means and the decay-weighted loss from summed [3, K] depth sums.
cudaError_t launch_depth_sums_combine(int K, double decay, const double* sums, float* loss_d, float* acc_d,
                                      int* valid_d, float* loss, cudaStream_t st);
cudaError_t launch_ce_merge(int rows, int part_ld, int row0, const float* p_max, const float* p_sum,
                            const float* p_lab, const int* p_idx, const int* row_label, float* row_ce, int* row_am,
                            cudaStream_t st);
cudaError_t launch_lm_argmax_final(int rows, int nchunks, const float* pval, const int* pidx, const int* d2t,
                                   int* tokens, cudaStream_t st);
cudaError_t launch_train_meta(const TrainMetaArgs& a, cudaStream_t st);
cudaError_t launch_verify(int B, int K, const int* d, const int* t, int* acc, int* next, cudaStream_t st);
struct NextContextArgs {
  int B, K;
  const int *drafts, *accept, *next, *cur_off, *cur_pos;
  int *kv_lens, *next_off, *next_tok, *next_pos;
  int* status;
};
cudaError_t launch_next_context(const NextContextArgs& a, cudaStream_t st);
cudaError_t launch_cod_select(const CodArgs& a, cudaStream_t st);
cudaError_t launch_sum_splits(const GemmOut& in, int M, int N, float* D, cudaStream_t st);

// Stochastic verification (rejection sampling) of B requests' K drafts.
struct SampleArgs {
  int B, K, V;
  const int* drafts;       // [B, K] target ids
  const float* q;          // [B, K, V] draft probabilities
  const float* p;          // [B, K+1, V] target probabilities
  const float* u;          // [B, K] acceptance uniforms in [0, 1)
  const uint32_t* draws;   // [B] uniform 32-bit draws
  int *accept, *next;      // [B]
  int* status;             // PEAGLE_DEV_BOUNDS for a draft id outside [0, V)
};
cudaError_t launch_verify_sample(const SampleArgs& a, cudaStream_t st);

void decode_attn_plan(int B, int nkv, int max_kv_len, int* chunk, int* nsplit);
cudaError_t launch_decode_attn(int dtype, const DecodeAttnArgs& a, int probe_op, cudaStream_t st);
// Query tiles of the tensor-core training attention: 64 rows of one depth.
struct TrainTileArgs {
  int K;
  int row_off[17];   // depth d rows [row_off[d], row_off[d+1])
  int tile_off[17];  // depth d tiles [tile_off[d], tile_off[d+1]) (filled by the launcher)
};
// Backward of the depth-masked training attention: a query-major pass (dQ,
// and each (row, head)'s log-sum-exp and D = dO . O) and a key-major pass
// (dK, dV) over the rows that see each key.
struct AttnBwdArgs {
  int R, n, K, nq, nkv, hd;
  const void *Q, *Kr, *Vr, *O, *dO;   // model dtype, [R, nq|nkv, hd]
  const int *row_anchor, *row_depth, *row_start, *row_end, *row_of;
  int off[17];                        // depth d rows [off[d], off[d+1])
  float scale;
  float *dQ, *dK, *dV;                // fp32 [R, nq|nkv, hd]
  float *lse, *Dv;                    // fp32 [R, nq]: log-sum-exp (natural units) and dO . O
  const float* lse2;                  // bf16 tensor-core path: the forward's base-2 log-sum-exp [R, nq], else NULL
};
cudaError_t launch_attn_bwd(int dtype, const AttnBwdArgs& a, cudaStream_t st);
// bf16 tensor-core form (needs lse2 from the forward; hd 64 or 128)
bool attn_bwd_mma_supported(int dtype, const AttnBwdArgs& a);
cudaError_t launch_attn_bwd_mma(const AttnBwdArgs& a, cudaStream_t st);
cudaError_t launch_transpose(int dtype, const void* src, int rows, int cols, int lds, void* dst, int ldd, int rows_pad,
                             cudaStream_t st);
cudaError_t launch_cast(int dtype, const float* src, void* dst, long long count, cudaStream_t st);
cudaError_t launch_gather_masked(int es, const void* src, int n, int rows, int cols, void* dst, cudaStream_t st);
cudaError_t launch_colsum(const float* src, int ld, int r0, int r1, int cols, float* dst, cudaStream_t st);
cudaError_t launch_ce_bwd(int dtype, const float* logits, int rows, int V, const int* row_label, const int* row_depth,
                          const int* valid_d, const float* row_ce, double decay, void* dlogits, int ldd,
                          cudaStream_t st);
cudaError_t launch_add_rows(const float* a, int lda, const float* b, int ldb, float* out, int ldo, int rows, int cols,
                            cudaStream_t st);
cudaError_t launch_rms_bwd(int x_es, const void* x, int ldx, const void* gain, int gain_bf16, const float* dy, int ldy,
                           const float* add, int ld_add, float* dx, int ldd, float* r_out, int rows, int H, float eps,
                           cudaStream_t st);
cudaError_t launch_gain_grad(int x_es, const void* x, int ldx, const int* map, int map_mod, int map_const, const float* dy,
                             int ldy, const float* r, int rows, int H, float* dg, cudaStream_t st);
cudaError_t launch_rms_of_rows(int x_es, const void* x, int ldx, const int* map, int map_mod, int map_const, int rows, int H,
                               float eps, float* r_out, cudaStream_t st);
cudaError_t launch_swiglu_bwd(int dtype, const float* gu, const float* dact, int rows, int I, void* dgu, cudaStream_t st);
cudaError_t launch_rope_bwd(int dtype, int hd, const float* dq, const float* dk, const float* dv, const int* row_pos,
                            const float* rcos, const float* rsin, int max_pos, int rows, int nq, int nkv, void* dqkv,
                            cudaStream_t st);

cudaError_t launch_train_attn(int dtype, const TrainAttnArgs& a, const TrainTileArgs& tt, int probe_op,
                              cudaStream_t st);
// tcgen05 training attention (bf16, hd = 128); false when it does not apply
bool train_attn_tc_supported(int dtype, const TrainAttnArgs& a);
cudaError_t launch_train_attn_tc(const TrainAttnArgs& a, const TrainTileArgs& tt, cudaStream_t st);

// Copy between mapped page-locked host memory and device memory as a
// kernel in the launch chain (dst / src: addresses the device can use).
cudaError_t launch_stage_copy(void* dst, const void* src, long long bytes, bool to_device, cudaStream_t st);

}  // namespace pe

/*
 * peagle.h -- C ABI of the P-EAGLE parallel-drafting library for GB300
 * (sm_103a). One process, one GPU.
 *
 * P-EAGLE drafts all K future tokens of an anchor in one forward pass of an
 * EAGLE-3 style draft model ("P-EAGLE" user guide, How It Works /
 * Architecture; "feat(speculative): add P-EAGLE parallel-drafting training
 * for EAGLE-3 drafts - #2376", PR description and Changelog):
 *   - the target's aux hidden states from the selected layers are
 *     concatenated and projected through fc and fc_norm;
 *   - every masked depth d >= 1 takes the learnable mask_hidden row, projected
 *     the same way, and the embedding of the reserved ptd_token_id;
 *   - rotary phases are looked up at the actual position values (anchor + d),
 *     not the sequence index (#2376, RoPE fix commit);
 *   - Llama-style decoder layers attend over the context plus each anchor's
 *     own depth chain (the diagonal-extension mask, #2376 "Equivalence to
 *     vLLM inference"); packed conversations never attend across their
 *     cu_seqlens boundaries ("P_Eagle" README, variable-length attention);
 *   - a draft-vocab lm_head and argmax run per depth.
 * Greedy verification accepts the longest prefix of drafts that matches the
 * target's argmax tokens (user guide, Inference Process). The training-shaped
 * pass keeps all n positions at depth 0 and about n*r^d (floored by
 * n*r_min) at depth d (user guide, COD Sampling) and weights the per-depth
 * cross-entropy by 0.8^d (#2376, Changelog).
 *
 * Conventions for every entry point:
 *   - The return value is a peagle_status. Nothing throws or aborts across
 *     the ABI. peagle_last_error() returns a one-line description of the last
 *     failure on the calling thread.
 *   - Arguments are validated on the host before any launch. A failed
 *     validation returns PEAGLE_ERR_INVALID_ARG (or _UNSUPPORTED) and leaves
 *     every output untouched.
 *   - Pointers marked "device" are CUDA device pointers owned by the caller;
 *     "host" pointers are ordinary host memory. Every array is contiguous and
 *     row-major. Floating-point tensors use the model's dtype (fp32 or bf16)
 *     unless the signature says float.
 *   - `stream` is a cudaStream_t (passed as void*). Work is enqueued
 *     asynchronously on it; calls return before the GPU finishes unless the
 *     comment says the call synchronizes.
 *   - Hot calls never allocate device memory: the caller passes a workspace
 *     of at least the size the matching *_workspace_size call reports, 256-byte
 *     aligned. Workspaces must not be shared by calls that may overlap on the GPU.
 *   - Faults the device detects (an index out of range, a bounded wait that
 *     ran out) set bits of the model's sticky device status word instead of
 *     trapping; read it with peagle_get_device_status.
 */
#ifndef PEAGLE_H_
#define PEAGLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum peagle_status {
  PEAGLE_OK = 0,
  PEAGLE_ERR_INVALID_ARG = 1,    /* a size, pointer, id or option is invalid */
  PEAGLE_ERR_UNSUPPORTED = 2,    /* valid, but outside what this build handles */
  PEAGLE_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
  PEAGLE_ERR_WORKSPACE = 4,      /* workspace NULL, misaligned or too small */
  PEAGLE_ERR_DEVICE = 5          /* the device status word is non-zero */
} peagle_status;

/* Bits of the sticky device status word. */
#define PEAGLE_DEV_BOUNDS  0x1   /* token id, position or KV range out of range */
#define PEAGLE_DEV_TIMEOUT 0x2   /* a bounded wait inside a kernel gave up */

typedef enum peagle_dtype { PEAGLE_F32 = 0, PEAGLE_BF16 = 1 } peagle_dtype;

/* Draft model configuration; mirrors the draft's config.json (#2376,
 * Checkpoint contract: ptd_token_id rides in config.json). */
typedef struct peagle_config {
  int32_t hidden;               /* H, draft hidden size */
  int32_t target_hidden;        /* Ht, width of one aux hidden state */
  int32_t num_aux;              /* A, aux states concatenated (3 in EAGLE-3) */
  int32_t num_layers;           /* draft decoder layers (>= 1) */
  int32_t num_q_heads;          /* nq */
  int32_t num_kv_heads;         /* nkv, nq % nkv == 0 */
  int32_t head_dim;             /* hd in {64, 128} */
  int32_t intermediate;         /* I, SwiGLU width */
  int32_t target_vocab;         /* Vt, rows of the embedding */
  int32_t draft_vocab;          /* Vd, rows of lm_head */
  int32_t ptd_token_id;         /* required, 0 <= id < Vt (#2376: no silent default) */
  int32_t norm_before_residual; /* 1 (default): layer-0 residual = normed hidden */
  int32_t max_position;         /* rows of the rotary table; positions must be < it */
  int32_t dtype;                /* peagle_dtype of weights, activations, KV cache */
  double rope_theta;            /* rotary base */
  double rms_eps;               /* RMSNorm epsilon */
} peagle_config;

/* Weights of one decoder layer, nn.Linear layout [out, in], device. */
typedef struct peagle_layer_weights {
  const void* in_norm_w;        /* [H] gain of the input RMSNorm */
  const void* hidden_norm_w;    /* [H] gain of the hidden RMSNorm; layer 0 only, else NULL */
  const void* qkv_w;            /* [(nq+2nkv)*hd, 2H] for layer 0, [(nq+2nkv)*hd, H] after;
                                   rows: q heads, then k heads, then v heads */
  const void* o_w;              /* [H, nq*hd] */
  const void* post_norm_w;      /* [H] gain of the post-attention RMSNorm */
  const void* gate_up_w;        /* [2I, H]: rows 0..I-1 gate, rows I..2I-1 up */
  const void* down_w;           /* [H, I] */
} peagle_layer_weights;

/* Model weights, device pointers borrowed by the model: they must stay valid
 * and unchanged until peagle_model_destroy. */
typedef struct peagle_weights {
  const void* embed;            /* [Vt, H] */
  const void* fc_w;             /* [H, A*Ht] */
  const void* fc_norm_w;        /* [H] */
  const void* mask_hidden;      /* [1, A*Ht] learnable placeholder (#2376, Changelog) */
  const void* final_norm_w;     /* [H] */
  const void* lm_head_w;        /* [Vd, H] draft-vocab head */
  const int32_t* d2t;           /* [Vd] draft id -> target id, or NULL = identity */
  const int32_t* t2d;           /* [Vt] target id -> draft id, -1 = not in the draft
                                   vocab (label ignored), or NULL = identity */
  const peagle_layer_weights* layers; /* HOST array of num_layers entries */
} peagle_weights;

typedef struct peagle_model peagle_model;

/* ---- library ------------------------------------------------------------ */
const char* peagle_version(void);
const char* peagle_status_string(peagle_status s);
/* One-line description of the last failure on this thread ("" if none). */
const char* peagle_last_error(void);
/* Number of kernels this library has launched in this process. */
uint64_t peagle_kernel_launches(void);

/* ---- model -------------------------------------------------------------- */
/* Validates the config, borrows the weights, allocates the model's own small
 * device state (rotary table, status word, constants, and the zeroed
 * arrival counters of the draft step's contractions, which every launch
 * leaves zero again) and precomputes what
 * every masked row shares: fc_norm(fc(mask_hidden)), the ptd embedding, the
 * layer-0 pre-rotary q/k/v and residual of a masked row (#2376, Changelog:
 * masked_projected_hidden). Synchronizes `stream` before returning. */
peagle_status peagle_model_create(const peagle_config* cfg, const peagle_weights* w,
                                  void* stream, peagle_model** out);
/* Frees what create allocated (synchronizes the device first). NULL is a no-op. */
peagle_status peagle_model_destroy(peagle_model* model);
/* Synchronizes `stream`, then copies the sticky device status word
 * (PEAGLE_DEV_* bits) to *host_status. */
peagle_status peagle_get_device_status(const peagle_model* model, void* stream,
                                       int32_t* host_status);
/* Clears the device status word and re-zeroes the model's arrival counters
 * (a launch that timed out may leave them set); enqueued on `stream`. */
peagle_status peagle_clear_device_status(const peagle_model* model, void* stream);

/* ---- draft step (decode) ------------------------------------------------ */
peagle_status peagle_draft_step_workspace_size(const peagle_model* model, int32_t B,
                                               int32_t K, int32_t max_kv_len, size_t* bytes);
/* One parallel draft step for B independent requests: all K depths of every
 * request in one pass (user guide, Inference Process step 1).
 * Row (b, d), d in [0, K), is depth d of request b (user guide: depth d
 * predicts position anchor + d):
 *   depth 0 takes anchor_tokens[b] and fc_norm(fc(aux[b])); depths >= 1 take
 *   ptd_token_id and fc_norm(fc(mask_hidden)); rotary position anchor_pos[b]+d.
 * Attention of row (b, d) at every layer reads the request's context rows
 * k_cache[l][kv_offsets[b] + t], t < kv_lens[b] (post-rotary, written by
 * earlier steps), then the chain rows (b, 0..d) of this pass.
 *   aux            device [B, A*Ht]
 *   anchor_tokens  device int32 [B], target ids < Vt
 *   anchor_pos     device int32 [B], anchor_pos[b] + K - 1 < max_position
 *   k_cache/v_cache HOST arrays of num_layers device pointers, each
 *                  [kv_capacity, nkv, hd]; rows kv_offsets[b].. belong to b
 *   kv_offsets     device int64 [B+1], kv_lens device int32 [B],
 *                  kv_lens[b] <= max_kv_len (host bound used to size the grid),
 *                  kv_offsets[b] + kv_lens[b] + append_anchor_kv <= kv_offsets[b+1]
 *                  <= kv_capacity
 *   append_anchor_kv  if 1, the anchor row's post-rotary K/V of every layer is
 *                  written to row kv_offsets[b] + kv_lens[b] (kv_lens unchanged)
 *   draft_tokens   device int32 [B, K] out: d2t(argmax over the draft vocab),
 *                  lowest index among equal maxima
 *   logits         device float [B, K, Vd] out, or NULL
 * K in [1, 16]. Violations of the device-side ranges set PEAGLE_DEV_BOUNDS
 * and the offending row is skipped. The step uses the model's arrival
 * counters: draft steps of one model must not run concurrently (enqueue them
 * on one stream, or order their streams). */
peagle_status peagle_draft_step(const peagle_model* model, int32_t B, int32_t K,
                                const void* aux, const int32_t* anchor_tokens,
                                const int32_t* anchor_pos, void* const* k_cache,
                                void* const* v_cache, const int64_t* kv_offsets,
                                const int32_t* kv_lens, int64_t kv_capacity,
                                int32_t max_kv_len, int32_t append_anchor_kv,
                                int32_t* draft_tokens, float* logits, void* workspace,
                                size_t workspace_bytes, void* stream);

/* ---- draft step over new context rows ------------------------------------ */
peagle_status peagle_draft_step_ctx_workspace_size(const peagle_model* model, int32_t B, int32_t K,
                                                   int32_t total_new, int32_t max_new,
                                                   int32_t max_kv_len, size_t* bytes);
/* One parallel draft step in which every request brings n_b >= 1 new rows:
 * the tokens that joined its sequence since the last step (the accepted
 * drafts and the target's next token: user guide, Inference Process), with
 * the target's aux hidden states. The last new row is the anchor (depth 0);
 * K - 1 masked rows follow it. In the flat layout [context, new rows,
 * mask_1..mask_{K-1}] ("feat(speculative) ... #2376", Equivalence to vLLM
 * inference) new row j attends to the cached context and new rows 0..j;
 * masked depth d attends to the context, every new row and depths 1..d. The
 * new rows' post-rotary K/V of every layer are written to cache rows
 * kv_offsets[b] + kv_lens[b] + j when append_new_kv (kv_lens unchanged: the
 * caller advances it, e.g. with peagle_next_context). With n_b = 1 this is
 * peagle_draft_step.
 *   total_new    HOST sum of n_b (= new_offsets[B]); max_new HOST bound on
 *                n_b (1..64)
 *   new_offsets  device int32 [B+1], new_offsets[0] = 0, n_b = new_offsets[b+1] -
 *                new_offsets[b] in [1, max_new]
 *   new_aux      device [total_new, A*Ht]; new_tokens, new_pos device int32
 *                [total_new] (target ids, rotary positions; masked depth d of
 *                request b is at the position of its last new row + d)
 *   caches, kv_offsets, kv_lens, kv_capacity, max_kv_len: as peagle_draft_step;
 *                kv_offsets[b] + kv_lens[b] + n_b <= kv_offsets[b+1]
 *   draft_tokens device int32 [B, K] out; logits device float [B, K, Vd] or NULL
 * A malformed new-row range sets PEAGLE_DEV_BOUNDS and the request is skipped. */
peagle_status peagle_draft_step_ctx(const peagle_model* model, int32_t B, int32_t K, int32_t total_new,
                                    int32_t max_new, const int32_t* new_offsets, const void* new_aux,
                                    const int32_t* new_tokens, const int32_t* new_pos,
                                    void* const* k_cache, void* const* v_cache,
                                    const int64_t* kv_offsets, const int32_t* kv_lens,
                                    int64_t kv_capacity, int32_t max_kv_len, int32_t append_new_kv,
                                    int32_t* draft_tokens, float* logits, void* workspace,
                                    size_t workspace_bytes, void* stream);
/* Closes the draft -> verify loop (user guide, Inference Process, steps 3-4:
 * accepted drafts are kept and the next round starts from the target's
 * token). After a peagle_draft_step_ctx whose new rows were cur_offsets /
 * cur_pos (and appended) and a verification with accept_len / next_token:
 *   kv_lens[b] += cur n_b (the appended rows are context now);
 *   the next step's rows of request b are n_b' = accept_len[b] + 1 new rows:
 *   tokens draft_tokens[b, 0..a-1] then next_token[b], at positions
 *   p + 1 .. p + a + 1 with p the position of the current anchor (the last
 *   current new row); next_offsets / next_tokens / next_pos receive them.
 * All arrays device int32: draft_tokens [B, K]; accept_len, next_token, kv_lens
 * [B]; cur_offsets, next_offsets [B+1]; cur_pos [cur total]; next_tokens,
 * next_pos [at most B*(K+1)]. One CTA; B in [0, 65536], K in [1, 16]. The
 * new total (next_offsets[B]) is on the device; read it before sizing the
 * next step. */
peagle_status peagle_next_context(int32_t B, int32_t K, const int32_t* draft_tokens,
                                  const int32_t* accept_len, const int32_t* next_token,
                                  const int32_t* cur_offsets, const int32_t* cur_pos, int32_t* kv_lens,
                                  int32_t* next_offsets, int32_t* next_tokens, int32_t* next_pos,
                                  void* stream);

/* ---- greedy verification ------------------------------------------------ */
/* accept_len[b] = the largest a <= K with draft_tokens[b, i] ==
 * target_tokens[b, i] for all i < a; next_token[b] = target_tokens[b, a]
 * (the target's correction, or its bonus token when all K match). The next
 * round starts from that token (user guide, Inference Process steps 3-4).
 *   draft_tokens device int32 [B, K]; target_tokens device int32 [B, K+1];
 *   accept_len, next_token device int32 [B]. B >= 0, K in [1, 64]. */
peagle_status peagle_verify_accept(int32_t B, int32_t K, const int32_t* draft_tokens,
                                   const int32_t* target_tokens, int32_t* accept_len,
                                   int32_t* next_token, void* stream);

/* ---- host staging inside the launch chain ------------------------------ */
/* Copies `bytes` between page-locked host memory and device memory with a
 * kernel instead of a copy-engine transfer, so that the copy joins the
 * stream's chain of programmatically dependent launches like the kernels of
 * a step: the next kernel launches while the copy runs, and a copy to the
 * device loads its source before it waits for the previous kernel (only its
 * stores wait). On GB300 the device reads and writes host memory over
 * NVLink-C2C. Serving plumbing; the pages have no counterpart for it.
 *   host   page-locked host memory mapped into the device's address space
 *          (cudaHostAlloc / cudaMallocHost, or a pinned torch tensor);
 *          anything else returns PEAGLE_ERR_INVALID_ARG and launches nothing
 *   dev    device memory
 *   bytes  >= 0; a multiple of 16 with 16-byte aligned addresses moves in
 *          16-byte vectors, anything else byte by byte
 * Ordering is the stream's, as for cudaMemcpyAsync: do not rewrite `host`
 * before a copy to the device that reads it has completed, and read a copy
 * to the host only after synchronizing the stream. One difference: a copy
 * to the device reads `host` before the previous kernel has finished, so
 * its source must not be written by an earlier kernel still in the launch
 * chain (e.g. a copy to the host into the same buffer): use separate
 * buffers for the two directions. */
peagle_status peagle_copy_to_device(void* dev, const void* host, size_t bytes, void* stream);
peagle_status peagle_copy_to_host(void* host, const void* dev, size_t bytes, void* stream);

/* ---- stochastic verification ------------------------------------------- */
/* Rejection sampling of the drafts ("P_Eagle" README, How Speculative
 * Decoding Works: accepted tokens are used, rejected ones resampled, and the
 * output is distributed as the target's), by the published speculative-
 * sampling rule (Leviathan, Kalman, Matias, ICML 2023; Chen et al. 2023):
 *   depth i keeps draft x = draft_tokens[b, i] iff
 *     fl32(accept_u[b, i] * q_i(x)) < p_i(x)          (fp32 product)
 *   accept_len[b] = number of depths kept before the first rejection;
 *   next_token[b] = a draw from max(0, p_a - q_a) at the first rejection a,
 *   or from p_K when all K are kept (the bonus token).
 * The draw is exact integer inverse-CDF: each weight (clamped to [0, 1], NaN
 * as 0) becomes W_j = floor(w_j * 2^40), S = sum W_j, T = (draws[b] * S) >> 32,
 * and the token is the smallest j whose inclusive prefix sum of W exceeds T.
 * If S == 0 the token is the lowest-index argmax of p_a.
 *   draft_tokens device int32 [B, K], target vocab ids
 *   draft_probs  device float [B, K, V]: q_i, the draft distribution of depth
 *                i over the target vocab (0 outside the draft vocab)
 *   target_probs device float [B, K+1, V]: p_i, the target's distribution at
 *                the position of depth i; row K is the bonus position
 *   accept_u     device float [B, K], uniform in [0, 1)
 *   draws        device uint32 [B], uniform 32-bit integers
 *   accept_len, next_token device int32 [B]
 * B >= 0, K in [1, 64], V in [1, 2^23]. A draft id outside [0, V) counts as
 * rejected and sets PEAGLE_DEV_BOUNDS in the library status word. */
peagle_status peagle_verify_sample(int32_t B, int32_t K, int32_t V, const int32_t* draft_tokens,
                                   const float* draft_probs, const float* target_probs,
                                   const float* accept_u, const uint32_t* draws, int32_t* accept_len,
                                   int32_t* next_token, void* stream);

/* ---- COD selection ------------------------------------------------------ */
/* Host only: counts[0] = n, counts[d] = min(counts[d-1], max(floor(n*r^d),
 * floor(n*r_min))) with r^d formed by repeated multiplication in double
 * (user guide, COD Sampling and Key Parameters). 0 < r_min <= r <= 1. */
peagle_status peagle_cod_counts(int32_t n, int32_t K, double r, double r_min,
                                int32_t* counts_host);
peagle_status peagle_cod_select_workspace_size(int32_t n, int32_t K, size_t* bytes);
/* Position i gets key_i = output i of SplitMix64 seeded with `seed` (Steele,
 * Lea, Flood, OOPSLA 2014: mix(seed + (i+1) * 0x9E3779B97F4A7C15)); keys are
 * distinct. S_d = the counts[d] positions with the smallest keys, so S_d is
 * a subset of S_{d-1}, and over random seeds each S_d is a uniform subset.
 *   counts_host  HOST int32 [K] out (as peagle_cod_counts)
 *   indices      device int32 [sum counts] out: S_0 = 0..n-1, then S_1, ...,
 *                each ascending (depth-major)
 *   row_of       device int32 [K, n] out or NULL: row_of[d*n + i] = index of
 *                position i within `indices` at depth d, or -1
 * n in [0, 2^24], K in [1, 16]. */
peagle_status peagle_cod_select(int32_t n, int32_t K, double r, double r_min,
                                uint64_t seed, int32_t* counts_host, int32_t* indices,
                                int32_t* row_of, void* workspace, size_t workspace_bytes,
                                void* stream);

/* ---- training-shaped parallel forward ----------------------------------- */
peagle_status peagle_parallel_forward_workspace_size(const peagle_model* model, int32_t n,
                                                     int32_t K, double r, double r_min,
                                                     size_t* bytes);
/* Forward of one packed sequence of n tokens split into num_seqs
 * conversations by cu_seqlens (#2376, PR description: depth 0 consumes the
 * real token and projected aux states, depths >= 1 the ptd token and
 * mask_hidden, no recurrence). Rows are depth-major: depth 0 anchors
 * 0..n-1, then the COD-kept anchors of each depth, ascending (the order of
 * peagle_cod_select's indices with the same n, K, r, r_min, seed).
 * Row (i, d) has rotary position position_ids[i] + d and attends to the
 * depth-0 rows s(i)..i of its conversation and to its own chain rows
 * (i, 1..d). Its label is labels[i+d] when i+d is inside the conversation,
 * loss_mask[i+d] != 0 (if given) and t2d maps it into the draft vocab;
 * otherwise the row has no label.
 *   aux          device [n, A*Ht]; input_ids, position_ids, labels device int32 [n]
 *   cu_seqlens   device int32 [num_seqs+1], 0 = cu[0] <= ... <= cu[num_seqs] = n
 *   loss_mask    device uint8 [n] or NULL
 * Outputs (device, float unless noted):
 *   per_depth_loss [K] mean CE over labelled rows of depth d (0 if none)
 *   per_depth_acc  [K] fraction of labelled rows whose argmax is the label
 *   per_depth_valid int32 [K] labelled rows per depth
 *   loss [1]       sum_d depth_decay^d * per_depth_loss[d]
 *   row_argmax     int32 [R] or NULL (draft-vocab argmax, lowest index on ties)
 *   row_ce         [R] or NULL (CE of the row, NaN if it has no label)
 *   logits         [R, Vd] or NULL
 *   depth_sums     double [3, K] or NULL: the sequence's sum of CE, correct
 *                  rows and labelled rows per depth are ADDED to it (see
 *                  peagle_combine_depth_sums)
 * R = sum of the COD counts. */
peagle_status peagle_parallel_forward(const peagle_model* model, int32_t n, const void* aux,
                                      const int32_t* input_ids, const int32_t* position_ids,
                                      const int32_t* cu_seqlens, int32_t num_seqs,
                                      const int32_t* labels, const uint8_t* loss_mask,
                                      int32_t K, double r, double r_min, uint64_t seed,
                                      double depth_decay, float* per_depth_loss,
                                      float* per_depth_acc, int32_t* per_depth_valid,
                                      float* loss, int32_t* row_argmax, float* row_ce,
                                      float* logits, double* depth_sums, void* workspace,
                                      size_t workspace_bytes, void* stream);
/* Data-parallel training over several packed sequences (#2376, Validation:
 * the 8-GPU run): the sequences are independent, so each rank runs its own
 * whole sequences, each call adding its per-depth sums to depth_sums, and
 * the ranks exchange those K*3 numbers in one all-reduce (sum). This call
 * turns the summed depth_sums [3, K] (row 0: sum of CE over labelled rows,
 * row 1: rows whose argmax is the label, row 2: labelled rows) into the
 * per-depth means, counts and the loss sum_d depth_decay^d * mean_d, with
 * the arithmetic of the single-sequence reduction (a depth without labelled
 * rows contributes 0). All pointers device. K in [1, 16]. */
/* ---- backward of the training-shaped forward ----------------------------- */
peagle_status peagle_parallel_backward_workspace_size(const peagle_model* model, int32_t n, int32_t K,
                                                      double r, double r_min, size_t* bytes);
/* Gradients of the training loss sum_d depth_decay^d * mean_d CE (the loss
 * of peagle_parallel_forward on the same arguments; #2376, PR description
 * and Changelog: the trainer runs the parallel masked-depth loss) with
 * respect to every weight except the token embedding (frozen: the draft
 * shares the target's). The call runs the forward again, keeping every
 * layer's activations in the workspace, then the backward: cross-entropy,
 * lm_head, final norm, each layer (MLP, post-attention norm, O projection,
 * depth-masked attention, RoPE, QKV, input norm), the layer-0 inputs, then
 * fc_norm / fc over the depth-0 rows and the shared masked row, which gives
 * mask_hidden its gradient.
 *   inputs        as peagle_parallel_forward (n >= 1)
 *   loss          device float [1] out: the loss
 *   grads         HOST struct of device float (fp32) buffers shaped like the
 *                 weights, written (not accumulated): fc_w, fc_norm_w,
 *                 mask_hidden, final_norm_w, lm_head_w and every layer's
 *                 fields (hidden_norm_w for layer 0 only); embed, d2t, t2d
 *                 are ignored and may be NULL
 * The contractions run on the library's GEMM over transposed copies; the
 * workspace holds the activations of every layer (about R * (10 H + 3 I)
 * elements per layer, plus R * Vd floats of logits). */
peagle_status peagle_parallel_backward(const peagle_model* model, int32_t n, const void* aux,
                                       const int32_t* input_ids, const int32_t* position_ids,
                                       const int32_t* cu_seqlens, int32_t num_seqs,
                                       const int32_t* labels, const uint8_t* loss_mask, int32_t K,
                                       double r, double r_min, uint64_t seed, double depth_decay,
                                       float* loss, const peagle_weights* grads, void* workspace,
                                       size_t workspace_bytes, void* stream);

peagle_status peagle_combine_depth_sums(int32_t K, double depth_decay, const double* depth_sums,
                                        float* per_depth_loss, float* per_depth_acc,
                                        int32_t* per_depth_valid, float* loss, void* stream);

/* ---- dense contraction --------------------------------------------------- */
peagle_status peagle_gemm_workspace_size(int32_t dtype, int32_t M, int32_t N, int32_t K,
                                         size_t* bytes);
/* D = X W^T accumulated and stored in float: the contraction behind every
 * projection of the draft (fc, QKV, O, gate/up, down, lm_head; user guide,
 * Architecture). X device [M, K] and W device [N, K] of `dtype` (nn.Linear
 * layout), D device float [M, N]. bf16 runs on the tcgen05 tensor cores
 * (K % 8 == 0, 16-byte aligned X and W), fp32 on the CUDA cores.
 * Asynchronous: a bounded wait that runs out inside the kernel sets
 * PEAGLE_DEV_TIMEOUT in the library status word (peagle_get_library_status)
 * and leaves D undefined.
 * Concurrency: a bf16 contraction of 129-1024 rows may cut K into slices
 * whose CTAs (at most one per SM) wait for one another to share the sum of
 * each tile. They all become resident unless other work holds SMs for the
 * whole wait bound (1 s by default, peagle_set_wait_limit_ns); a kernel on
 * another stream that does makes the call fail as above. */
peagle_status peagle_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* X,
                          const void* W, float* D, void* workspace, size_t workspace_bytes,
                          void* stream);

/* ---- dense contraction without allocation -------------------------------- */
/* peagle_gemm for callers that cannot allocate device memory. Examples:
 * serving engines whose allocator already owns the device heap; plugins
 * whose host framework forbids allocation; latency-critical loops that
 * cannot take cudaMalloc's implicit synchronisation. The pages have no
 * counterpart for this entry point.
 * Same operands and result as peagle_gemm, but the split-K partial sums and
 * tile counters live in a fixed device array inside the library: 8 MiB of
 * partial sums plus 16 KiB of counters, held on every GPU that loads the
 * library until the process exits. No workspace is taken and nothing is
 * allocated.
 *   - Contractions whose partial sums exceed the array (more than 2^21
 *     floats, e.g. a few hundred rows of a 32000-wide head) return
 *     PEAGLE_ERR_UNSUPPORTED.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current. Make that first call
 *     before any stream capture.
 *   - The looked-up address is cached per device and does not survive a
 *     device reset (cudaDeviceReset); restart the process after one.
 *   - Every call clears the counters before use. Calls share the array, so
 *     calls that may overlap on the GPU race: serialise them, e.g. on one
 *     stream.
 *   - As for peagle_gemm, a bounded wait that runs out sets
 *     PEAGLE_DEV_TIMEOUT in the library status word. */
peagle_status peagle_gemm_noalloc(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* X,
                                  const void* W, float* D, void* stream);

/* ---- checkpoint I/O ------------------------------------------------------ */
/* Where the weight buffers of a checkpoint call live. */
typedef enum peagle_memory { PEAGLE_MEM_DEVICE = 0, PEAGLE_MEM_HOST = 1 } peagle_memory;
/* Writes `dir`/config.json and `dir`/model.safetensors in the layout vLLM's
 * parallel-drafting loader reads: a standard EAGLE-3 draft checkpoint with
 * the placeholder saved under the key "mask_hidden" ([1, A*Ht]) and
 * "parallel_drafting": true plus "ptd_token_id" in config.json (#2376,
 * Checkpoint contract). Tensor names: embed_tokens.weight, fc.weight,
 * fc_norm.weight, mask_hidden, layers.<l>.{input_layernorm, hidden_norm (layer 0),
 * self_attn.{q,k,v,o}_proj, post_attention_layernorm, mlp.{gate,up,down}_proj}.weight,
 * norm.weight, lm_head.weight, d2t (int64 [Vd], target id - draft id) and t2d
 * (bool [Vt], target id in the draft vocab). The fused q/k/v and gate/up
 * matrices of peagle_layer_weights are split into their row blocks.
 *   w       the weights, in `memory` (device pointers are read with
 *           cudaMemcpyAsync on `stream`, which is synchronized); d2t / t2d
 *           may be NULL (identity)
 * The directory must exist. Host memory only is touched on the way; nothing
 * is allocated on the device. */
peagle_status peagle_checkpoint_save(const char* dir, const peagle_config* cfg, const peagle_weights* w,
                                     int32_t memory, void* stream);
/* Reads `dir`/config.json into *cfg. Requires "parallel_drafting": true and a
 * "ptd_token_id" (#2376: no silent default). The number of aux states comes
 * from num_aux_hidden_states, else the length of
 * eagle_aux_hidden_state_layer_ids, else the width of fc.weight; dtype from
 * torch_dtype (float32, else bf16); max_position from max_position_embeddings. */
peagle_status peagle_checkpoint_load_config(const char* dir, peagle_config* cfg);
/* Fills caller-owned buffers `w` (sized for *cfg, all in `memory`) from
 * `dir`/model.safetensors: every tensor must be present with the shape *cfg
 * implies; F32 and BF16 files convert to the model dtype on the host. d2t /
 * t2d are rebuilt from the stored offsets (t2d = the inverse map, checked
 * against the stored membership mask); they may be NULL only if the stored
 * map is the identity. Synchronizes `stream` (device memory). */
peagle_status peagle_checkpoint_load(const char* dir, const peagle_config* cfg, const peagle_weights* w,
                                     int32_t memory, void* stream);

/* ---- library status word -------------------------------------------------- */
/* The calls that take no model handle (peagle_gemm, peagle_gemm_noalloc)
 * report faults their kernels detect (PEAGLE_DEV_* bits) in one sticky
 * status word per device, a device variable of the library (no allocation).
 * get synchronizes `stream`, then copies the word of the current device to
 * *host_status; clear zeroes it, enqueued on `stream`. */
peagle_status peagle_get_library_status(void* stream, int32_t* host_status);
peagle_status peagle_clear_library_status(void* stream);
/* Test hook for the timeout path: every in-kernel wait of the tensor-core
 * contractions launched after this call gives up after `ns` nanoseconds
 * (default 1e9; 0 = at the first try that finds the awaited phase still
 * open) and sets PEAGLE_DEV_TIMEOUT. Process-wide. A contraction whose wait
 * gave up drains the copies and products it issued before it exits. */
peagle_status peagle_set_wait_limit_ns(uint64_t ns);

/* ---- per-kernel timing probe -------------------------------------------- */
/* Operation classes the probe can time (one class at a time). */
typedef enum peagle_op {
  PEAGLE_OP_FC = 0, PEAGLE_OP_QKV = 1, PEAGLE_OP_ATTN = 2, PEAGLE_OP_O = 3,
  PEAGLE_OP_GATE_UP = 4, PEAGLE_OP_DOWN = 5, PEAGLE_OP_LM_HEAD = 6,
  PEAGLE_OP_VERIFY = 7, PEAGLE_OP_COD = 8, PEAGLE_OP_CE = 9,
  PEAGLE_OP_BWD_GEMM = 10,   /* every contraction of peagle_parallel_backward */
  PEAGLE_OP_COUNT = 11
} peagle_op;
const char* peagle_op_name(int32_t op);
/* Starts recording a CUDA event pair around every launch of the main kernel
 * of operation `op` (the GEMM of a projection, the attention kernel, ...) on
 * the stream it runs on, for up to `capacity` launches. Process-wide. */
peagle_status peagle_probe_begin(int32_t op, int32_t capacity);
/* Synchronizes the recorded events and writes up to `capacity` per-launch
 * durations (ms) to HOST ms_out; *count = launches recorded. Ends recording. */
peagle_status peagle_probe_end(float* ms_out, int32_t capacity, int32_t* count);

#ifdef __cplusplus
}
#endif
#endif /* PEAGLE_H_ */

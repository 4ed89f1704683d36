"""Python binding of libpeagle, the GB300 (sm_103a) P-EAGLE drafting library.

Argument marshalling only: every function below forwards to the C entry
point of the same name declared in include/peagle.h. Tensors are passed as
raw device pointers (torch tensors are accepted and must already live on the
GPU); every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: importing this package fails if libpeagle.so has
not been built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpeagle.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libpeagle.so is missing at {LIB_PATH}: build it first with "
        "python -c 'import __graft_entry__ as g; g.build()'")

_lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------------ constants
PEAGLE_OK = 0
PEAGLE_ERR_INVALID_ARG = 1
PEAGLE_ERR_UNSUPPORTED = 2
PEAGLE_ERR_CUDA = 3
PEAGLE_ERR_WORKSPACE = 4
PEAGLE_ERR_DEVICE = 5
PEAGLE_DEV_BOUNDS = 0x1
PEAGLE_DEV_TIMEOUT = 0x2
PEAGLE_F32 = 0
PEAGLE_BF16 = 1
PEAGLE_MEM_DEVICE = 0
PEAGLE_MEM_HOST = 1
OPS = {"fc": 0, "qkv": 1, "attn": 2, "o_proj": 3, "gate_up": 4, "down": 5, "lm_head": 6,
       "verify": 7, "cod": 8, "ce": 9}

c_int32 = ctypes.c_int32
c_int64 = ctypes.c_int64
c_size_t = ctypes.c_size_t
c_void_p = ctypes.c_void_p
c_double = ctypes.c_double


class peagle_config(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("target_hidden", c_int32), ("num_aux", c_int32),
                ("num_layers", c_int32), ("num_q_heads", c_int32), ("num_kv_heads", c_int32),
                ("head_dim", c_int32), ("intermediate", c_int32), ("target_vocab", c_int32),
                ("draft_vocab", c_int32), ("ptd_token_id", c_int32),
                ("norm_before_residual", c_int32), ("max_position", c_int32), ("dtype", c_int32),
                ("rope_theta", c_double), ("rms_eps", c_double)]


class peagle_layer_weights(ctypes.Structure):
    _fields_ = [("in_norm_w", c_void_p), ("hidden_norm_w", c_void_p), ("qkv_w", c_void_p),
                ("o_w", c_void_p), ("post_norm_w", c_void_p), ("gate_up_w", c_void_p),
                ("down_w", c_void_p)]


class peagle_weights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("fc_w", c_void_p), ("fc_norm_w", c_void_p),
                ("mask_hidden", c_void_p), ("final_norm_w", c_void_p), ("lm_head_w", c_void_p),
                ("d2t", c_void_p), ("t2d", c_void_p),
                ("layers", ctypes.POINTER(peagle_layer_weights))]


def _sig(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_sig("peagle_version", ctypes.c_char_p)
_sig("peagle_status_string", ctypes.c_char_p, c_int32)
_sig("peagle_last_error", ctypes.c_char_p)
_sig("peagle_kernel_launches", ctypes.c_uint64)
_sig("peagle_model_create", c_int32, ctypes.POINTER(peagle_config), ctypes.POINTER(peagle_weights),
     c_void_p, ctypes.POINTER(c_void_p))
_sig("peagle_model_destroy", c_int32, c_void_p)
_sig("peagle_get_device_status", c_int32, c_void_p, c_void_p, ctypes.POINTER(c_int32))
_sig("peagle_clear_device_status", c_int32, c_void_p, c_void_p)
_sig("peagle_draft_step_workspace_size", c_int32, c_void_p, c_int32, c_int32, c_int32,
     ctypes.POINTER(c_size_t))
_sig("peagle_draft_step", c_int32, c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
     ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p), c_void_p, c_void_p, c_int64, c_int32,
     c_int32, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p)
_sig("peagle_draft_step_ctx_workspace_size", c_int32, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32,
     ctypes.POINTER(c_size_t))
_sig("peagle_draft_step_ctx", c_int32, c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p,
     c_void_p, c_void_p, ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p), c_void_p, c_void_p, c_int64,
     c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p)
_sig("peagle_next_context", c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p)
_sig("peagle_verify_accept", c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
     c_void_p)
_sig("peagle_copy_to_device", c_int32, c_void_p, c_void_p, c_size_t, c_void_p)
_sig("peagle_copy_to_host", c_int32, c_void_p, c_void_p, c_size_t, c_void_p)
_sig("peagle_verify_sample", c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
     c_void_p, c_void_p, c_void_p, c_void_p)
_sig("peagle_cod_counts", c_int32, c_int32, c_int32, c_double, c_double, ctypes.POINTER(c_int32))
_sig("peagle_cod_select_workspace_size", c_int32, c_int32, c_int32, ctypes.POINTER(c_size_t))
_sig("peagle_cod_select", c_int32, c_int32, c_int32, c_double, c_double, ctypes.c_uint64,
     ctypes.POINTER(c_int32), c_void_p, c_void_p, c_void_p, c_size_t, c_void_p)
_sig("peagle_parallel_forward_workspace_size", c_int32, c_void_p, c_int32, c_int32, c_double,
     c_double, ctypes.POINTER(c_size_t))
_sig("peagle_parallel_forward", c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
     c_int32, c_void_p, c_void_p, c_int32, c_double, c_double, ctypes.c_uint64, c_double,
     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
     c_size_t, c_void_p)
_sig("peagle_parallel_backward_workspace_size", c_int32, c_void_p, c_int32, c_int32, c_double, c_double,
     ctypes.POINTER(c_size_t))
_sig("peagle_parallel_backward", c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
     c_void_p, c_void_p, c_int32, c_double, c_double, ctypes.c_uint64, c_double, c_void_p,
     ctypes.POINTER(peagle_weights), c_void_p, c_size_t, c_void_p)
_sig("peagle_combine_depth_sums", c_int32, c_int32, c_double, c_void_p, c_void_p, c_void_p, c_void_p,
     c_void_p, c_void_p)
_sig("peagle_gemm_workspace_size", c_int32, c_int32, c_int32, c_int32, c_int32,
     ctypes.POINTER(c_size_t))
_sig("peagle_gemm", c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
     c_void_p, c_size_t, c_void_p)
_sig("peagle_gemm_noalloc", c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p,
     c_void_p, c_void_p)
_sig("peagle_checkpoint_save", c_int32, ctypes.c_char_p, ctypes.POINTER(peagle_config),
     ctypes.POINTER(peagle_weights), c_int32, c_void_p)
_sig("peagle_checkpoint_load_config", c_int32, ctypes.c_char_p, ctypes.POINTER(peagle_config))
_sig("peagle_checkpoint_load", c_int32, ctypes.c_char_p, ctypes.POINTER(peagle_config),
     ctypes.POINTER(peagle_weights), c_int32, c_void_p)
_sig("peagle_get_library_status", c_int32, c_void_p, ctypes.POINTER(c_int32))
_sig("peagle_clear_library_status", c_int32, c_void_p)
_sig("peagle_set_wait_limit_ns", c_int32, ctypes.c_uint64)
_sig("peagle_op_name", ctypes.c_char_p, c_int32)
_sig("peagle_probe_begin", c_int32, c_int32, c_int32)
_sig("peagle_probe_end", c_int32, ctypes.POINTER(ctypes.c_float), c_int32, ctypes.POINTER(c_int32))


class PeagleError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.peagle_last_error().decode()
        super().__init__(f"{where}: {_lib.peagle_status_string(status).decode()} ({status}): {msg}")


def _check(status, where):
    if status != PEAGLE_OK:
        raise PeagleError(status, where)


def ptr(x):
    """Address of a torch tensor (device or host), a numpy array (host), an
    int, or None (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


# --------------------------------------------------------------- the ABI calls
def peagle_version():
    return _lib.peagle_version().decode()


def peagle_last_error():
    return _lib.peagle_last_error().decode()


def peagle_kernel_launches():
    return int(_lib.peagle_kernel_launches())


def peagle_model_create(cfg: peagle_config, weights: peagle_weights, stream=None):
    h = c_void_p()
    _check(_lib.peagle_model_create(ctypes.byref(cfg), ctypes.byref(weights), _stream(stream),
                                    ctypes.byref(h)), "peagle_model_create")
    return h.value


def peagle_model_destroy(model):
    _check(_lib.peagle_model_destroy(model), "peagle_model_destroy")


def peagle_get_device_status(model, stream=None):
    v = c_int32()
    _check(_lib.peagle_get_device_status(model, _stream(stream), ctypes.byref(v)),
           "peagle_get_device_status")
    return v.value


def peagle_clear_device_status(model, stream=None):
    _check(_lib.peagle_clear_device_status(model, _stream(stream)), "peagle_clear_device_status")


def peagle_draft_step_workspace_size(model, B, K, max_kv_len):
    n = c_size_t()
    _check(_lib.peagle_draft_step_workspace_size(model, B, K, max_kv_len, ctypes.byref(n)),
           "peagle_draft_step_workspace_size")
    return n.value


def peagle_draft_step(model, B, K, aux, anchor_tokens, anchor_pos, k_cache, v_cache, kv_offsets,
                      kv_lens, kv_capacity, max_kv_len, append_anchor_kv, draft_tokens, logits,
                      workspace, workspace_bytes, stream=None):
    L = len(k_cache)
    karr = (c_void_p * L)(*[ptr(t) for t in k_cache])
    varr = (c_void_p * L)(*[ptr(t) for t in v_cache])
    _check(_lib.peagle_draft_step(model, B, K, ptr(aux), ptr(anchor_tokens), ptr(anchor_pos), karr,
                                  varr, ptr(kv_offsets), ptr(kv_lens), kv_capacity, max_kv_len,
                                  int(append_anchor_kv), ptr(draft_tokens), ptr(logits),
                                  ptr(workspace), workspace_bytes, _stream(stream)),
           "peagle_draft_step")


def peagle_draft_step_ctx_workspace_size(model, B, K, total_new, max_new, max_kv_len):
    n = c_size_t()
    _check(_lib.peagle_draft_step_ctx_workspace_size(model, B, K, total_new, max_new, max_kv_len,
                                                     ctypes.byref(n)), "peagle_draft_step_ctx_workspace_size")
    return n.value


def peagle_draft_step_ctx(model, B, K, total_new, max_new, new_offsets, new_aux, new_tokens, new_pos, k_cache,
                          v_cache, kv_offsets, kv_lens, kv_capacity, max_kv_len, append_new_kv, draft_tokens,
                          logits, workspace, workspace_bytes, stream=None):
    L = len(k_cache)
    karr = (c_void_p * L)(*[ptr(t) for t in k_cache])
    varr = (c_void_p * L)(*[ptr(t) for t in v_cache])
    _check(_lib.peagle_draft_step_ctx(model, B, K, total_new, max_new, ptr(new_offsets), ptr(new_aux),
                                      ptr(new_tokens), ptr(new_pos), karr, varr, ptr(kv_offsets), ptr(kv_lens),
                                      kv_capacity, max_kv_len, int(append_new_kv), ptr(draft_tokens), ptr(logits),
                                      ptr(workspace), workspace_bytes, _stream(stream)), "peagle_draft_step_ctx")


def peagle_next_context(B, K, draft_tokens, accept_len, next_token, cur_offsets, cur_pos, kv_lens, next_offsets,
                        next_tokens, next_pos, stream=None):
    _check(_lib.peagle_next_context(B, K, ptr(draft_tokens), ptr(accept_len), ptr(next_token), ptr(cur_offsets),
                                    ptr(cur_pos), ptr(kv_lens), ptr(next_offsets), ptr(next_tokens), ptr(next_pos),
                                    _stream(stream)), "peagle_next_context")


def peagle_verify_accept(B, K, draft_tokens, target_tokens, accept_len, next_token, stream=None):
    _check(_lib.peagle_verify_accept(B, K, ptr(draft_tokens), ptr(target_tokens), ptr(accept_len),
                                     ptr(next_token), _stream(stream)), "peagle_verify_accept")


def peagle_copy_to_device(dev, host, nbytes, stream=None):
    _check(_lib.peagle_copy_to_device(ptr(dev), ptr(host), nbytes, _stream(stream)), "peagle_copy_to_device")


def peagle_copy_to_host(host, dev, nbytes, stream=None):
    _check(_lib.peagle_copy_to_host(ptr(host), ptr(dev), nbytes, _stream(stream)), "peagle_copy_to_host")


def peagle_verify_sample(B, K, V, draft_tokens, draft_probs, target_probs, accept_u, draws, accept_len,
                         next_token, stream=None):
    _check(_lib.peagle_verify_sample(B, K, V, ptr(draft_tokens), ptr(draft_probs), ptr(target_probs),
                                     ptr(accept_u), ptr(draws), ptr(accept_len), ptr(next_token),
                                     _stream(stream)), "peagle_verify_sample")


def peagle_cod_counts(n, K, r, r_min):
    out = (c_int32 * K)()
    _check(_lib.peagle_cod_counts(n, K, r, r_min, out), "peagle_cod_counts")
    return list(out)


def peagle_cod_select_workspace_size(n, K):
    s = c_size_t()
    _check(_lib.peagle_cod_select_workspace_size(n, K, ctypes.byref(s)),
           "peagle_cod_select_workspace_size")
    return s.value


def peagle_cod_select(n, K, r, r_min, seed, indices, row_of=None, workspace=None,
                      workspace_bytes=0, stream=None):
    counts = (c_int32 * K)()
    _check(_lib.peagle_cod_select(n, K, r, r_min, seed & ((1 << 64) - 1), counts, ptr(indices),
                                  ptr(row_of), ptr(workspace), workspace_bytes, _stream(stream)),
           "peagle_cod_select")
    return list(counts)


def peagle_parallel_forward_workspace_size(model, n, K, r, r_min):
    s = c_size_t()
    _check(_lib.peagle_parallel_forward_workspace_size(model, n, K, r, r_min, ctypes.byref(s)),
           "peagle_parallel_forward_workspace_size")
    return s.value


def peagle_parallel_forward(model, n, aux, input_ids, position_ids, cu_seqlens, num_seqs, labels,
                            loss_mask, K, r, r_min, seed, depth_decay, per_depth_loss,
                            per_depth_acc, per_depth_valid, loss, row_argmax, row_ce, logits,
                            workspace, workspace_bytes, stream=None, depth_sums=None):
    _check(_lib.peagle_parallel_forward(
        model, n, ptr(aux), ptr(input_ids), ptr(position_ids), ptr(cu_seqlens), num_seqs,
        ptr(labels), ptr(loss_mask), K, r, r_min, seed & ((1 << 64) - 1), depth_decay,
        ptr(per_depth_loss), ptr(per_depth_acc), ptr(per_depth_valid), ptr(loss), ptr(row_argmax),
        ptr(row_ce), ptr(logits), ptr(depth_sums), ptr(workspace), workspace_bytes, _stream(stream)),
        "peagle_parallel_forward")


def peagle_parallel_backward_workspace_size(model, n, K, r, r_min):
    s = c_size_t()
    _check(_lib.peagle_parallel_backward_workspace_size(model, n, K, r, r_min, ctypes.byref(s)),
           "peagle_parallel_backward_workspace_size")
    return s.value


def peagle_parallel_backward(model, n, aux, input_ids, position_ids, cu_seqlens, num_seqs, labels, loss_mask, K,
                             r, r_min, seed, depth_decay, loss, grads, workspace, workspace_bytes, stream=None):
    _check(_lib.peagle_parallel_backward(
        model, n, ptr(aux), ptr(input_ids), ptr(position_ids), ptr(cu_seqlens), num_seqs, ptr(labels),
        ptr(loss_mask), K, r, r_min, seed & ((1 << 64) - 1), depth_decay, ptr(loss), ctypes.byref(grads),
        ptr(workspace), workspace_bytes, _stream(stream)), "peagle_parallel_backward")


def peagle_combine_depth_sums(K, depth_decay, depth_sums, per_depth_loss, per_depth_acc, per_depth_valid,
                              loss, stream=None):
    _check(_lib.peagle_combine_depth_sums(K, depth_decay, ptr(depth_sums), ptr(per_depth_loss),
                                          ptr(per_depth_acc), ptr(per_depth_valid), ptr(loss),
                                          _stream(stream)), "peagle_combine_depth_sums")


def peagle_gemm_workspace_size(dtype, M, N, K):
    s = c_size_t()
    _check(_lib.peagle_gemm_workspace_size(dtype, M, N, K, ctypes.byref(s)),
           "peagle_gemm_workspace_size")
    return s.value


def peagle_gemm(dtype, M, N, K, X, W, D, workspace, workspace_bytes, stream=None):
    _check(_lib.peagle_gemm(dtype, M, N, K, ptr(X), ptr(W), ptr(D), ptr(workspace),
                            workspace_bytes, _stream(stream)), "peagle_gemm")


def peagle_gemm_noalloc(dtype, M, N, K, X, W, D, stream=None):
    _check(_lib.peagle_gemm_noalloc(dtype, M, N, K, ptr(X), ptr(W), ptr(D), _stream(stream)),
           "peagle_gemm_noalloc")


def _stream_or_null(stream, memory):
    # host-memory checkpoint calls make no CUDA call and need no stream
    return None if memory == PEAGLE_MEM_HOST and stream is None else _stream(stream)


def peagle_checkpoint_save(directory, cfg, weights, memory=PEAGLE_MEM_DEVICE, stream=None):
    _check(_lib.peagle_checkpoint_save(os.fsencode(directory), ctypes.byref(cfg), ctypes.byref(weights), memory,
                                       _stream_or_null(stream, memory)), "peagle_checkpoint_save")


def peagle_checkpoint_load_config(directory):
    cfg = peagle_config()
    _check(_lib.peagle_checkpoint_load_config(os.fsencode(directory), ctypes.byref(cfg)),
           "peagle_checkpoint_load_config")
    return cfg


def peagle_checkpoint_load(directory, cfg, weights, memory=PEAGLE_MEM_DEVICE, stream=None):
    _check(_lib.peagle_checkpoint_load(os.fsencode(directory), ctypes.byref(cfg), ctypes.byref(weights), memory,
                                       _stream_or_null(stream, memory)), "peagle_checkpoint_load")


def peagle_get_library_status(stream=None):
    v = c_int32()
    _check(_lib.peagle_get_library_status(_stream(stream), ctypes.byref(v)), "peagle_get_library_status")
    return v.value


def peagle_clear_library_status(stream=None):
    _check(_lib.peagle_clear_library_status(_stream(stream)), "peagle_clear_library_status")


def peagle_set_wait_limit_ns(ns):
    _check(_lib.peagle_set_wait_limit_ns(int(ns)), "peagle_set_wait_limit_ns")


def peagle_op_name(op):
    return _lib.peagle_op_name(op).decode()


def peagle_probe_begin(op, capacity):
    _check(_lib.peagle_probe_begin(op, capacity), "peagle_probe_begin")


def peagle_probe_end(capacity):
    buf = (ctypes.c_float * max(1, capacity))()
    n = c_int32()
    _check(_lib.peagle_probe_end(buf, capacity, ctypes.byref(n)), "peagle_probe_end")
    return [buf[i] for i in range(min(n.value, capacity))]


from .model import Model, make_config  # noqa: E402  (convenience wrapper over the calls above)

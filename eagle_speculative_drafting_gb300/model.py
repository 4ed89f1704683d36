"""Convenience handle over the C ABI: keeps the weight tensors alive, builds
the config/weight structs, and hands out workspaces from PyTorch's device
allocator. It only marshals arguments; the calls themselves are the ABI
functions of the package."""
import ctypes

import torch

from . import (PEAGLE_BF16, PEAGLE_F32, peagle_config, peagle_layer_weights, peagle_weights,
               peagle_model_create, peagle_model_destroy, peagle_draft_step,
               peagle_draft_step_workspace_size, peagle_parallel_forward,
               peagle_parallel_forward_workspace_size, ptr)


def make_config(hidden, target_hidden, num_aux, num_layers, num_q_heads, num_kv_heads, head_dim,
                intermediate, target_vocab, draft_vocab, ptd_token_id, dtype,
                norm_before_residual=1, max_position=16384, rope_theta=5e5, rms_eps=1e-5):
    return peagle_config(hidden, target_hidden, num_aux, num_layers, num_q_heads, num_kv_heads,
                         head_dim, intermediate, target_vocab, draft_vocab, ptd_token_id,
                         int(norm_before_residual), max_position,
                         PEAGLE_BF16 if dtype in ("bf16", PEAGLE_BF16) else PEAGLE_F32,
                         float(rope_theta), float(rms_eps))


def weights_struct(weights: dict):
    """peagle_weights over a dict of buffers (torch tensors or numpy arrays,
    all in one kind of memory) named like the struct's fields;
    ``weights["layers"]`` is a list of per-layer dicts. Returns the struct and
    the per-layer array it points to (keep both alive)."""
    Ls = weights["layers"]
    layers = (peagle_layer_weights * len(Ls))(*[
        peagle_layer_weights(ptr(L["in_norm_w"]), ptr(L.get("hidden_norm_w")), ptr(L["qkv_w"]),
                             ptr(L["o_w"]), ptr(L["post_norm_w"]), ptr(L["gate_up_w"]),
                             ptr(L["down_w"])) for L in Ls])
    w = peagle_weights(ptr(weights.get("embed")), ptr(weights["fc_w"]), ptr(weights["fc_norm_w"]),
                       ptr(weights["mask_hidden"]), ptr(weights["final_norm_w"]),
                       ptr(weights["lm_head_w"]), ptr(weights.get("d2t")), ptr(weights.get("t2d")),
                       ctypes.cast(layers, ctypes.POINTER(peagle_layer_weights)))
    return w, layers


def weight_shapes(cfg: peagle_config) -> dict:
    """Shape of every weight buffer a config implies (same keys as
    weights_struct; d2t / t2d are int32)."""
    H, A, Ht, I = cfg.hidden, cfg.num_aux, cfg.target_hidden, cfg.intermediate
    qkv = (cfg.num_q_heads + 2 * cfg.num_kv_heads) * cfg.head_dim
    out = {"embed": (cfg.target_vocab, H), "fc_w": (H, A * Ht), "fc_norm_w": (H,),
           "mask_hidden": (1, A * Ht), "final_norm_w": (H,), "lm_head_w": (cfg.draft_vocab, H),
           "d2t": (cfg.draft_vocab,), "t2d": (cfg.target_vocab,), "layers": []}
    for l in range(cfg.num_layers):
        out["layers"].append({
            "in_norm_w": (H,), "hidden_norm_w": (H,) if l == 0 else None,
            "qkv_w": (qkv, 2 * H if l == 0 else H), "o_w": (H, cfg.num_q_heads * cfg.head_dim),
            "post_norm_w": (H,), "gate_up_w": (2 * I, H), "down_w": (H, I)})
    return out


def load_checkpoint(directory, stream=None):
    """Reads a P-EAGLE draft checkpoint (config.json + model.safetensors) into
    fresh device tensors and creates the model over them."""
    import torch
    from . import peagle_checkpoint_load, peagle_checkpoint_load_config
    cfg = peagle_checkpoint_load_config(directory)
    dt = torch.bfloat16 if cfg.dtype == PEAGLE_BF16 else torch.float32
    shapes = weight_shapes(cfg)
    W = {}
    for k, v in shapes.items():
        if k == "layers":
            W["layers"] = [{kk: (None if sh is None else torch.empty(sh, dtype=dt, device="cuda"))
                            for kk, sh in L.items()} for L in v]
        elif k in ("d2t", "t2d"):
            W[k] = torch.empty(v, dtype=torch.int32, device="cuda")
        else:
            W[k] = torch.empty(v, dtype=dt, device="cuda")
    w, keep = weights_struct(W)
    peagle_checkpoint_load(directory, cfg, w, stream=stream)
    return Model(cfg, W, stream)


class Model:
    """A created draft model. ``weights`` maps the names of peagle_weights /
    peagle_layer_weights to device tensors; ``weights["layers"]`` is a list
    of per-layer dicts."""

    def __init__(self, cfg: peagle_config, weights: dict, stream=None):
        self.cfg = cfg
        self._keep = weights
        self._w, self._layers = weights_struct(weights)
        self.handle = peagle_model_create(cfg, self._w, stream)
        self._ws = {}

    def workspace(self, key, nbytes):
        buf = self._ws.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
            self._ws[key] = buf
        return buf

    def draft_step(self, K, aux, anchor_tokens, anchor_pos, k_cache, v_cache, kv_offsets, kv_lens,
                   kv_capacity, max_kv_len, append_anchor_kv=False, draft_tokens=None, logits=None,
                   stream=None):
        B = anchor_tokens.numel()
        nbytes = peagle_draft_step_workspace_size(self.handle, B, K, max_kv_len)
        ws = self.workspace(("draft", B, K, max_kv_len), nbytes)
        if draft_tokens is None:
            draft_tokens = torch.empty((B, K), dtype=torch.int32, device="cuda")
        peagle_draft_step(self.handle, B, K, aux, anchor_tokens, anchor_pos, k_cache, v_cache,
                          kv_offsets, kv_lens, kv_capacity, max_kv_len, append_anchor_kv,
                          draft_tokens, logits, ws, nbytes, stream)
        return draft_tokens

    def parallel_forward(self, aux, input_ids, position_ids, cu_seqlens, labels, K, r, r_min, seed,
                         depth_decay=0.8, loss_mask=None, row_argmax=None, row_ce=None,
                         logits=None, stream=None, depth_sums=None):
        n = input_ids.numel()
        nbytes = peagle_parallel_forward_workspace_size(self.handle, n, K, r, r_min)
        ws = self.workspace(("train", n, K, r, r_min), nbytes)
        dev = dict(device="cuda")
        out = {
            "per_depth_loss": torch.empty(K, dtype=torch.float32, **dev),
            "per_depth_acc": torch.empty(K, dtype=torch.float32, **dev),
            "per_depth_valid": torch.empty(K, dtype=torch.int32, **dev),
            "loss": torch.empty(1, dtype=torch.float32, **dev),
        }
        peagle_parallel_forward(self.handle, n, aux, input_ids, position_ids, cu_seqlens,
                                cu_seqlens.numel() - 1, labels, loss_mask, K, r, r_min, seed,
                                depth_decay, out["per_depth_loss"], out["per_depth_acc"],
                                out["per_depth_valid"], out["loss"], row_argmax, row_ce, logits,
                                ws, nbytes, stream, depth_sums=depth_sums)
        return out

    def parallel_backward(self, aux, input_ids, position_ids, cu_seqlens, labels, K, r, r_min, seed,
                          depth_decay=0.8, loss_mask=None, stream=None):
        """Loss and fp32 gradients of every trainable weight (dict named like
        the weights; grads["layers"][l][key])."""
        import torch
        from . import peagle_parallel_backward, peagle_parallel_backward_workspace_size
        n = input_ids.numel()
        nbytes = peagle_parallel_backward_workspace_size(self.handle, n, K, r, r_min)
        ws = self.workspace(("backward", n, K, r, r_min), nbytes)
        shapes = weight_shapes(self.cfg)
        f32 = dict(dtype=torch.float32, device="cuda")
        grads = {k: torch.empty(shapes[k], **f32) for k in ("fc_w", "fc_norm_w", "mask_hidden", "final_norm_w",
                                                               "lm_head_w")}
        grads["embed"] = None
        grads["layers"] = [{k: (None if sh is None else torch.empty(sh, **f32)) for k, sh in L.items()}
                           for L in shapes["layers"]]
        gw, keep = weights_struct(grads)
        loss = torch.empty(1, **f32)
        peagle_parallel_backward(self.handle, n, aux, input_ids, position_ids, cu_seqlens, cu_seqlens.numel() - 1,
                                 labels, loss_mask, K, r, r_min, seed, depth_decay, loss, gw, ws, nbytes, stream)
        return loss, grads

    def save_checkpoint(self, directory, stream=None):
        """Writes the model's weights as a vLLM-loadable P-EAGLE checkpoint."""
        from . import peagle_checkpoint_save
        peagle_checkpoint_save(directory, self.cfg, self._w, stream=stream)

    def close(self):
        if getattr(self, "handle", None):
            peagle_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

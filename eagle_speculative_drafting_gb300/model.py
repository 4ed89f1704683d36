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


class Model:
    """A created draft model. ``weights`` maps the names of peagle_weights /
    peagle_layer_weights to device tensors; ``weights["layers"]`` is a list
    of per-layer dicts."""

    def __init__(self, cfg: peagle_config, weights: dict, stream=None):
        self.cfg = cfg
        self._keep = weights
        Ls = weights["layers"]
        self._layers = (peagle_layer_weights * len(Ls))(*[
            peagle_layer_weights(ptr(L["in_norm_w"]), ptr(L.get("hidden_norm_w")), ptr(L["qkv_w"]),
                                 ptr(L["o_w"]), ptr(L["post_norm_w"]), ptr(L["gate_up_w"]),
                                 ptr(L["down_w"])) for L in Ls])
        self._w = peagle_weights(ptr(weights["embed"]), ptr(weights["fc_w"]),
                                 ptr(weights["fc_norm_w"]), ptr(weights["mask_hidden"]),
                                 ptr(weights["final_norm_w"]), ptr(weights["lm_head_w"]),
                                 ptr(weights.get("d2t")), ptr(weights.get("t2d")),
                                 ctypes.cast(self._layers, ctypes.POINTER(peagle_layer_weights)))
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
                         logits=None, stream=None):
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
                                ws, nbytes, stream)
        return out

    def close(self):
        if getattr(self, "handle", None):
            peagle_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

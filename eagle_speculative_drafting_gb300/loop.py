"""The closed draft -> verify loop of P-EAGLE decoding ("P-EAGLE" user
guide, Inference Process): draft K tokens per request in one pass, verify
them against the target, keep the accepted prefix and the target's token,
and start the next round from there.

Every step runs in the library: peagle_draft_step_ctx drafts over each
request's new rows (appending their K/V to the cache), peagle_verify_accept
or peagle_verify_sample verifies, and peagle_next_context turns the result
into the next round's new rows and advances the cache lengths. This class
only holds the device buffers and reads back the next round's row count,
which sizes the next draft step (one small device-to-host copy per round).
The target model is the caller's: it supplies the aux hidden states of the
new rows and the target tokens (or distributions) to verify against.
"""
import numpy as np
import torch

from . import (peagle_draft_step_ctx, peagle_draft_step_ctx_workspace_size, peagle_next_context,
               peagle_verify_accept)


class DraftLoop:
    """B requests, each with a cache region [kv_offsets[b], kv_offsets[b+1])
    of every layer's k_cache / v_cache holding kv_lens[b] context rows."""

    def __init__(self, model, K, k_cache, v_cache, kv_offsets, kv_lens, kv_capacity, stream=None):
        self.model, self.K = model, K
        self.k_cache, self.v_cache = k_cache, v_cache
        self.kv_offsets = kv_offsets
        self.kv_lens = kv_lens.clone()
        self.kv_capacity = int(kv_capacity)
        self.stream = stream
        self.B = kv_lens.numel()
        B = self.B
        dev = dict(device="cuda", dtype=torch.int32)
        self.max_kv_len = int(kv_lens.max().item()) if B else 0
        cap = B * (K + 1)
        self._off = [torch.zeros(B + 1, **dev), torch.zeros(B + 1, **dev)]
        self._tok = [torch.zeros(max(cap, 1), **dev), torch.zeros(max(cap, 1), **dev)]
        self._pos = [torch.zeros(max(cap, 1), **dev), torch.zeros(max(cap, 1), **dev)]
        self.cur = 0
        self.total_new, self.max_new = 0, 1
        self.drafts = torch.zeros((B, K), **dev)
        self.accept = torch.zeros(B, **dev)
        self.next = torch.zeros(B, **dev)
        self._ws = None

    # the current round's new rows (the caller's target supplies their aux)
    @property
    def new_offsets(self):
        return self._off[self.cur]

    @property
    def new_tokens(self):
        return self._tok[self.cur][:self.total_new]

    @property
    def new_pos(self):
        return self._pos[self.cur][:self.total_new]

    def start(self, tokens, positions):
        """First round: one new row per request (its last prompt token)."""
        B = self.B
        self._off[0].copy_(torch.arange(B + 1, dtype=torch.int32))
        self._tok[0][:B].copy_(torch.as_tensor(tokens, dtype=torch.int32))
        self._pos[0][:B].copy_(torch.as_tensor(positions, dtype=torch.int32))
        self.cur, self.total_new, self.max_new = 0, B, 1

    def _workspace(self, nbytes):
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        return self._ws

    def draft(self, new_aux, logits=None):
        """Drafts K tokens per request from the current new rows, whose aux
        hidden states are new_aux [total_new, A*Ht]; their K/V join the cache."""
        m = self.model
        nbytes = peagle_draft_step_ctx_workspace_size(m.handle, self.B, self.K, self.total_new, self.max_new,
                                                      self.max_kv_len)
        ws = self._workspace(nbytes)
        peagle_draft_step_ctx(m.handle, self.B, self.K, self.total_new, self.max_new, self.new_offsets, new_aux,
                              self.new_tokens, self.new_pos, self.k_cache, self.v_cache, self.kv_offsets,
                              self.kv_lens, self.kv_capacity, self.max_kv_len, 1, self.drafts, logits, ws,
                              nbytes, self.stream)
        return self.drafts

    def verify_greedy(self, target_tokens):
        """Greedy verification against target_tokens [B, K+1], then the next
        round's new rows. Returns (accept_len, next_token)."""
        peagle_verify_accept(self.B, self.K, self.drafts, target_tokens, self.accept, self.next, self.stream)
        self._advance()
        return self.accept, self.next

    def advance_after(self, accept_len, next_token):
        """The next round after a verification done elsewhere (e.g. sampled)."""
        self.accept.copy_(accept_len)
        self.next.copy_(next_token)
        self._advance()

    def _advance(self):
        nxt = 1 - self.cur
        peagle_next_context(self.B, self.K, self.drafts, self.accept, self.next, self._off[self.cur],
                            self._pos[self.cur], self.kv_lens, self._off[nxt], self._tok[nxt], self._pos[nxt],
                            self.stream)
        off = self._off[nxt].cpu().numpy()   # sizes the next draft step
        self.max_kv_len += self.max_new      # every request gained at most max_new context rows
        self.cur = nxt
        self.total_new = int(off[-1])
        self.max_new = int(np.max(np.diff(off))) if self.B else 1

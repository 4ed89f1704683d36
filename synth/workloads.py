"""The five workload shapes of the P-EAGLE drafting step.

Each entry is named by what it is. Model dimensions follow the EAGLE-3 style
draft layer the P-EAGLE pages describe (aux states from three target layers,
Llama-style decoder layers, draft-vocab head). Where a workload leaves a value
open the plainest reading is used: rope_theta 5e5, rms_eps 1e-5,
target vocab equal to draft vocab, ptd_token_id = vocab - 1.
"""
from dataclasses import dataclass, field, replace
from typing import Optional


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16"
    hidden: int                # draft hidden H
    target_hidden: int         # target hidden Ht
    num_aux: int               # A, aux layers concatenated
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    intermediate: int          # SwiGLU width I
    vocab: int                 # draft vocab = target vocab here
    K: int                     # depths
    kind: str                  # "decode" or "train"
    # decode shape
    batch: int = 0
    kv_len: int = 0            # fixed context length (0: drawn per request)
    kv_len_range: Optional[tuple] = None
    accept_p: float = 0.7      # geometric accept-length parameter (decode)
    accept_uniform: bool = False
    # train shape
    n_tokens: int = 0
    conv_len_uniform: Optional[tuple] = None
    conv_len_lognormal: Optional[tuple] = None   # (median, sigma)
    cod_r: float = 0.7
    cod_r_min: float = 0.2
    depth_decay: float = 0.8
    # shared
    rope_theta: float = 5e5
    rms_eps: float = 1e-5
    max_position: int = 16384
    seed: int = 1234

    @property
    def ptd_token_id(self) -> int:
        return self.vocab - 1

    @property
    def qkv_out(self) -> int:
        return (self.num_q_heads + 2 * self.num_kv_heads) * self.head_dim

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # fp32, one request, 64 context tokens, K=4, MHA 4x64, SwiGLU 688, vocab 1024
    "tiny_f32_decode": Workload(
        name="tiny_f32_decode", dtype="f32", hidden=256, target_hidden=256,
        num_aux=3, num_layers=1, num_q_heads=4, num_kv_heads=4, head_dim=64,
        intermediate=688, vocab=1024, K=4, kind="decode", batch=1, kv_len=64,
        accept_uniform=True, max_position=1024, seed=1235),
    # bf16 decode, one request, 2048 context, Llama-3-8B-sized draft layer
    "decode_b1_ctx2048_k4": Workload(
        name="decode_b1_ctx2048_k4", dtype="bf16", hidden=4096,
        target_hidden=4096, num_aux=3, num_layers=1, num_q_heads=32,
        num_kv_heads=8, head_dim=128, intermediate=14336, vocab=32000, K=4,
        kind="decode", batch=1, kv_len=2048, max_position=16384, seed=1236),
    # bf16 batched decode, 64 requests with ragged context U[512, 8192], K=8
    "decode_b64_ragged_k8": Workload(
        name="decode_b64_ragged_k8", dtype="bf16", hidden=4096,
        target_hidden=4096, num_aux=3, num_layers=1, num_q_heads=32,
        num_kv_heads=8, head_dim=128, intermediate=14336, vocab=32000, K=8,
        kind="decode", batch=64, kv_len_range=(512, 8192),
        max_position=16384, seed=1237),
    # bf16 training-shaped forward, one packed 4096-token sequence
    "train_n4096_k4": Workload(
        name="train_n4096_k4", dtype="bf16", hidden=2560, target_hidden=2560,
        num_aux=3, num_layers=4, num_q_heads=20, num_kv_heads=4, head_dim=128,
        intermediate=10240, vocab=32000, K=4, kind="train", n_tokens=4096,
        conv_len_uniform=(128, 1024), max_position=16384, seed=1238),
    # bf16 long-context training shape, one packed 32768-token sequence
    "train_n32768_k8": Workload(
        name="train_n32768_k8", dtype="bf16", hidden=4096, target_hidden=4096,
        num_aux=3, num_layers=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
        intermediate=14336, vocab=32000, K=8, kind="train", n_tokens=32768,
        conv_len_lognormal=(2048.0, 0.75), max_position=65536, seed=1239),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]

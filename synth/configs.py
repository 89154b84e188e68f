"""Workload shapes and the seeded input recipe for each of them.

Shapes follow the Llama configurations the pages describe: the toy 8Q/2KV
block, a small 512-wide block, the Llama-3-8B block ("LLaMA-3 8B ..." page, section 一 table), the
original LLaMA-7B MHA block ("LLaMA Architecture > Model Architecture" page, configuration table), and a 32-layer
Llama-3-8B stack decoding one token per sequence against 8192 cached positions.

Recipe (all draws from synth's counter-based generator):
  weights   ~ N(0, 0.02), no biases, stored [out, in]
  x, x_emb  ~ N(0, 1)
  KV cache  ~ N(0, 1), treated as already rotated
  gains     ones, except the small block: N(1, 0.1)
The seed of a workload is 1000 * (index + 1); tensor ids are in synth/__init__.py.
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import (BF16, F32, LAYER_STRIDE, TID_ATTN_G, TID_FFN_G, TID_FINAL_G, TID_KCACHE,
               TID_VCACHE, TID_WDOWN, TID_WGATE, TID_WK, TID_WLM, TID_WO, TID_WQ, TID_WUP,
               TID_WV, TID_X)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dtype: int                 # F32 or BF16
    B: int
    S: int
    d_model: int
    n_q: int
    n_kv: int
    head_dim: int
    d_ff: int
    theta_base: float
    eps: float
    gain_std: float = 0.0      # 0 -> gains are exactly one
    n_layers: int = 1
    t_cache: int = 0           # decode: cached positions per sequence
    vocab: int = 0             # decode: LM head rows
    w_std: float = 0.02

    @property
    def seed(self) -> int:
        return 1000 * (self.index + 1)

    @property
    def dims(self):
        return (self.B, self.S, self.d_model, self.n_q, self.n_kv, self.head_dim, self.d_ff,
                self.theta_base, self.eps)

    @property
    def tokens(self) -> int:
        return self.B * self.S


TOY = Workload("toy-fp32-B1-S4-d16-8q2kv", 0, F32, 1, 4, 16, 8, 2, 2, 48, 1e4, 1e-5)
SMALL = Workload("small-bf16-B2-S256-d512-8q2kv", 1, BF16, 2, 256, 512, 8, 2, 64, 1280, 1e4, 1e-5,
                 gain_std=0.1)
LLAMA3_8B_PREFILL = Workload("llama3-8b-block-prefill-B1-S8192", 2, BF16, 1, 8192, 4096, 32, 8, 128,
                             14336, 5e5, 1e-5)
LLAMA_7B_MHA_PREFILL = Workload("llama-7b-mha-block-prefill-B4-S2048", 3, BF16, 4, 2048, 4096, 32, 32,
                                128, 11008, 1e4, 1e-5)
LLAMA3_8B_DECODE = Workload("llama3-8b-32L-decode-B64-T8192", 4, BF16, 64, 1, 4096, 32, 8, 128, 14336,
                            5e5, 1e-5, n_layers=32, t_cache=8192, vocab=128256)

ALL = [TOY, SMALL, LLAMA3_8B_PREFILL, LLAMA_7B_MHA_PREFILL, LLAMA3_8B_DECODE]


def tensor_specs(w: Workload, layer: int = 0):
    """(name, tensor id, shape, mean, std) for one layer's inputs, in [out, in] layout."""
    d, hq, hkv, dff = w.d_model, w.n_q * w.head_dim, w.n_kv * w.head_dim, w.d_ff
    base = LAYER_STRIDE * layer
    gmean, gstd = 1.0, w.gain_std
    return [
        ("attn_norm_g", base + TID_ATTN_G, (d,), gmean, gstd),
        ("wq", base + TID_WQ, (hq, d), 0.0, w.w_std),
        ("wk", base + TID_WK, (hkv, d), 0.0, w.w_std),
        ("wv", base + TID_WV, (hkv, d), 0.0, w.w_std),
        ("wo", base + TID_WO, (d, hq), 0.0, w.w_std),
        ("ffn_norm_g", base + TID_FFN_G, (d,), gmean, gstd),
        ("w_gate", base + TID_WGATE, (dff, d), 0.0, w.w_std),
        ("w_up", base + TID_WUP, (dff, d), 0.0, w.w_std),
        ("w_down", base + TID_WDOWN, (d, dff), 0.0, w.w_std),
    ]


def x_spec(w: Workload):
    return ("x", TID_X, (w.B, w.S, w.d_model), 0.0, 1.0)


def cache_spec(w: Workload, which: str, cap: int):
    """Cache [n_layers, B, cap, n_kv, hd]; layer l is drawn as its own tensor id."""
    tid = TID_KCACHE if which == "k" else TID_VCACHE
    return (which + "_cache", tid, (w.n_layers, w.B, cap, w.n_kv, w.head_dim), 0.0, 1.0)


def final_specs(w: Workload):
    return [("final_g", TID_FINAL_G, (w.d_model,), 1.0, w.gain_std),
            ("w_lm", TID_WLM, (w.vocab, w.d_model), 0.0, w.w_std)]

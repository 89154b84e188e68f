"""GPU vs oracle parity for llama_stack_decode_step.

A small 3-layer stack is checked in full; the 32-layer Llama-3-8B stack (batch 64, 8192
cached positions, 128256-row LM head) is checked on sequences 0, 31 and 63 (decode rows are
independent across the batch, so the oracle runs those three alone).
"""
import numpy as np
import pytest

import llama_decoder_block_fwd_gb300 as L
import oracle as O
from synth import configs as C
from synth import workloads as W
from tests.helpers import assert_parity, oracle_dims, to_f64

pytestmark = pytest.mark.gpu


def _decode(wl, cap):
    import torch
    layers = [W.device_layer(wl, l) for l in range(wl.n_layers)]
    kc, vc = W.device_caches(wl, cap)
    final_g, w_lm = W.device_final(wl)
    x = W.device_x_emb(wl)
    logits = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    dims = wl.dims
    ws = torch.empty(L.llama_workspace_bytes(L.OP_STACK_DECODE_STEP, dims, wl.dtype, wl.n_layers, wl.vocab, cap),
                     dtype=torch.uint8, device="cuda")
    L.llama_stack_decode_step(dims, wl.dtype, layers, final_g, w_lm, wl.vocab, x, kc, vc, cap, wl.t_cache, logits, ws)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    return logits, kc, vc


def _oracle(wl, rows, cap):
    d = oracle_dims(wl, B=len(rows))
    fg, wlm = W.host_final(wl)
    x = W.host_x_emb(wl, rows)

    def caches(l):
        k = np.stack([W.host_cache(wl, "k", l, b, cap, wl.t_cache) for b in rows])
        v = np.stack([W.host_cache(wl, "v", l, b, cap, wl.t_cache) for b in rows])
        return k, v

    return O.stack_decode_step(x, lambda l: O.BlockWeights(**W.host_layer(wl, l)), wl.n_layers, d, wl.t_cache,
                               caches, fg, wlm)


@pytest.mark.parametrize("hd,vocab", [(128, 1000), (128, 1024), (64, 1000)])
def test_decode_small_stack_full(hd, vocab):
    # hd 128: the tensor-core decode path (split-K hi/lo GEMMs, finishers, split-K attention with a
    # ragged last tile of 301 keys); a 1024-row LM head runs on the hi/lo GEMM, a 1000-row one on
    # the generic GEMM.  hd 64: the per-block path with CUDA-core attention.
    nq, nkv = (4, 1) if hd == 128 else (8, 2)
    wl = C.Workload("small-stack", 6, C.BF16, 5, 1, 512, nq, nkv, hd, 384, 1e4, 1e-5, gain_std=0.1, n_layers=3,
                    t_cache=300, vocab=vocab)
    cap = 333
    logits, kc, vc = _decode(wl, cap)
    ref = _oracle(wl, list(range(wl.B)), cap)
    assert_parity(to_f64(logits), ref, wl.dtype, "small stack logits")
    # the new token's K/V were appended at position t_cache; other positions untouched
    for l in range(wl.n_layers):
        for b in (0, wl.B - 1):
            before = W.host_cache(wl, "k", l, b, cap, cap)
            got = to_f64(kc[l, b])
            np.testing.assert_array_equal(got[:wl.t_cache], before[:wl.t_cache])
            np.testing.assert_array_equal(got[wl.t_cache + 1:], before[wl.t_cache + 1:])
            assert not np.array_equal(got[wl.t_cache], before[wl.t_cache])


def test_decode_stack_narrow_model():
    """d_model 128 with 4 query heads and 1 KV head of 128 (so n_q * head_dim = 512 != d_model, a
    general W_O) and d_ff 256: every weight-streaming projection is one or a few 128-row tiles with
    short K ranges, and the LM head 256 rows; three layers against the oracle."""
    wl = C.Workload("tiny-stack", 8, C.BF16, 5, 1, 128, 4, 1, 128, 256, 1e4, 1e-5, gain_std=0.1, n_layers=3,
                    t_cache=200, vocab=256)
    cap = 256
    logits, _, _ = _decode(wl, cap)
    ref = _oracle(wl, list(range(wl.B)), cap)
    assert_parity(to_f64(logits), ref, wl.dtype, "tiny stack logits")


def test_decode_fp32_toy_stack():
    wl = C.Workload("toy-stack", 7, C.F32, 2, 1, 16, 8, 2, 2, 48, 1e4, 1e-5, n_layers=2, t_cache=5, vocab=11)
    cap = 8
    logits, _, _ = _decode(wl, cap)
    ref = _oracle(wl, [0, 1], cap)
    assert_parity(to_f64(logits), ref, wl.dtype, "toy stack logits")


@pytest.mark.slow
def test_decode_llama3_8b_32_layers_sampled_sequences():
    wl = C.LLAMA3_8B_DECODE
    cap = wl.t_cache + 1
    logits, _, _ = _decode(wl, cap)
    rows = [0, 31, 63]
    ref = _oracle(wl, rows, cap)
    assert_parity(to_f64(logits[rows]), ref, wl.dtype, "llama3-8b decode logits")


def test_decode_llama3_8b_32_layers_32k_context_sampled_sequences():
    """The long-context decode bench line: the 32-layer 8B stack for 16 sequences holding 32768 cached
    positions each (RoPE base 5e5, a new token at position 32768); sequences 0 and 15 against the
    oracle."""
    import dataclasses
    wl = dataclasses.replace(C.LLAMA3_8B_DECODE, B=16, t_cache=32768, name="llama3-8b-32L-decode-B16-T32768")
    cap = wl.t_cache + 1
    logits, kc, vc = _decode(wl, cap)
    got = to_f64(logits)
    del kc, vc
    rows = [0, 15]
    ref = _oracle(wl, rows, cap)
    assert_parity(got[rows], ref, wl.dtype, "llama3-8b decode logits, 32768 cached")

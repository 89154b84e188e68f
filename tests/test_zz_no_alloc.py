"""llama_gqa_attention_decode_noalloc: the one-token attention call that brings its own fixed
scratch, for callers that cannot allocate device memory where they call (an allocator that owns
all of device memory, or a loop where cudaMalloc/cudaFree would synchronise the device).

It is checked against llama_gqa_attention with a caller workspace and against the oracle's
attention on the same seeded q/k/v ("LLaMA-3 8B ...", section 4.4; "Llama Architecture ...",
Mathematical Foundations 4), within the bf16 bar the other GPU tests use, on two calls in a row with
different shapes, so that anything a call left behind in the shared scratch would show.  This file
is collected last on purpose.
"""
import ctypes

import pytest

import llama_decoder_block_fwd_gb300 as L
import oracle as O
import synth
from tests.helpers import assert_parity, dev_tensor, host_tensor, to_f64

pytestmark = pytest.mark.gpu


def _inputs(B, nq, nkv, cap, seed):
    q = dev_tensor(synth.BF16, (B, 1, nq, 128), seed, 1, 0.0, 1.0)
    k = dev_tensor(synth.BF16, (B, cap, nkv, 128), seed, 2, 0.0, 1.0)
    v = dev_tensor(synth.BF16, (B, cap, nkv, 128), seed, 3, 0.0, 1.0)
    return q, k, v


def test_noalloc_matches_workspace_call_twice_in_a_row():
    import torch
    cases = [  # (B, n_q, n_kv, capacity, pos0): a long cache first, then a shorter, wider one
        (64, 32, 8, 8193, 8192),
        (7, 16, 4, 900, 777),
    ]
    for call, (B, nq, nkv, cap, pos0) in enumerate(cases):
        q, k, v = _inputs(B, nq, nkv, cap, 4242 + call)
        dims = (B, 1, nq * 128, nq, nkv, 128, 1, 5e5, 1e-5)
        ws = torch.empty(L.llama_workspace_bytes(L.OP_GQA_ATTENTION, dims, L.BF16, kv_capacity=cap),
                         dtype=torch.uint8, device="cuda")
        o_ws = torch.empty_like(q)
        L.llama_gqa_attention(dims, L.BF16, q, k, v, cap, pos0, o_ws, ws)
        o_na = torch.full_like(q, float("nan"))
        L.llama_gqa_attention_decode_noalloc(dims, L.BF16, q, k, v, cap, pos0, o_na)
        torch.cuda.synchronize()
        assert L.llama_get_device_status() == 0
        assert_parity(to_f64(o_na), to_f64(o_ws), synth.BF16, f"noalloc call {call}")
        # the oracle on the same seeded inputs, sequence by sequence (first, middle and last of a
        # large batch; every sequence of a small one)
        seqs = sorted({0, B // 2, B - 1}) if B > 8 else list(range(B))
        row = nkv * 128
        for b in seqs:
            qh = host_tensor(synth.BF16, (1, 1, nq, 128), 4242 + call, 1, 0.0, 1.0, offset=b * nq * 128)
            kh = host_tensor(synth.BF16, (1, pos0 + 1, nkv, 128), 4242 + call, 2, 0.0, 1.0, offset=b * cap * row)
            vh = host_tensor(synth.BF16, (1, pos0 + 1, nkv, 128), 4242 + call, 3, 0.0, 1.0, offset=b * cap * row)
            ref = O.gqa_attention(qh, kh, vh, pos0)
            assert_parity(to_f64(o_na[b:b + 1]), ref, synth.BF16, f"noalloc call {call} seq {b} vs oracle")
            assert_parity(to_f64(o_ws[b:b + 1]), ref, synth.BF16, f"workspace call {call} seq {b} vs oracle")


def test_noalloc_rejects_batches_beyond_its_scratch():
    lib = L.lib()
    fake = 0x10000
    d = L.dims_of(800, 1, 32 * 128, 32, 8, 128, 1, 5e5, 1e-5)   # (800*8 + 256)*4*520 B > 12 MiB
    assert lib.llama_gqa_attention_decode_noalloc(ctypes.byref(d), L.BF16, fake, fake, fake, 10, 9, fake,
                                                  None) == 4   # LLAMA_ERR_WORKSPACE, nothing launched

"""GPU vs oracle parity for the standalone calls (llama_rmsnorm, llama_rope,
llama_gqa_attention, llama_swiglu_ffn), through the C ABI, on seeded inputs.

Sizes span several tiles and a ragged tail; edge cases: empty input, a single token,
one query against a long cache (decode shape), MHA (n_kv == n_q), pos0 > 0.
"""
import numpy as np
import pytest

import llama_decoder_block_fwd_gb300 as L
import oracle as O
import synth
from synth import configs as C
from tests.helpers import assert_parity, dev_tensor, host_tensor, to_f64

pytestmark = pytest.mark.gpu

SEED = 777


def _sync():
    import torch
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0


def test_synth_device_matches_host_bitwise():
    import torch
    for dtype in (synth.F32, synth.BF16):
        t = dev_tensor(dtype, (1 << 16) + 7, 5, 3, 0.0, 0.02, offset=12345)
        _sync()
        got = t.view(torch.int32 if dtype == synth.F32 else torch.int16).cpu().numpy()
        ref = synth.host_bits(dtype, ((1 << 16) + 7,), 5, 3, 0.0, 0.02, offset=12345)
        np.testing.assert_array_equal(got.view(ref.dtype), ref)


@pytest.mark.parametrize("dtype,rows,d", [(synth.F32, 4, 16), (synth.BF16, 512, 512), (synth.BF16, 37, 4096),
                                          (synth.F32, 9, 4096), (synth.BF16, 3, 520), (synth.F32, 5, 12),
                                          # the streaming kernel (bf16, >= 304 rows of 1024..4096): ragged
                                          # last round over the SMs, the narrowest and widest rows, and the
                                          # 8B block's 8192 x 4096 activations
                                          (synth.BF16, 305, 1024), (synth.BF16, 1001, 2056),
                                          (synth.BF16, 2000, 4096), (synth.BF16, 8192, 4096)])
def test_rmsnorm(dtype, rows, d):
    import torch
    x = dev_tensor(dtype, (rows, d), SEED, 1, 0.0, 1.0)
    g = dev_tensor(dtype, (d,), SEED, 2, 1.0, 0.1)
    y = torch.empty_like(x)
    L.llama_rmsnorm((1, rows, d, 1, 1, 2, 1, 1e4, 1e-5), dtype, x, g, y)
    _sync()
    ref = O.rmsnorm(host_tensor(dtype, (rows, d), SEED, 1, 0.0, 1.0), host_tensor(dtype, (d,), SEED, 2, 1.0, 0.1), 1e-5)
    assert_parity(to_f64(y), ref, dtype, "rmsnorm")


def test_rmsnorm_tiny_rows_eps_inside():
    import torch
    x = torch.full((2, 64), 1e-4, device="cuda")
    g = torch.ones(64, device="cuda")
    y = torch.empty_like(x)
    L.llama_rmsnorm((1, 2, 64, 1, 1, 2, 1, 1e4, 1e-5), L.F32, x, g, y)
    _sync()
    np.testing.assert_allclose(to_f64(y), 1e-4 / np.sqrt(1e-8 + 1e-5), rtol=1e-5)


@pytest.mark.parametrize("dtype,B,S,nq,nkv,hd,theta,pos0", [
    (synth.F32, 1, 4, 8, 2, 2, 1e4, 0),
    (synth.BF16, 2, 256, 8, 2, 64, 1e4, 0),
    (synth.BF16, 1, 33, 32, 8, 128, 5e5, 8160),      # positions 8160..8192
    (synth.F32, 1, 3, 2, 1, 128, 5e5, 300000),       # far positions
])
def test_rope(dtype, B, S, nq, nkv, hd, theta, pos0):
    q = dev_tensor(dtype, (B, S, nq, hd), SEED, 3, 0.0, 1.0)
    k = dev_tensor(dtype, (B, S, nkv, hd), SEED, 4, 0.0, 1.0)
    L.llama_rope((B, S, 64, nq, nkv, hd, 1, theta, 1e-5), dtype, q, k, pos0)
    _sync()
    pos = pos0 + np.arange(S)
    qr = O.rope(host_tensor(dtype, (B, S, nq, hd), SEED, 3, 0.0, 1.0), pos, theta)
    kr = O.rope(host_tensor(dtype, (B, S, nkv, hd), SEED, 4, 0.0, 1.0), pos, theta)
    assert_parity(to_f64(q), qr, dtype, "rope q")
    assert_parity(to_f64(k), kr, dtype, "rope k")


def _attn_case(dtype, B, S, nq, nkv, hd, cap, pos0):
    import torch
    q = dev_tensor(dtype, (B, S, nq, hd), SEED, 5, 0.0, 1.0)
    k = dev_tensor(dtype, (B, cap, nkv, hd), SEED, 6, 0.0, 1.0)
    v = dev_tensor(dtype, (B, cap, nkv, hd), SEED, 7, 0.0, 1.0)
    o = torch.empty_like(q)
    dims = (B, S, nq * hd, nq, nkv, hd, 1, 1e4, 1e-5)
    need = L.llama_workspace_bytes(L.OP_GQA_ATTENTION, dims, dtype, kv_capacity=cap)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda") if need else None
    L.llama_gqa_attention(dims, dtype, q, k, v, cap, pos0, o, ws)
    _sync()
    qh = host_tensor(dtype, (B, S, nq, hd), SEED, 5, 0.0, 1.0)
    kh = host_tensor(dtype, (B, cap, nkv, hd), SEED, 6, 0.0, 1.0)[:, :pos0 + S]
    vh = host_tensor(dtype, (B, cap, nkv, hd), SEED, 7, 0.0, 1.0)[:, :pos0 + S]
    ref = O.gqa_attention(qh, kh, vh, pos0)
    assert_parity(to_f64(o), ref, dtype, "gqa_attention")


@pytest.mark.parametrize("dtype,B,S,nq,nkv,hd,cap,pos0", [
    (synth.F32, 1, 4, 8, 2, 2, 4, 0),              # toy shape
    (synth.BF16, 2, 256, 8, 2, 64, 256, 0),        # small block shape
    (synth.BF16, 1, 300, 8, 2, 128, 300, 0),       # ragged tail (300 = 2*128 + 44)
    (synth.BF16, 2, 130, 4, 4, 128, 130, 0),       # MHA, ragged
    (synth.BF16, 2, 77, 8, 2, 64, 300, 200),       # chunk after a 200-token cache
    (synth.BF16, 3, 1, 32, 8, 128, 1100, 1040),    # decode shape: one query, long cache (split-K kernel)
    (synth.BF16, 2, 1, 8, 1, 128, 4000, 3999),     # decode, r = 8, cache full to capacity
    (synth.BF16, 2, 1, 4, 4, 128, 130, 128),       # decode, MHA (r = 1), 129 keys: ragged tile
    (synth.BF16, 1, 1, 16, 1, 128, 1, 0),          # decode, first token: one key
    (synth.F32, 2, 5, 6, 3, 8, 9, 4),
])
def test_gqa_attention(dtype, B, S, nq, nkv, hd, cap, pos0):
    _attn_case(dtype, B, S, nq, nkv, hd, cap, pos0)


@pytest.mark.parametrize("dtype,T,d,dff", [(synth.F32, 4, 16, 48), (synth.BF16, 512, 512, 1280),
                                           (synth.BF16, 200, 256, 384), (synth.BF16, 5, 512, 1280)])
def test_swiglu_ffn(dtype, T, d, dff):
    import torch
    x = dev_tensor(dtype, (T, d), SEED, 8, 0.0, 1.0)
    wg = dev_tensor(dtype, (dff, d), SEED, 9, 0.0, 0.02)
    wu = dev_tensor(dtype, (dff, d), SEED, 10, 0.0, 0.02)
    wd = dev_tensor(dtype, (d, dff), SEED, 11, 0.0, 0.02)
    y = torch.empty_like(x)
    dims = (1, T, d, 1, 1, 2, dff, 1e4, 1e-5)
    ws = torch.empty(L.llama_workspace_bytes(L.OP_SWIGLU_FFN, dims, dtype), dtype=torch.uint8, device="cuda")
    L.llama_swiglu_ffn(dims, dtype, x, wg, wu, wd, y, ws)
    _sync()
    ref = O.swiglu_ffn(host_tensor(dtype, (T, d), SEED, 8, 0.0, 1.0), host_tensor(dtype, (dff, d), SEED, 9, 0.0, 0.02),
                       host_tensor(dtype, (dff, d), SEED, 10, 0.0, 0.02), host_tensor(dtype, (d, dff), SEED, 11, 0.0, 0.02))
    assert_parity(to_f64(y), ref, dtype, "swiglu_ffn")


def test_empty_calls_are_no_ops():
    L.llama_rmsnorm((0, 4, 16, 1, 1, 2, 1, 1e4, 1e-5), L.F32, None, None, None)
    L.llama_block_forward((2, 0, 16, 8, 2, 2, 48, 1e4, 1e-5), L.F32, L.BlockWeights(*[16] * 9), 16, 32)
    _sync()


def test_bounded_wait_times_out_cleanly_and_the_context_survives():
    """A kernel's mbarrier wait on a phase that nothing completes gives up after its limit: the host
    reads LLAMA_ERR_TIMEOUT (and the word is cleared), and the next call still computes correctly."""
    import time

    import torch
    t0 = time.perf_counter()
    L.llama_selftest_bounded_wait()
    assert L.llama_get_device_status() == 6                       # LLAMA_ERR_TIMEOUT
    assert 1.0 < time.perf_counter() - t0 < 30.0                  # the 2 s limit, not a hang
    assert L.llama_get_device_status() == 0                       # read-and-clear
    rows, d = 7, 64
    x = torch.randn(rows, d, dtype=torch.float32, device="cuda")
    g = torch.randn(d, dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    L.llama_rmsnorm(L.dims_of(1, rows, d, 1, 1, 64, 128, 1e4, 1e-5), L.F32, x, g, y)
    torch.cuda.synchronize()
    ref = x * torch.rsqrt((x * x).mean(-1, keepdim=True) + 1e-5) * g
    assert torch.allclose(y, ref, rtol=1e-5, atol=1e-5)
    assert L.llama_get_device_status() == 0

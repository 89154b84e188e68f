"""GPU vs oracle for the 8-bit (E4M3) KV cache: the encoding kernel (codes must be identical: both
sides divide in fp32 and round to nearest even), the decode attention over codes, and the decode
stack with an 8-bit cache, whose new K/V are encoded before the token attends to them."""
import numpy as np
import pytest

import llama_decoder_block_fwd_gb300 as L
import oracle as O
from oracle import fp8
from synth import BF16, TID_KCACHE
from synth import configs as C
from synth import host_f64
from synth import workloads as W
from tests.helpers import assert_parity, oracle_dims, to_f64

pytestmark = pytest.mark.gpu


def _scales(n_kv, base):
    return (base * (1.0 + 0.25 * np.arange(n_kv) / max(1, n_kv))).astype(np.float32)


def _dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def test_kv_quantize_codes_are_exact():
    import torch
    T, n_kv, hd = 4099, 8, 128
    x = W.device_tensor(BF16, (T, n_kv, hd), 77, TID_KCACHE, 0.0, 3.0)
    xh = host_f64(BF16, (T, n_kv, hd), 77, TID_KCACHE, 0.0, 3.0)
    xh[0, 0, :4] = [1000.0, -1000.0, 0.0, -0.0]           # saturation and signed zero
    x[0, 0, :4] = torch.tensor([1000.0, -1000.0, 0.0, -0.0], dtype=torch.bfloat16)
    scale = _scales(n_kv, 0.021)
    codes = torch.empty((T, n_kv, hd), dtype=torch.uint8, device="cuda")
    L.llama_kv_quantize(x, _dev(scale), codes)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(codes.cpu().numpy(), fp8.quantize(xh, scale))


def _codes_cache(B, cap, n_kv, hd, seed, tid, scale):
    """Synthetic N(0,1) cache values, encoded on the GPU by llama_kv_quantize and by the oracle."""
    import torch
    x = W.device_tensor(BF16, (B, cap, n_kv, hd), seed, tid, 0.0, 1.0)
    codes = torch.empty((B, cap, n_kv, hd), dtype=torch.uint8, device="cuda")
    L.llama_kv_quantize(x, _dev(scale), codes)
    xh = host_f64(BF16, (B, cap, n_kv, hd), seed, tid, 0.0, 1.0)
    return codes, fp8.dequantize(fp8.quantize(xh, scale), scale)


@pytest.mark.parametrize("B,n_q,n_kv,pos0", [(3, 32, 8, 1039), (2, 8, 1, 3999), (2, 4, 4, 129), (1, 16, 1, 0),
                                             (2, 16, 8, 500), (1, 16, 1, 777)])
def test_decode_attention_over_codes(B, n_q, n_kv, pos0):
    import torch
    hd, cap = 128, pos0 + 5
    ks, vs = _scales(n_kv, 0.03), _scales(n_kv, 0.025)
    kc, kref = _codes_cache(B, cap, n_kv, hd, 31, 11, ks)
    vc, vref = _codes_cache(B, cap, n_kv, hd, 32, 12, vs)
    q = W.device_tensor(BF16, (B, n_q, hd), 33, 1, 0.0, 1.0)
    qh = host_f64(BF16, (B, n_q, hd), 33, 1, 0.0, 1.0)
    dims = L.dims_of(B, 1, n_q * hd, n_q, n_kv, hd, 128, 1e4, 1e-5)
    ws = torch.empty(L.llama_workspace_bytes(L.OP_GQA_ATTENTION, dims, BF16, 0, 0, cap), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty((B, n_q, hd), dtype=torch.bfloat16, device="cuda")
    L.llama_gqa_attention_decode_kv8(dims, q, kc, vc, _dev(ks), _dev(vs), cap, pos0, o, ws)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    ref = O.gqa_attention(qh[:, None], kref[:, :pos0 + 1], vref[:, :pos0 + 1], pos0)[:, 0]
    assert_parity(to_f64(o).reshape(B * n_q, hd), ref.reshape(B * n_q, hd), BF16, "kv8 decode attention")


def _stack_kv8(wl, cap, base_k=0.03, base_v=0.025):
    import torch
    layers = [W.device_layer(wl, l) for l in range(wl.n_layers)]
    hkv = wl.n_kv * wl.head_dim
    scales = np.stack([np.stack([_scales(wl.n_kv, base_k * (1 + 0.1 * l)), _scales(wl.n_kv, base_v * (1 + 0.1 * l))])
                       for l in range(wl.n_layers)]).astype(np.float32)          # [L, 2, n_kv]
    kc = torch.empty((wl.n_layers, wl.B, cap, wl.n_kv, wl.head_dim), dtype=torch.uint8, device="cuda")
    vc = torch.empty_like(kc)
    for l in range(wl.n_layers):
        for which, dst, s in (("k", kc, scales[l, 0]), ("v", vc, scales[l, 1])):
            x = W.device_tensor(wl.dtype, (wl.B, cap, wl.n_kv, wl.head_dim), wl.seed, W.cache_tid(which, l), 0.0, 1.0)
            L.llama_kv_quantize(x, _dev(s), dst[l])
            del x
    final_g, w_lm = W.device_final(wl)
    x = W.device_x_emb(wl)
    logits = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.llama_workspace_bytes(L.OP_STACK_DECODE_STEP, wl.dims, wl.dtype, wl.n_layers, wl.vocab, cap),
                     dtype=torch.uint8, device="cuda")
    L.llama_stack_decode_step_kv8(wl.dims, layers, final_g, w_lm, wl.vocab, x, kc, vc, _dev(scales), cap, wl.t_cache,
                                  logits, ws)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    return logits, kc, vc, scales


def _oracle_kv8(wl, rows, cap, scales):
    d = oracle_dims(wl, B=len(rows))
    fg, wlm = W.host_final(wl)
    x = W.host_x_emb(wl, rows)

    def caches(l):
        out = []
        for which, s in (("k", scales[l, 0]), ("v", scales[l, 1])):
            raw = np.stack([W.host_cache(wl, which, l, b, cap, wl.t_cache) for b in rows])
            out.append(fp8.dequantize(fp8.quantize(raw, s), s))
        return tuple(out)

    return O.stack_decode_step(x, lambda l: O.BlockWeights(**W.host_layer(wl, l)), wl.n_layers, d, wl.t_cache, caches,
                               fg, wlm, kv_store=lambda l: fp8.kv_quant_fn(scales[l, 0], scales[l, 1]))


def test_decode_small_stack_kv8():
    wl = C.Workload("small-stack-kv8", 10, C.BF16, 5, 1, 512, 4, 1, 128, 384, 1e4, 1e-5, gain_std=0.1, n_layers=3,
                    t_cache=300, vocab=1024)
    cap = 333
    logits, kc, vc, scales = _stack_kv8(wl, cap)
    ref = _oracle_kv8(wl, list(range(wl.B)), cap, scales)
    assert_parity(to_f64(logits), ref, wl.dtype, "small stack kv8 logits")
    # positions other than t_cache keep their codes; position t_cache received the new token's
    for l in range(wl.n_layers):
        raw = np.stack([W.host_cache(wl, "k", l, b, cap, cap) for b in range(wl.B)])
        before = fp8.quantize(raw, scales[l, 0])
        got = kc[l].cpu().numpy()
        np.testing.assert_array_equal(got[:, :wl.t_cache], before[:, :wl.t_cache])
        np.testing.assert_array_equal(got[:, wl.t_cache + 1:], before[:, wl.t_cache + 1:])
        assert not np.array_equal(got[:, wl.t_cache], before[:, wl.t_cache])


@pytest.mark.slow
def test_decode_llama3_8b_32_layers_kv8_sampled_sequences():
    import dataclasses
    wl = dataclasses.replace(C.LLAMA3_8B_DECODE, name="llama3-8b-decode-kv8")
    cap = wl.t_cache + 1
    logits, _, _, scales = _stack_kv8(wl, cap)
    rows = [0, 31, 63]
    ref = _oracle_kv8(wl, rows, cap, scales)
    assert_parity(to_f64(logits[rows]), ref, wl.dtype, "llama3-8b kv8 decode logits")

"""Pins of the 8-bit KV-cache oracle: the E4M3 code table of the OCP 8-bit floating-point format
(values the format's definition fixes, and the same casts in torch's float8_e4m3fn, a library
routine), round-to-nearest-even and saturation, the per-head scaling, and how the block uses the
encoded K/V (attention reads the stored values, including the decoded token's own)."""
import numpy as np
import pytest

import oracle as O
from oracle import fp8


def test_code_table_values_fixed_by_the_format():
    d = fp8.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x3F, 0x7E, 0x80, 0xFE], dtype=np.uint8))
    assert list(d[:7]) == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.875, 448.0]
    assert d[7] == 0.0 and np.signbit(d[7]) and d[8] == -448.0
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_decode_and_encode_agree_with_torch_float8_e4m3fn():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    mine = fp8.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    x = np.random.default_rng(0).normal(0, 40, 200000).astype(np.float32).astype(np.float64)
    x = np.concatenate([np.clip(x, -448, 448), np.ldexp(np.arange(-40, 40) / 8.0, -6)])   # incl. subnormal ties
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), ref)


def test_round_to_nearest_even_and_saturation():
    enc = lambda v: int(fp8.e4m3_encode(np.array([v]))[0])
    assert enc(1.0625) == 0x38            # halfway between 1.0 (even) and 1.125
    assert enc(1.1875) == 0x3A            # halfway between 1.125 and 1.25 (even)
    assert enc(2.0 ** -10) == 0x00        # halfway between 0 and the smallest subnormal
    assert enc(3 * 2.0 ** -10) == 0x02    # halfway between 0x01 and 0x02 (even)
    assert enc(1000.0) == 0x7E and enc(-1000.0) == 0xFE and enc(464.0) == 0x7E
    assert enc(float("nan")) == 0x7F
    assert enc(-0.0) == 0x80 and enc(-1e-9) == 0x80


def test_scaled_round_trip():
    codes = np.arange(0, 256, dtype=np.uint8).reshape(2, 128)
    codes = np.where(np.isnan(fp8.e4m3_decode(codes)), 0, codes).astype(np.uint8)
    scale = np.array([0.03125, 0.75], dtype=np.float32)            # a power of two and not
    x = fp8.dequantize(codes, scale)
    assert np.array_equal(fp8.quantize(x, scale)[0], codes[0])      # exact with a power-of-two scale
    err = np.abs(fp8.dequantize(fp8.quantize(x, scale), scale) - x)
    assert np.all(err <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * 0.75)
    # per-head scaling: head 1 of a [.., 2, hd] tensor uses scale[1]
    y = np.ones((3, 2, 4))
    assert np.allclose(fp8.dequantize(fp8.quantize(y, scale), scale), 1.0, rtol=2.0 ** -4)


def _tiny():
    rng = np.random.default_rng(4)
    d = O.Dims(1, 1, 16, 4, 2, 4, 24, 1e4, 1e-5)
    w = O.BlockWeights(np.ones(16), rng.normal(0, .3, (16, 16)), rng.normal(0, .3, (8, 16)),
                       rng.normal(0, .3, (8, 16)), rng.normal(0, .3, (16, 16)), np.ones(16),
                       rng.normal(0, .3, (24, 16)), rng.normal(0, .3, (24, 16)), rng.normal(0, .3, (16, 24)))
    return d, w, rng


def test_attention_reads_the_stored_kv_of_the_new_token():
    d, w, rng = _tiny()
    x = rng.normal(size=(1, 1, 16))
    ks, vs = np.array([0.02, 0.05], np.float32), np.array([0.01, 0.04], np.float32)
    store = fp8.kv_quant_fn(ks, vs)
    y, k_new, v_new = O.block_forward(x, w, d, kv_store=store)
    k_raw, v_raw = O.project_kv(x, w, d)
    assert np.array_equal(k_new, fp8.dequantize(fp8.quantize(k_raw, ks), ks))
    assert np.array_equal(v_new, fp8.dequantize(fp8.quantize(v_raw, vs), vs))
    # one key: attention returns its value, so h = x + v_stored (per head group) W_O^T
    o = np.repeat(v_new[0, 0], 2, axis=0).reshape(1, 16)
    h = x[0] + o @ w.wo.T
    want = h + O.swiglu_ffn(O.rmsnorm(h, w.ffn_norm_g, d.eps), w.w_gate, w.w_up, w.w_down)
    assert np.allclose(y[0], want, rtol=0, atol=1e-12)
    # without a store the raw values are used, and the outputs differ
    y0, _, _ = O.block_forward(x, w, d)
    assert not np.allclose(y0, y, atol=1e-6)


def test_stack_passes_each_layer_its_store():
    d, w, rng = _tiny()
    x = rng.normal(size=(1, 16))
    cache = rng.normal(size=(1, 3, 2, 4))
    seen = []

    def store(l):
        seen.append(l)
        return fp8.kv_quant_fn(np.full(2, 0.05, np.float32), np.full(2, 0.05, np.float32))

    O.stack_decode_step(x, lambda l: w, 2, d, 3, lambda l: (cache, cache), np.ones(16), np.eye(16), kv_store=store)
    assert seen == [0, 1]

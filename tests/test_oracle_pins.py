"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test names the passage it follows.  They are chosen so that a plausible
mistake in the oracle (eps outside the root, a sign flip in the rotation,
half-split instead of interleaved pairs, head_dim vs d_model in theta_k,
h mod n_kv instead of floor(h/r), a missing causal mask, a transposed weight,
a dropped residual) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ---------------------------------------------------------------- GQA toy example
# "LLaMA-3 8B 现代 LLM 架构、计算规模与能耗", section 四.4, subsections 4.3-4.6.
def _toy():
    with open(os.path.join(GOLDEN, "gqa_toy_8q2kv.json")) as f:
        t = json.load(f)
    k = np.array(t["k"], dtype=np.float64)[None]          # [1, 4 tokens, 2 kv heads, 2]
    v = np.array(t["v"], dtype=np.float64)[None]
    q = np.zeros((1, 4, 8, 2))
    q[0, 3] = np.array(t["q_token4"], dtype=np.float64)   # only token 4's queries are printed
    return t, q, k, v


def test_toy_head_map():
    t, *_ = _toy()
    assert [O.kv_head_of(h, 8, 2) for h in range(8)] == t["kv_head_of_query_head"]


def test_toy_softmax_rows_match_page():
    t, q, k, v = _toy()
    for h in range(8):
        g = O.kv_head_of(h, 8, 2)
        p = O.causal_probs(q[0, 3:4, h], k[0, :, g], np.array([3]))[0]
        np.testing.assert_allclose(p, t["softmax_printed"][h], atol=5e-4)


def test_toy_outputs_match_page_and_closed_form():
    t, q, k, v = _toy()
    o = O.gqa_attention(q, k, v, pos0=0)[0, 3]            # [8, 2]
    np.testing.assert_allclose(o, t["output_printed"], atol=5e-4)
    # Closed form: softmax weights (e^a, 1, e^-a, 1)/(e^a + e^-a + 2) with a = sqrt(2), so the
    # group-0 magnitude is sinh(a)/(cosh(a)+1) = tanh(1/sqrt(2)); group 1 has twice the values.
    m = math.tanh(1 / math.sqrt(2))
    expect = np.array([[m, 0], [0, m], [-m, 0], [0, -m], [2 * m, 0], [0, 2 * m], [-2 * m, 0], [0, -2 * m]])
    np.testing.assert_allclose(o, expect, atol=1e-12)


def test_toy_wrong_head_map_would_fail():
    # With h mod n_kv, Q1 would read KV head 1: its output would no longer be [0, 0.609].
    t, q, k, v = _toy()
    p = O.causal_probs(q[0, 3:4, 1], k[0, :, 1 % 2], np.array([3]))[0]
    assert not np.allclose(p @ v[0, :, 1], t["output_printed"][1], atol=5e-3)


# ---------------------------------------------------------------- d_ff rule
# "Llama Architecture: RMSNorm, SwiGLU, RoPE, GQA ..." section 2 prints
# d_ff = floor(8d / (3*256)) * 256 and says it gives 14336 at d = 4096.
def test_ffn_dim_floor_rule():
    assert O.ffn_dim_floor(512) == 1280           # the small block's d_ff
    # The printed rule does NOT give 14336 at d = 4096: it gives 10752.  14336 is the Llama-3-8B
    # value (a separate multiplier); the library takes d_ff as an explicit parameter.
    assert O.ffn_dim_floor(4096) == 10752
    assert O.ffn_dim_floor(4096) != 14336


def test_ffn_dim_ceil_rule_matches_llama1_table():
    # "LLaMA Architecture > Model Architecture", configuration table: 11008, 13824, 17920, 22016.
    assert [O.ffn_dim_ceil(d) for d in (4096, 5120, 6656, 8192)] == [11008, 13824, 17920, 22016]


# ---------------------------------------------------------------- RoPE
# "Llama Architecture ..." section 3: R_{theta_k, m} = [[cos, -sin], [sin, cos]], theta_k =
# theta_base^(-2k/d) on interleaved pairs (x_2k, x_2k+1); norm preserved; q.k depends on m - n.
def test_rope_hd2_is_rotation_by_m():
    x = np.zeros((1, 1, 1, 2)); x[..., 0] = 1.0
    for m in (0, 1, 3, 17):
        y = O.rope(x[0], np.array([m]), 1e4)[0, 0]
        np.testing.assert_allclose(y, [math.cos(m), math.sin(m)], atol=1e-15)


def test_rope_interleaved_pairs_and_theta_uses_head_dim():
    # hd = 4: pair 0 = (x0, x1) turns by m*1, pair 1 = (x2, x3) by m*theta_base^(-2/4).
    x = np.array([[[[0.0, 0.0, 1.0, 0.0]]]])[0]           # [T=1, H=1, 4]
    y = O.rope(x, np.array([100]), 1e4)[0, 0]
    np.testing.assert_allclose(y, [0, 0, math.cos(1.0), math.sin(1.0)], atol=1e-13)
    x = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    y = O.rope(x, np.array([2]), 1e4)[0, 0]
    np.testing.assert_allclose(y, [math.cos(2), math.sin(2), 0, 0], atol=1e-15)


def test_rope_norm_preserved_and_identity_at_zero():
    x = rng.standard_normal((7, 3, 128))
    pos = rng.integers(0, 200000, size=7)
    y = O.rope(x, pos, 5e5)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    np.testing.assert_array_equal(O.rope(x, np.zeros(7, dtype=int), 5e5), x)


def test_rope_relative_position():
    q = rng.standard_normal((1, 1, 64)); k = rng.standard_normal((1, 1, 64))
    for m, n in ((5, 3), (100, 7), (8192, 8000)):
        ref = np.sum(O.rope(q, np.array([m]), 5e5) * O.rope(k, np.array([n]), 5e5))
        for c in (1, 37, 4096):
            got = np.sum(O.rope(q, np.array([m + c]), 5e5) * O.rope(k, np.array([n + c]), 5e5))
            assert abs(got - ref) < 1e-9 * (1 + abs(ref))
        # and it does change with the difference
        other = np.sum(O.rope(q, np.array([m + 1]), 5e5) * O.rope(k, np.array([n]), 5e5))
        assert abs(other - ref) > 1e-6


def test_rope_composes():
    x = rng.standard_normal((1, 2, 16))
    a = O.rope(O.rope(x, np.array([11]), 1e4), np.array([30]), 1e4)
    np.testing.assert_allclose(a, O.rope(x, np.array([41]), 1e4), atol=1e-12)


# ---------------------------------------------------------------- RMSNorm
# "RMSNorm" study note, "How it works": x * (mean(x^2) + eps)^(-1/2), gain g; "LLaMA Architecture >
# Model Architecture", "Key Architectural Choices": outputs have RMS near 1.
def test_rmsnorm_unit_gain_rms():
    x = rng.standard_normal((5, 4096)) * 3.0
    y = O.rmsnorm(x, np.ones(4096), 1e-5)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), np.sqrt(ms / (ms + 1e-5)), rtol=1e-13)
    assert np.all(np.abs(np.sqrt(np.mean(y * y, axis=-1)) - 1) < 1e-5)


def test_rmsnorm_eps_inside_sqrt():
    # A row of 1e-4s: eps inside gives 1e-4/sqrt(1e-8 + 1e-5) ~ 0.0316; outside would give ~0.909.
    y = O.rmsnorm(np.full((1, 64), 1e-4), np.ones(64), 1e-5)
    np.testing.assert_allclose(y, 1e-4 / math.sqrt(1e-8 + 1e-5), rtol=1e-14)
    assert abs(y[0, 0] - 0.0316) < 1e-3


def test_rmsnorm_zero_row_gain_and_scale():
    assert np.all(O.rmsnorm(np.zeros((1, 8)), np.ones(8), 1e-5) == 0)
    x = rng.standard_normal((3, 32)); g = rng.standard_normal(32)
    np.testing.assert_allclose(O.rmsnorm(x, g, 1e-5), O.rmsnorm(x, np.ones(32), 1e-5) * g, rtol=1e-14)
    np.testing.assert_allclose(O.rmsnorm(1e3 * x, g, 1e-5), O.rmsnorm(x, g, 1e-5), rtol=1e-5)
    # mean is NOT removed (no centring): a constant row maps to sign * sqrt(c^2/(c^2+eps))
    c = 2.0
    np.testing.assert_allclose(O.rmsnorm(np.full((1, 8), c), np.ones(8), 1e-5), c / math.sqrt(c * c + 1e-5))


# ---------------------------------------------------------------- SiLU
# "Llama Architecture ..." section 2: SiLU(z) = z / (1 + e^-z).
def test_silu_closed_form():
    assert O.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(O.silu(np.array([1.0])), 1 / (1 + math.exp(-1)), rtol=1e-15)
    np.testing.assert_allclose(O.silu(np.array([-1.0])), -1 / (1 + math.e), rtol=1e-15)
    np.testing.assert_allclose(O.silu(np.array([40.0])), 40.0, rtol=1e-15)
    assert abs(O.silu(np.array([-40.0]))[0]) < 1e-15


def test_swiglu_gate_and_up_roles():
    # x = e_0, W_gate row 0 = 2 e_0, W_up row 0 = 3 e_0, W_down column 0 = e_1:
    # the output is SiLU(2) * 3 on feature 1, zero elsewhere.  Swapping gate and up gives SiLU(3)*2.
    d, dff = 4, 2
    x = np.zeros((1, d)); x[0, 0] = 1
    wg = np.zeros((dff, d)); wg[0, 0] = 2
    wu = np.zeros((dff, d)); wu[0, 0] = 3
    wd = np.zeros((d, dff)); wd[1, 0] = 1
    y = O.swiglu_ffn(x, wg, wu, wd)
    np.testing.assert_allclose(y, [[0, 2 / (1 + math.exp(-2)) * 3, 0, 0]], rtol=1e-15)


# ---------------------------------------------------------------- attention reductions
def _mha_loop(q, k, v):
    """Independent per-head MHA with explicit loops (n_kv == n_q), full causal softmax."""
    B, S, H, hd = q.shape
    o = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            for i in range(S):
                s = [sum(q[b, i, h, t] * k[b, j, h, t] for t in range(hd)) / math.sqrt(hd) for j in range(i + 1)]
                mx = max(s)
                e = [math.exp(z - mx) for z in s]
                tot = sum(e)
                for t in range(hd):
                    o[b, i, h, t] = sum(e[j] / tot * v[b, j, h, t] for j in range(i + 1))
    return o


def test_gqa_with_nkv_eq_nq_is_mha():
    # "Llama Architecture ..." section 4: MHA is the case h = g.
    q = rng.standard_normal((2, 5, 3, 4)); k = rng.standard_normal((2, 5, 3, 4)); v = rng.standard_normal((2, 5, 3, 4))
    np.testing.assert_allclose(O.gqa_attention(q, k, v), _mha_loop(q, k, v), atol=1e-13)


def test_gqa_equals_mha_on_repeat_interleaved_kv():
    # Section 4: K~ = repeat_interleave(K, r, dim=heads), same for V.
    q = rng.standard_normal((1, 6, 8, 4)); k = rng.standard_normal((1, 6, 2, 4)); v = rng.standard_normal((1, 6, 2, 4))
    kr, vr = np.repeat(k, 4, axis=2), np.repeat(v, 4, axis=2)
    np.testing.assert_allclose(O.gqa_attention(q, k, v), _mha_loop(q, kr, vr), atol=1e-13)


def test_causal_mask_brute_force_and_future_independence():
    B, S, H, hd = 1, 6, 2, 3
    q = rng.standard_normal((B, S, H, hd)); k = rng.standard_normal((B, S, H, hd)); v = rng.standard_normal((B, S, H, hd))
    # explicit -inf mask matrix + full softmax
    mask = np.where(np.tril(np.ones((S, S))) > 0, 0.0, -np.inf)
    for h in range(H):
        sc = q[0, :, h] @ k[0, :, h].T / math.sqrt(hd) + mask
        p = np.exp(sc - sc.max(-1, keepdims=True)); p /= p.sum(-1, keepdims=True)
        np.testing.assert_allclose(O.gqa_attention(q, k, v)[0, :, h], p @ v[0, :, h], atol=1e-14)
    base = O.gqa_attention(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[:, 4:] += 5.0; v2[:, 4:] -= 3.0
    after = O.gqa_attention(q, k2, v2)
    np.testing.assert_array_equal(after[:, :4], base[:, :4])
    assert not np.allclose(after[:, 4:], base[:, 4:])


def test_first_token_attends_only_to_itself():
    q = rng.standard_normal((1, 3, 4, 8)); k = rng.standard_normal((1, 3, 2, 8)); v = rng.standard_normal((1, 3, 2, 8))
    o = O.gqa_attention(q, k, v)
    for h in range(4):
        np.testing.assert_allclose(o[0, 0, h], v[0, 0, h // 2], atol=1e-15)


# ---------------------------------------------------------------- block
def _rand_weights(d, nq, nkv, hd, dff, scale=0.1):
    return O.BlockWeights(
        attn_norm_g=1 + 0.1 * rng.standard_normal(d), wq=scale * rng.standard_normal((nq * hd, d)),
        wk=scale * rng.standard_normal((nkv * hd, d)), wv=scale * rng.standard_normal((nkv * hd, d)),
        wo=scale * rng.standard_normal((d, nq * hd)), ffn_norm_g=1 + 0.1 * rng.standard_normal(d),
        w_gate=scale * rng.standard_normal((dff, d)), w_up=scale * rng.standard_normal((dff, d)),
        w_down=scale * rng.standard_normal((d, dff)))


def test_block_identity_when_sublayers_output_zero():
    # "LLaMA Architecture > Model Architecture", The Transformer Block: a sublayer that outputs
    # zero leaves the input unchanged through the residual path.
    dims = O.Dims(2, 5, 16, 4, 2, 4, 24, 1e4, 1e-5)
    w = _rand_weights(16, 4, 2, 4, 24)
    w.wo[:] = 0; w.w_down[:] = 0
    x = rng.standard_normal((2, 5, 16))
    y, _, _ = O.block_forward(x, w, dims)
    np.testing.assert_array_equal(y, x)


def test_block_residual_structure():
    # zero FFN -> y = h = x + Attn(RMSNorm(x)); check against a hand composition with a loop MHA
    dims = O.Dims(1, 4, 8, 2, 2, 4, 8, 1e4, 1e-5)
    w = _rand_weights(8, 2, 2, 4, 8)
    w.w_down[:] = 0
    x = rng.standard_normal((1, 4, 8))
    u = O.rmsnorm(x, w.attn_norm_g, 1e-5)
    pos = np.arange(4)
    q = O.rope((u @ w.wq.T).reshape(1, 4, 2, 4), pos, 1e4)
    k = O.rope((u @ w.wk.T).reshape(1, 4, 2, 4), pos, 1e4)
    v = (u @ w.wv.T).reshape(1, 4, 2, 4)
    h = x + _mha_loop(q, k, v).reshape(1, 4, 8) @ w.wo.T
    y, _, _ = O.block_forward(x, w, dims)
    np.testing.assert_allclose(y, h, atol=1e-13)


def test_block_rows_subset_matches_full():
    dims = O.Dims(2, 9, 16, 4, 2, 4, 24, 1e4, 1e-5)
    w = _rand_weights(16, 4, 2, 4, 24)
    x = rng.standard_normal((2, 9, 16))
    full, kf, vf = O.block_forward(x, w, dims)
    rows = np.array([0, 4, 8])
    part, kp, vp = O.block_forward(x, w, dims, rows=rows)
    np.testing.assert_allclose(part, full[:, rows], atol=1e-13)
    np.testing.assert_array_equal(kp, kf)


def test_prefill_then_decode_equals_longer_prefill():
    # A decode step at position S against the cache of an S-token prefill gives the same output
    # as the last row of an (S+1)-token prefill ("LLaMA-3 8B ..." page, section 九: KV cache reuse).
    dims1 = O.Dims(2, 7, 16, 4, 2, 4, 24, 1e4, 1e-5)
    w = _rand_weights(16, 4, 2, 4, 24)
    x = rng.standard_normal((2, 7, 16))
    y_full, _, _ = O.block_forward(x, w, dims1)
    dims0 = O.Dims(2, 6, 16, 4, 2, 4, 24, 1e4, 1e-5)
    _, kc, vc = O.block_forward(x[:, :6], w, dims0)
    dims_step = O.Dims(2, 1, 16, 4, 2, 4, 24, 1e4, 1e-5)
    y_step, _, _ = O.block_forward(x[:, 6:7], w, dims_step, pos0=6, k_past=kc, v_past=vc)
    np.testing.assert_allclose(y_step[:, 0], y_full[:, 6], atol=1e-12)


def test_stack_decode_two_layers_matches_manual_chain():
    d, nq, nkv, hd, dff = 16, 4, 2, 4, 24
    dims = O.Dims(3, 1, d, nq, nkv, hd, dff, 1e4, 1e-5)
    ws = [_rand_weights(d, nq, nkv, hd, dff) for _ in range(2)]
    caches = [(rng.standard_normal((3, 5, nkv, hd)), rng.standard_normal((3, 5, nkv, hd))) for _ in range(2)]
    fg = 1 + 0.1 * rng.standard_normal(d)
    wlm = 0.1 * rng.standard_normal((11, d))
    x = rng.standard_normal((3, d))
    logits = O.stack_decode_step(x, lambda l: ws[l], 2, dims, 5, lambda l: caches[l], fg, wlm)
    h = x[:, None]
    for l in range(2):
        h, _, _ = O.block_forward(h, ws[l], dims, pos0=5, k_past=caches[l][0], v_past=caches[l][1])
    np.testing.assert_allclose(logits, O.rmsnorm(h[:, 0], fg, 1e-5) @ wlm.T, atol=1e-13)
    assert logits.shape == (3, 11)


# ---------------------------------------------------------------- sizes
# "LLaMA-3 8B ..." page, section 六 (parameter counts) and section 七 (KV cache per token).
def test_parameter_counts():
    assert O.block_param_count(4096, 32, 8, 128, 14336) == 218_112_000
    assert O.model_param_count(32, 4096, 32, 8, 128, 14336, 128256) == 8_030_261_248
    assert 4096 * 32 * 128 + 2 * 4096 * 8 * 128 + 32 * 128 * 4096 == 41_943_040
    assert 3 * 4096 * 14336 == 176_160_768
    # MHA attention would be 4 * 4096^2; GQA is 37.5% smaller
    assert 4 * 4096 ** 2 == 67_108_864 and abs(1 - 41_943_040 / 67_108_864 - 0.375) < 1e-12


def test_kv_cache_bytes():
    assert O.kv_bytes_per_token(1, 8, 128, 2) == 4096
    assert O.kv_bytes_per_token(32, 8, 128, 2) == 128 * 1024
    assert O.kv_bytes_per_token(32, 8, 128, 2) * 8192 == 1 << 30
    assert O.kv_bytes_per_token(32, 32, 128, 2) == 512 * 1024     # MHA: 4x ("Llama Architecture ..." page, Mathematical Foundations 4: g/h = 1/r)

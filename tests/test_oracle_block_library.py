"""A pin of the whole block: the fp64 oracle against torch's own routines in float64 on the CPU.

No page prints a block output, so the oracle's block is checked here against a second,
independent formulation built from library routines: `scaled_dot_product_attention` (causal mask
with a position offset, `enable_gqa` for the query-head to KV-head map), `rms_norm` for RMSNorm,
`silu` for SiLU, and RoPE written as multiplication of complex numbers (each interleaved pair
(x_2k, x_2k+1) taken as x_2k + i x_2k+1 and multiplied by e^{i m theta_k}), a formulation the
oracle does not use.  The block structure follows "Llama Architecture ...", Mathematical
Foundations 1-5 (pre-norm, residual around attention and around the SwiGLU FFN) and
"LLaMA-3 8B ...", section 四 (GQA, causal attention with a cache).  A mistake in the oracle's
composition (a dropped residual, a transposed weight, a wrong head map, a mask off by one, pairs
split by halves) moves the output by far more than the tolerance."""
import numpy as np
import pytest

import oracle as O

torch = pytest.importorskip("torch")
F = torch.nn.functional


def _weights(rng, d, n_q, n_kv, hd, d_ff):
    def m(o, i):
        return rng.normal(0.0, 1.0 / np.sqrt(i), (o, i))
    return O.BlockWeights(attn_norm_g=rng.normal(1.0, 0.2, d), wq=m(n_q * hd, d), wk=m(n_kv * hd, d),
                          wv=m(n_kv * hd, d), wo=m(d, n_q * hd), ffn_norm_g=rng.normal(1.0, 0.2, d),
                          w_gate=m(d_ff, d), w_up=m(d_ff, d), w_down=m(d, d_ff))


def _torch_block(x, w, dims, pos0=0, k_past=None, v_past=None):
    """y, k, v of one block for tokens at positions pos0 .. pos0+S-1 (float64, library routines)."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    B, S, d = x.shape
    n_q, n_kv, hd = dims.n_q, dims.n_kv, dims.head_dim
    X = t(x)
    u = F.rms_norm(X, (d,), weight=t(w.attn_norm_g), eps=dims.eps)
    q = (u @ t(w.wq).T).reshape(B, S, n_q, hd)
    k = (u @ t(w.wk).T).reshape(B, S, n_kv, hd)
    v = (u @ t(w.wv).T).reshape(B, S, n_kv, hd)
    theta = dims.theta_base ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    ang = (pos0 + torch.arange(S, dtype=torch.float64))[:, None] * theta[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)                       # e^{i m theta_k}, [S, hd/2]

    def rope(a, heads):
        c = torch.view_as_complex(a.reshape(B, S, heads, hd // 2, 2).contiguous())
        return torch.view_as_real(c * rot[None, :, None, :]).reshape(B, S, heads, hd)

    q, k = rope(q, n_q), rope(k, n_kv)
    K = k if k_past is None else torch.cat([k_past, k], dim=1)
    V = v if v_past is None else torch.cat([v_past, v], dim=1)
    visible = torch.arange(pos0 + S)[None, :] <= (pos0 + torch.arange(S))[:, None]   # key j <= query position
    o = F.scaled_dot_product_attention(q.transpose(1, 2), K.transpose(1, 2), V.transpose(1, 2),
                                       attn_mask=visible, enable_gqa=True)
    h = X + o.transpose(1, 2).reshape(B, S, n_q * hd) @ t(w.wo).T
    z = F.rms_norm(h, (d,), weight=t(w.ffn_norm_g), eps=dims.eps)
    y = h + (F.silu(z @ t(w.w_gate).T) * (z @ t(w.w_up).T)) @ t(w.w_down).T
    return y, k, v


@pytest.mark.parametrize("n_q,n_kv", [(4, 2), (8, 1), (4, 4)])
def test_block_prefill_matches_library_formulation(n_q, n_kv):
    rng = np.random.default_rng(20 + n_q * 3 + n_kv)
    B, S, d, hd, d_ff = 2, 9, 32, 8, 48
    dims = O.Dims(B, S, d, n_q, n_kv, hd, d_ff, 1e4, 1e-5)
    w = _weights(rng, d, n_q, n_kv, hd, d_ff)
    x = rng.normal(0.0, 1.0, (B, S, d))
    y_ref, k_ref, v_ref = _torch_block(x, w, dims)
    y, k, v = O.block_forward(x, w, dims)
    np.testing.assert_allclose(y, y_ref.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(k, k_ref.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(v, v_ref.numpy(), rtol=0, atol=1e-10)


@pytest.mark.parametrize("S1", [1, 4])
def test_block_against_a_cache_matches_library_formulation(S1):
    """Chunked prefill (S1 = 4) and one decode step (S1 = 1) after 6 cached positions, RoPE base
    5e5; each side builds its cache from the same 6 prefix tokens with its own formulation."""
    rng = np.random.default_rng(77 + S1)
    B, S0, d, n_q, n_kv, hd, d_ff = 2, 6, 32, 4, 2, 8, 40
    w = _weights(rng, d, n_q, n_kv, hd, d_ff)
    x0 = rng.normal(0.0, 1.0, (B, S0, d))
    x1 = rng.normal(0.0, 1.0, (B, S1, d))
    d0 = O.Dims(B, S0, d, n_q, n_kv, hd, d_ff, 5e5, 1e-6)
    d1 = O.Dims(B, S1, d, n_q, n_kv, hd, d_ff, 5e5, 1e-6)
    _, k0_ref, v0_ref = _torch_block(x0, w, d0)
    y_ref, _, _ = _torch_block(x1, w, d1, pos0=S0, k_past=k0_ref, v_past=v0_ref)
    _, k0, v0 = O.block_forward(x0, w, d0)
    y, _, _ = O.block_forward(x1, w, d1, pos0=S0, k_past=k0, v_past=v0)
    np.testing.assert_allclose(y, y_ref.numpy(), rtol=0, atol=1e-10)


def test_stack_decode_matches_library_formulation():
    """The decode stack ("LLaMA-3 8B ...", sections 二, 九 and 十: blocks, then the final RMSNorm and
    the untied LM head) in the library formulation: two layers of one-token decode after 5 cached
    positions per layer (the same cached K/V on both sides), torch's rms_norm for the final norm and
    a plain product with the head.  A wrong layer order, a skipped final norm or a transposed head
    moves the logits far past the tolerance."""
    rng = np.random.default_rng(5)
    B, S0, d, n_q, n_kv, hd, d_ff, vocab, eps = 2, 5, 32, 4, 2, 8, 40, 13, 1e-6
    ws = [_weights(rng, d, n_q, n_kv, hd, d_ff) for _ in range(2)]
    caches = [(rng.normal(0.0, 1.0, (B, S0, n_kv, hd)), rng.normal(0.0, 1.0, (B, S0, n_kv, hd))) for _ in range(2)]
    fg = rng.normal(1.0, 0.2, d)
    wlm = rng.normal(0.0, 1.0 / np.sqrt(d), (vocab, d))
    x_emb = rng.normal(0.0, 1.0, (B, d))
    dims = O.Dims(B, 1, d, n_q, n_kv, hd, d_ff, 5e5, eps)
    logits = O.stack_decode_step(x_emb, lambda l: ws[l], 2, dims, S0, lambda l: caches[l], fg, wlm)
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    h = x_emb[:, None, :]
    for l in range(2):
        y, _, _ = _torch_block(h, ws[l], dims, pos0=S0, k_past=t(caches[l][0]), v_past=t(caches[l][1]))
        h = y.numpy()
    ref = F.rms_norm(t(h[:, 0, :]), (d,), weight=t(fg), eps=eps) @ t(wlm).T
    np.testing.assert_allclose(logits, ref.numpy(), rtol=0, atol=1e-10)
    assert logits.shape == (B, vocab)

"""GPU vs oracle for the next-token choice (llama_sample) and the embedding lookup (llama_embed),
and a three-step greedy generation loop (embed -> decode step -> choice -> embed).

Where the choice is decided by comparisons alone (argmax, top-k membership) the GPU must agree
exactly.  Where it is decided by sums of probabilities (the top-p cut, the inverse CDF) the GPU
sums fp32 exponentials exactly in fixed point and the oracle sums fp64 ones, so a row may differ
only where u or p sits within a rounding error of a boundary: each such row must still be a valid
draw within EPS of probability mass, and most rows must match exactly."""
import numpy as np
import pytest

import llama_decoder_block_fwd_gb300 as L
import oracle as O
from oracle import sampling as S
from synth import BF16, F32, TID_LOGITS
from synth import configs as C
from synth import host_f64
from synth import workloads as W
from tests.helpers import assert_parity, oracle_dims, to_f64

pytestmark = pytest.mark.gpu

EPS = 2e-5      # probability mass: fp32 exp error (~2e-6 per term) with headroom


def _logits(B, V, std, seed=4242, mean=0.0):
    import torch
    z = W.device_tensor(F32, (B, V), seed, TID_LOGITS, mean, std)
    return z, host_f64(F32, (B, V), seed, TID_LOGITS, mean, std)


def _uniforms(B, seed=99):
    import torch
    u = np.random.default_rng(seed).random(B).astype(np.float32)
    return torch.from_numpy(u).cuda(), u.astype(np.float64)


def _run(z, T, k, p, u, vocab=None):
    import torch
    tok = torch.full((z.shape[0],), -1, dtype=torch.int32, device="cuda")
    L.llama_sample(z, T, k, p, u, tok, vocab=vocab)
    torch.cuda.synchronize()
    return tok.cpu().numpy()


def _valid(z, T, k, p, u, g):
    u = min(u, 0.99999994)
    ps = [p] if p >= 1 else [p * (1 - EPS), p, min(1.0, p * (1 + EPS))]
    for pp in ps:
        kept = S.kept_set(z, T, k, pp)
        if g not in set(kept.tolist()):
            continue
        if kept.shape[0] == 1:
            return True
        ids = np.sort(kept)
        m = np.exp((z[ids] - z.max()) / T)
        c = np.cumsum(m) / m.sum()
        j = int(np.searchsorted(ids, g))
        lo = c[j - 1] if j else 0.0
        if lo - EPS <= u < c[j] + EPS:
            return True
    return False


def _check(zh, T, k, p, uh, got, min_exact=0.75):
    exact = 0
    for b in range(zh.shape[0]):
        ref = S.sample(zh[b], T, k, p, min(uh[b], 0.99999994))
        if got[b] == ref:
            exact += 1
        else:
            assert _valid(zh[b], T, k, p, uh[b], int(got[b])), (b, int(got[b]), ref)
    assert exact >= min_exact * zh.shape[0], exact
    return exact


def test_argmax_is_exact():
    B, V = 64, 128256
    z, zh = _logits(B, V, 3.0)
    u, _ = _uniforms(B)
    want = np.array([S.argmax(zh[b]) for b in range(B)])
    np.testing.assert_array_equal(_run(z, 0.0, 0, 1.0, u), want)          # T = 0
    np.testing.assert_array_equal(_run(z, 0.8, 1, 0.9, u), want)          # top-k = 1
    np.testing.assert_array_equal(_run(z, 1.0, 50, 0.0, u), want)         # top-p = 0


def test_argmax_ties_go_to_the_lowest_id():
    import torch
    B, V = 8, 5000
    zh = np.round(np.random.default_rng(5).normal(0, 1, (B, V)))     # integers: many equal maxima
    z = torch.from_numpy(zh.astype(np.float32)).cuda()
    u, _ = _uniforms(B)
    got = _run(z, 0.0, 0, 1.0, u)
    np.testing.assert_array_equal(got, [int(np.flatnonzero(zh[b] == zh[b].max())[0]) for b in range(B)])


def test_rows_split_over_a_cluster_ties_across_parts():
    """Few rows over a large vocabulary: each row is split over a cluster of up to eight CTAs.  Equal
    maxima that sit in different CTAs' parts still go to the lowest id, and small top-k draws
    (candidates gathered by every CTA, ranked by the leader) match the oracle."""
    import torch
    B, V = 8, 65536
    zh = np.round(np.random.default_rng(21).normal(0, 1, (B, V)))     # integers: equal maxima far apart
    zh[3, 5] = zh[3, V - 3] = zh[3].max() + 1.0                       # first and last part
    z = torch.from_numpy(zh.astype(np.float32)).cuda()
    u, uh = _uniforms(B, seed=21)
    got = _run(z, 0.0, 0, 1.0, u)
    np.testing.assert_array_equal(got, [int(np.flatnonzero(zh[b] == zh[b].max())[0]) for b in range(B)])
    for k, p in ((50, 0.95), (1024, 0.9), (2, 1.0)):
        got = _run(z, 1.0, k, p, u)
        for b in range(B):
            assert int(got[b]) in set(S.order_desc(zh[b])[:k].tolist())
        _check(zh, 1.0, k, p, uh, got)
    z1, z1h = _logits(1, 128256, 2.5)                                 # one row: eight CTAs
    u1, u1h = _uniforms(1, seed=3)
    for T, k, p in ((0.8, 50, 0.95), (0.0, 0, 1.0)):
        got = _run(z1, T, k, p, u1)
        want = S.argmax(z1h[0]) if T == 0.0 else S.sample(z1h[0], T, k, p, min(u1h[0], 0.99999994))
        assert int(got[0]) == want or (T > 0 and _valid(z1h[0], T, k, p, u1h[0], int(got[0])))


@pytest.mark.parametrize("T,k,p", [(1.0, 0, 1.0), (0.7, 50, 1.0), (1.0, 0, 0.9), (0.8, 40, 0.95),
                                   (1.3, 1000, 0.5), (2.0, 0, 0.99), (0.5, 0, 1e-4)])
def test_draws_match_the_oracle_llama3_vocab(T, k, p):
    B, V = 64, 128256
    z, zh = _logits(B, V, 2.5)
    u, uh = _uniforms(B, seed=int(T * 100) + k + int(p * 1000))
    got = _run(z, T, k, p, u)
    if 0 < k < V:
        for b in range(B):                                   # membership is exact
            assert int(got[b]) in set(S.order_desc(zh[b])[:k].tolist())
    _check(zh, T, k, p, uh, got)
    np.testing.assert_array_equal(_run(z, T, k, p, u), got)  # same inputs, same tokens


@pytest.mark.parametrize("k,p", [(1000, 1.0), (0, 0.3), (700, 0.6), (3, 1.0)])
def test_ties_at_the_top_k_and_top_p_cuts(k, p):
    import torch
    B, V = 16, 20000
    zh = np.round(np.random.default_rng(11).normal(0, 2, (B, V)))    # integer logits: the cuts fall in ties
    z = torch.from_numpy(zh.astype(np.float32)).cuda()
    u, uh = _uniforms(B, seed=k + 1)
    got = _run(z, 1.0, k, p, u)
    if 0 < k < V:
        for b in range(B):
            assert int(got[b]) in set(S.order_desc(zh[b])[:k].tolist())
    _check(zh, 1.0, k, p, uh, got)


@pytest.mark.parametrize("V", [5, 100, 1031, 2049, 4099, 50001])
def test_small_top_k_over_small_and_masked_vocabularies(V):
    """Top-k up to 1024 ranks a gathered candidate set: vocabularies below one token per thread
    (threads holding no token), ragged rows (V % 4 != 0) and rows that are mostly -inf."""
    import torch
    rng = np.random.default_rng(V)
    B = 8
    zh = rng.normal(0, 2, (B, V))
    zh[4:][rng.random((4, V)) < 0.97] = -np.inf                       # rows 4-7: mostly masked
    zh[4:, 0] = rng.normal(0, 2, 4)
    z = torch.from_numpy(zh.astype(np.float32)).cuda()
    zh = to_f64(z)
    for k in sorted({2, 3, 50, min(V - 1, 1024)}):
        if k >= V or k < 2:
            continue
        u, uh = _uniforms(B, seed=k)
        got = _run(z, 0.9, k, 0.97, u)
        for b in range(B):
            assert int(got[b]) in set(S.order_desc(zh[b])[:k].tolist())
            assert np.isfinite(zh[b, got[b]])
        _check(zh, 0.9, k, 0.97, uh, got)


def test_small_top_k_when_the_gather_bound_holds_too_many_tokens():
    """Equal logits: the gather bound (or the top-p bucket) admits more tokens than shared memory
    holds, and the radix-selection path must take over with the same result (lowest ids kept)."""
    import torch
    B, V = 4, 128256
    zh = np.zeros((B, V))
    zh[1, 7::1000] = 0.5                                              # a few above an equal plateau
    zh[2, :] = np.round(np.random.default_rng(8).normal(0, 0.3, V))
    z = torch.from_numpy(zh.astype(np.float32)).cuda()
    for k, p in ((2, 1.0), (700, 1.0), (1024, 1.0), (0, 0.5), (1500, 0.9)):
        u, uh = _uniforms(B, seed=k + 5)
        got = _run(z, 1.0, k, p, u)
        if k:
            for b in range(B):
                assert int(got[b]) in set(S.order_desc(zh[b])[:k].tolist())
        _check(zh, 1.0, k, p, uh, got)


@pytest.mark.parametrize("k,p", [(0, 0.9), (50, 0.95), (0, 1.0), (2000, 0.8)])
def test_rows_not_16_byte_aligned(k, p):
    """Row stride of 1001 floats: every other row starts off a 16-byte boundary (scalar loads)."""
    import torch
    B, V = 6, 1001
    zh = np.random.default_rng(k + 17).normal(0, 2, (B, V))
    z = torch.from_numpy(zh.astype(np.float32)).cuda()
    zh = to_f64(z)
    u, uh = _uniforms(B, seed=k + 3)
    got = _run(z, 0.9, k, p, u)
    if 0 < k < V:
        for b in range(B):
            assert int(got[b]) in set(S.order_desc(zh[b])[:k].tolist())
    _check(zh, 0.9, k, p, uh, got)


def test_masked_tokens_strided_rows_and_small_vocabularies():
    import torch
    rng = np.random.default_rng(2)
    B, V, ld = 16, 3000, 3072
    zh = rng.normal(0, 2, (B, ld))
    zh[rng.random((B, ld)) < 0.9] = -np.inf                           # masked tokens
    zh[:, 0] = rng.normal(0, 2, B)                                    # at least one finite per row
    z = torch.from_numpy(zh.astype(np.float32)).cuda()
    u, uh = _uniforms(B, seed=3)
    got = _run(z, 1.0, 0, 0.95, u, vocab=V)                           # row stride ld > vocab
    zv = zh[:, :V]
    for b in range(B):
        assert np.isfinite(zv[b, got[b]])
    _check(zv, 1.0, 0, 0.95, uh, got)
    for V in (1, 2, 7):
        zs = torch.from_numpy(rng.normal(0, 1, (4, V)).astype(np.float32)).cuda()
        zsh = to_f64(zs)
        us, ush = _uniforms(4, seed=V)
        _check(zsh, 1.0, 0, 1.0, ush, _run(zs, 1.0, 0, 1.0, us), min_exact=1.0)


def test_empty_batch_is_a_no_op():
    import torch
    z = torch.empty((0, 10), dtype=torch.float32, device="cuda")
    tok = torch.empty((0,), dtype=torch.int32, device="cuda")
    L.llama_sample(z, 1.0, 0, 1.0, torch.empty(0, device="cuda"), tok)


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_embedding_rows_are_exact(dtype):
    import torch
    wl = C.Workload("embed", 8, dtype, 64, 1, 512, 8, 2, 64, 1280, 1e4, 1e-5, vocab=3000)
    E = W.device_embed(wl)
    tokens = np.random.default_rng(1).integers(0, wl.vocab, 64).astype(np.int32)
    tok = torch.from_numpy(tokens).cuda()
    x = torch.empty((64, wl.d_model), dtype=E.dtype, device="cuda")
    L.llama_embed(dtype, E, tok, x)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    np.testing.assert_array_equal(to_f64(x), W.host_embed_rows(wl, tokens))
    np.testing.assert_array_equal(to_f64(x), S.embed(to_f64(E), tokens))


def test_embedding_rejects_out_of_range_ids_on_the_device():
    import torch
    wl = C.Workload("embed", 8, BF16, 4, 1, 256, 8, 2, 32, 512, 1e4, 1e-5, vocab=100)
    E = W.device_embed(wl)
    tok = torch.tensor([5, 100, -1, 99], dtype=torch.int32, device="cuda")
    x = torch.full((4, wl.d_model), 7.0, dtype=E.dtype, device="cuda")
    L.llama_embed(BF16, E, tok, x)
    assert L.llama_get_device_status() == 1                      # LLAMA_ERR_INVALID_ARG latched
    assert L.llama_get_device_status() == 0                      # and cleared by the read
    got = to_f64(x)
    np.testing.assert_array_equal(got[0], W.host_embed_rows(wl, [5])[0])
    np.testing.assert_array_equal(got[3], W.host_embed_rows(wl, [99])[0])
    assert not got[1].any() and not got[2].any()


def test_greedy_generation_loop_three_steps():
    """embed -> 3-layer decode step -> argmax -> embed, three times, against the oracle's own loop
    per sequence (decode rows are independent).  A sequence is followed while the oracle's top-1
    logit leads the runner-up by more than the logits' tolerance; after a closer call the two
    loops may legitimately pick different tokens, so that sequence stops being compared."""
    import torch
    wl = C.Workload("gen-stack", 9, BF16, 6, 1, 512, 4, 1, 128, 384, 1e4, 1e-5, gain_std=0.1, n_layers=3,
                    t_cache=200, vocab=1024)
    steps, cap = 3, 208
    layers = [W.device_layer(wl, l) for l in range(wl.n_layers)]
    kc, vc = W.device_caches(wl, cap)
    final_g, w_lm = W.device_final(wl)
    E = W.device_embed(wl)
    tokens0 = np.random.default_rng(17).integers(0, wl.vocab, wl.B).astype(np.int32)
    tok = torch.from_numpy(tokens0).cuda()
    x = torch.empty((wl.B, wl.d_model), dtype=torch.bfloat16, device="cuda")
    logits = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.llama_workspace_bytes(L.OP_STACK_DECODE_STEP, wl.dims, wl.dtype, wl.n_layers, wl.vocab, cap),
                     dtype=torch.uint8, device="cuda")
    u = torch.zeros(wl.B, device="cuda")
    gpu_logits, gpu_tokens = [], [tokens0]
    for s in range(steps):
        L.llama_embed(BF16, E, tok, x)
        L.llama_stack_decode_step(wl.dims, wl.dtype, layers, final_g, w_lm, wl.vocab, x, kc, vc, cap,
                                  wl.t_cache + s, logits, ws)
        L.llama_sample(logits, 0.0, 0, 1.0, u, tok)
        gpu_logits.append(to_f64(logits))
        gpu_tokens.append(tok.cpu().numpy().copy())
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0

    d = oracle_dims(wl, B=1)
    hw = [O.BlockWeights(**W.host_layer(wl, l)) for l in range(wl.n_layers)]
    fg, wlm = W.host_final(wl)
    compared = 0
    for b in range(wl.B):
        caches = [[W.host_cache(wl, "k", l, b, cap, wl.t_cache)[None], W.host_cache(wl, "v", l, b, cap, wl.t_cache)[None]]
                  for l in range(wl.n_layers)]
        t = int(tokens0[b])
        for s in range(steps):
            h = W.host_embed_rows(wl, [t])[:, None, :]
            for l in range(wl.n_layers):
                h, k_new, v_new = O.block_forward(h, hw[l], d, pos0=wl.t_cache + s, k_past=caches[l][0],
                                                  v_past=caches[l][1])
                caches[l][0] = np.concatenate([caches[l][0], k_new], axis=1)
                caches[l][1] = np.concatenate([caches[l][1], v_new], axis=1)
            ref = O.rmsnorm(h[:, 0, :], fg, d.eps) @ wlm.T
            assert_parity(gpu_logits[s][b:b + 1], ref, wl.dtype, f"logits seq {b} step {s}")
            compared += 1
            t = S.argmax(ref[0])
            top2 = np.sort(ref[0])[-2:]
            if top2[1] - top2[0] <= 2e-2 * np.sqrt(np.mean(ref[0] ** 2)):
                break                                         # a close call: the loops may part here
            assert int(gpu_tokens[s + 1][b]) == t, (b, s)
    assert compared >= wl.B

"""Long contexts and the paged KV cache against the oracle.

Paged: every sequence has its own length and its K/V sit in 128-position pages scattered through a
pool (a random page order); the unused rows of each last page, and every page nobody uses, are
filled with NaN, so a kernel that read a position past a sequence's end would fail the test.
Long: decode attention over 32769 and 131073 keys, RoPE at positions past 128K, and (slow) a full
8B block prefill over 32768 tokens."""
import numpy as np
import pytest

import llama_decoder_block_fwd_gb300 as L
import oracle as O
from synth import BF16, TID_KCACHE, TID_VCACHE
from synth import configs as C
from synth import host_f64
from synth import workloads as W
from tests.helpers import assert_parity, oracle_dims, sample_rows, to_f64

pytestmark = pytest.mark.gpu


def _pages_for(lengths, extra_pages=5, seed=0):
    """A block table with a random page order; returns (table [B, max_pages] int32, n_pages)."""
    need = [(n + 127) // 128 for n in lengths]
    max_pages = max(need)
    n_pages = sum(need) + extra_pages
    perm = np.random.default_rng(seed).permutation(n_pages).astype(np.int32)
    table = np.full((len(lengths), max_pages), -1, dtype=np.int32)
    k = 0
    for b, nb in enumerate(need):
        table[b, :nb] = perm[k:k + nb]
        k += nb
    table[table < 0] = perm[-1]      # unused entries point at a page no sequence uses
    return table, n_pages


def _fill_pool(pool, table, lengths, make_rows):
    """pool [n_pages, 128, n_kv, hd] <- NaN, then sequence b's rows 0..len_b-1 into its pages."""
    import torch
    pool.fill_(float("nan"))
    for b, n in enumerate(lengths):
        rows = make_rows(b, n)                     # device tensor [n, n_kv, hd]
        for j in range((n + 127) // 128):
            m = min(128, n - 128 * j)
            pool[int(table[b, j]), :m] = rows[128 * j:128 * j + m]


def _seq_cache(seed, tid, n_kv, hd, b, n):
    return W.device_tensor(BF16, (n, n_kv, hd), seed + 17 * b, tid, 0.0, 1.0)


def _seq_cache_host(seed, tid, n_kv, hd, b, n):
    return host_f64(BF16, (n, n_kv, hd), seed + 17 * b, tid, 0.0, 1.0)


@pytest.mark.parametrize("lengths,n_q,n_kv", [([1, 300, 4097, 128], 32, 8), ([129, 2000], 8, 1), ([257, 33], 16, 16)])
def test_paged_decode_attention(lengths, n_q, n_kv):
    import torch
    hd = 128
    B = len(lengths)
    table, n_pages = _pages_for(lengths, seed=len(lengths))
    kp = torch.empty((n_pages, 128, n_kv, hd), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    _fill_pool(kp, table, lengths, lambda b, n: _seq_cache(40, TID_KCACHE, n_kv, hd, b, n))
    _fill_pool(vp, table, lengths, lambda b, n: _seq_cache(40, TID_VCACHE, n_kv, hd, b, n))
    q = W.device_tensor(BF16, (B, n_q, hd), 41, 1, 0.0, 1.0)
    pos = np.array([n - 1 for n in lengths], dtype=np.int32)
    max_pos = int(pos.max())
    dims = L.dims_of(B, 1, n_q * hd, n_q, n_kv, hd, 128, 5e5, 1e-5)
    ws = torch.empty(L.llama_workspace_bytes(L.OP_GQA_ATTENTION, dims, BF16, 0, 0, max_pos + 1), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty((B, n_q, hd), dtype=torch.bfloat16, device="cuda")
    L.llama_gqa_attention_decode_paged(dims, q, kp, vp, torch.from_numpy(table).cuda(), torch.from_numpy(pos).cuda(),
                                       max_pos, o, ws)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    qh = host_f64(BF16, (B, n_q, hd), 41, 1, 0.0, 1.0)
    for b, n in enumerate(lengths):
        k = _seq_cache_host(40, TID_KCACHE, n_kv, hd, b, n)[None]
        v = _seq_cache_host(40, TID_VCACHE, n_kv, hd, b, n)[None]
        ref = O.gqa_attention(qh[b][None, None], k, v, n - 1)[0, 0]
        assert_parity(to_f64(o[b]), ref, BF16, f"paged attention seq {b} ({n} keys)")


@pytest.mark.parametrize("n_keys", [32769, 131073])
def test_long_context_decode_attention(n_keys):
    """One new token against 32K / 128K cached keys (dense layout), two sequences."""
    import torch
    B, n_q, n_kv, hd = 2, 32, 8, 128
    cap = n_keys + 7
    k = W.device_tensor(BF16, (B, cap, n_kv, hd), 50, TID_KCACHE, 0.0, 1.0)
    v = W.device_tensor(BF16, (B, cap, n_kv, hd), 50, TID_VCACHE, 0.0, 1.0)
    q = W.device_tensor(BF16, (B, 1, n_q, hd), 51, 1, 0.0, 1.0)
    dims = L.dims_of(B, 1, n_q * hd, n_q, n_kv, hd, 128, 5e5, 1e-5)
    ws = torch.empty(L.llama_workspace_bytes(L.OP_GQA_ATTENTION, dims, BF16, 0, 0, cap), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty((B, 1, n_q, hd), dtype=torch.bfloat16, device="cuda")
    L.llama_gqa_attention(dims, BF16, q, k, v, cap, n_keys - 1, o, ws)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    qh = host_f64(BF16, (B, 1, n_q, hd), 51, 1, 0.0, 1.0)
    n = B * cap * n_kv * hd
    kh = host_f64(BF16, (B, cap, n_kv, hd), 50, TID_KCACHE, 0.0, 1.0)[:, :n_keys]
    vh = host_f64(BF16, (B, cap, n_kv, hd), 50, TID_VCACHE, 0.0, 1.0)[:, :n_keys]
    ref = O.gqa_attention(qh, kh, vh, n_keys - 1)
    assert_parity(to_f64(o).reshape(B * n_q, hd), ref.reshape(B * n_q, hd), BF16, f"decode attention {n_keys} keys")


def test_rope_beyond_128k_positions():
    import torch
    B, S, n_q, n_kv, hd = 1, 64, 4, 2, 128
    pos0 = 131000
    q = W.device_tensor(BF16, (B, S, n_q, hd), 52, 1, 0.0, 1.0)
    k = W.device_tensor(BF16, (B, S, n_kv, hd), 52, 2, 0.0, 1.0)
    qh = host_f64(BF16, (B, S, n_q, hd), 52, 1, 0.0, 1.0)
    kh = host_f64(BF16, (B, S, n_kv, hd), 52, 2, 0.0, 1.0)
    dims = L.dims_of(B, S, n_q * hd, n_q, n_kv, hd, 128, 5e5, 1e-5)
    L.llama_rope(dims, BF16, q, k, pos0)
    torch.cuda.synchronize()
    pos = pos0 + np.arange(S)
    assert_parity(to_f64(q).reshape(-1, hd), O.rope(qh, pos, 5e5).reshape(-1, hd), BF16, "rope q at 131K")
    assert_parity(to_f64(k).reshape(-1, hd), O.rope(kh, pos, 5e5).reshape(-1, hd), BF16, "rope k at 131K")


def test_paged_decode_stack_variable_lengths():
    import torch
    wl = C.Workload("paged-stack", 11, C.BF16, 4, 1, 512, 4, 1, 128, 384, 5e5, 1e-5, gain_std=0.1, n_layers=3,
                    t_cache=0, vocab=1024)
    lengths = [1, 200, 5000, 129]          # cached positions per sequence (the new token is at that index)
    hkv = wl.n_kv * wl.head_dim
    table, n_pages = _pages_for([n + 1 for n in lengths], seed=3)
    kp = torch.empty((wl.n_layers, n_pages, 128, wl.n_kv, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    for l in range(wl.n_layers):
        _fill_pool(kp[l], table, lengths, lambda b, n: _seq_cache(60 + l, TID_KCACHE, wl.n_kv, wl.head_dim, b, n))
        _fill_pool(vp[l], table, lengths, lambda b, n: _seq_cache(60 + l, TID_VCACHE, wl.n_kv, wl.head_dim, b, n))
    layers = [W.device_layer(wl, l) for l in range(wl.n_layers)]
    final_g, w_lm = W.device_final(wl)
    x = W.device_x_emb(wl)
    pos = np.array(lengths, dtype=np.int32)
    max_pos = int(pos.max())
    logits = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.llama_workspace_bytes(L.OP_STACK_DECODE_STEP, wl.dims, wl.dtype, wl.n_layers, wl.vocab,
                                             max_pos + 1), dtype=torch.uint8, device="cuda")
    tt = torch.from_numpy(table).cuda()
    L.llama_stack_decode_step_paged(wl.dims, layers, final_g, w_lm, wl.vocab, x, kp, vp, tt,
                                    torch.from_numpy(pos).cuda(), max_pos, logits, ws)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    fg, wlm = W.host_final(wl)
    for b, n in enumerate(lengths):
        d = oracle_dims(wl, B=1)
        ref = O.stack_decode_step(
            W.host_x_emb(wl, [b]), lambda l: O.BlockWeights(**W.host_layer(wl, l)), wl.n_layers, d, n,
            lambda l: (_seq_cache_host(60 + l, TID_KCACHE, wl.n_kv, wl.head_dim, b, n)[None],
                       _seq_cache_host(60 + l, TID_VCACHE, wl.n_kv, wl.head_dim, b, n)[None]),
            fg, wlm)
        assert_parity(to_f64(logits[b:b + 1]), ref, wl.dtype, f"paged stack seq {b} at position {n}")
    # the new token's K landed in its page at its position; nothing else in its pages changed
    for b, n in enumerate(lengths):
        page, row = int(table[b, n // 128]), n % 128
        assert torch.isfinite(kp[0, page, row]).all()
        if row + 1 < 128:
            assert torch.isnan(kp[0, page, row + 1:]).all()


def test_llama3_8b_32_layers_paged_sampled_sequences():
    """The paged decode bench line: the 32-layer 8B stack, batch 64, each sequence's 8193 positions in
    128-position pages spread over one pool in a random order, the pool drawn per page as the bench
    draws it.  Logits of sequences 0, 31 and 63 against the oracle, which reads each sequence's
    positions back from the pages its block table names."""
    import torch
    wl = C.LLAMA3_8B_DECODE
    max_pos = wl.t_cache
    per_seq = (max_pos + 1 + 127) // 128
    n_pages = wl.B * per_seq + 1
    perm = np.random.default_rng(wl.seed).permutation(n_pages).astype(np.int32)
    table = perm[:wl.B * per_seq].reshape(wl.B, per_seq).copy()
    page_shape = (128, wl.n_kv, wl.head_dim)
    kp = torch.empty((wl.n_layers, n_pages) + page_shape, dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    for l in range(wl.n_layers):
        W.device_tensor(BF16, (n_pages,) + page_shape, wl.seed + l, TID_KCACHE, 0.0, 1.0, out=kp[l])
        W.device_tensor(BF16, (n_pages,) + page_shape, wl.seed + l, TID_VCACHE, 0.0, 1.0, out=vp[l])
    layers = [W.device_layer(wl, l) for l in range(wl.n_layers)]
    final_g, w_lm = W.device_final(wl)
    x = W.device_x_emb(wl)
    logits = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.llama_workspace_bytes(L.OP_STACK_DECODE_STEP, wl.dims, wl.dtype, wl.n_layers, wl.vocab,
                                             max_pos + 1), dtype=torch.uint8, device="cuda")
    pos = torch.full((wl.B,), max_pos, dtype=torch.int32, device="cuda")
    L.llama_stack_decode_step_paged(wl.dims, layers, final_g, w_lm, wl.vocab, x, kp, vp,
                                    torch.from_numpy(table).cuda(), pos, max_pos, logits, ws)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    got = to_f64(logits)
    del kp, vp, layers, ws
    torch.cuda.empty_cache()
    rows = [0, 31, 63]
    page_elems = 128 * wl.n_kv * wl.head_dim
    n_full = max_pos // 128                # pages 0 .. n_full-1 hold positions 0 .. max_pos-1

    def seq_cache(l, tid, b):
        return np.concatenate([host_f64(BF16, page_shape, wl.seed + l, tid, 0.0, 1.0,
                                        offset=int(table[b, j]) * page_elems) for j in range(n_full)])

    fg, wlm = W.host_final(wl)
    ref = O.stack_decode_step(W.host_x_emb(wl, rows), lambda l: O.BlockWeights(**W.host_layer(wl, l)), wl.n_layers,
                              oracle_dims(wl, B=len(rows)), max_pos,
                              lambda l: (np.stack([seq_cache(l, TID_KCACHE, b) for b in rows]),
                                         np.stack([seq_cache(l, TID_VCACHE, b) for b in rows])),
                              fg, wlm)
    assert_parity(got[rows], ref, wl.dtype, "llama3-8b paged decode logits")


@pytest.mark.slow
def test_llama3_8b_block_prefill_32k_tokens():
    """The 8B block over one 32768-token sequence (RoPE theta 5e5), 48 sampled rows."""
    import dataclasses
    import torch
    wl = dataclasses.replace(C.LLAMA3_8B_PREFILL, S=32768, name="llama3-8b-block-prefill-S32768")
    T = wl.B * wl.S
    w = W.device_layer(wl)
    x = W.device_x(wl).reshape(T, wl.d_model)
    y = torch.empty(x.shape, dtype=torch.float32, device="cuda")       # fp32 output, as the bench runs it
    ws = torch.empty(L.llama_workspace_bytes(L.OP_BLOCK_FORWARD, wl.dims, wl.dtype), dtype=torch.uint8, device="cuda")
    L.llama_block_forward(wl.dims, wl.dtype | L.Y_F32, L.block_weights(w), x, y, 0, None, None, 0, ws)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    rows = sample_rows(wl.S, 48)
    hw = O.BlockWeights(**W.host_layer(wl))
    xh = W.host_x(wl, 0)[None]
    ref, _, _ = O.block_forward(xh, hw, oracle_dims(wl), rows=rows)
    assert_parity(to_f64(y)[rows], ref[0], wl.dtype, "8B block prefill S=32768")

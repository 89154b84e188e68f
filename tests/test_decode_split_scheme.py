"""A model of the bf16 decode attention's work split, written out in Python, and the invariants the
kernel and its combine pass rely on: the 128-key tiles of all (sequence, KV group) pairs, in
(b, g, tile) order, are cut into one equal contiguous range per CTA; every tile lands in exactly one
piece; the piece of pair q cut by CTA c writes slot q + c, and those slots are distinct and below
B n_kv + G; and the combine's CTA span c0..c1 of a pair (skipping empty ranges) is exactly the set
of CTAs that wrote one of its pieces.  Dense caches (every sequence the same length) and paged
ones (a length per sequence).  This checks the scheme; the GPU parity tests check the kernel."""
import random

import pytest

def seq_tiles(seq_pos, kv_tiles, b):
    """Tiles of sequence b: a paged cache holds seq_pos[b] + 1 keys, a dense one kv_tiles tiles."""
    return (seq_pos[b] + 1 + 127) // 128 if seq_pos is not None else kv_tiles


def all_tiles(seq_pos, kv_tiles, B, n_kv):
    if seq_pos is None:
        return B * n_kv * kv_tiles
    return sum(seq_tiles(seq_pos, kv_tiles, b) for b in range(B)) * n_kv


def range_begin(T, G, c):
    return c * T // G


def cta_of(T, G, x):
    """The CTA whose range holds tile x (the last of several with the same start)."""
    c = min(G - 1, x * G // T)
    while c + 1 < G and range_begin(T, G, c + 1) <= x:
        c += 1
    while c > 0 and range_begin(T, G, c) > x:
        c -= 1
    return c


def pair_span(seq_pos, kv_tiles, n_kv, b, g):
    """First tile of pair (b, g) in the sequence, and its tile count."""
    if seq_pos is None:
        return (b * n_kv + g) * kv_tiles, kv_tiles
    before = sum(seq_tiles(seq_pos, kv_tiles, bb) for bb in range(b))
    nt = seq_tiles(seq_pos, kv_tiles, b)
    return before * n_kv + g * nt, nt


def pieces(B, n_kv, kv_tiles, seq_pos, G, c):
    """CTA c's pieces: (b, g, first tile, end tile, partial slot)."""
    T = all_tiles(seq_pos, kv_tiles, B, n_kv)
    x, end = range_begin(T, G, c), range_begin(T, G, c + 1)
    out = []
    if x >= end:
        return out
    if seq_pos is None:
        pair = x // kv_tiles
        b, g, nt, off = pair // n_kv, pair % n_kv, kv_tiles, pair * kv_tiles
    else:
        o, b = 0, 0
        while True:
            nt = seq_tiles(seq_pos, kv_tiles, b)
            if x < o + n_kv * nt:
                break
            o += n_kv * nt
            b += 1
        g = (x - o) // nt
        off = o + g * nt
    while x < end:
        t0, t1 = x - off, min(nt, end - off)
        out.append((b, g, t0, t1, b * n_kv + g + c))
        x = off + t1
        if t1 == nt:
            off += nt
            g += 1
            if g == n_kv:
                g, b = 0, b + 1
                if b < B:
                    nt = seq_tiles(seq_pos, kv_tiles, b)
    return out


def check(B, n_kv, kv_tiles, seq_pos, G):
    T = all_tiles(seq_pos, kv_tiles, B, n_kv)
    covered, slots, writers = {}, set(), {}
    for c in range(G):
        for b, g, t0, t1, slot in pieces(B, n_kv, kv_tiles, seq_pos, G, c):
            assert 0 <= t0 < t1, (b, g, t0, t1)
            for t in range(t0, t1):
                assert (b, g, t) not in covered            # no tile twice
                covered[(b, g, t)] = c
            assert slot not in slots and 0 <= slot < B * n_kv + G
            slots.add(slot)
            writers.setdefault((b, g), set()).add(c)
    for b in range(B):
        for g in range(n_kv):
            off, nt = pair_span(seq_pos, kv_tiles, n_kv, b, g)
            for t in range(nt):
                assert (b, g, t) in covered, (b, g, t)     # every tile once
            c0, c1 = cta_of(T, G, off), cta_of(T, G, off + nt - 1)
            span = {c for c in range(c0, c1 + 1) if range_begin(T, G, c) < range_begin(T, G, c + 1)}
            assert span == writers[(b, g)], (b, g, span, writers[(b, g)])
    assert len(covered) == T

@pytest.mark.parametrize("B,n_kv,kv_len", [(64, 8, 8193), (16, 8, 32769), (2, 8, 131073), (3, 8, 1040),
                                          (1, 1, 1), (2, 1, 4000), (5, 4, 300), (1, 16, 777), (2, 2, 129)])
@pytest.mark.parametrize("G", [152, 151, 7, 1, 256])
def test_dense_split_invariants(B, n_kv, kv_len, G):
    kt = (kv_len + 127) // 128
    check(B, n_kv, kt, None, max(1, min(G, B * n_kv * kt)))   # a dense grid has at most one CTA per tile


def test_paged_split_invariants_random_lengths():
    rnd = random.Random(1)
    for _ in range(300):
        B = rnd.randint(1, 12)
        n_kv = rnd.choice([1, 2, 4, 8])
        G = rnd.choice([1, 3, 17, 152, 256])
        lens = [rnd.choice([0, 1, 127, 128, 129, 4096, rnd.randint(0, 20000)]) for _ in range(B)]
        check(B, n_kv, None, lens, G)

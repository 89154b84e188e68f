"""Pins of the sampling and embedding oracle ("LLaMA-3 8B 现代 LLM 架构、计算规模与能耗", sections
三 and 十) against what the page states and what the mathematics fixes: argmax picks the most
probable token, top-k keeps the k most probable, top-p the smallest set reaching mass p, the
temperature sharpens (T -> 0: argmax) or flattens (T -> inf: uniform) the distribution, and the
draw reproduces the softmax probabilities.  A plausible slip (ties to the higher id, top-p
cutting one token early or late, the temperature multiplying instead of dividing, u compared on
the wrong side) fails one of them."""
import math

import numpy as np
import pytest

from oracle import sampling as S


def test_argmax_and_ties_to_lower_id():
    z = np.array([1.0, 3.0, 3.0, 2.0])
    assert S.argmax(z) == 1
    assert S.sample(z, 0.0, 0, 1.0, 0.99) == 1          # T = 0 is argmax whatever u
    assert S.sample(z, 1.0, 1, 1.0, 0.99) == 1          # top-k = 1 is argmax whatever u
    assert list(S.order_desc(z)) == [1, 2, 3, 0]


def test_top_k_keeps_the_k_largest_with_ties_by_id():
    z = np.array([1.0, 3.0, 3.0, 2.0])
    assert list(S.kept_set(z, 1.0, 2, 1.0)) == [1, 2]
    assert list(S.kept_set(z, 1.0, 3, 1.0)) == [1, 2, 3]
    assert list(S.kept_set(z, 1.0, 0, 1.0)) == [1, 2, 3, 0]     # k <= 0: no filter
    assert list(S.kept_set(z, 1.0, 99, 1.0)) == [1, 2, 3, 0]    # k >= vocab: no filter
    # a draw never leaves the top-k set
    for u in np.linspace(0, 0.999, 50):
        assert S.sample(z, 1.0, 2, 1.0, u) in (1, 2)


def test_top_p_smallest_prefix_reaching_p():
    p = np.array([0.5, 0.2, 0.2, 0.1])
    z = np.log(p)
    assert list(S.kept_set(z, 1.0, 0, 0.6)) == [0, 1]       # 0.5 < 0.6 <= 0.7; tie 1/2 -> id 1
    assert list(S.kept_set(z, 1.0, 0, 0.45)) == [0]         # 0.5 already reaches 0.45
    assert list(S.kept_set(z, 1.0, 0, 0.75)) == [0, 1, 2]
    assert list(S.kept_set(z, 1.0, 0, 0.95)) == [0, 1, 2, 3]
    # top-p after top-k: the mass is the top-k set's (0.5 / 0.7 = 0.714 >= 0.7)
    assert list(S.kept_set(z, 1.0, 2, 0.7)) == [0]
    # renormalised draw over {0, 1}: token 0 for u < 5/7, token 1 above
    assert S.sample(z, 1.0, 0, 0.6, 0.70) == 0
    assert S.sample(z, 1.0, 0, 0.6, 0.72) == 1


def test_draw_frequencies_reproduce_softmax():
    rng = np.random.default_rng(7)
    z = rng.normal(0, 1.5, 12)
    N = 20000
    us = (np.arange(N) + 0.5) / N
    counts = np.bincount([S.sample(z, 1.0, 0, 1.0, u) for u in us], minlength=12)
    p = np.exp(z - z.max())
    p /= p.sum()
    assert np.all(np.abs(counts - N * p) <= 1.0)
    # the same with top-p 0.6 on the page-style example: 5/7 and 2/7
    z2 = np.log(np.array([0.5, 0.2, 0.2, 0.1]))
    c2 = np.bincount([S.sample(z2, 1.0, 0, 0.6, u) for u in us], minlength=4)
    assert abs(c2[0] - N * 5 / 7) <= 1 and abs(c2[1] - N * 2 / 7) <= 1 and c2[2] == c2[3] == 0


def test_temperature_limits():
    z = np.array([0.3, 2.0, -1.0, 1.9, 0.0])
    # T -> 0+: every u picks the argmax
    for u in np.linspace(0, 0.999, 40):
        assert S.sample(z, 1e-4, 0, 1.0, u) == 1
    # T -> inf: uniform over the vocabulary, walked in id order: token floor(u * V)
    V = z.shape[0]
    for i in range(V):
        u = (i + 0.5) / V
        assert S.sample(z, 1e9, 0, 1.0, u) == i
    # T divides the logits: T = 2 on z equals T = 1 on z / 2 (and differs from T = 1 on 2z)
    us = np.linspace(0.01, 0.99, 60)
    a = [S.sample(z, 2.0, 0, 1.0, u) for u in us]
    assert a == [S.sample(z / 2, 1.0, 0, 1.0, u) for u in us]
    assert a != [S.sample(2 * z, 1.0, 0, 1.0, u) for u in us]


def test_minus_infinity_logits_are_never_drawn():
    z = np.array([-np.inf, 0.0, -np.inf, 1.0])
    for u in np.linspace(0, 0.999, 40):
        assert S.sample(z, 1.0, 0, 1.0, u) in (1, 3)
    assert S.sample(z, 1.0, 0, 1.0, 0.0) == 1
    assert S.sample(z, 1.0, 0, 1.0, 0.999) == 3


def test_margins_flag_boundaries():
    z = np.log(np.array([0.5, 0.2, 0.2, 0.1]))
    # u * kept mass exactly on the 5/7 boundary of the {0, 1} draw
    _, m_u = S.sample_margins(z, 1.0, 0, 0.6, 5 / 7)
    assert m_u < 1e-12
    m_cut, _ = S.sample_margins(z, 1.0, 0, 0.7, 0.1)
    assert m_cut < 1e-12                                   # 0.5 + 0.2 sits on p = 0.7
    m_cut, m_u = S.sample_margins(z, 1.0, 0, 0.6, 0.3)
    assert m_cut == pytest.approx(0.1) and m_u > 0.1


def test_embedding_is_a_row_lookup():
    rng = np.random.default_rng(3)
    E = rng.normal(size=(10, 6))
    tokens = [3, 0, 9, 3]
    x = S.embed(E, tokens)
    onehot = np.zeros((4, 10))
    onehot[np.arange(4), tokens] = 1.0
    assert np.array_equal(x, onehot @ E)
    assert x.shape == (4, 6) and math.isclose(x[0, 2], E[3, 2])

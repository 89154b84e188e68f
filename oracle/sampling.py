"""fp64 CPU oracle for the steps either side of the decode stack: the embedding lookup that turns
token ids into input rows, and the choice of the next token from the LM head's logits.

TEST INFRASTRUCTURE ONLY (the same rule as llama_oracle.py): only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs may import it.

Sources (page title, section):
  [P3] "LLaMA-3 8B 现代 LLM 架构、计算规模与能耗": section 三 (the embedding is a row lookup in
       the [vocab, d_model] table), section 十 (softmax over the vocabulary, then argmax, or
       sampling shaped by temperature, top-k and top-p; the sampled token goes back to the
       embedding for the next step).

The page names the four rules without formulas.  Readings taken:
  * temperature T > 0 divides the logits before the softmax; T <= 0 means argmax.
  * argmax and every "most probable" ordering rank tokens by logit, larger first, and break
    ties by the lower token id (the order is total, so every set below is unique).
  * top-k keeps the first k tokens of that order (k <= 0 or k >= vocab keeps all).
  * top-p is applied after top-k: it keeps the shortest prefix of the order whose share of the
    top-k set's probability mass reaches p (p >= 1 keeps all).
  * the token is drawn by inverse CDF with a caller-supplied uniform u in [0, 1), walking the
    kept tokens in increasing token id: the first id whose cumulative mass exceeds u times the
    kept mass.
"""
import numpy as np


def embed(table: np.ndarray, tokens) -> np.ndarray:
    """[P3 三] x[b] = E[token_b]: row token_b of the [vocab, d_model] table."""
    return np.asarray(table, dtype=np.float64)[np.asarray(tokens, dtype=np.int64)]


def order_desc(z: np.ndarray) -> np.ndarray:
    """Token ids ranked by logit, larger first, ties by the lower id."""
    z = np.asarray(z, dtype=np.float64)
    ids = np.arange(z.shape[0])
    return np.lexsort((ids, -z))


def argmax(z: np.ndarray) -> int:
    """[P3 十] argmax: the most probable token (the lowest id among equal maxima)."""
    return int(order_desc(z)[0])


def kept_set(z: np.ndarray, temperature: float, top_k: int, top_p: float) -> np.ndarray:
    """[P3 十] The candidate tokens after top-k and top-p, in ranked order."""
    z = np.asarray(z, dtype=np.float64)
    order = order_desc(z)
    V = z.shape[0]
    if temperature <= 0 or top_k == 1:
        return order[:1]
    n = V if (top_k <= 0 or top_k >= V) else int(top_k)
    kept = order[:n]
    if top_p < 1.0:
        # softmax over the top-k set at temperature T (unnormalised: the shift by the max cancels)
        mass = np.exp((z[kept] - z[order[0]]) / temperature)
        cum = np.cumsum(mass)
        need = top_p * cum[-1]
        n_p = 1
        while cum[n_p - 1] < need:
            n_p += 1
        kept = kept[:n_p]
    return kept


def sample(z: np.ndarray, temperature: float, top_k: int, top_p: float, u: float) -> int:
    """[P3 十] One draw from softmax(z / T) restricted to the kept set, by inverse CDF in token-id
    order with the uniform u in [0, 1)."""
    z = np.asarray(z, dtype=np.float64)
    kept = kept_set(z, temperature, top_k, top_p)
    if kept.shape[0] == 1:
        return int(kept[0])
    ids = np.sort(kept)
    mass = np.exp((z[ids] - z.max()) / temperature)
    total = mass.sum()
    acc = 0.0
    for i, m in zip(ids, mass):
        acc += m
        if acc > u * total:
            return int(i)
    return int(ids[-1])


def sample_margins(z: np.ndarray, temperature: float, top_k: int, top_p: float, u: float):
    """How far the draw is from changing: the relative gap between the top-p cut and its target,
    and between u * kept mass and the nearest cumulative boundary (inf when the rule does not
    apply).  A float32 implementation that agrees with this oracle only up to rounding can
    choose differently only where one of these is of the order of its rounding error."""
    z = np.asarray(z, dtype=np.float64)
    order = order_desc(z)
    V = z.shape[0]
    if temperature <= 0 or top_k == 1:
        return np.inf, np.inf
    n = V if (top_k <= 0 or top_k >= V) else int(top_k)
    topk = order[:n]
    m_cut = np.inf
    kept = topk
    if top_p < 1.0:
        mass = np.exp((z[topk] - z[order[0]]) / temperature)
        cum = np.cumsum(mass)
        need = top_p * cum[-1]
        m_cut = float(np.min(np.abs(cum - need)) / cum[-1])
        kept = kept_set(z, temperature, top_k, top_p)
    if kept.shape[0] == 1:
        return m_cut, np.inf
    ids = np.sort(kept)
    mass = np.exp((z[ids] - z.max()) / temperature)
    cum = np.cumsum(mass)
    m_u = float(np.min(np.abs(cum - u * cum[-1])) / cum[-1])
    return m_cut, m_u

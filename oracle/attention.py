"""Single-token decode attention over a gathered KV context, in fp64.

Test infrastructure only (see the package docstring).

What is computed is the plain definition of scaled dot-product attention for
one new query token against every cached key and value of its sequence
([B] §3.1: the new token's query attends to the cached K and V of all
previous tokens; [E] §1: each decode step reads the whole cache):

    s_t = (q_h . k_t) * sm_scale
    w   = softmax(s)            (max-subtracted, fp64)
    o_h = sum_t w_t v_t

Grouped-query attention ([A] §2: eight KV heads thanks to GQA): query head h
reads kv head h // (Hq / Hkv) -- contiguous groups, the plainest reading; the
pages do not say which grouping. sm_scale is passed in (1/sqrt(head_dim) by
default in callers).

Paging, splitting the context and online softmax are ways of reaching this
same result faster ([C] §2, the FlashAttention tiling idea); the oracle does
none of them. ``partial_state`` and ``merge_partials`` are the plain
definitions a split computation has to agree with: the softmax of a whole
context equals the merge of the softmax states of any partition of it.
"""

from __future__ import annotations

import numpy as np


def kv_head_of(q_head: int, num_q_heads: int, num_kv_heads: int) -> int:
    if num_q_heads % num_kv_heads:
        raise ValueError("Hq must be a multiple of Hkv")
    return q_head // (num_q_heads // num_kv_heads)


def decode_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float,
                     return_weights: bool = False):
    """Attention of one query token per head over a contiguous context.

    q: [Hq, d]; k, v: [n, Hkv, d] (any float dtype; computed in fp64).
    Returns out [Hq, d] fp64 (and the softmax weights [Hq, n] if asked).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    hq, d = q.shape
    n, hkv, dk = k.shape
    if n < 1:
        raise ValueError("a decode step attends over at least one token")
    if dk != d or v.shape != k.shape:
        raise ValueError("shape mismatch")
    out = np.empty((hq, d), dtype=np.float64)
    weights = np.empty((hq, n), dtype=np.float64)
    for h in range(hq):
        g = kv_head_of(h, hq, hkv)
        s = (k[:, g, :] @ q[h]) * float(sm_scale)
        e = np.exp(s - np.max(s))
        w = e / np.sum(e)
        weights[h] = w
        out[h] = w @ v[:, g, :]
    return (out, weights) if return_weights else out


def partial_state(q_h: np.ndarray, k_g: np.ndarray, v_g: np.ndarray, sm_scale: float,
                  base: float = np.e):
    """Unnormalised softmax state of one query head over part of a context.

    With x_t = s_t / ln(base) (so that base**x_t == e**s_t):
    m = max_t x_t, l = sum_t base**(x_t - m), o = sum_t base**(x_t - m) v_t.
    """
    q_h = np.asarray(q_h, dtype=np.float64)
    k_g = np.asarray(k_g, dtype=np.float64)
    v_g = np.asarray(v_g, dtype=np.float64)
    x = (k_g @ q_h) * float(sm_scale) / np.log(base)
    m = np.max(x)
    p = np.power(base, x - m)
    return m, np.sum(p), p @ v_g


def merge_partials(ms, ls, os_, base: float = np.e) -> np.ndarray:
    """Normalised output from the softmax states of the parts of a partition.

    M = max_j m_j;  L = sum_j l_j base**(m_j - M);  O = sum_j o_j base**(m_j - M) / L.
    """
    ms = np.asarray(ms, dtype=np.float64)
    ls = np.asarray(ls, dtype=np.float64)
    os_ = np.asarray(os_, dtype=np.float64)
    big = np.max(ms)
    c = np.power(base, ms - big)
    return (c @ os_) / np.sum(c * ls)

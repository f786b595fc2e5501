"""Oracle for the draft model's sliding-window self-attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this module; the product path never
does. Plain numpy in fp64, one (sequence, query, head) at a time.

What the pages fix ("LongSpec: Long-Context Lossless Speculative Decoding with
Efficient Drafting and Verification", Korean summary section 2.A and Dutch
summary Methodologie section 1, "Self-Attention"): the draft model's
self-attention uses a sliding window of 512 positions so that its KV cache
stays the same size whatever the context length. Readings taken where the
pages are silent: the cache is a ring of S slots per sequence and KV head
(position j in slot j mod S); a query at position p attends causally to the W
most recent positions up to its own, max(0, p - W + 1) .. p. With T new
queries per call the ring needs S >= W + T - 1 slots: the first query still
reads W - 1 positions that the last T - 1 new ones would otherwise overwrite.
Softmax scale 1/sqrt(d) unless given; the log-sum-exp is the natural log of
the softmax denominator of the scaled scores; query head hq reads KV head
hq // (Hq / Hkv).
"""
from __future__ import annotations

import math

import numpy as np


def _f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64: a bf16 is the top half of an fp32."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def window_attention(q, k_ring, v_ring, pos, window: int, scale: float = 0.0):
    """q [B][T][Hq][d], k_ring/v_ring [B][Hkv][S][d] (uint16 bf16 bits),
    pos [B] (position of query 0), window W with W + T - 1 <= S. Returns
    (o [B][T][Hq][d], lse [B][T][Hq]) in float64."""
    qf, kf, vf = _f64(q), _f64(k_ring), _f64(v_ring)
    B, T, Hq, d = qf.shape
    _, Hkv, S, _ = kf.shape
    W = int(window)
    if W < 1 or W + T - 1 > S:
        raise ValueError("need 1 <= window and window + T - 1 <= ring slots")
    G = Hq // Hkv
    s = scale if scale > 0 else 1.0 / math.sqrt(d)
    o = np.zeros((B, T, Hq, d))
    lse = np.zeros((B, T, Hq))
    for b in range(B):
        P = int(pos[b])
        for t in range(T):
            p = P + t
            js = np.arange(max(0, p - W + 1), p + 1)  # visible positions
            slots = js % S
            for hq in range(Hq):
                kv = hq // G
                sc = s * (kf[b, kv, slots] @ qf[b, t, hq])
                m = sc.max()
                e = np.exp(sc - m)
                o[b, t, hq] = (e @ vf[b, kv, slots]) / e.sum()
                lse[b, t, hq] = m + math.log(e.sum())
    return o, lse

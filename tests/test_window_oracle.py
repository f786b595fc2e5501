"""Pins for the sliding-window oracle (oracle/window.py), on CPU.

The window rule ("LongSpec: Long-Context Lossless Speculative Decoding with
Efficient Drafting and Verification", Korean summary 2.A, Dutch summary
section 1): a query at position p sees positions max(0, p - W + 1) .. p. The
references here unroll the ring into a linear sequence of positions and use
torch's fp64 scaled-dot-product attention with an explicitly built band mask,
or closed forms, or explicit fsum sums.
"""
import math

import numpy as np
import pytest
import torch

from oracle.window import window_attention
from speculative_decoding_tree_hybrid_gb300 import workloads as wl


def _f64(bits):
    return torch.from_numpy((np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)).double()


def _linear(inp, b):
    """Positions lo .. end-1 of sequence b as [Hkv][n][d] (read from the ring), and lo."""
    S = inp.S
    end = int(inp.pos[b]) + inp.q.shape[1]
    lo = max(0, end - S)
    js = np.arange(lo, end)
    return _f64(inp.k_ring[b][:, js % S]), _f64(inp.v_ring[b][:, js % S]), lo


def _sdpa_band(inp, b, window):
    """Attention of sequence b's queries over its linear positions with mask
    allowed[t][j] = (p_t - window < j <= p_t), p_t = pos + t."""
    B, T, Hq, d = inp.q.shape
    k, v, lo = _linear(inp, b)
    Hkv = k.shape[0]
    G = Hq // Hkv
    n = k.shape[1]
    j = torch.arange(lo, lo + n)[None, :]
    p = (int(inp.pos[b]) + torch.arange(T))[:, None]
    allowed = (j <= p) & (j > p - window)
    q = _f64(inp.q[b]).permute(1, 0, 2)  # [Hq][T][d]
    kk = k.repeat_interleave(G, 0)
    vv = v.repeat_interleave(G, 0)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=allowed)
    sc = (q @ kk.transpose(1, 2)) / math.sqrt(d)
    sc = sc.masked_fill(~allowed, -math.inf)
    lse = torch.logsumexp(sc, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("T,pos", [(1, [0, 5]), (4, [0, 12]), (6, [3, 50]), (8, [0, 0])])
def test_window_covering_everything_is_causal_attention(T, pos):
    # W >= pos + T: the last query, and so every query, sees every earlier position
    W = max(pos) + T
    S = W + T - 1
    inp = wl.window_inputs(2, T, 4, 2, 16, S, pos, seed=T * 100 + S)
    o, lse = window_attention(inp.q, inp.k_ring, inp.v_ring, inp.pos, W)
    for b in range(2):
        assert int(inp.pos[b]) + T <= W
        ro, rl = _sdpa_band(inp, b, window=10 ** 9)
        np.testing.assert_allclose(o[b], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl, rtol=1e-13)


@pytest.mark.parametrize("T,W,pos", [(1, 4, [9, 100]), (5, 8, [20, 3]), (16, 16, [40, 31]), (3, 32, [1000, 0]),
                                     (7, 1, [12, 0])])
def test_short_window_is_banded_causal_attention(T, W, pos):
    S = W + T - 1 + 3  # a ring a little longer than needed
    inp = wl.window_inputs(2, T, 6, 3, 32, S, pos, seed=7 * T + W)
    o, lse = window_attention(inp.q, inp.k_ring, inp.v_ring, inp.pos, W)
    for b in range(2):
        ro, rl = _sdpa_band(inp, b, window=W)
        np.testing.assert_allclose(o[b], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl, rtol=1e-13)


def test_window_of_one_returns_own_value():
    inp = wl.window_inputs(2, 3, 4, 4, 8, 3, [17, 0], seed=3)
    o, lse = window_attention(inp.q, inp.k_ring, inp.v_ring, inp.pos, 1)
    q, k, v = _f64(inp.q).numpy(), _f64(inp.k_ring).numpy(), _f64(inp.v_ring).numpy()
    for b in range(2):
        for t in range(3):
            slot = (int(inp.pos[b]) + t) % 3
            for h in range(4):
                np.testing.assert_array_equal(o[b, t, h], v[b, h, slot])
                assert lse[b, t, h] == pytest.approx(q[b, t, h] @ k[b, h, slot] / math.sqrt(8), rel=1e-14)


def test_slots_outside_the_window_are_never_read():
    # a ring longer than W + T - 1 holds live positions no query sees: making
    # them NaN changes nothing; the oldest position query 1 sees is not seen by
    # query 0
    T, W, S, P = 2, 8, 12, 100
    inp = wl.window_inputs(1, T, 2, 1, 8, S, [P], seed=5)
    o1, l1 = window_attention(inp.q, inp.k_ring, inp.v_ring, inp.pos, W)
    assert np.isfinite(o1).all() and np.isfinite(l1).all()
    k2, v2 = inp.k_ring.copy(), inp.v_ring.copy()
    unseen = [j % S for j in range(P + T - S, P - W + 1)]  # live, older than any window
    assert unseen
    k2[0][:, unseen] = wl.BF16_NAN
    v2[0][:, unseen] = wl.BF16_NAN
    o2, l2 = window_attention(inp.q, k2, v2, inp.pos, W)
    np.testing.assert_array_equal(o2, o1)
    k3, v3 = inp.k_ring.copy(), inp.v_ring.copy()
    only_q1 = (P + 1 - W + 1) - 1  # position P - W + 1: seen by query 0 only
    k3[0][:, only_q1 % S] = wl.BF16_NAN
    o3, _ = window_attention(inp.q, k3, v3, inp.pos, W)
    assert np.isnan(o3[0, 0]).all() and np.isfinite(o3[0, 1]).all()


def test_brute_force_tiny_with_fsum():
    inp = wl.window_inputs(1, 3, 2, 1, 4, 5, [2], seed=11)
    W, S, d = 3, 5, 4
    o, lse = window_attention(inp.q, inp.k_ring, inp.v_ring, inp.pos, W)
    q, k, v = _f64(inp.q).numpy(), _f64(inp.k_ring).numpy(), _f64(inp.v_ring).numpy()
    for t in range(3):
        p = 2 + t
        for h in range(2):
            keys = [j for j in range(p + 1) if j > p - W]
            sc = [math.fsum(q[0, t, h, c] * k[0, 0, j % S, c] for c in range(d)) / 2.0 for j in keys]
            den = math.fsum(math.exp(x) for x in sc)
            for c in range(d):
                num = math.fsum(math.exp(x) * v[0, 0, j % S, c] for x, j in zip(sc, keys))
                assert o[0, t, h, c] == pytest.approx(num / den, rel=1e-12, abs=1e-14)
            assert lse[0, t, h] == pytest.approx(math.log(den), rel=1e-12)


def test_ring_too_short_is_rejected():
    inp = wl.window_inputs(1, 4, 2, 1, 8, 6, [10], seed=1)
    with pytest.raises(ValueError):
        window_attention(inp.q, inp.k_ring, inp.v_ring, inp.pos, 4)  # needs 4 + 3 = 7 slots

"""Pins of the CPU oracle against facts the pages and the mathematics fix.

No test here re-types the oracle's own loop. Each compares the oracle with
something independent of it:
  * the exactness claim of the split method (cached part + speculative part
    merged by log-sum-exp equals the single softmax), with the merge formula
    applied here to two separate oracle calls over disjoint key sets;
  * library routines (torch SDPA / logsumexp in fp64, networkx ancestors) on
    trees whose mask has a textbook form (chain = causal, star, single node);
  * brute force over every tree with T <= 4 and short prefixes, with sets
    built by recursion and sums taken by math.fsum without a max shift;
  * hand-derived closed forms in tests/golden/;
  * invariants (weights sum to one, convex hull, LSE bounds, permutation
    and relabelling symmetry, GQA replication, empty prefix).
Sources: "LongSpec: Long-Context Lossless Speculative Decoding with Efficient
Drafting and Verification" (Korean summary section 2.C, Dutch summary
Methodologie section 3) and "LogitSpec: Accelerating Retrieval-based
Speculative Decoding via Next Next Token Speculation" (section 2, step 2).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from speculative_decoding_tree_hybrid_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def expand_kv(x, G):
    # [B][Hkv][L][d] -> [B][Hq][L][d], head hq reads kv head hq // G
    return np.repeat(x, G, axis=1)


def sdpa_reference(inp, visible_spec, scale=None):
    """torch fp64 attention over [prefix || spec] with an explicit bool mask.

    visible_spec[b][t] is the set of spec indices node t may see, built by the
    caller from the tree's textbook shape (not from a parent walk).
    Returns (o [B][T][Hq][d], lse [B][T][Hq]).
    """
    B, T, Hq, d = inp.q.shape
    Hkv = inp.k_cache.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = np.zeros((B, T, Hq, d))
    lse = np.zeros((B, T, Hq))
    for b in range(B):
        L = int(inp.cache_lens[b])
        k = np.concatenate([f64(inp.k_cache[b, :, :L]), f64(inp.k_spec[b])], axis=1)
        v = np.concatenate([f64(inp.v_cache[b, :, :L]), f64(inp.v_spec[b])], axis=1)
        k = torch.from_numpy(expand_kv(k[None], G)[0])  # [Hq][L+T][d]
        v = torch.from_numpy(expand_kv(v[None], G)[0])
        q = torch.from_numpy(f64(inp.q[b])).permute(1, 0, 2)  # [Hq][T][d]
        allow = torch.zeros(T, L + T, dtype=torch.bool)
        allow[:, :L] = True
        for t in range(T):
            for j in visible_spec[b][t]:
                allow[t, L + j] = True
        out = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=allow, scale=scale)
        scores = (q @ k.transpose(-1, -2)) * scale
        scores = scores.masked_fill(~allow, float("-inf"))
        o[b] = out.permute(1, 0, 2).numpy()
        lse[b] = torch.logsumexp(scores, dim=-1).permute(1, 0).numpy()
    return o, lse


def run_oracle(oracle_mod, inp, mask=None, lens=None, scale=0.0):
    if mask is None:
        mask, bad = oracle_mod.build_mask(inp.parents)
        assert bad == 0
    lens = inp.cache_lens if lens is None else lens
    return oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, lens, inp.k_spec,
                                inp.v_spec, mask, scale=scale)


def lse_merge(o1, l1, o2, l2):
    """The log-sum-exp merge of two partial softmaxes (merge step of the method)."""
    m = np.maximum(l1, l2)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w1 = np.exp(l1 - m_safe)
    w2 = np.exp(l2 - m_safe)
    o = (w1[..., None] * o1 + w2[..., None] * o2) / (w1 + w2)[..., None]
    return o, m_safe + np.log(w1 + w2)


# ------------------------------------------------------------------ exactness

@pytest.mark.parametrize("lens", [[37, 0], [1, 64], [64, 5]])
def test_split_plus_merge_equals_single_softmax(oracle_mod, lens):
    inp = wl.random_inputs(2, 12, 6, 2, 16, lens, seed=3, Lmax=64)
    mask, _ = oracle_mod.build_mask(inp.parents)
    o_full, lse_full = run_oracle(oracle_mod, inp, mask)
    # cached part: no tree key visible; speculative part: no cache key visible
    o_c, lse_c = run_oracle(oracle_mod, inp, np.zeros_like(mask))
    o_s, lse_s = run_oracle(oracle_mod, inp, mask, lens=np.zeros(2, np.int32))
    o_m, lse_m = lse_merge(o_c, lse_c, o_s, lse_s)
    assert np.abs(o_m - o_full).max() <= 1e-12
    assert np.abs(lse_m - lse_full).max() <= 1e-12 * max(1.0, np.abs(lse_full).max())
    # an empty prefix gives LSE_c = -inf and O_c = 0
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(np.isneginf(lse_c[b])) and np.all(o_c[b] == 0)


# ------------------------------------------------------------------ textbook trees

@pytest.mark.parametrize("T,L,Hq,Hkv,d", [(16, 40, 4, 2, 32), (5, 0, 2, 2, 8), (33, 7, 3, 1, 64)])
def test_chain_tree_is_causal_attention(oracle_mod, T, L, Hq, Hkv, d):
    inp = wl.random_inputs(1, T, Hq, Hkv, d, [L], seed=T + L,
                           parents=wl.tree_chain(T)[None])
    o, lse = run_oracle(oracle_mod, inp)
    causal = [[list(range(t + 1)) for t in range(T)]]
    o_ref, lse_ref = sdpa_reference(inp, causal)
    assert np.abs(o - o_ref).max() <= 1e-12
    assert np.abs(lse - lse_ref).max() <= 1e-12


@pytest.mark.parametrize("T", [2, 9, 40])
def test_star_tree(oracle_mod, T):
    inp = wl.random_inputs(2, T, 4, 4, 16, [25, 3], seed=T, parents=np.stack([wl.tree_star(T)] * 2))
    mask, bad = oracle_mod.build_mask(inp.parents)
    assert bad == 0
    pop = np.array([[sum(bin(int(w)).count("1") for w in row) for row in mb] for mb in mask])
    assert pop[:, 0].tolist() == [1, 1] and (pop[:, 1:] == 2).all()
    o, lse = run_oracle(oracle_mod, inp, mask)
    star = [[[0]] + [[0, t] for t in range(1, T)]] * 2
    o_ref, lse_ref = sdpa_reference(inp, star)
    assert np.abs(o - o_ref).max() <= 1e-12
    assert np.abs(lse - lse_ref).max() <= 1e-12


def test_single_node_is_plain_decode(oracle_mod):
    inp = wl.random_inputs(3, 1, 8, 2, 64, [100, 1, 0], seed=11, Lmax=100)
    o, lse = run_oracle(oracle_mod, inp)
    o_ref, lse_ref = sdpa_reference(inp, [[[0]]] * 3)
    assert np.abs(o - o_ref).max() <= 1e-12
    assert np.abs(lse - lse_ref).max() <= 1e-12


# ------------------------------------------------------------------ brute force

def _all_trees(T):
    choices = [[-1]] + [list(range(-1, i)) for i in range(1, T)]
    for par in itertools.product(*choices):
        yield np.array(par, dtype=np.int32)


def _anc(par, i):
    return set() if i == -1 else {i} | _anc(par, int(par[i]))


@pytest.mark.parametrize("L", [0, 1, 16])
def test_brute_force_every_small_tree(oracle_mod, L):
    d, Hq, Hkv = 4, 2, 1
    count = 0
    for T in range(1, 5):
        for par in _all_trees(T):
            inp = wl.random_inputs(1, T, Hq, Hkv, d, [L], seed=count, parents=par[None], Lmax=16)
            o, lse = run_oracle(oracle_mod, inp)
            q = f64(inp.q[0])
            kc, vc = f64(inp.k_cache[0, 0]), f64(inp.v_cache[0, 0])
            ks, vs = f64(inp.k_spec[0, 0]), f64(inp.v_spec[0, 0])
            for t in range(T):
                keys = [kc[j] for j in range(L)] + [ks[j] for j in sorted(_anc(par, t))]
                vals = [vc[j] for j in range(L)] + [vs[j] for j in sorted(_anc(par, t))]
                for h in range(Hq):
                    s = [math.fsum(q[t, h, c] * k[c] for c in range(d)) / math.sqrt(d) for k in keys]
                    e = [math.exp(x) for x in s]
                    z = math.fsum(e)
                    ref_o = [math.fsum(e[j] * vals[j][c] for j in range(len(e))) / z for c in range(d)]
                    assert abs(lse[0, t, h] - math.log(z)) <= 1e-12
                    assert max(abs(o[0, t, h, c] - ref_o[c]) for c in range(d)) <= 1e-12
            count += 1
    assert count == 1 + 2 + 6 + 24


# ------------------------------------------------------------------ closed forms

def _golden_inputs(case):
    B, T, Hq, Hkv, d = (case[k] for k in ("B", "T", "Hq", "Hkv", "d"))
    bits = lambda a: wl.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))
    inp = wl.Inputs(None, bits(case["q"]), bits(case["k_cache"]), bits(case["v_cache"]),
                    np.asarray(case["cache_lens"], np.int32), bits(case["k_spec"]),
                    bits(case["v_spec"]), np.asarray(case["parents"], np.int32))
    assert inp.q.shape == (B, T, Hq, d) and inp.k_spec.shape == (B, Hkv, T, d)
    return inp


def test_golden_closed_forms(oracle_mod):
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) >= 3
    for case in cases:
        inp = _golden_inputs(case)
        mask, bad = oracle_mod.build_mask(inp.parents)
        assert bad == 0
        assert mask.tolist() == case["expected_mask_rows"], case["name"]
        o, lse = run_oracle(oracle_mod, inp, mask, scale=case["scale"])
        assert np.abs(o - np.asarray(case["expected_o"])).max() <= 1e-12, case["name"]
        assert np.abs(lse - np.asarray(case["expected_lse"])).max() <= 1e-12, case["name"]


# ------------------------------------------------------------------ invariants

def test_weights_sum_to_one_and_convex_hull(oracle_mod):
    inp = wl.random_inputs(2, 20, 4, 2, 16, [30, 0], seed=5, Lmax=30)
    ones = inp.v_cache.copy()
    ones[...] = wl.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    ones_s = np.full_like(inp.v_spec, ones.flat[0])
    mask, _ = oracle_mod.build_mask(inp.parents)
    o1, _ = oracle_mod.attention(inp.q, inp.k_cache, ones, inp.cache_lens, inp.k_spec, ones_s, mask)
    assert np.abs(o1 - 1.0).max() <= 1e-14
    o, lse = run_oracle(oracle_mod, inp, mask)
    G = 2
    for b in range(2):
        L = inp.cache_lens[b]
        for t in range(20):
            spec = [j for j in range(20) if (mask[b, t, j // 32] >> (j % 32)) & 1]
            for h in range(4):
                vis = np.concatenate([f64(inp.v_cache[b, h // G, :L]), f64(inp.v_spec[b, h // G, spec])])
                assert (o[b, t, h] >= vis.min(0) - 1e-12).all() and (o[b, t, h] <= vis.max(0) + 1e-12).all()
                keys = np.concatenate([f64(inp.k_cache[b, h // G, :L]), f64(inp.k_spec[b, h // G, spec])])
                s = keys @ f64(inp.q[b, t, h]) / 4.0
                assert s.max() - 1e-12 <= lse[b, t, h] <= s.max() + math.log(len(s)) + 1e-12


def test_prefix_permutation_invariance(oracle_mod):
    inp = wl.random_inputs(1, 10, 4, 1, 32, [50], seed=8)
    o, lse = run_oracle(oracle_mod, inp)
    perm = np.random.default_rng(1).permutation(50)
    inp.k_cache[:, :, :50] = inp.k_cache[:, :, perm]
    inp.v_cache[:, :, :50] = inp.v_cache[:, :, perm]
    o2, lse2 = run_oracle(oracle_mod, inp)
    assert np.abs(o - o2).max() <= 1e-12 and np.abs(lse - lse2).max() <= 1e-12


def test_topological_relabelling_permutes_outputs(oracle_mod):
    T = 12
    inp = wl.random_inputs(1, T, 2, 1, 16, [9], seed=21)
    par = inp.parents[0]
    o, lse = run_oracle(oracle_mod, inp)
    # another topological order: sort nodes by (depth, -index)
    depth = np.zeros(T, int)
    for i in range(1, T):
        depth[i] = depth[par[i]] + 1 if par[i] >= 0 else 0
    order = sorted(range(T), key=lambda i: (depth[i], -i))  # new position -> old node
    new_of = {old: new for new, old in enumerate(order)}
    new_par = np.array([-1 if par[old] < 0 else new_of[int(par[old])] for old in order], np.int32)
    assert all(new_par[i] < i for i in range(T))
    inp2 = wl.Inputs(None, inp.q[:, order], inp.k_cache, inp.v_cache, inp.cache_lens,
                     inp.k_spec[:, :, order], inp.v_spec[:, :, order], new_par[None])
    o2, lse2 = run_oracle(oracle_mod, inp2)
    assert np.abs(o2 - o[:, order]).max() <= 1e-12
    assert np.abs(lse2 - lse[:, order]).max() <= 1e-12


def test_gqa_equals_replicated_mha(oracle_mod):
    inp = wl.random_inputs(2, 7, 6, 2, 16, [13, 4], seed=31)
    o, lse = run_oracle(oracle_mod, inp)
    G = 3
    mha = wl.Inputs(None, inp.q, expand_kv(inp.k_cache, G), expand_kv(inp.v_cache, G),
                    inp.cache_lens, expand_kv(inp.k_spec, G), expand_kv(inp.v_spec, G), inp.parents)
    o2, lse2 = run_oracle(oracle_mod, mha)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_empty_prefix_is_tree_only_attention(oracle_mod):
    inp = wl.random_inputs(1, 9, 2, 2, 16, [0], seed=41)
    o, lse = run_oracle(oracle_mod, inp)
    mask, _ = oracle_mod.build_mask(inp.parents)
    vis = [[[j for j in range(9) if (mask[0, t, 0] >> j) & 1] for t in range(9)]]
    o_ref, lse_ref = sdpa_reference(inp, vis)
    assert np.abs(o - o_ref).max() <= 1e-12 and np.abs(lse - lse_ref).max() <= 1e-12


def test_row_subset_matches_full(oracle_mod):
    inp = wl.random_inputs(2, 6, 4, 2, 8, [11, 3], seed=51)
    o, lse = run_oracle(oracle_mod, inp)
    rows = np.array([0, 7, 30, 47, 25], np.int64)
    mask, _ = oracle_mod.build_mask(inp.parents)
    o_r, lse_r = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens,
                                      inp.k_spec, inp.v_spec, mask, rows=rows)
    assert np.array_equal(o_r, o.reshape(-1, 8)[rows]) and np.array_equal(lse_r, lse.reshape(-1)[rows])


# ------------------------------------------------------------------ mask

def _nx_mask(par):
    import networkx as nx
    T = len(par)
    g = nx.DiGraph()
    g.add_nodes_from(range(T))
    g.add_edges_from((int(p), i) for i, p in enumerate(par) if p >= 0)
    W = (T + 31) // 32
    m = np.zeros((T, W), np.uint32)
    for i in range(T):
        for j in nx.ancestors(g, i) | {i}:
            m[i, j // 32] |= np.uint32(1 << (j % 32))
    return m


@pytest.mark.parametrize("T", [1, 2, 31, 32, 33, 64, 100, 256])
def test_mask_matches_graph_ancestors(oracle_mod, T):
    rng = np.random.default_rng(T)
    trees = [wl.tree_uniform(T, rng), wl.tree_window8_depth8(T, rng), wl.tree_chain(T), wl.tree_star(T)]
    forest = wl.tree_uniform(T, rng)
    forest[rng.random(T) < 0.2] = -1
    trees.append(forest)
    par = np.stack(trees)
    mask, bad = oracle_mod.build_mask(par)
    assert bad == 0
    for b in range(len(trees)):
        assert np.array_equal(mask[b], _nx_mask(par[b]))
        depth = np.zeros(T, int)
        for i in range(T):
            depth[i] = 0 if par[b, i] < 0 else depth[par[b, i]] + 1
            pop = sum(bin(int(w)).count("1") for w in mask[b, i])
            assert pop == depth[i] + 1
            if par[b, i] >= 0:
                assert np.array_equal(mask[b, i] & mask[b, par[b, i]], mask[b, par[b, i]])
        # bits at or beyond T stay clear
        if T % 32:
            assert (mask[b, :, -1] >> np.uint32(T % 32) == 0).all()


@pytest.mark.parametrize("bad_par", [[0, 0, 1], [-1, 1, 0], [-1, 0, 5], [-1, -2, 0], [-1, 0, 2]])
def test_mask_rejects_invalid_trees(oracle_mod, bad_par):
    good = [-1, 0, 0]
    mask, bad = oracle_mod.build_mask(np.array([good, bad_par], np.int32))
    assert bad == 1
    assert mask[1].sum() == 0 and mask[0].sum() > 0


def test_config_trees_follow_their_recipes():
    for name, cfg in wl.CONFIGS.items():
        par = wl.make_trees(cfg)
        assert par.shape == (cfg.B, cfg.T)
        for row in par:
            assert row[0] == -1 and all(-1 <= row[i] < i for i in range(cfg.T))
            depth = [0] * cfg.T
            for i in range(1, cfg.T):
                depth[i] = depth[row[i]] + 1
            if cfg.tree == "window8_depth8":
                assert max(depth) <= 8
                assert (row[1:] >= 0).all()
    lens = wl.cache_lengths(wl.CONFIGS["ragged_b32"])
    assert lens.min() >= 4096 and lens.max() <= 65536 and len(set(lens.tolist())) > 16


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-40, 3.0e38], np.float32)
    got = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(x))
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(got, ref)

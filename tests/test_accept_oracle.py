"""Pins of the accept-walk / KV-commit oracle (CPU only).

The oracle walks forward from the root; these checks use other formulations:
hand-derived cases (tests/golden/accept_cases.json), a per-node ancestor test
(a node is accepted iff every edge on its root path matches, which for trees
with distinct sibling tokens is exactly the walk), and direct reads of the
appended cache rows.
"""
import json
import os

import numpy as np
import pytest

from oracle.accept import accept_commit, accept_walk
from speculative_decoding_tree_hybrid_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_walk_matches_hand_derived_cases(case):
    path, nxt = accept_walk(np.array(case["parents"]), np.array(case["draft"]), np.array(case["target"]))
    assert path == case["path"]
    assert nxt == case["next_token"]


def _tree_with_distinct_sibling_tokens(T, rng):
    par = wl.tree_window8_depth8(T, rng) if T > 1 else np.array([-1], np.int32)
    draft = np.zeros(T, np.int64)
    for p in range(T):
        kids = [c for c in range(p + 1, T) if par[c] == p]
        draft[kids] = rng.choice(1000, size=len(kids), replace=False) + 1
    target = np.zeros(T, np.int64)
    for p in range(T):
        kids = [c for c in range(p + 1, T) if par[c] == p]
        # follow a random child with probability 0.7, else predict a token no child has
        target[p] = draft[rng.choice(kids)] if kids and rng.random() < 0.7 else 5000 + p
    return par, draft, target


@pytest.mark.parametrize("seed", range(20))
def test_walk_equals_per_node_ancestor_test(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 65))
    par, draft, target = _tree_with_distinct_sibling_tokens(T, rng)
    # a node is accepted iff its root path starts at node 0 and every edge on it matches
    acc = []
    for n in range(T):
        x, ok = n, True
        while par[x] >= 0:
            ok = ok and draft[x] == target[par[x]]
            x = par[x]
        if x == 0 and ok:
            acc.append(n)
    depth = {n: 0 for n in acc}
    for n in acc:
        x = n
        while par[x] >= 0:
            depth[n] += 1
            x = par[x]
    expected = sorted(acc, key=lambda n: depth[n])
    assert sorted(depth.values()) == list(range(len(acc)))  # a chain: one node per depth
    path, nxt = accept_walk(par, draft, target)
    assert path == expected
    assert nxt == target[expected[-1]]


def test_commit_appends_path_rows_and_leaves_the_rest():
    rng = np.random.default_rng(3)
    B, T, Hkv, d, Lmax = 3, 12, 2, 8, 40
    par = np.stack([wl.tree_uniform(T, rng) for _ in range(B)]).astype(np.int32)
    draft = rng.integers(0, 3, size=(B, T)).astype(np.int32)
    target = rng.integers(0, 3, size=(B, T)).astype(np.int32)
    ks = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
    vs = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
    kc = rng.standard_normal((B, Hkv, Lmax, d)).astype(np.float32)
    vc = rng.standard_normal((B, Hkv, Lmax, d)).astype(np.float32)
    lens = np.array([0, 17, Lmax - 1], np.int32)
    acc, n, nxt, kc2, vc2, lens2, clamped = accept_commit(par, draft, target, ks, vs, kc, vc, lens)
    for b in range(B):
        path = [int(x) for x in acc[b] if x >= 0]
        assert len(path) == n[b] and path[0] == 0
        assert (path, nxt[b]) == accept_walk(par[b], draft[b], target[b])
        nc = min(len(path), Lmax - lens[b])
        assert lens2[b] == lens[b] + nc
        for j in range(nc):
            assert np.array_equal(kc2[b, :, lens[b] + j], ks[b, :, path[j]])
            assert np.array_equal(vc2[b, :, lens[b] + j], vs[b, :, path[j]])
        keep = np.ones(Lmax, bool)
        keep[lens[b]:lens[b] + nc] = False
        assert np.array_equal(kc2[b][:, keep], kc[b][:, keep])
        assert np.array_equal(vc2[b][:, keep], vc[b][:, keep])
    assert clamped == int(n[2] > 1)  # the last sequence has room for one row

"""Pins for the LogitSpec draft-tree oracle (oracle/logitspec.py), on CPU:
hand-derived cases (tests/golden/logitspec_cases.json) and properties checked
by brute force on random streams ("LogitSpec: Accelerating Retrieval-based
Speculative Decoding via Next Next Token Speculation", section 2)."""
import json
import pathlib

import numpy as np
import pytest

from oracle.logitspec import build_tree, build_trees, latest_match, ranked

CASES = json.loads((pathlib.Path(__file__).parent / "golden" / "logitspec_cases.json").read_text())["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_derived_cases(case):
    par, tok, n, x1 = build_tree(np.array(case["logits"]), case["hist"], case["k"], case["m"], case["keep"], case["T"])
    assert par.tolist() == case["parents"]
    assert tok.tolist() == case["tokens"]
    assert n == case["n_nodes"] and x1 == case["x_next"]


def test_ranking_is_value_then_id():
    rng = np.random.default_rng(0)
    for _ in range(50):
        V = int(rng.integers(2, 200))
        logits = rng.integers(-3, 4, size=V).astype(np.float64)  # many ties
        K = int(rng.integers(1, V + 1))
        want = sorted(range(V), key=lambda t: (-logits[t], t))[:K]
        assert ranked(logits, K) == want


def _stream(rng, n, vocab):
    """A token stream with repeats: copies of earlier spans mixed with noise."""
    out = list(rng.integers(0, vocab, size=8))
    while len(out) < n:
        if rng.random() < 0.6 and len(out) > 4:
            a = int(rng.integers(0, len(out) - 2))
            out += out[a:a + int(rng.integers(2, 9))]
        else:
            out.append(int(rng.integers(0, vocab)))
    return out[:n]


@pytest.mark.parametrize("seed", range(25))
def test_tree_properties_by_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    vocab = int(rng.integers(4, 12))
    n = int(rng.integers(0, 80))
    hist = _stream(rng, n, vocab) if n else []
    m = int(rng.integers(2, 5))
    k = int(rng.integers(0, vocab - 1))
    T = int(rng.integers(1, 40))
    keep = [int(x) for x in rng.integers(0, 6, size=k + 1)]
    logits = rng.standard_normal(vocab)
    par, tok, nn, x1 = build_tree(logits, hist, k, m, keep, T)
    order = sorted(range(vocab), key=lambda t: (-logits[t], t))
    assert x1 == order[0] and tok[0] == x1 and par[0] == -1
    # topological, padding after the real nodes
    assert all(0 <= par[i] < i for i in range(1, nn))
    assert all(par[i] == 0 and tok[i] == -1 for i in range(nn, T))
    # children of the root: the g1 branch head (if any) and the guesses in rank order
    kids = [i for i in range(1, nn) if par[i] == 0]
    guess_nodes = [i for i in kids if tok[i] in order[1:k + 1]]

    def brute_latest(gram):
        best = -1
        for s in range(len(hist) - len(gram)):  # s + m <= len - 1
            if hist[s:s + len(gram)] == list(gram):
                best = s
        return best

    # every chain below a branch head is the history right after the branch's latest match
    def chain_from(head):
        out, cur = [], head
        while True:
            nxt = [i for i in range(cur + 1, nn) if par[i] == cur]
            if not nxt:
                return out
            assert len(nxt) == 1
            cur = nxt[0]
            out.append(int(tok[cur]))

    # the g1 branch: nodes 1 .. c form one chain under the root, holding the
    # history right after the latest match of (last m-1 tokens, x_{i+1})
    want_g1 = []
    if len(hist) >= m - 1:
        g1 = (hist[len(hist) - (m - 1):] if m > 1 else []) + [x1]
        s1 = brute_latest(g1)
        if s1 >= 0:
            want_g1 = hist[s1 + m:s1 + m + keep[0]]
    c = min(len(want_g1), T - 1)
    assert tok[1:1 + c].tolist() == want_g1[:c]
    assert all(par[i] == (0 if i == 1 else i - 1) for i in range(1, 1 + c))
    if 1 + c < nn and k >= 1:  # the first guess comes right after the g1 chain
        assert par[1 + c] == 0 and tok[1 + c] == order[1]

    for r, g in enumerate(order[1:k + 1], start=1):
        nodes = [i for i in guess_nodes if tok[i] == g and i >= 1]
        if not nodes:
            break  # the tree filled up before this guess
        gnode = nodes[-1] if len(nodes) > 1 else nodes[0]
        gram = (hist[len(hist) - (m - 2):] if m > 2 else []) + [x1, g] if len(hist) >= m - 2 else None
        s = brute_latest(gram) if gram is not None else -1
        assert s == (latest_match(hist, gram) if gram is not None else -1)
        got = chain_from(gnode)
        if s < 0:
            assert got == []
        else:
            want = hist[s + m:s + m + keep[r]]
            assert got == want[:len(got)] and (len(got) == len(want) or nn == T)
    assert nn <= T


def test_batch_form_matches_single():
    rng = np.random.default_rng(7)
    B, V, L = 4, 30, 60
    logits = rng.standard_normal((B, V))
    hist = np.zeros((B, L), np.int32)
    lens = np.array([0, 5, 33, 60], np.int32)
    for b in range(B):
        hist[b, :lens[b]] = _stream(rng, int(lens[b]), 6) if lens[b] else []
    par, tok, nn, nxt = build_trees(logits, hist, lens, 3, 3, [4, 3, 2, 1], 12)
    for b in range(B):
        p, t, n, x = build_tree(logits[b], hist[b][:lens[b]], 3, 3, [4, 3, 2, 1], 12)
        assert par[b].tolist() == p.tolist() and tok[b].tolist() == t.tolist() and nn[b] == n and nxt[b] == x

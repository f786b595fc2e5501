"""Oracle for the LogitSpec draft-tree builder.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this module; the product path never
does. Plain Python and numpy, one sequence at a time.

What the pages fix ("LogitSpec: Accelerating Retrieval-based Speculative
Decoding via Next Next Token Speculation", section 2, workflow steps 1 and 2):
the target's last logits give the next token x_{i+1}; the top-k entries of
the same logits other than x_{i+1} are guesses of the next-next token; two
kinds of n-gram queries are looked up in the reference token stream,
g1 = (x_{i-m+2}, ..., x_i, x_{i+1}) and, per guess,
g2 = (x_{i-m+3}, ..., x_i, x_{i+1}, guess); the retrieved tokens form a draft
tree rooted at x_{i+1} whose branches belong to different guesses; a
rank-based pruning keeps more retrieved tokens for better-ranked guesses.

Readings taken where the pages are silent (each stated once here):
  * order of the logits: value descending, ties by the smaller token id; x_{i+1}
    is the first, the guesses are ranks 1 .. k after it;
  * the reference stream is the sequence's own tokens x_0 .. x_i (the
    retrieval source of prompt-lookup style methods);
  * a query matches at start s when hist[s .. s+m-1] equals it and at least one
    token follows (s + m <= len - 1); the latest such s is used;
  * the retrieved continuation of a match at s is hist[s+m ..], truncated at
    the end of the history;
  * pruning is a per-rank budget keep[r] (r = 0: the g1 branch; r >= 1: the
    tokens after guess r), given by the caller;
  * tree layout: node 0 = x_{i+1} (parent -1); then the g1 continuation as a
    chain under the root; then, for r = 1 .. k, the guess as a child of the
    root followed by its continuation as a chain; nodes are added until T;
    unused nodes are padding (parent 0, token -1, never accepted);
  * a query that needs more history than there is finds nothing.
"""
from __future__ import annotations

import numpy as np


def ranked(logits: np.ndarray, K: int) -> list[int]:
    """Token ids of the K largest logits, value descending, ties by id."""
    order = np.argsort(-np.asarray(logits, dtype=np.float64), kind="stable")
    return [int(x) for x in order[:K]]


def latest_match(hist: list[int], gram: list[int]) -> int:
    """Latest start s with hist[s:s+m] == gram and a token after it, else -1."""
    m = len(gram)
    for s in range(len(hist) - m - 1, -1, -1):
        if hist[s:s + m] == gram:
            return s
    return -1


def build_tree(logits, hist, k: int, m: int, keep, T: int):
    """One sequence. Returns (parents [T], tokens [T], n_nodes, x_next)."""
    hist = [int(x) for x in hist]
    top = ranked(logits, k + 1)
    x1, guesses = top[0], top[1:]
    parents, tokens = [-1], [x1]

    def add(tok: int, par: int) -> int:
        parents.append(par)
        tokens.append(tok)
        return len(tokens) - 1

    def chain(start: int, budget: int, par: int):
        for j in range(budget):
            pos = start + j
            if pos >= len(hist) or len(tokens) >= T:
                return
            par = add(hist[pos], par)

    n = len(hist)
    if n >= m - 1:  # g1: the last m-1 history tokens and x_{i+1}
        g1 = hist[n - (m - 1):] + [x1] if m > 1 else [x1]
        s = latest_match(hist, g1)
        if s >= 0:
            chain(s + m, int(keep[0]), 0)
    for r, g in enumerate(guesses, start=1):
        if len(tokens) >= T:
            break
        node = add(g, 0)
        if n >= m - 2:  # g2: the last m-2 history tokens, x_{i+1} and the guess
            g2 = (hist[n - (m - 2):] if m > 2 else []) + [x1, g]
            s = latest_match(hist, g2)
            if s >= 0:
                chain(s + m, int(keep[r]), node)
    n_nodes = len(tokens)
    parents += [0] * (T - n_nodes)
    tokens += [-1] * (T - n_nodes)
    return np.array(parents, np.int32), np.array(tokens, np.int32), n_nodes, x1


def build_trees(logits, hist, hist_len, k: int, m: int, keep, T: int):
    """Batch form: logits [B][V], hist [B][Lh_max], hist_len [B]."""
    B = len(hist_len)
    par = np.zeros((B, T), np.int32)
    tok = np.zeros((B, T), np.int32)
    nn = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    for b in range(B):
        par[b], tok[b], nn[b], nxt[b] = build_tree(logits[b], hist[b][:int(hist_len[b])], k, m, keep, T)
    return par, tok, nn, nxt

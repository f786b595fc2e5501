"""Oracle for the accept walk and KV commit that follow tree verification.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this module; the product path never
does. Plain Python loops over the (small) tree and numpy copies for the KV
rows.

What the pages fix ("LogitSpec: Accelerating Retrieval-based Speculative
Decoding via Next Next Token Speculation", section 2, workflow step 2; the
speculative decoding setting of "LongSpec: Long-Context Lossless Speculative
Decoding with Efficient Drafting and Verification", Korean summary section 1):
the draft tree is rooted at x_{i+1}, the token the target itself predicted,
and the target checks every branch in one pass. The acceptance rule is not
given; the reading used here is greedy verification:

  * node 0 (the root) is always accepted;
  * a child c of the last accepted node p is accepted when its draft token
    equals the target's greedy prediction at p (target[p]); if several
    children qualify, the one with the smallest index;
  * the walk stops at the first node with no qualifying child, and the
    target's prediction there is the next step's root token.

The K/V rows of the accepted nodes (from the speculative buffers, in path
order) are then appended to the cache of their sequence at positions
L_b, L_b + 1, ...; cache_lens[b] grows by the number appended. Rows that
would pass Lmax are not written (the count is clamped, and the call reports
it).
"""
from __future__ import annotations

import numpy as np


def accept_walk(parents: np.ndarray, draft: np.ndarray, target: np.ndarray) -> tuple[list[int], int]:
    """The accepted path of one tree (node indices, root first) and the
    target's prediction after its last node."""
    T = len(parents)
    path = [0]
    cur = 0
    while True:
        nxt = -1
        for c in range(cur + 1, T):  # children come after their parent
            if int(parents[c]) == cur and int(draft[c]) == int(target[cur]):
                nxt = c
                break
        if nxt < 0:
            return path, int(target[cur])
        path.append(nxt)
        cur = nxt


def accept_commit(parents, draft, target, k_spec, v_spec, k_cache, v_cache, cache_lens):
    """Runs the walk for every sequence and appends the accepted rows.

    parents, draft, target: int32 [B][T]; k_spec, v_spec: [B][Hkv][T][d];
    k_cache, v_cache: [B][Hkv][Lmax][d] (any dtype, copied, not modified);
    cache_lens: int32 [B].
    Returns (accepted int32 [B][T] padded with -1, n_accepted int32 [B],
    next_token int32 [B], new k_cache, new v_cache, new cache_lens int32 [B],
    clamped: number of sequences whose path did not fit under Lmax).
    """
    B, T = parents.shape
    Lmax = k_cache.shape[2]
    acc = np.full((B, T), -1, np.int32)
    n_acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    kc, vc = k_cache.copy(), v_cache.copy()
    lens = np.array(cache_lens, np.int32).copy()
    clamped = 0
    for b in range(B):
        path, nt = accept_walk(parents[b], draft[b], target[b])
        n = len(path)
        acc[b, :n] = path
        n_acc[b] = n
        nxt[b] = nt
        L = int(min(max(int(cache_lens[b]), 0), Lmax))
        nc = min(n, Lmax - L)
        if nc < n:
            clamped += 1
        if nc > 0:
            idx = np.array(path[:nc])
            kc[b, :, L:L + nc, :] = k_spec[b][:, idx, :]
            vc[b, :, L:L + nc, :] = v_spec[b][:, idx, :]
        lens[b] = L + nc
    return acc, n_acc, nxt, kc, vc, lens, clamped

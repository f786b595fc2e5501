"""GPU parity of hta_accept_commit against the oracle (oracle/accept.py):
integer outputs bit-exact, appended K/V rows bit-exact, the rest of the cache
untouched."""
import numpy as np
import pytest

from speculative_decoding_tree_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle.accept import accept_commit as oracle_accept  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import build as hbuild  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import hta  # noqa: E402

hbuild.build()
DEV = torch.device("cuda:0")


def tokens(parents, rng, follow=0.8):
    """Draft tokens (distinct per sibling set only by chance: duplicates are
    allowed and exercise the smallest-index rule) and target predictions
    that follow a random child with probability `follow`."""
    B, T = parents.shape
    draft = rng.integers(0, 6, size=(B, T)).astype(np.int32)
    target = np.zeros((B, T), np.int32)
    for b in range(B):
        for p in range(T):
            kids = np.nonzero(parents[b] == p)[0]
            target[b, p] = draft[b, rng.choice(kids)] if len(kids) and rng.random() < follow else 100 + p
    return draft, target


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)


def run_case(B, T, Hkv, d, lens, Lmax, tree, seed, follow=0.8):
    rng = np.random.default_rng(seed)
    par = None
    if tree in ("chain", "star"):
        par = np.stack([wl.tree_chain(T) if tree == "chain" else wl.tree_star(T)] * B)
    inp = wl.random_inputs(B, T, Hkv, Hkv, d, list(lens), seed=seed, Lmax=Lmax, tree=tree, parents=par)
    parents = inp.parents.astype(np.int32)
    draft, target = tokens(parents, rng, follow)
    lens_np = np.array(lens, np.int32)
    acc, n, nxt, kc2, vc2, lens2, clamped = oracle_accept(parents, draft, target, inp.k_spec, inp.v_spec,
                                                          inp.k_cache, inp.v_cache, lens_np)
    t = {k: torch.from_numpy(v).to(DEV) for k, v in (("parents", parents), ("draft", draft), ("target", target))}
    kc, vc = bf16(inp.k_cache), bf16(inp.v_cache)
    lens_t = torch.from_numpy(lens_np.copy()).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    g_acc, g_n, g_nxt = hta.accept_commit(t["parents"], t["draft"], t["target"], bf16(inp.k_spec), bf16(inp.v_spec),
                                          kc, vc, lens_t, dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(g_acc.cpu().numpy(), acc)
    assert np.array_equal(g_n.cpu().numpy(), n)
    assert np.array_equal(g_nxt.cpu().numpy(), nxt)
    assert np.array_equal(lens_t.cpu().numpy(), lens2)
    assert np.array_equal(kc.cpu().view(torch.int16).numpy().view(np.uint16), kc2)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy().view(np.uint16), vc2)
    assert bool(int(err.item()) & hta.DEVERR_CACHE_LEN) == (clamped > 0)
    return n


@pytest.mark.parametrize("case", [
    # (B, T, Hkv, d, lens, Lmax, tree)
    (1, 8, 1, 64, [256], 300, "uniform"),
    (1, 64, 8, 128, [3000], 3200, "window8_depth8"),      # LLaMA layer shape, short cache
    (4, 32, 32, 128, [700, 0, 1, 333], 800, "uniform"),   # Vicuna-like, one empty cache
    (3, 256, 2, 128, [10, 20, 30], 400, "chain"),         # the longest possible paths
    (2, 64, 8, 128, [5, 6], 64, "star"),
])
def test_accept_commit_matches_oracle(case):
    B, T, Hkv, d, lens, Lmax, tree = case
    for seed in (1, 2):
        run_case(B, T, Hkv, d, lens, Lmax, tree, seed)


def test_accept_commit_long_paths_follow_every_match():
    # target always follows a child: the path runs to a leaf
    n = run_case(2, 128, 4, 128, [100, 900], 1200, "window8_depth8", seed=5, follow=1.0)
    assert (n > 1).all()


def test_accept_commit_clamps_at_lmax():
    # cache one row short of full, and full: the path is cut, the flag set
    run_case(2, 64, 2, 64, [63, 64], 64, "chain", seed=7, follow=1.0)


def test_accept_commit_full_size_ragged_batch():
    run_case(32, 64, 8, 128, list(np.random.default_rng(11).integers(4096, 8192, size=32)), 8192,
             "window8_depth8", seed=11)

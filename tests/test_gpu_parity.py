"""GPU parity of every libhta entry point against the CPU fp64 oracle.

The CUDA path is called through the C ABI (ctypes binding); the expected
values come only from oracle/ on the same seeded inputs. Small cases compare
every output element at sizes that span several key tiles and a ragged tail;
the full-size workloads compare sampled rows the oracle computes one by one.
"""
import numpy as np
import pytest

from speculative_decoding_tree_hybrid_gb300 import workloads as wl

from _util import assert_close, mask_to_torch, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from speculative_decoding_tree_hybrid_gb300 import build as hbuild  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import hta  # noqa: E402

hbuild.build()
DEV = torch.device("cuda:0")
PATHS = ["auto", "cc", "tc", "tc2"]


@pytest.fixture
def path(request, monkeypatch):
    p = request.param
    if p == "auto":
        monkeypatch.delenv("HTA_FORCE_PATH", raising=False)
    else:
        monkeypatch.setenv("HTA_FORCE_PATH", p)
    return p


def run_verify(inp, path_name, mask=None, scale=0.0):
    t = to_device(inp, DEV)
    if mask is None:
        mask = hta.build_mask(t["parents"])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    try:
        o, lse = hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"],
                            t["v_spec"], mask, scale=scale, dev_err=err)
    except hta.HtaError as e:
        if path_name in ("tc", "tc2") and e.status == -2:
            pytest.skip("this tensor-core path does not take this shape")
        raise
    torch.cuda.synchronize()
    if path_name == "tc":
        assert hta.last_path() == hta.PATH_TC
    if path_name == "tc2":
        assert hta.last_path() == hta.PATH_TC2
    if path_name == "cc":
        assert hta.last_path() == hta.PATH_CC
    assert int(err.item()) == 0
    return o, lse


def oracle_full(oracle_mod, inp, scale=0.0):
    mask, bad = oracle_mod.build_mask(inp.parents)
    assert bad == 0
    return oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec,
                                inp.v_spec, mask, scale=scale)


# ---------------------------------------------------------------- mask

def _adversarial_trees(T, rng):
    forest = wl.tree_uniform(T, rng)
    forest[rng.random(T) < 0.25] = -1
    forest[0] = -1
    return [wl.tree_uniform(T, rng), wl.tree_window8_depth8(T, rng), wl.tree_chain(T),
            wl.tree_star(T), forest]


@pytest.mark.parametrize("T", [1, 2, 8, 31, 32, 33, 64, 100, 128, 255, 256])
def test_mask_bit_exact(oracle_mod, T):
    par = np.stack(_adversarial_trees(T, np.random.default_rng(T)))
    ref, bad = oracle_mod.build_mask(par)
    assert bad == 0
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = hta.build_mask(torch.from_numpy(par).to(DEV), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(got.cpu().numpy().view(np.uint32), ref)


def test_mask_bit_exact_on_config_trees(oracle_mod):
    for name, cfg in wl.CONFIGS.items():
        par = wl.make_trees(cfg)
        ref, _ = oracle_mod.build_mask(par)
        got = hta.build_mask(torch.from_numpy(par).to(DEV))
        assert np.array_equal(got.cpu().numpy().view(np.uint32), ref), name


@pytest.mark.parametrize("bad_par", [[0, 0, 1, 2], [-1, 1, 0, 0], [-1, 0, 7, 1], [-1, -2, 0, 1]])
def test_mask_flags_invalid_tree(oracle_mod, bad_par):
    par = np.array([[-1, 0, 0, 1], bad_par, [-1, 0, 1, 2]], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = hta.build_mask(torch.from_numpy(par).to(DEV), dev_err=err).cpu().numpy().view(np.uint32)
    torch.cuda.synchronize()
    assert int(err.item()) & hta.DEVERR_BAD_TREE
    ref, nbad = oracle_mod.build_mask(par)
    assert nbad == 1
    assert np.array_equal(got, ref)  # the bad tree's rows are zero on both sides


# ---------------------------------------------------------------- small cases, every element

SMALL = [
    # (B, T, Hq, Hkv, d, lens, tree)
    (1, 8, 4, 1, 64, [256], "uniform"),            # Tiny shape
    (1, 64, 32, 8, 128, [1000], "window8_depth8"),  # LLaMA shape, short cache, ragged tail
    (2, 32, 8, 8, 128, [700, 333], "uniform"),      # MHA (Vicuna-like), two lengths
    (1, 64, 40, 8, 128, [515], "window8_depth8"),   # QwQ shape (G = 5, 320 rows)
    (3, 64, 32, 8, 128, [129, 0, 1], "window8_depth8"),  # ragged incl. empty cache
    (2, 1, 8, 2, 128, [300, 5], "uniform"),         # single node: plain decode
    (1, 200, 4, 2, 64, [90], "uniform"),            # large tree, several tree tiles
    (2, 33, 10, 2, 128, [128, 256], "uniform"),     # G = 5, T not a multiple of 32
    (1, 100, 16, 4, 128, [900], "window8_depth8"),  # two row groups of 200 rows (two 100-row halves)
    (1, 65, 16, 4, 128, [600], "uniform"),          # short last row group, odd nodes per group
    (1, 64, 64, 8, 128, [777], "window8_depth8"),   # G = 8: 512 rows, clusters of four CTAs
    (3, 64, 40, 8, 128, [300, 1029, 0], "window8_depth8"),  # QwQ shape, ragged incl. an empty cache
    (1, 256, 32, 8, 128, [700], "window8_depth8"),  # largest tree: 1024 rows, two groups of four CTAs
    (1, 256, 64, 8, 128, [300], "uniform"),         # largest tree at G = 8: 2048 rows, four row groups
    # largest batch, ragged lengths 0 .. 299 (a few empty caches)
    (1024, 4, 8, 2, 128, [int(x) for x in np.random.default_rng(3).integers(0, 300, 1024)], "uniform"),
]


@pytest.mark.parametrize("path", PATHS, indirect=True)
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_verify_small_every_element(oracle_mod, path, case):
    B, T, Hq, Hkv, d, lens, tree = SMALL[case]
    if path in ("tc", "tc2") and d != 128:
        pytest.skip("tensor-core paths need d = 128")
    inp = wl.random_inputs(B, T, Hq, Hkv, d, lens, seed=100 + case, tree=tree)
    o, lse = run_verify(inp, path)
    o_ref, lse_ref = oracle_full(oracle_mod, inp)
    assert_close(o, lse, o_ref, lse_ref, f"case {SMALL[case]} path {path}")


@pytest.mark.parametrize("path", PATHS, indirect=True)
def test_verify_explicit_scale(oracle_mod, path):
    inp = wl.random_inputs(1, 16, 8, 2, 128, [400], seed=7)
    o, lse = run_verify(inp, path, scale=0.05)
    o_ref, lse_ref = oracle_full(oracle_mod, inp, scale=0.05)
    assert_close(o, lse, o_ref, lse_ref, "scale 0.05")


@pytest.mark.parametrize("path", PATHS, indirect=True)
@pytest.mark.parametrize("scale", [1.0, 4.0])
def test_verify_large_scale_near_one_hot(oracle_mod, path, scale):
    """Large softmax scales make the softmax nearly one-hot and the running
    max move by tens of units between tiles: a wrong reference max would
    overflow, and the rescale of O runs on many tiles."""
    inp = wl.random_inputs(2, 64, 16, 4, 128, [1500, 777], seed=29, tree="window8_depth8")
    o, lse = run_verify(inp, path, scale=scale)
    o_ref, lse_ref = oracle_full(oracle_mod, inp, scale=scale)
    assert_close(o, lse, o_ref, lse_ref, f"scale {scale}")


@pytest.mark.parametrize("path", PATHS, indirect=True)
def test_verify_growing_keys_force_rescale(oracle_mod, path):
    """Cache keys grow in magnitude with position, so every new tile raises
    the running max (the O rescale path runs on most tiles)."""
    inp = wl.random_inputs(1, 32, 8, 2, 128, [2048], seed=31)
    kf = wl.bf16_bits_to_f32(inp.k_cache)
    growth = (1.0 + np.arange(kf.shape[2], dtype=np.float32) / 128.0)[None, None, :, None]
    inp.k_cache[...] = wl.f32_to_bf16_bits(np.nan_to_num(kf, nan=0.0) * growth)
    o, lse = run_verify(inp, path)
    o_ref, lse_ref = oracle_full(oracle_mod, inp)
    assert_close(o, lse, o_ref, lse_ref, "growing keys")


@pytest.mark.parametrize("path", ["cc", "tc", "tc2"], indirect=True)
def test_verify_is_deterministic(path):
    inp = wl.random_inputs(2, 64, 32, 8, 128, [3000, 1700], seed=9, tree="window8_depth8")
    o1, l1 = run_verify(inp, path)
    o2, l2 = run_verify(inp, path)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("path", ["cc", "tc", "tc2"], indirect=True)
def test_cooperative_launch_matches_default(oracle_mod, path, monkeypatch):
    """HTA_COOPERATIVE=1 launches the persistent grids cooperatively instead of
    as ordinary programmatically dependent grids: same oracle parity and
    bit-identical outputs (the schedule and the merge order do not depend on
    the launch mode)."""
    inp = wl.random_inputs(2, 64, 32, 8, 128, [3000, 1700], seed=19, tree="window8_depth8")
    o1, l1 = run_verify(inp, path)
    monkeypatch.setenv("HTA_COOPERATIVE", "1")
    o2, l2 = run_verify(inp, path)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, lse_ref = oracle_full(oracle_mod, inp)
    assert_close(o2, l2, o_ref, lse_ref, f"cooperative {path}")


def test_prefix_tree_merge_entry_points(oracle_mod):
    inp = wl.random_inputs(2, 24, 8, 2, 128, [777, 0], seed=13)
    t = to_device(inp, DEV)
    mask_np, _ = oracle_mod.build_mask(inp.parents)
    mask = mask_to_torch(mask_np, DEV)
    o_c, lse_c = hta.prefix_attn(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"])
    o_s, lse_s = hta.tree_attn(t["q"], t["k_spec"], t["v_spec"], mask)
    o, lse = hta.merge(o_c, lse_c, o_s, lse_s)
    torch.cuda.synchronize()
    zero_mask = np.zeros_like(mask_np)
    rc = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec,
                              inp.v_spec, zero_mask)
    rs = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, np.zeros(2, np.int32), inp.k_spec,
                              inp.v_spec, mask_np)
    rf = oracle_full(oracle_mod, inp)
    assert_close(o_c, lse_c, *rc, "prefix")
    assert_close(o_s, lse_s, *rs, "tree")
    assert_close(o, lse, *rf, "merge")
    # empty cache: LSE_c = -inf and O_c = 0 exactly
    assert torch.isneginf(lse_c[1]).all() and (o_c[1] == 0).all()


def test_merge_of_oracle_partials(oracle_mod):
    """hta_merge alone, fed the oracle's own fp64 partials (rounded to fp32)."""
    inp = wl.random_inputs(1, 16, 4, 2, 64, [50], seed=17)
    mask_np, _ = oracle_mod.build_mask(inp.parents)
    rc = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec,
                              inp.v_spec, np.zeros_like(mask_np))
    rs = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, np.zeros(1, np.int32), inp.k_spec,
                              inp.v_spec, mask_np)
    f = lambda a: torch.from_numpy(a.astype(np.float32)).to(DEV)
    o, lse = hta.merge(f(rc[0]), f(rc[1]), f(rs[0]), f(rs[1]))
    rf = oracle_full(oracle_mod, inp)
    assert_close(o, lse, *rf, "merge")
    # one side -inf: weight zero
    neg = torch.full_like(f(rc[1]), float("-inf"))
    o2, lse2 = hta.merge(f(rc[0]), neg, f(rs[0]), f(rs[1]))
    assert_close(o2, lse2, rs[0], rs[1], "merge with empty cached part")


def test_cache_len_out_of_range_is_flagged():
    inp = wl.random_inputs(1, 4, 4, 1, 64, [20], seed=19, Lmax=32)
    t = to_device(inp, DEV)
    t["cache_lens"][0] = 40  # > Lmax
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mask = hta.build_mask(t["parents"])
    inp.k_cache[...] = 0  # keep the clamped read finite
    t["k_cache"].zero_()
    t["v_cache"].zero_()
    hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"], t["v_spec"], mask,
               dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & hta.DEVERR_CACHE_LEN


def test_host_errors_on_gpu_tensors():
    inp = wl.random_inputs(1, 8, 4, 1, 64, [10], seed=23)
    t = to_device(inp, DEV)
    mask = hta.build_mask(t["parents"])
    small_ws = torch.zeros(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(hta.HtaError) as ei:
        hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"], t["v_spec"],
                   mask, ws=small_ws)
    assert ei.value.status == -5


# ---------------------------------------------------------------- full-size configs, sampled rows

_FULL_CACHE = {}


def full_inputs(name):
    if name not in _FULL_CACHE:
        _FULL_CACHE.clear()
        _FULL_CACHE[name] = wl.make_inputs(name, threads=16)
    return _FULL_CACHE[name]


def sample_rows(cfg, n, seed):
    rng = np.random.default_rng(seed)
    total = cfg.B * cfg.T * cfg.Hq
    corners = [0, cfg.Hq - 1, total - 1, total - cfg.Hq, (cfg.T // 2) * cfg.Hq + cfg.Hq // 2]
    rows = np.unique(np.concatenate([rng.choice(total, size=min(n, total), replace=False), corners]))
    return rows.astype(np.int64)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["tiny", "llama8b", "vicuna7b", "qwq32b", "ragged_b1",
                                  "ragged_b4", "ragged_b16", "ragged_b32"])
def test_verify_full_size_sampled_rows(oracle_mod, name, monkeypatch):
    monkeypatch.delenv("HTA_FORCE_PATH", raising=False)
    inp = full_inputs(name)
    cfg = inp.cfg
    o, lse = run_verify(inp, "auto")
    rows = sample_rows(cfg, 24 if name in ("qwq32b", "ragged_b32") else 48, seed=cfg.cfg_id)
    mask_np, _ = oracle_mod.build_mask(inp.parents)
    o_ref, lse_ref = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens,
                                          inp.k_spec, inp.v_spec, mask_np, rows=rows)
    rows_t = torch.from_numpy(rows).to(DEV)
    o_s = o.reshape(-1, cfg.d)[rows_t]
    l_s = lse.reshape(-1)[rows_t]
    assert_close(o_s, l_s, o_ref, lse_ref, name)
    # every row sees at least its own tree node, so every output is finite
    assert torch.isfinite(lse).all() and torch.isfinite(o.float()).all()

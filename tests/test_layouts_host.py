"""CPU checks of the cache-storage layouts: the seeded paging helper that the
GPU layout tests use, and the host-side rejection of layouts that break the
rules of hta_kv_layout (no kernel runs here)."""
import ctypes

import numpy as np
import pytest

from speculative_decoding_tree_hybrid_gb300 import build as hbuild
from speculative_decoding_tree_hybrid_gb300 import hta
from speculative_decoding_tree_hybrid_gb300 import workloads as wl


@pytest.mark.parametrize("order", ["hnd", "nhd"])
@pytest.mark.parametrize("P", [16, 64, 128, 256])
def test_paged_kv_round_trip(order, P):
    inp = wl.random_inputs(3, 4, 8, 2, 64, [300, 1029, 0], seed=7)
    kp, vp, table = wl.paged_kv(inp.k_cache, inp.v_cache, inp.cache_lens, P, order=order, seed=3)
    lens = inp.cache_lens
    used = [-(-int(L) // P) for L in lens]
    assert table.shape == (3, -(-inp.Lmax // P))
    pages = np.concatenate([table[b, :used[b]] for b in range(3)])
    assert len(set(pages.tolist())) == len(pages) == sum(used)  # each pool page holds one sequence page
    assert pages.min(initial=0) >= 0 and pages.max(initial=0) < kp.shape[0]
    for b in range(3):
        assert np.all(table[b, used[b]:] == -1)
    for pool, ref in ((kp, inp.k_cache), (vp, inp.v_cache)):
        back = wl.unpage_kv(pool, table, lens, inp.Lmax, order=order)
        for b in range(3):
            assert np.array_equal(back[b, :, :lens[b]], ref[b, :, :lens[b]])
    spare = sorted(set(range(kp.shape[0])) - set(pages.tolist()))
    assert len(spare) == 3 and np.all(kp[spare] == wl.BF16_NAN)
    if order == "nhd":
        assert kp.shape[1:] == (P, 2, 64)


def test_kv_nhd_is_a_transpose():
    x = np.arange(2 * 3 * 5 * 4, dtype=np.uint16).reshape(2, 3, 5, 4)
    y = wl.kv_nhd(x)
    assert y.shape == (2, 5, 3, 4)
    assert all(y[b, j, h, c] == x[b, h, j, c] for b in range(2) for j in range(5) for h in range(3)
               for c in range(4))


@pytest.fixture(scope="module")
def lib():
    hbuild.build()
    return hta.load()


def _call(lib, lay, Lmax=256):
    d = hta.HtaDims(1, 8, 4, 1, 64, Lmax, 0.0)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the call returns before any launch
    args = [fake] * 10  # q .. lse, workspace
    v = lib.hta_verify_kv(ctypes.byref(d), ctypes.byref(lay) if lay is not None else None, *args,
                          1 << 20, None, None)
    p = lib.hta_prefix_attn_kv(ctypes.byref(d), ctypes.byref(lay) if lay is not None else None,
                               *([fake] * 7), 1 << 20, None, None)
    return v, p


@pytest.mark.parametrize("order,P,max_pages,num_pages,table,Lmax", [
    (2, 0, 0, 0, None, 256),         # unknown order
    (0, -16, 0, 0, None, 256),       # negative page size
    (0, 48, 16, 4, 1 << 20, 256),    # a 128-key tile would straddle pages unevenly
    (1, 96, 16, 4, 1 << 20, 256),
    (0, 16, 16, 4, None, 256),       # paged without a block table
    (0, 16, 0, 4, 1 << 20, 256),     # no table columns
    (0, 16, 16, 0, 1 << 20, 256),    # empty pool
    (0, 16, 15, 4, 1 << 20, 256),    # Lmax beyond max_pages * page_size
])
def test_bad_layouts_rejected_on_host(lib, order, P, max_pages, num_pages, table, Lmax):
    lay = hta.HtaKvLayout(order, P, max_pages, num_pages, table)
    assert _call(lib, lay, Lmax) == (-1, -1)


def test_layout_checks_follow_dims_checks(lib):
    lay = hta.HtaKvLayout(1, 128, 4, 4, 1 << 20)
    d = hta.HtaDims(1, 8, 6, 4, 64, 256, 0.0)  # Hq % Hkv != 0
    fake = ctypes.c_void_p(1 << 20)
    assert lib.hta_verify_kv(ctypes.byref(d), ctypes.byref(lay), *([fake] * 10), 1 << 20, None, None) == -2
    # misaligned cache pointer under a valid layout
    d = hta.HtaDims(1, 8, 4, 1, 64, 256, 0.0)
    args = [fake] * 10
    args[1] = ctypes.c_void_p((1 << 20) + 8)
    assert lib.hta_verify_kv(ctypes.byref(d), ctypes.byref(lay), *args, 1 << 20, None, None) == -3
    args = [fake] * 10
    args[0] = None
    assert lib.hta_verify_kv(ctypes.byref(d), ctypes.byref(lay), *args, 1 << 20, None, None) == -1


def test_paged_kv_reserve_maps_every_page():
    inp = wl.random_inputs(2, 4, 8, 2, 64, [100, 0], seed=9, Lmax=256)
    kp, vp, table = wl.paged_kv(inp.k_cache, inp.v_cache, inp.cache_lens, 64, seed=1, reserve=True)
    assert np.all(table >= 0) and len(set(table.ravel().tolist())) == table.size == 8
    back = wl.unpage_kv(kp, table, inp.cache_lens, 256)
    assert np.array_equal(back[0, :, :100], inp.k_cache[0, :, :100])
    # pages past L_b are NaN: nothing was written into them
    assert np.all(kp[table[0, 2:]] == wl.BF16_NAN) and np.all(kp[table[1]] == wl.BF16_NAN)
    assert np.all(kp[table[0, 1], :, 36:] == wl.BF16_NAN)


def test_misaligned_block_table_rejected(lib):
    lay = hta.HtaKvLayout(0, 16, 16, 4, (1 << 20) + 2)
    assert _call(lib, lay) == (-3, -3)

"""GPU parity of the cache-storage layouts (hta_verify_kv, hta_prefix_attn_kv):
token-major (NHD) and paged caches, on every kernel path.

Storage changes only the addresses the K/V tiles come from, so each layout's
result must be bit-identical to the contiguous head-major call on the same
values (same kernel, same schedule: every case's Lmax is a multiple of every
page size, so the grid is the same), and within the parity tolerance of the
CPU fp64 oracle. Paged pools are scattered by a seeded permutation, with NaN
in the unused rows of a sequence's last page and in the spare pages.
"""
import numpy as np
import pytest

from speculative_decoding_tree_hybrid_gb300 import workloads as wl

from _util import assert_close, mask_to_torch, to_device, to_torch_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from speculative_decoding_tree_hybrid_gb300 import build as hbuild  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import hta  # noqa: E402

hbuild.build()
DEV = torch.device("cuda:0")
LMAX = 1536  # a multiple of every page size below

# (B, T, Hq, Hkv, d, lens, kernel path the shape takes)
CASES = {
    "clustered": (3, 64, 32, 8, 128, [300, 1029, 0], hta.PATH_TC2),
    "tensor-core": (2, 8, 32, 8, 128, [700, 129], hta.PATH_TC),
    "cuda-core": (2, 8, 8, 2, 64, [333, 64], hta.PATH_CC),
}
LAYOUTS = [("nhd", 0), ("hnd", 16), ("nhd", 16), ("hnd", 32), ("nhd", 64), ("hnd", 128), ("nhd", 256)]


def stored(inp, order, P, seed=11):
    """Device tensors of the cache (and tree K/V) stored as (order, P)."""
    if P == 0:
        kc, vc, table = inp.k_cache, inp.v_cache, None
        if order == "nhd":
            kc, vc = wl.kv_nhd(kc), wl.kv_nhd(vc)
    else:
        kc, vc, table = wl.paged_kv(inp.k_cache, inp.v_cache, inp.cache_lens, P, order=order, seed=seed)
    ks, vs = (wl.kv_nhd(inp.k_spec), wl.kv_nhd(inp.v_spec)) if order == "nhd" else (inp.k_spec, inp.v_spec)
    t = dict(k_cache=to_torch_bf16(kc, DEV), v_cache=to_torch_bf16(vc, DEV), k_spec=to_torch_bf16(ks, DEV),
             v_spec=to_torch_bf16(vs, DEV))
    t["block_table"] = None if table is None else torch.from_numpy(table).to(DEV)
    return t


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                       b.contiguous().view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))


@pytest.fixture(scope="module")
def contiguous(oracle_mod):
    """Per case: inputs, the contiguous call's (o, lse) and the oracle's."""
    out = {}
    for name, (B, T, Hq, Hkv, d, lens, path) in CASES.items():
        inp = wl.random_inputs(B, T, Hq, Hkv, d, lens, seed=40 + len(out), Lmax=LMAX, tree="window8_depth8")
        t = to_device(inp, DEV)
        mask = hta.build_mask(t["parents"])
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        o, lse = hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"], t["v_spec"],
                            mask, dev_err=err)
        torch.cuda.synchronize()
        assert hta.last_path() == path and int(err.item()) == 0
        m_np, _ = oracle_mod.build_mask(inp.parents)
        ref = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec, inp.v_spec,
                                   m_np)
        assert_close(o, lse, *ref, f"{name} contiguous")
        out[name] = (inp, t, mask, o, lse, ref, path)
    return out


@pytest.mark.parametrize("order,P", LAYOUTS)
@pytest.mark.parametrize("case", list(CASES))
def test_verify_layout_bit_identical(contiguous, case, order, P):
    inp, t, mask, o0, lse0, ref, path = contiguous[case]
    s = stored(inp, order, P)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = hta.verify_kv(t["q"], s["k_cache"], s["v_cache"], t["cache_lens"], s["k_spec"], s["v_spec"], mask,
                           order=order, block_table=s["block_table"], dev_err=err)
    torch.cuda.synchronize()
    assert hta.last_path() == path
    assert int(err.item()) == 0
    assert same_bits(o, o0) and same_bits(lse, lse0), f"{case} {order} P={P}: differs from contiguous"
    assert_close(o, lse, *ref, f"{case} {order} P={P}")


@pytest.mark.parametrize("order,P", [("hnd", 16), ("nhd", 64), ("nhd", 0)])
@pytest.mark.parametrize("case", list(CASES))
def test_verify_layout_in_workspace_sized_by_host_lengths(contiguous, case, order, P):
    # a workspace of exactly hta_verify_workspace_bytes(dims, lens): the call
    # runs with the split-KV workers it holds, within the oracle's tolerance
    inp, t, mask, o0, lse0, ref, path = contiguous[case]
    s = stored(inp, order, P)
    dims, _, _ = hta._kv_layout(t["q"], s["k_cache"], s["v_cache"], t["cache_lens"], order, s["block_table"])
    nbytes = hta.workspace_bytes(dims, inp.cache_lens)
    assert 0 < nbytes <= hta.workspace_bytes(dims)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        o, lse = hta.verify_kv(t["q"], s["k_cache"], s["v_cache"], t["cache_lens"], s["k_spec"], s["v_spec"],
                               mask, order=order, block_table=s["block_table"], ws=ws, dev_err=err)
    torch.cuda.synchronize()
    assert hta.last_path() == path
    assert int(err.item()) == 0
    assert_close(o, lse, *ref, f"{case} {order} P={P}, sized workspace")


@pytest.mark.parametrize("order,P", [("hnd", 16), ("nhd", 128), ("nhd", 0)])
def test_prefix_attn_layout_cross_attention(oracle_mod, order, P):
    """The draft model's cross-attention (a few queries over the target's
    cache) on a paged / token-major cache."""
    inp = wl.random_inputs(2, 1, 32, 8, 128, [1000, 1536], seed=51, Lmax=LMAX)
    t = to_device(inp, DEV)
    o0, lse0 = hta.prefix_attn(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"])
    s = stored(inp, order, P)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = hta.prefix_attn_kv(t["q"], s["k_cache"], s["v_cache"], t["cache_lens"], order=order,
                                block_table=s["block_table"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert same_bits(o, o0) and same_bits(lse, lse0)
    zero = np.zeros((2, 1, 1), np.uint32)
    ref = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec, inp.v_spec, zero)
    assert_close(o, lse, *ref, f"cross {order} P={P}")


@pytest.mark.parametrize("case", list(CASES))
def test_bad_page_entry_is_flagged(contiguous, case):
    """A block-table entry outside the pool is read as page 0 and flagged."""
    inp, t, mask, *_ = contiguous[case]
    s = stored(inp, "hnd", 64)
    bt = s["block_table"]
    bt[1, 0] = s["k_cache"].shape[0] + 5  # the first page of sequence 1 (every case has one)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = hta.verify_kv(t["q"], s["k_cache"], s["v_cache"], t["cache_lens"], s["k_spec"], s["v_spec"], mask,
                           block_table=bt, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & hta.DEVERR_PAGE
    # sequence 0 reads none of the bad entry's keys
    assert torch.isfinite(lse[0]).all()


def test_paged_full_llama_shape_sampled(oracle_mod):
    """LLaMA-3.1-8B layer shape at L = 32768 on 16-token pages, token-major:
    bit-identical to the contiguous call."""
    inp = wl.make_inputs("llama8b")
    t = to_device(inp, DEV)
    mask = hta.build_mask(t["parents"])
    o0, lse0 = hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"], t["v_spec"], mask)
    s = stored(inp, "nhd", 16, seed=2)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = hta.verify_kv(t["q"], s["k_cache"], s["v_cache"], t["cache_lens"], s["k_spec"], s["v_spec"], mask,
                           order="nhd", block_table=s["block_table"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert same_bits(o, o0) and same_bits(lse, lse0)


@pytest.mark.parametrize("order,P", [("hnd", 16), ("nhd", 64), ("nhd", 0), ("hnd", 128)])
def test_accept_commit_layout(order, P):
    """Accept walk + KV commit into a paged / token-major cache: the appended
    rows, lengths and walk results equal the oracle's (bit-exact), with one
    sequence clamped at Lmax."""
    from oracle.accept import accept_commit as accept_ref
    rng = np.random.default_rng(5)
    B, T, Hkv, d, Lmax = 3, 32, 2, 128, 256
    par = np.stack([wl.tree_window8_depth8(T, rng) for _ in range(B)]).astype(np.int32)
    draft = rng.integers(0, 2, size=(B, T)).astype(np.int32)
    target = rng.integers(0, 2, size=(B, T)).astype(np.int32)
    ks, vs = wl.normal_bf16(rng, (B, Hkv, T, d)), wl.normal_bf16(rng, (B, Hkv, T, d))
    kc, vc = wl.normal_bf16(rng, (B, Hkv, Lmax, d)), wl.normal_bf16(rng, (B, Hkv, Lmax, d))
    cl = np.array([0, 100, 254], np.int32)
    for b in range(B):
        kc[b, :, cl[b]:] = wl.BF16_NAN
        vc[b, :, cl[b]:] = wl.BF16_NAN
    r_acc, r_n, r_nxt, r_kc, r_vc, r_lens, clamped = accept_ref(par, draft, target, ks, vs, kc, vc, cl)

    if P:
        kp, vp, table = wl.paged_kv(kc, vc, cl, P, order=order, seed=4, reserve=True)
        bt = torch.from_numpy(table).to(DEV)
    else:
        kp, vp, bt = (wl.kv_nhd(kc), wl.kv_nhd(vc), None) if order == "nhd" else (kc, vc, None)
    ks_s, vs_s = (wl.kv_nhd(ks), wl.kv_nhd(vs)) if order == "nhd" else (ks, vs)
    kd, vd = to_torch_bf16(kp, DEV), to_torch_bf16(vp, DEV)
    lens = torch.from_numpy(cl.copy()).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    i32 = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    acc, n_acc, nxt = hta.accept_commit_kv(i32(par), i32(draft), i32(target), to_torch_bf16(ks_s, DEV),
                                           to_torch_bf16(vs_s, DEV), kd, vd, lens, order=order, block_table=bt,
                                           dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), r_acc) and np.array_equal(n_acc.cpu().numpy(), r_n)
    assert np.array_equal(nxt.cpu().numpy(), r_nxt) and np.array_equal(lens.cpu().numpy(), r_lens)
    assert bool(int(err.item()) & hta.DEVERR_CACHE_LEN) == (clamped > 0)
    assert not int(err.item()) & hta.DEVERR_PAGE
    for got_dev, ref in ((kd, r_kc), (vd, r_vc)):
        got = got_dev.cpu().view(torch.int16).numpy().view(np.uint16)
        if P:
            got = wl.unpage_kv(got, table, r_lens, Lmax, order=order)
        elif order == "nhd":
            got = np.ascontiguousarray(np.swapaxes(got, 1, 2))
        for b in range(B):
            assert np.array_equal(got[b, :, :r_lens[b]], ref[b, :, :r_lens[b]]), f"sequence {b}"


def test_accept_commit_bad_page_is_flagged():
    """An appended row whose page entry lies outside the pool is not written."""
    rng = np.random.default_rng(6)
    B, T, Hkv, d, Lmax = 1, 8, 1, 64, 128
    par = wl.tree_chain(T)[None].astype(np.int32)
    draft = np.zeros((B, T), np.int32)
    target = np.zeros((B, T), np.int32)  # the whole chain is accepted
    ks, vs = wl.normal_bf16(rng, (B, Hkv, T, d)), wl.normal_bf16(rng, (B, Hkv, T, d))
    kc, vc = wl.normal_bf16(rng, (B, Hkv, Lmax, d)), wl.normal_bf16(rng, (B, Hkv, Lmax, d))
    cl = np.array([60], np.int32)  # rows 60..67 cross from page 3 into page 4 (16-token pages)
    kp, vp, table = wl.paged_kv(kc, vc, cl, 16, seed=2, reserve=True)
    table[0, 4] = 10_000
    kd, vd = to_torch_bf16(kp, DEV), to_torch_bf16(vp, DEV)
    before = kd.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    hta.accept_commit_kv(i32(par), i32(draft), i32(target), to_torch_bf16(ks, DEV), to_torch_bf16(vs, DEV), kd, vd,
                         i32(cl.copy()), block_table=i32(table), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & hta.DEVERR_PAGE
    # rows 60..63 (page 3) written, nothing else in the pool changed
    pg3 = int(table[0, 3])
    changed = (kd.view(torch.int16) != before.view(torch.int16)).any(dim=-1).nonzero().tolist()
    assert changed and all(c[0] == pg3 and c[2] >= 12 for c in changed)

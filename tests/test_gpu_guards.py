"""Out-of-bounds writes, checked without a sanitizer: every buffer a kernel
writes (outputs, workspace, committed cache, accept outputs) is carved out of
a larger allocation whose head and tail are filled with a known byte pattern;
after the calls (which must also be parity-green) the guard bytes must be
unchanged."""
import numpy as np
import pytest

import oracle
from oracle.accept import accept_commit as accept_ref
from speculative_decoding_tree_hybrid_gb300 import workloads as wl

from _util import assert_close, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from speculative_decoding_tree_hybrid_gb300 import build as hbuild  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import hta  # noqa: E402

hbuild.build()
oracle.build()
DEV = torch.device("cuda:0")
GUARD = 4096  # bytes on each side
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape`/`dtype` in the middle of a byte buffer with guards."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device=DEV)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        head, tail = self.raw[:GUARD], self.raw[-GUARD:]
        return bool(torch.all(head == PATTERN)) and bool(torch.all(tail == PATTERN))


CASES = [
    (1, 64, 32, 8, 128, [3000], "window8_depth8", "tc2"),
    (2, 32, 8, 8, 128, [700, 129], "uniform", "tc"),
    (1, 8, 4, 1, 64, [256], "uniform", "cc"),
    (3, 16, 8, 2, 64, [0, 300, 1029], "uniform", "cc"),
]


@pytest.mark.parametrize("case", CASES)
def test_verify_and_prefix_write_nothing_outside_their_buffers(case, monkeypatch):
    B, T, Hq, Hkv, d, lens, tree, path = case
    monkeypatch.setenv("HTA_FORCE_PATH", path)
    inp = wl.random_inputs(B, T, Hq, Hkv, d, lens, seed=41, tree=tree)
    t = to_device(inp, DEV)
    mask = hta.build_mask(t["parents"])
    ref_mask, _ = oracle.build_mask(inp.parents)
    dims = hta.dims_of(t["q"], t["k_cache"])
    nbytes = hta.workspace_bytes(dims)
    ws = Guarded((nbytes,), torch.uint8, fill=torch.zeros(nbytes, dtype=torch.uint8, device=DEV))
    o = Guarded(tuple(t["q"].shape), torch.bfloat16)
    lse = Guarded(tuple(t["q"].shape[:3]), torch.float32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):  # twice: the second call starts from the first one's workspace
        hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"], t["v_spec"], mask,
                   ws=ws.t, dev_err=err, out=(o.t, lse.t))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, lse_ref = oracle.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec, inp.v_spec,
                                      ref_mask)
    assert_close(o.t, lse.t, o_ref, lse_ref, f"verify {case}")
    assert ws.intact() and o.intact() and lse.intact()

    oc = Guarded(tuple(t["q"].shape), torch.float32)
    lc = Guarded(tuple(t["q"].shape[:3]), torch.float32)
    hta.prefix_attn(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], ws=ws.t, dev_err=err, out=(oc.t, lc.t))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    zero_mask = np.zeros_like(ref_mask)
    oc_ref, lc_ref = oracle.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec, inp.v_spec,
                                      zero_mask)
    assert_close(oc.t, lc.t, oc_ref, lc_ref, f"prefix {case}")
    assert ws.intact() and oc.intact() and lc.intact()


# short lengths in a cache whose Lmax is far longer: the calls size their grid
# from Lmax, a workspace from the lengths' query holds fewer workers' records
SIZED_CASES = [
    (1, 64, 32, 8, 128, [300], 8192, "window8_depth8", "tc2"),
    (2, 32, 8, 8, 128, [40, 129], 8192, "uniform", "tc"),
    (3, 16, 8, 2, 64, [0, 30, 100], 4096, "uniform", "cc"),
]


@pytest.mark.parametrize("case", SIZED_CASES)
def test_workspace_sized_by_host_lengths_is_enough(case, monkeypatch):
    B, T, Hq, Hkv, d, lens, Lmax, tree, path = case
    monkeypatch.setenv("HTA_FORCE_PATH", path)
    inp = wl.random_inputs(B, T, Hq, Hkv, d, lens, seed=43, Lmax=Lmax, tree=tree)
    t = to_device(inp, DEV)
    mask = hta.build_mask(t["parents"])
    ref_mask, _ = oracle.build_mask(inp.parents)
    dims = hta.dims_of(t["q"], t["k_cache"])
    nbytes = hta.workspace_bytes(dims, inp.cache_lens)
    assert 0 < nbytes < hta.workspace_bytes(dims)  # the case really is below the Lmax bound
    ws = Guarded((nbytes,), torch.uint8, fill=torch.zeros(nbytes, dtype=torch.uint8, device=DEV))
    o = Guarded(tuple(t["q"].shape), torch.bfloat16)
    lse = Guarded(tuple(t["q"].shape[:3]), torch.float32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"], t["v_spec"], mask,
                   ws=ws.t, dev_err=err, out=(o.t, lse.t))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, lse_ref = oracle.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec, inp.v_spec,
                                      ref_mask)
    assert_close(o.t, lse.t, o_ref, lse_ref, f"verify, sized workspace {case}")
    assert ws.intact() and o.intact() and lse.intact()

    oc = Guarded(tuple(t["q"].shape), torch.float32)
    lc = Guarded(tuple(t["q"].shape[:3]), torch.float32)
    hta.prefix_attn(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], ws=ws.t, dev_err=err, out=(oc.t, lc.t))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oc_ref, lc_ref = oracle.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec, inp.v_spec,
                                      np.zeros_like(ref_mask))
    assert_close(oc.t, lc.t, oc_ref, lc_ref, f"prefix, sized workspace {case}")
    assert ws.intact() and oc.intact() and lc.intact()


def test_accept_commit_writes_nothing_outside_its_buffers():
    rng = np.random.default_rng(5)
    B, T, Hkv, d, Lmax = 3, 32, 2, 128, 96
    par = np.stack([wl.tree_window8_depth8(T, rng) for _ in range(B)]).astype(np.int32)
    draft = rng.integers(0, 4, size=(B, T)).astype(np.int32)
    target = rng.integers(0, 4, size=(B, T)).astype(np.int32)
    ks = wl.normal_bf16(rng, (B, Hkv, T, d))
    vs = wl.normal_bf16(rng, (B, Hkv, T, d))
    kc = wl.normal_bf16(rng, (B, Hkv, Lmax, d))
    vc = wl.normal_bf16(rng, (B, Hkv, Lmax, d))
    cl = np.array([3, 60, 90], np.int32)  # the last one reaches Lmax: clamped

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)
    kc_g = Guarded(kc.shape, torch.bfloat16, fill=bf(kc))
    vc_g = Guarded(vc.shape, torch.bfloat16, fill=bf(vc))
    cl_g = Guarded((B,), torch.int32, fill=torch.from_numpy(cl).to(DEV))
    acc = Guarded((B, T), torch.int32)
    n_acc = Guarded((B,), torch.int32)
    nxt = Guarded((B,), torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    hta.accept_commit(torch.from_numpy(par).to(DEV), torch.from_numpy(draft).to(DEV),
                      torch.from_numpy(target).to(DEV), bf(ks), bf(vs), kc_g.t, vc_g.t, cl_g.t, dev_err=err,
                      out=(acc.t, n_acc.t, nxt.t))
    torch.cuda.synchronize()
    r_acc, r_n, r_nxt, r_kc, r_vc, r_lens, _ = accept_ref(par, draft, target, ks, vs, kc, vc, cl)
    assert np.array_equal(acc.t.cpu().numpy(), r_acc) and np.array_equal(n_acc.t.cpu().numpy(), r_n)
    assert np.array_equal(nxt.t.cpu().numpy(), r_nxt) and np.array_equal(cl_g.t.cpu().numpy(), r_lens)
    assert np.array_equal(kc_g.t.cpu().view(torch.int16).numpy().view(np.uint16), r_kc)
    assert np.array_equal(vc_g.t.cpu().view(torch.int16).numpy().view(np.uint16), r_vc)
    for g in (kc_g, vc_g, cl_g, acc, n_acc, nxt):
        assert g.intact()

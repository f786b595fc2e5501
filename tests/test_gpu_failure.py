"""Failure detection on the GPU without a GPU fault: the bounded grid-barrier
wait before the merge is made to run out (HTA_TEST_BARRIER_WAIT_CYCLES=1, read
on every call). Every async copy of a CTA has completed before it waits there,
so a CTA that gives up has nothing in flight. Checked: the device flag
HTA_DEVERR_TIMEOUT is raised, the rows that could not be merged are NaN (no
silent wrong values: every other row still matches the oracle), and the
workspace counters are back at zero, so the next normal call on the same
workspace is parity-green."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_hybrid_gb300 import workloads as wl

from _util import LSE_REL_TOL, O_ABS_TOL, assert_close, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from speculative_decoding_tree_hybrid_gb300 import build as hbuild  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import hta  # noqa: E402

hbuild.build()
oracle.build()
DEV = torch.device("cuda:0")


# (B, T, lens): 256 packed rows per KV head; and one query per sequence (4
# rows per KV head, each split over many workers: several threads merge a row)
SHAPES = {"tree64": (2, 64, [6000, 2500]), "one_query": (1, 1, [9000])}


@pytest.mark.parametrize("path,shape", [("tc2", "tree64"), ("tc", "tree64"), ("cc", "tree64"),
                                        ("tc", "one_query"), ("cc", "one_query")])
def test_barrier_timeout_flags_nan_and_recovers(path, shape, monkeypatch):
    monkeypatch.setenv("HTA_FORCE_PATH", path)
    B, T, lens = SHAPES[shape]
    tree = "window8_depth8" if T > 1 else "uniform"
    inp = wl.random_inputs(B, T, 32, 8, 128, lens, seed=31, tree=tree)
    t = to_device(inp, DEV)
    mask = hta.build_mask(t["parents"])
    ref_mask, _ = oracle.build_mask(inp.parents)
    o_ref, lse_ref = oracle.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec, inp.v_spec,
                                      ref_mask)
    dims = hta.dims_of(t["q"], t["k_cache"])
    ws = hta.workspace(dims, DEV)

    def call():
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        o, lse = hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"], t["v_spec"], mask,
                            ws=ws, dev_err=err)
        torch.cuda.synchronize()
        return o, lse, int(err.item())

    monkeypatch.setenv("HTA_TEST_BARRIER_WAIT_CYCLES", "1")
    o, lse, err = call()
    assert err & hta.DEVERR_TIMEOUT, f"timeout not flagged (flags {err})"
    o64 = o.float().cpu().numpy().astype(np.float64)
    lse64 = lse.cpu().numpy().astype(np.float64)
    bad = np.isnan(lse64)
    assert bad.any(), "no row was left unmerged"
    assert np.all(np.isnan(o64[bad])), "an unmerged row holds a number"
    good = ~bad
    assert np.all(np.abs(o64[good] - o_ref[good]) <= O_ABS_TOL)
    assert np.all(np.abs(lse64[good] - lse_ref[good]) <= LSE_REL_TOL * np.maximum(1.0, np.abs(lse_ref[good])))

    monkeypatch.delenv("HTA_TEST_BARRIER_WAIT_CYCLES")
    o, lse, err = call()
    assert err == 0
    assert_close(o, lse, o_ref, lse_ref, f"{path}: call after the timed-out one")

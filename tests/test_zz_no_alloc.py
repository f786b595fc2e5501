"""hta_verify_noalloc: the verify entry point for callers that cannot allocate
device memory when they call it (fixed memory pools, framework plug-ins that
only receive tensors, code running under stream capture). It keeps its
split-KV partials in a static device array instead of a caller workspace.

Called through the C ABI twice in a row (the array keeps the previous call's
contents, so the second call checks that nothing stale leaks through) and
compared both with hta_verify and with the fp64 oracle on the same inputs,
within the parity tolerances of the other GPU tests. This file is collected
last on purpose.
"""
import ctypes

import numpy as np
import pytest

from speculative_decoding_tree_hybrid_gb300 import workloads as wl

from _util import assert_close, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from speculative_decoding_tree_hybrid_gb300 import build as hbuild  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import hta  # noqa: E402

hbuild.build()
DEV = torch.device("cuda:0")
SCRATCH_BYTES = 32 << 20  # HTA_NOALLOC_SCRATCH_BYTES in include/hta.h


def call_noalloc(t, mask, o, lse, err):
    lib = hta.load()
    dims = hta.dims_of(t["q"], t["k_cache"])
    stream = torch.cuda.current_stream(DEV).cuda_stream
    return lib.hta_verify_noalloc(ctypes.byref(dims), t["q"].data_ptr(), t["k_cache"].data_ptr(),
                                  t["v_cache"].data_ptr(), t["cache_lens"].data_ptr(),
                                  t["k_spec"].data_ptr(), t["v_spec"].data_ptr(), mask.data_ptr(),
                                  o.data_ptr(), lse.data_ptr(), err.data_ptr(), stream)


@pytest.mark.parametrize("shape", [
    (1, 64, 32, 8, 128, [3000], "window8_depth8"),   # LLaMA-3.1-8B layer shape, tensor-core path
    (1, 8, 4, 1, 64, [256], "uniform"),              # tiny shape, CUDA-core path
    (2, 32, 8, 8, 128, [700, 129], "uniform"),       # two sequences of different lengths
])
def test_noalloc_matches_verify_twice(oracle_mod, shape):
    B, T, Hq, Hkv, d, lens, tree = shape
    outs = []
    for call, seed in enumerate((71, 72)):  # two calls in a row, different inputs
        inp = wl.random_inputs(B, T, Hq, Hkv, d, lens, seed=seed, tree=tree)
        t = to_device(inp, DEV)
        mask = hta.build_mask(t["parents"])
        o_ref, lse_ref = hta.verify(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], t["k_spec"],
                                    t["v_spec"], mask)
        o = torch.full_like(t["q"], float("nan"))
        lse = torch.full(t["q"].shape[:3], float("nan"), dtype=torch.float32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        st = call_noalloc(t, mask, o, lse, err)
        torch.cuda.synchronize()
        assert st == 0, hta.status_string(st)
        assert int(err.item()) == 0
        assert_close(o, lse, o_ref.double().cpu().numpy(), lse_ref.double().cpu().numpy(),
                     f"no-alloc call {call} vs hta_verify")
        ref_mask, bad = oracle_mod.build_mask(inp.parents)
        assert bad == 0
        o_or, lse_or = oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens,
                                            inp.k_spec, inp.v_spec, ref_mask)
        assert_close(o, lse, o_or, lse_or, f"no-alloc call {call} vs oracle")
        outs.append(o)
    assert not torch.equal(outs[0], outs[1])  # the second call really recomputed


def test_noalloc_rejects_dims_beyond_the_scratch():
    # 1024 sequences x 64 KV heads of 256 packed rows need far more than 32 MiB
    dims = hta.HtaDims(1024, 64, 256, 64, 128, 4096, 0.0)
    assert hta.workspace_bytes(dims) > SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)  # rejected before any pointer is used
    st = hta.load().hta_verify_noalloc(ctypes.byref(dims), *([fake] * 9), None, None)
    assert st == -5  # HTA_ERR_WORKSPACE

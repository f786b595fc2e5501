"""CPU checks of the C-ABI boundary: the library builds for sm_103a, loads,
exports every function include/hta.h declares, and rejects bad arguments on
the host before any launch. No kernel runs here."""
import ctypes
import os
import re

import pytest

from speculative_decoding_tree_hybrid_gb300 import build as hbuild
from speculative_decoding_tree_hybrid_gb300 import hta

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "hta.h")


@pytest.fixture(scope="module")
def lib():
    hbuild.build()
    return hta.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hta_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for required in ("hta_build_mask", "hta_prefix_attn", "hta_tree_attn", "hta_merge",
                     "hta_verify", "hta_verify_workspace_bytes", "hta_status_string"):
        assert required in names
    assert set(names) == set(hta.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(0, -8, -1):
        s = hta.status_string(code)
        assert s and s != "unknown status"
    assert hta.status_string(-99) == "unknown status"


def _dims(**kw):
    base = dict(B=1, T=8, Hq=4, Hkv=1, d=64, Lmax=256, scale=0.0)
    base.update(kw)
    return hta.HtaDims(base["B"], base["T"], base["Hq"], base["Hkv"], base["d"], base["Lmax"], base["scale"])


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), -1), (dict(T=0), -1), (dict(Hq=0), -1), (dict(Lmax=-1), -1), (dict(scale=-1.0), -1),
    (dict(Hq=6, Hkv=4), -2), (dict(d=96), -2), (dict(T=257), -2), (dict(B=1025), -2),
])
def test_verify_rejects_bad_dims_on_host(lib, kw, status):
    d = _dims(**kw)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the call returns before any launch
    st = lib.hta_verify(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                        1 << 20, None, None)
    assert st == status


def test_verify_rejects_null_and_misaligned_pointers(lib):
    d = _dims()
    good = ctypes.c_void_p(1 << 20)
    args = [good] * 10
    for i in range(9):
        a = list(args)
        a[i] = None
        assert lib.hta_verify(ctypes.byref(d), *a, 1 << 20, None, None) == -1
    a = list(args)
    a[0] = ctypes.c_void_p((1 << 20) + 2)
    assert lib.hta_verify(ctypes.byref(d), *a, 1 << 20, None, None) == -3


def test_build_mask_rejects_bad_sizes(lib):
    p = ctypes.c_void_p(1 << 20)
    assert lib.hta_build_mask(None, 1, 8, p, None, None) == -1
    assert lib.hta_build_mask(p, 0, 8, p, None, None) == -1
    assert lib.hta_build_mask(p, 1, 257, p, None, None) == -2


def test_merge_and_tree_reject_bad_args(lib):
    d = _dims()
    p = ctypes.c_void_p(1 << 20)
    assert lib.hta_merge(ctypes.byref(d), None, p, p, p, p, p, None) == -1
    assert lib.hta_tree_attn(ctypes.byref(d), p, p, p, p, p, None, None) == -1
    assert lib.hta_prefix_attn(None, p, p, p, p, p, p, p, 0, None, None) == -1


def test_workspace_query_without_device_is_zero_or_sized(lib):
    n = hta.workspace_bytes(_dims())
    assert n == 0 or n >= 256
    assert hta.workspace_bytes(_dims(d=96)) == 0


def test_verify_workspace_bytes_signature(lib):
    """hta_verify_workspace_bytes(dims, host_cache_lens): NULL bounds every
    length <= Lmax; host lengths give a size no larger than that bound; the
    old name is the NULL form."""
    import numpy as np
    d = _dims(B=2, Lmax=4096)
    lens = np.array([100, 4096], np.int32)
    bound = int(lib.hta_verify_workspace_bytes(ctypes.byref(d), None))
    sized = int(lib.hta_verify_workspace_bytes(ctypes.byref(d), lens.ctypes.data))
    assert bound == int(lib.hta_workspace_bytes(ctypes.byref(d)))
    assert sized <= bound
    assert hta.workspace_bytes(d, lens) == sized and hta.workspace_bytes(d) == bound
    with pytest.raises(ValueError):
        hta.workspace_bytes(d, np.zeros(3, np.int32))
    assert int(lib.hta_verify_workspace_bytes(None, None)) == 0


def test_verify_refuses_memory_that_is_not_on_the_current_device(lib):
    """Valid dims, aligned pointers that are not device allocations of the
    current device (or no device at all): refused on the host with
    HTA_ERR_INVALID_ARG before any launch."""
    d = _dims()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.hta_verify(ctypes.byref(d), *([fake] * 10), 1 << 20, None, None) == -1
    assert lib.hta_prefix_attn(ctypes.byref(d), *([fake] * 7), 1 << 20, None, None) == -1
    assert lib.hta_tree_attn(ctypes.byref(d), *([fake] * 6), None) == -1


def test_binding_refuses_host_tensors():
    """The binding has no CPU path: host tensors are rejected before any call."""
    torch = pytest.importorskip("torch")
    q = torch.zeros((1, 8, 4, 64), dtype=torch.bfloat16)
    kc = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16)
    lens = torch.zeros(1, dtype=torch.int32)
    ks = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    mask = torch.zeros((1, 8, 1), dtype=torch.int32)
    parents = torch.zeros((1, 8), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        hta.verify(q, kc, kc, lens, ks, ks, mask)
    with pytest.raises(ValueError, match="CUDA"):
        hta.verify_kv(q, kc, kc, lens, ks, ks, mask, order="nhd")
    with pytest.raises(ValueError, match="CUDA"):
        hta.prefix_attn(q, kc, kc, lens)
    with pytest.raises(ValueError, match="CUDA"):
        hta.build_mask(parents)


def test_int32_arrays_must_be_4_byte_aligned(lib):
    """A misaligned int32 / fp32 array is refused on the host (the device
    would fault on it)."""
    d = _dims()
    good = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)
    # hta_verify: q, kc, vc, cache_lens, ks, vs, mask, o, lse, ws
    for idx in (3, 6, 8):  # cache_lens, mask, lse
        a = [good] * 10
        a[idx] = odd
        assert lib.hta_verify(ctypes.byref(d), *a, 1 << 20, None, None) == -3
    # dev_err
    assert lib.hta_verify(ctypes.byref(d), *([good] * 10), 1 << 20, odd, None) == -3
    assert lib.hta_build_mask(odd, 1, 8, good, None, None) == -3
    assert lib.hta_build_mask(good, 1, 8, odd, None, None) == -3
    # hta_merge: o_c, lse_c, o_s, lse_s, o, lse
    assert lib.hta_merge(ctypes.byref(d), good, odd, good, good, good, good, None) == -3

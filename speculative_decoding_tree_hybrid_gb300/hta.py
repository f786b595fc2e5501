"""Thin ctypes binding of libhta (C ABI declared in include/hta.h).

Argument marshalling only: every function checks tensor devices, dtypes and
shapes, allocates outputs through torch, and passes raw device pointers and
torch's current CUDA stream to the library. All computation happens in the
library's CUDA kernels; there is no fallback of any kind, and loading fails
loudly when libhta.so has not been built.

bf16 tensors are torch.bfloat16; masks are int32 tensors holding the uint32
mask words bit for bit.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None
_ws_cache: dict = {}

PATH_CC, PATH_TC, PATH_TC2 = 1, 2, 3
DEVERR_BAD_TREE, DEVERR_CACHE_LEN, DEVERR_TIMEOUT, DEVERR_LAUNCH, DEVERR_PAGE = 1, 2, 4, 8, 16
KV_HND, KV_NHD = 0, 1
TMAX, BMAX = 256, 1024

# every exported symbol of include/hta.h
EXPORTS = ("hta_build_mask", "hta_verify_workspace_bytes", "hta_workspace_bytes", "hta_prefix_attn",
           "hta_tree_attn",
           "hta_merge", "hta_verify", "hta_verify_noalloc", "hta_accept_commit", "hta_window_attn",
           "hta_logitspec_tree", "hta_verify_kv", "hta_prefix_attn_kv", "hta_accept_commit_kv",
           "hta_status_string",
           "hta_last_path")


class HtaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class HtaDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("Lmax", ctypes.c_int64),
                ("scale", ctypes.c_float)]


class HtaKvLayout(ctypes.Structure):
    _fields_ = [("order", ctypes.c_int32), ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("block_table", ctypes.c_void_p)]


def library_path() -> str:
    return _build.LIB


def load():
    """Loads libhta.so from the package's build folder (raises if absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libhta.so is not built ({path}); call "
                               "speculative_decoding_tree_hybrid_gb300.build.build() first")
        lib = ctypes.CDLL(path)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(HtaDims)
        lib.hta_build_mask.argtypes = [P, I32, I32, P, P, P]
        lib.hta_verify_workspace_bytes.argtypes = [D, P]
        lib.hta_verify_workspace_bytes.restype = SZ
        lib.hta_workspace_bytes.argtypes = [D]
        lib.hta_workspace_bytes.restype = SZ
        lib.hta_prefix_attn.argtypes = [D, P, P, P, P, P, P, P, SZ, P, P]
        lib.hta_tree_attn.argtypes = [D, P, P, P, P, P, P, P]
        lib.hta_merge.argtypes = [D, P, P, P, P, P, P, P]
        lib.hta_verify.argtypes = [D, P, P, P, P, P, P, P, P, P, P, SZ, P, P]
        lib.hta_verify_noalloc.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P]
        lib.hta_accept_commit.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, P, P]
        lib.hta_window_attn.argtypes = [D, I32, P, P, P, P, P, P, P, P]
        lib.hta_logitspec_tree.argtypes = [I32, I32, I64, I32, I32, I32, P, P, P, P, P, P, P, P, P, P]
        KL = ctypes.POINTER(HtaKvLayout)
        lib.hta_verify_kv.argtypes = [D, KL, P, P, P, P, P, P, P, P, P, P, SZ, P, P]
        lib.hta_prefix_attn_kv.argtypes = [D, KL, P, P, P, P, P, P, P, SZ, P, P]
        lib.hta_accept_commit_kv.argtypes = [D, KL, P, P, P, P, P, P, P, P, P, P, P, P, P]
        lib.hta_status_string.argtypes = [ctypes.c_int]
        lib.hta_status_string.restype = ctypes.c_char_p
        lib.hta_last_path.restype = I32
        for name in ("hta_build_mask", "hta_prefix_attn", "hta_tree_attn", "hta_merge", "hta_verify",
                     "hta_verify_noalloc", "hta_accept_commit", "hta_window_attn", "hta_logitspec_tree"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().hta_status_string(int(status)).decode()


def last_path() -> int:
    return int(load().hta_last_path())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(t, name, dtype, ndim, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def dims_of(q, k_cache, scale: float = 0.0) -> HtaDims:
    B, T, Hq, d = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    return HtaDims(B, T, Hq, Hkv, d, Lmax, float(scale))


def workspace_bytes(dims: HtaDims, host_cache_lens=None) -> int:
    """hta_verify_workspace_bytes: host_cache_lens is None (bound over every
    length <= Lmax) or a host int32 array of the B cache lengths."""
    if host_cache_lens is None:
        return int(load().hta_verify_workspace_bytes(ctypes.byref(dims), None))
    import numpy as np
    lens = np.ascontiguousarray(host_cache_lens, dtype=np.int32)
    if lens.shape != (dims.B,):
        raise ValueError("host_cache_lens must hold B lengths")
    return int(load().hta_verify_workspace_bytes(ctypes.byref(dims), lens.ctypes.data))


def workspace(dims: HtaDims, device) -> torch.Tensor:
    """A zero-initialised workspace for these dims, cached per device and stream.

    Calls that share it must run in stream order (the library resets its
    barrier counters at the end of every call).
    """
    device = torch.device(device)
    nbytes = workspace_bytes(dims)
    if nbytes == 0:
        raise HtaError(-1, "hta_workspace_bytes")
    key = (device, _stream(device))
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _raise(status: int, what: str):
    if status != 0:
        raise HtaError(status, what)


def build_mask(parents: torch.Tensor, dev_err: torch.Tensor | None = None,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """parents int32 [B][T] -> ancestor-or-self mask words int32 [B][T][ceil(T/32)]."""
    _check(parents, "parents", torch.int32, 2)
    B, T = parents.shape
    if out is None:
        mask = torch.empty((B, T, (T + 31) // 32), dtype=torch.int32, device=parents.device)
    else:
        _check(out, "out", torch.int32, 3, parents.device)
        if tuple(out.shape) != (B, T, (T + 31) // 32):
            raise ValueError("out must be [B][T][ceil(T/32)]")
        mask = out
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, 1, parents.device)
    with torch.cuda.device(parents.device):
        _raise(load().hta_build_mask(_ptr(parents), B, T, _ptr(mask), _ptr(dev_err),
                                     _stream(parents.device)), "hta_build_mask")
    return mask


def _check_qkv(q, k_cache, v_cache, cache_lens):
    _check(q, "q", torch.bfloat16, 4)
    dev = q.device
    _check(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _check(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _check(cache_lens, "cache_lens", torch.int32, 1, dev)
    B, T, Hq, d = q.shape
    if k_cache.shape[0] != B or k_cache.shape[3] != d or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [B][Hkv][Lmax][d] matching q")
    if cache_lens.shape[0] != B:
        raise ValueError("cache_lens must be [B]")


def _check_spec(q, k_spec, v_spec, mask, Hkv):
    B, T, Hq, d = q.shape
    dev = q.device
    _check(k_spec, "k_spec", torch.bfloat16, 4, dev)
    _check(v_spec, "v_spec", torch.bfloat16, 4, dev)
    _check(mask, "mask", torch.int32, 3, dev)
    if tuple(k_spec.shape) != (B, Hkv, T, d) or v_spec.shape != k_spec.shape:
        raise ValueError("k_spec/v_spec must be [B][Hkv][T][d]")
    if tuple(mask.shape) != (B, T, (T + 31) // 32):
        raise ValueError("mask must be [B][T][ceil(T/32)]")


def verify(q, k_cache, v_cache, cache_lens, k_spec, v_spec, mask, *, scale: float = 0.0,
           ws: torch.Tensor | None = None, dev_err: torch.Tensor | None = None,
           out: tuple | None = None):
    """Fused hybrid tree attention. Returns (o bf16 [B][T][Hq][d], lse fp32 [B][T][Hq])."""
    _check_qkv(q, k_cache, v_cache, cache_lens)
    _check_spec(q, k_spec, v_spec, mask, k_cache.shape[1])
    dims = dims_of(q, k_cache, scale)
    dev = q.device
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    else:
        o, lse = out
    if ws is None:
        ws = workspace(dims, dev)
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, 1, dev)
    with torch.cuda.device(dev):
        _raise(load().hta_verify(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(cache_lens), _ptr(k_spec), _ptr(v_spec), _ptr(mask), _ptr(o),
                                 _ptr(lse), _ptr(ws), ws.numel(), _ptr(dev_err), _stream(dev)),
               "hta_verify")
    return o, lse


def prefix_attn(q, k_cache, v_cache, cache_lens, *, scale: float = 0.0,
                ws: torch.Tensor | None = None, dev_err: torch.Tensor | None = None, out: tuple | None = None):
    """Cached part alone. Returns (o_c fp32 [B][T][Hq][d], lse_c fp32 [B][T][Hq]),
    written into `out` when given."""
    _check_qkv(q, k_cache, v_cache, cache_lens)
    dims = dims_of(q, k_cache, scale)
    dev = q.device
    if out is None:
        o_c = torch.empty(q.shape, dtype=torch.float32, device=dev)
        lse_c = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    else:
        o_c, lse_c = out
        _check(o_c, "o_c", torch.float32, 4, dev)
        _check(lse_c, "lse_c", torch.float32, 3, dev)
        if o_c.shape != q.shape or lse_c.shape != q.shape[:3]:
            raise ValueError("out must be (o_c [B][T][Hq][d], lse_c [B][T][Hq])")
    if ws is None:
        ws = workspace(dims, dev)
    with torch.cuda.device(dev):
        _raise(load().hta_prefix_attn(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(cache_lens), _ptr(o_c), _ptr(lse_c), _ptr(ws), ws.numel(),
                                      _ptr(dev_err), _stream(dev)), "hta_prefix_attn")
    return o_c, lse_c


def _kv_layout(q, k_cache, v_cache, cache_lens, order: str, block_table):
    """Checks a cache stored as `order` ("hnd" or "nhd"), contiguous
    (block_table None: [B][Hkv][Lmax][d] or [B][Lmax][Hkv][d]) or paged
    (a pool [pages][Hkv][P][d] or [pages][P][Hkv][d] and block_table int32
    [B][max_pages]). Returns (dims, HtaKvLayout, Hkv)."""
    if order not in ("hnd", "nhd"):
        raise ValueError("order must be 'hnd' or 'nhd'")
    nhd = order == "nhd"
    _check(q, "q", torch.bfloat16, 4)
    dev = q.device
    _check(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _check(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _check(cache_lens, "cache_lens", torch.int32, 1, dev)
    B, T, Hq, d = q.shape
    if v_cache.shape != k_cache.shape or k_cache.shape[3] != d:
        raise ValueError("k_cache/v_cache must have the same shape, head dimension last")
    if cache_lens.shape[0] != B:
        raise ValueError("cache_lens must be [B]")
    rows, Hkv = (k_cache.shape[1], k_cache.shape[2]) if nhd else (k_cache.shape[2], k_cache.shape[1])
    lay = HtaKvLayout(KV_NHD if nhd else KV_HND, 0, 0, 0, None)
    if block_table is None:
        if k_cache.shape[0] != B:
            raise ValueError("a contiguous cache has one block of Lmax rows per sequence")
        Lmax = rows
    else:
        _check(block_table, "block_table", torch.int32, 2, dev)
        if block_table.shape[0] != B:
            raise ValueError("block_table must be [B][max_pages]")
        lay.page_size, lay.max_pages, lay.num_pages = rows, block_table.shape[1], k_cache.shape[0]
        lay.block_table = block_table.data_ptr()
        Lmax = rows * block_table.shape[1]
    return HtaDims(B, T, Hq, Hkv, d, Lmax, 0.0), lay, Hkv


def verify_kv(q, k_cache, v_cache, cache_lens, k_spec, v_spec, mask, *, order: str = "hnd",
              block_table: torch.Tensor | None = None, scale: float = 0.0,
              ws: torch.Tensor | None = None, dev_err: torch.Tensor | None = None,
              out: tuple | None = None):
    """verify() over a token-major and/or paged cache (see _kv_layout);
    k_spec/v_spec are [B][Hkv][T][d] ("hnd") or [B][T][Hkv][d] ("nhd").
    Returns (o bf16 [B][T][Hq][d], lse fp32 [B][T][Hq])."""
    dims, lay, Hkv = _kv_layout(q, k_cache, v_cache, cache_lens, order, block_table)
    dims.scale = float(scale)
    B, T, Hq, d = q.shape
    dev = q.device
    _check(k_spec, "k_spec", torch.bfloat16, 4, dev)
    _check(v_spec, "v_spec", torch.bfloat16, 4, dev)
    _check(mask, "mask", torch.int32, 3, dev)
    want = (B, T, Hkv, d) if order == "nhd" else (B, Hkv, T, d)
    if tuple(k_spec.shape) != want or v_spec.shape != k_spec.shape:
        raise ValueError(f"k_spec/v_spec must be {want}")
    if tuple(mask.shape) != (B, T, (T + 31) // 32):
        raise ValueError("mask must be [B][T][ceil(T/32)]")
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    else:
        o, lse = out
    if ws is None:
        ws = workspace(dims, dev)
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, 1, dev)
    with torch.cuda.device(dev):
        _raise(load().hta_verify_kv(ctypes.byref(dims), ctypes.byref(lay), _ptr(q), _ptr(k_cache),
                                    _ptr(v_cache), _ptr(cache_lens), _ptr(k_spec), _ptr(v_spec), _ptr(mask),
                                    _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _ptr(dev_err), _stream(dev)),
               "hta_verify_kv")
    return o, lse


def prefix_attn_kv(q, k_cache, v_cache, cache_lens, *, order: str = "hnd",
                   block_table: torch.Tensor | None = None, scale: float = 0.0,
                   ws: torch.Tensor | None = None, dev_err: torch.Tensor | None = None):
    """prefix_attn() over a token-major and/or paged cache (see _kv_layout).
    Returns (o_c fp32 [B][T][Hq][d], lse_c fp32 [B][T][Hq])."""
    dims, lay, _ = _kv_layout(q, k_cache, v_cache, cache_lens, order, block_table)
    dims.scale = float(scale)
    dev = q.device
    o_c = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse_c = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(dims, dev)
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, 1, dev)
    with torch.cuda.device(dev):
        _raise(load().hta_prefix_attn_kv(ctypes.byref(dims), ctypes.byref(lay), _ptr(q), _ptr(k_cache),
                                         _ptr(v_cache), _ptr(cache_lens), _ptr(o_c), _ptr(lse_c), _ptr(ws),
                                         ws.numel(), _ptr(dev_err), _stream(dev)), "hta_prefix_attn_kv")
    return o_c, lse_c


def tree_attn(q, k_spec, v_spec, mask, *, scale: float = 0.0):
    """Speculative part alone. Returns (o_s fp32 [B][T][Hq][d], lse_s fp32 [B][T][Hq])."""
    _check(q, "q", torch.bfloat16, 4)
    Hkv = k_spec.shape[1]
    _check_spec(q, k_spec, v_spec, mask, Hkv)
    B, T, Hq, d = q.shape
    dims = HtaDims(B, T, Hq, Hkv, d, 0, float(scale))
    dev = q.device
    o_s = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse_s = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _raise(load().hta_tree_attn(ctypes.byref(dims), _ptr(q), _ptr(k_spec), _ptr(v_spec),
                                    _ptr(mask), _ptr(o_s), _ptr(lse_s), _stream(dev)), "hta_tree_attn")
    return o_s, lse_s


def merge(o_c, lse_c, o_s, lse_s):
    """Log-sum-exp merge of two partial softmaxes. Returns (o bf16, lse fp32)."""
    _check(o_c, "o_c", torch.float32, 4)
    dev = o_c.device
    _check(o_s, "o_s", torch.float32, 4, dev)
    _check(lse_c, "lse_c", torch.float32, 3, dev)
    _check(lse_s, "lse_s", torch.float32, 3, dev)
    B, T, Hq, d = o_c.shape
    if o_s.shape != o_c.shape or tuple(lse_c.shape) != (B, T, Hq) or lse_s.shape != lse_c.shape:
        raise ValueError("partials must share [B][T][Hq][d] / [B][T][Hq]")
    dims = HtaDims(B, T, Hq, 1, d, 0, 0.0)
    o = torch.empty(o_c.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(lse_c.shape, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _raise(load().hta_merge(ctypes.byref(dims), _ptr(o_c), _ptr(lse_c), _ptr(o_s), _ptr(lse_s),
                                _ptr(o), _ptr(lse), _stream(dev)), "hta_merge")
    return o, lse


def accept_commit(parents, draft, target, k_spec, v_spec, k_cache, v_cache, cache_lens,
                  dev_err: torch.Tensor | None = None, out=None):
    """Greedy accept walk over each draft tree and append of the accepted
    nodes' K/V rows to the cache (k_cache, v_cache and cache_lens change in
    place). Returns (accepted int32 [B][T] padded with -1, n_accepted int32
    [B], next_token int32 [B])."""
    _check(parents, "parents", torch.int32, 2)
    dev = parents.device
    _check(draft, "draft", torch.int32, 2, dev)
    _check(target, "target", torch.int32, 2, dev)
    _check(k_spec, "k_spec", torch.bfloat16, 4, dev)
    _check(v_spec, "v_spec", torch.bfloat16, 4, dev)
    _check(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _check(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _check(cache_lens, "cache_lens", torch.int32, 1, dev)
    B, T = parents.shape
    _, Hkv, Lmax, d = k_cache.shape
    if draft.shape != parents.shape or target.shape != parents.shape:
        raise ValueError("parents, draft and target must share [B][T]")
    if tuple(k_spec.shape) != (B, Hkv, T, d) or v_spec.shape != k_spec.shape or v_cache.shape != k_cache.shape:
        raise ValueError("k_spec/v_spec must be [B][Hkv][T][d] and k_cache/v_cache [B][Hkv][Lmax][d]")
    if tuple(cache_lens.shape) != (B,):
        raise ValueError("cache_lens must be [B]")
    dims = HtaDims(B, T, Hkv, Hkv, d, Lmax, 0.0)
    if out is None:
        accepted = torch.empty((B, T), dtype=torch.int32, device=dev)
        n_acc = torch.empty((B,), dtype=torch.int32, device=dev)
        nxt = torch.empty((B,), dtype=torch.int32, device=dev)
    else:
        accepted, n_acc, nxt = out
    with torch.cuda.device(dev):
        _raise(load().hta_accept_commit(ctypes.byref(dims), _ptr(parents), _ptr(draft), _ptr(target),
                                        _ptr(k_spec), _ptr(v_spec), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(cache_lens), _ptr(accepted), _ptr(n_acc), _ptr(nxt),
                                        _ptr(dev_err) if dev_err is not None else None, _stream(dev)),
               "hta_accept_commit")
    return accepted, n_acc, nxt


def accept_commit_kv(parents, draft, target, k_spec, v_spec, k_cache, v_cache, cache_lens, *,
                     order: str = "hnd", block_table: torch.Tensor | None = None,
                     dev_err: torch.Tensor | None = None, out=None):
    """accept_commit() into a token-major and/or paged cache (storage as for
    verify_kv; the pages the appended rows fall in must be in block_table).
    Returns (accepted, n_accepted, next_token)."""
    if order not in ("hnd", "nhd"):
        raise ValueError("order must be 'hnd' or 'nhd'")
    nhd = order == "nhd"
    _check(parents, "parents", torch.int32, 2)
    dev = parents.device
    for t, n in ((draft, "draft"), (target, "target")):
        _check(t, n, torch.int32, 2, dev)
    for t, n in ((k_spec, "k_spec"), (v_spec, "v_spec"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4, dev)
    _check(cache_lens, "cache_lens", torch.int32, 1, dev)
    B, T = parents.shape
    if draft.shape != parents.shape or target.shape != parents.shape:
        raise ValueError("parents, draft and target must share [B][T]")
    rows, Hkv = (k_cache.shape[1], k_cache.shape[2]) if nhd else (k_cache.shape[2], k_cache.shape[1])
    d = k_cache.shape[3]
    want = (B, T, Hkv, d) if nhd else (B, Hkv, T, d)
    if tuple(k_spec.shape) != want or v_spec.shape != k_spec.shape or v_cache.shape != k_cache.shape:
        raise ValueError(f"k_spec/v_spec must be {want}, v_cache shaped as k_cache")
    if tuple(cache_lens.shape) != (B,):
        raise ValueError("cache_lens must be [B]")
    lay = HtaKvLayout(KV_NHD if nhd else KV_HND, 0, 0, 0, None)
    if block_table is None:
        if k_cache.shape[0] != B:
            raise ValueError("a contiguous cache has one block of Lmax rows per sequence")
        Lmax = rows
    else:
        _check(block_table, "block_table", torch.int32, 2, dev)
        if block_table.shape[0] != B:
            raise ValueError("block_table must be [B][max_pages]")
        lay.page_size, lay.max_pages, lay.num_pages = rows, block_table.shape[1], k_cache.shape[0]
        lay.block_table = block_table.data_ptr()
        Lmax = rows * block_table.shape[1]
    dims = HtaDims(B, T, Hkv, Hkv, d, Lmax, 0.0)
    if out is None:
        accepted = torch.empty((B, T), dtype=torch.int32, device=dev)
        n_acc = torch.empty((B,), dtype=torch.int32, device=dev)
        nxt = torch.empty((B,), dtype=torch.int32, device=dev)
    else:
        accepted, n_acc, nxt = out
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, 1, dev)
    with torch.cuda.device(dev):
        _raise(load().hta_accept_commit_kv(ctypes.byref(dims), ctypes.byref(lay), _ptr(parents), _ptr(draft),
                                           _ptr(target), _ptr(k_spec), _ptr(v_spec), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(cache_lens), _ptr(accepted), _ptr(n_acc), _ptr(nxt),
                                           _ptr(dev_err), _stream(dev)), "hta_accept_commit_kv")
    return accepted, n_acc, nxt


def window_attn(q, k_ring, v_ring, pos, window: int, *, scale: float = 0.0,
                dev_err: torch.Tensor | None = None, out: tuple | None = None):
    """Draft-model sliding-window self-attention: window W over a ring of S
    slots (k_ring/v_ring [B][Hkv][S][d], position j in slot j mod S,
    W + T - 1 <= S); the T queries are positions pos[b] .. pos[b] + T - 1.
    Returns (o bf16 [B][T][Hq][d], lse fp32 [B][T][Hq])."""
    _check(q, "q", torch.bfloat16, 4)
    dev = q.device
    _check(k_ring, "k_ring", torch.bfloat16, 4, dev)
    _check(v_ring, "v_ring", torch.bfloat16, 4, dev)
    _check(pos, "pos", torch.int32, 1, dev)
    B, T, Hq, d = q.shape
    _, Hkv, S, d2 = k_ring.shape
    if k_ring.shape[0] != B or d2 != d or v_ring.shape != k_ring.shape or tuple(pos.shape) != (B,):
        raise ValueError("k_ring/v_ring must be [B][Hkv][W][d] and pos [B]")
    dims = HtaDims(B, T, Hq, Hkv, d, S, float(scale))
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=dev)
    else:
        o, lse = out
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, 1, dev)
    with torch.cuda.device(dev):
        _raise(load().hta_window_attn(ctypes.byref(dims), int(window), _ptr(q), _ptr(k_ring), _ptr(v_ring), _ptr(pos),
                                      _ptr(o), _ptr(lse), _ptr(dev_err), _stream(dev)),
               "hta_window_attn")
    return o, lse


def logitspec_tree(logits, hist, hist_len, k: int, m: int, keep, T: int, *,
                   dev_err: torch.Tensor | None = None, out: tuple | None = None):
    """LogitSpec draft trees, one per sequence: logits fp32 [B][V], hist int32
    [B][Lh_max] (the token stream), hist_len int32 [B]; keep: k + 1 ints (the
    per-rank budget). Returns (parents int32 [B][T], tokens int32 [B][T],
    n_nodes int32 [B], next_token int32 [B])."""
    _check(logits, "logits", torch.float32, 2)
    dev = logits.device
    _check(hist, "hist", torch.int32, 2, dev)
    _check(hist_len, "hist_len", torch.int32, 1, dev)
    B, V = logits.shape
    if hist.shape[0] != B or tuple(hist_len.shape) != (B,):
        raise ValueError("hist must be [B][Lh_max] and hist_len [B]")
    if len(keep) != k + 1:
        raise ValueError("keep needs k + 1 entries")
    keep_arr = (ctypes.c_int32 * (k + 1))(*[int(x) for x in keep])
    if out is None:
        parents = torch.empty((B, T), dtype=torch.int32, device=dev)
        tokens = torch.empty((B, T), dtype=torch.int32, device=dev)
        n_nodes = torch.empty((B,), dtype=torch.int32, device=dev)
        nxt = torch.empty((B,), dtype=torch.int32, device=dev)
    else:
        parents, tokens, n_nodes, nxt = out
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, 1, dev)
    with torch.cuda.device(dev):
        _raise(load().hta_logitspec_tree(B, V, hist.shape[1], T, k, m, _ptr(logits), _ptr(hist), _ptr(hist_len),
                                         keep_arr, _ptr(parents), _ptr(tokens), _ptr(n_nodes), _ptr(nxt),
                                         _ptr(dev_err), _stream(dev)),
               "hta_logitspec_tree")
    return parents, tokens, n_nodes, nxt

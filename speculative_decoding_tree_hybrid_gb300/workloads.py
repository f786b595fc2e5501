"""Seeded synthetic workloads for Hybrid Tree Attention.

This module only draws inputs: draft trees (parent arrays), post-RoPE Q/K/V
values rounded to bf16, and cache lengths. It holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle may consume what it makes.

Shapes follow the layer shapes of the target models the LongSpec summaries
evaluate (LLaMA-3.1-8B, Vicuna/LongChat-7B, QwQ-32B); the pages' datasets
(LongBench-type, AIME/MATH-type) are not available here and N(0,1) values
stand in for the activations. Every tensor comes from a PCG64 stream keyed by
(config id, batch size, sequence, stream, head), so every platform draws the
same bytes.

Layouts (bf16 kept as uint16 bit patterns, row-major):
  q        [B][T][Hq][d]
  k_cache  [B][Hkv][Lmax][d]   (tokens j >= cache_lens[b] hold NaN)
  v_cache  [B][Hkv][Lmax][d]
  k_spec   [B][Hkv][T][d]
  v_spec   [B][Hkv][T][d]
  parents  [B][T] int32, parents[b][0] = -1, -1 <= parents[b][i] < i
  cache_lens [B] int32
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BF16_NAN = np.uint16(0x7FC0)

# stream ids of the seed sequence
S_TREE, S_Q, S_KC, S_VC, S_KS, S_VS, S_LEN = 0, 1, 2, 3, 4, 5, 6


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    cfg_id: int
    B: int
    Hq: int
    Hkv: int
    d: int
    T: int
    L: int | None          # fixed cache length, or None for ragged
    tree: str              # "uniform" | "window8_depth8"
    L_range: tuple[int, int] | None = None  # inclusive range for ragged lengths

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


CONFIGS: dict[str, Config] = {
    # parent[i] ~ U{0..i-1} drawn with default_rng(0)
    "tiny": Config("tiny", 0, B=1, Hq=4, Hkv=1, d=64, T=8, L=256, tree="uniform"),
    # LLaMA-3.1-8B layer shape, 32K context, 64-node tree of depth <= 8
    "llama8b": Config("llama8b", 1, B=1, Hq=32, Hkv=8, d=128, T=64, L=32768,
                      tree="window8_depth8"),
    # Vicuna/LongChat-7B MHA layer shape, 4 sequences of 16K, 32-node trees
    "vicuna7b": Config("vicuna7b", 2, B=4, Hq=32, Hkv=32, d=128, T=32, L=16384,
                       tree="uniform"),
    # QwQ-32B layer shape, 128K reasoning context, 64-node tree of depth <= 8
    "qwq32b": Config("qwq32b", 3, B=1, Hq=40, Hkv=8, d=128, T=64, L=131072,
                     tree="window8_depth8"),
}
for _B in (1, 4, 16, 32):
    CONFIGS[f"ragged_b{_B}"] = Config(f"ragged_b{_B}", 4, B=_B, Hq=32, Hkv=8, d=128, T=64,
                                      L=None, tree="window8_depth8", L_range=(4096, 65536))


def _rng(cfg_id: int, B: int, b: int, stream: int, h: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([cfg_id, B, b, stream, h]))


# --------------------------------------------------------------------------- trees

def tree_uniform(T: int, rng: np.random.Generator) -> np.ndarray:
    """parent[0] = -1, parent[i] ~ U{0..i-1}."""
    par = np.empty(T, dtype=np.int32)
    par[0] = -1
    for i in range(1, T):
        par[i] = rng.integers(0, i)
    return par


def tree_window8_depth8(T: int, rng: np.random.Generator, window: int = 8,
                        max_depth: int = 8) -> np.ndarray:
    """parent[i] ~ U{max(0,i-8)..i-1} restricted to nodes whose depth is < 8.

    The root has depth 0. If no node of the window qualifies, the parent is
    drawn uniformly among all earlier nodes of depth < 8 (the root always
    qualifies), so every tree has depth <= 8.
    """
    par = np.empty(T, dtype=np.int32)
    depth = np.zeros(T, dtype=np.int32)
    par[0] = -1
    for i in range(1, T):
        cand = [j for j in range(max(0, i - window), i) if depth[j] <= max_depth - 1]
        if not cand:
            cand = [j for j in range(i) if depth[j] <= max_depth - 1]
        p = cand[int(rng.integers(0, len(cand)))]
        par[i] = p
        depth[i] = depth[p] + 1
    return par


def tree_chain(T: int) -> np.ndarray:
    return np.arange(-1, T - 1, dtype=np.int32)


def tree_star(T: int) -> np.ndarray:
    par = np.zeros(T, dtype=np.int32)
    par[0] = -1
    return par


def make_trees(cfg: Config) -> np.ndarray:
    if cfg.name == "tiny":
        return tree_uniform(cfg.T, np.random.default_rng(0))[None]
    out = np.empty((cfg.B, cfg.T), dtype=np.int32)
    for b in range(cfg.B):
        rng = _rng(cfg.cfg_id, cfg.B, b, S_TREE)
        if cfg.tree == "uniform":
            out[b] = tree_uniform(cfg.T, rng)
        elif cfg.tree == "window8_depth8":
            out[b] = tree_window8_depth8(cfg.T, rng)
        else:
            raise ValueError(cfg.tree)
    return out


# --------------------------------------------------------------------------- values

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
            >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def cache_lengths(cfg: Config) -> np.ndarray:
    if cfg.L is not None:
        return np.full(cfg.B, cfg.L, dtype=np.int32)
    lo, hi = cfg.L_range
    rng = _rng(cfg.cfg_id, cfg.B, 0, S_LEN)
    return rng.integers(lo, hi, size=cfg.B, endpoint=True).astype(np.int32)


@dataclasses.dataclass
class Inputs:
    cfg: Config
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    cache_lens: np.ndarray
    k_spec: np.ndarray
    v_spec: np.ndarray
    parents: np.ndarray

    @property
    def Lmax(self) -> int:
        return int(self.k_cache.shape[2])


def _fill_cache(out: np.ndarray, cfg: Config, lens: np.ndarray, stream: int, salt: int,
                threads: int) -> None:
    B, Hkv, Lmax, d = out.shape

    def job(bh):
        b, h = divmod(bh, Hkv)
        L = int(lens[b])
        rng = _rng(cfg.cfg_id, cfg.B, b, stream + 16 * salt, h)
        out[b, h, :L] = normal_bf16(rng, (L, d))
        out[b, h, L:] = BF16_NAN

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(job, range(B * Hkv)))


def make_inputs(cfg: Config | str, *, kv_set: int = 0, lmax: int | None = None,
                threads: int = 8) -> Inputs:
    """Draw one full set of inputs for a configuration.

    kv_set > 0 draws an independent K/V cache (same q, tree and lengths), used
    to rotate several caches through the timed loop so they are read from HBM.
    lmax pads the cache allocation beyond the longest sequence.
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    lens = cache_lengths(cfg)
    Lmax = int(lmax) if lmax is not None else int(lens.max())
    if Lmax < int(lens.max()):
        raise ValueError("lmax shorter than a sequence")
    parents = make_trees(cfg)
    q = np.empty((cfg.B, cfg.T, cfg.Hq, cfg.d), dtype=np.uint16)
    ks = np.empty((cfg.B, cfg.Hkv, cfg.T, cfg.d), dtype=np.uint16)
    vs = np.empty_like(ks)
    for b in range(cfg.B):
        q[b] = normal_bf16(_rng(cfg.cfg_id, cfg.B, b, S_Q), q.shape[1:])
        ks[b] = normal_bf16(_rng(cfg.cfg_id, cfg.B, b, S_KS), ks.shape[1:])
        vs[b] = normal_bf16(_rng(cfg.cfg_id, cfg.B, b, S_VS), vs.shape[1:])
    kc = np.empty((cfg.B, cfg.Hkv, Lmax, cfg.d), dtype=np.uint16)
    vc = np.empty_like(kc)
    _fill_cache(kc, cfg, lens, S_KC, kv_set, threads)
    _fill_cache(vc, cfg, lens, S_VC, kv_set, threads)
    return Inputs(cfg, q, kc, vc, lens, ks, vs, parents)


def random_inputs(B: int, T: int, Hq: int, Hkv: int, d: int, lens, *, seed: int,
                  parents: np.ndarray | None = None, Lmax: int | None = None,
                  tree: str = "uniform") -> Inputs:
    """Small ad-hoc inputs for edge-case tests (same value recipe as the configs)."""
    lens = np.asarray(lens, dtype=np.int32).reshape(B)
    Lmax = int(Lmax if Lmax is not None else max(1, int(lens.max())))
    cfg = Config(f"adhoc{seed}", 1000 + seed, B=B, Hq=Hq, Hkv=Hkv, d=d, T=T, L=None,
                 tree=tree)
    rng = np.random.default_rng(np.random.SeedSequence([1000, seed]))
    if parents is None:
        parents = np.stack([
            tree_uniform(T, rng) if tree == "uniform" else tree_window8_depth8(T, rng)
            for _ in range(B)])
    parents = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, T)
    q = normal_bf16(rng, (B, T, Hq, d))
    kc = normal_bf16(rng, (B, Hkv, Lmax, d))
    vc = normal_bf16(rng, (B, Hkv, Lmax, d))
    for b in range(B):
        kc[b, :, lens[b]:] = BF16_NAN
        vc[b, :, lens[b]:] = BF16_NAN
    ks = normal_bf16(rng, (B, Hkv, T, d))
    vs = normal_bf16(rng, (B, Hkv, T, d))
    return Inputs(cfg, q, kc, vc, lens, ks, vs, parents)


# --------------------------------------------------------------------------- cache storage

def kv_nhd(x: np.ndarray) -> np.ndarray:
    """Head-major [outer][Hkv][rows][d] -> token-major [outer][rows][Hkv][d]."""
    return np.ascontiguousarray(np.swapaxes(x, 1, 2))


def paged_kv(k_cache: np.ndarray, v_cache: np.ndarray, lens, page_size: int, *, order: str = "hnd",
             seed: int = 0, spare: int = 3, reserve: bool = False):
    """Scatters contiguous caches [B][Hkv][Lmax][d] into a pool of pages.

    Page i of sequence b (tokens i*P .. i*P + P - 1) goes to pool page
    block_table[b][i]; the used pages of all sequences are spread over
    n_used + spare pool pages by a seeded permutation. Rows past L_b in a
    sequence's last page, and the pool pages no sequence uses, hold NaN;
    table entries past a sequence's pages are -1; max_pages = ceil(Lmax / P).
    order "nhd" stores each page token-major. reserve: every sequence gets
    pages for all Lmax tokens (room to append rows). Returns (k_pool, v_pool,
    block_table int32 [B][max_pages])."""
    B, Hkv, Lmax, d = k_cache.shape
    P = int(page_size)
    lens = np.asarray(lens, dtype=np.int64).reshape(B)
    max_pages = max(1, -(-Lmax // P))
    used = [max_pages if reserve else -(-int(L) // P) for L in lens]
    n_pool = sum(used) + spare
    perm = np.random.default_rng(np.random.SeedSequence([5000, seed])).permutation(n_pool)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    kp = np.full((n_pool, Hkv, P, d), BF16_NAN, dtype=np.uint16)
    vp = np.full_like(kp, BF16_NAN)
    n = 0
    for b in range(B):
        for i in range(used[b]):
            pg = int(perm[n])
            n += 1
            table[b, i] = pg
            lo, hi = i * P, min((i + 1) * P, int(lens[b]))
            if hi > lo:  # a reserved page past L_b stays NaN
                kp[pg, :, :hi - lo] = k_cache[b, :, lo:hi]
                vp[pg, :, :hi - lo] = v_cache[b, :, lo:hi]
    if order == "nhd":
        kp, vp = kv_nhd(kp), kv_nhd(vp)
    return kp, vp, table


def unpage_kv(pool: np.ndarray, table: np.ndarray, lens, Lmax: int, *, order: str = "hnd") -> np.ndarray:
    """Inverse of paged_kv for one pool: contiguous [B][Hkv][Lmax][d], NaN past L_b."""
    if order == "nhd":
        pool = np.swapaxes(pool, 1, 2)
    _, Hkv, P, d = pool.shape
    B = table.shape[0]
    out = np.full((B, Hkv, Lmax, d), BF16_NAN, dtype=np.uint16)
    for b in range(B):
        L = int(lens[b])
        for i in range(-(-L // P)):
            lo, hi = i * P, min((i + 1) * P, L)
            out[b, :, lo:hi] = pool[int(table[b, i]), :, :hi - lo]
    return out


# --------------------------------------------------------------------------- draft model

@dataclasses.dataclass
class WindowInputs:
    q: np.ndarray       # [B][T][Hq][d] bf16 bits
    k_ring: np.ndarray  # [B][Hkv][S][d] bf16 bits, position j in slot j mod S
    v_ring: np.ndarray
    pos: np.ndarray     # [B] int32: position of query 0

    @property
    def S(self) -> int:
        return int(self.k_ring.shape[2])


def window_inputs(B: int, T: int, Hq: int, Hkv: int, d: int, S: int, pos, *, seed: int) -> WindowInputs:
    """Queries at positions pos[b] .. pos[b] + T - 1 and a ring of S slots
    holding positions max(0, pos[b] + T - S) .. pos[b] + T - 1 (N(0,1) values
    rounded to bf16, like every other input); slots that hold no position yet
    are NaN, so a read of one shows up."""
    pos = np.asarray(pos, dtype=np.int32).reshape(B)
    rng = np.random.default_rng(np.random.SeedSequence([2000, seed]))
    q = normal_bf16(rng, (B, T, Hq, d))
    kr = np.full((B, Hkv, S, d), BF16_NAN, dtype=np.uint16)
    vr = np.full((B, Hkv, S, d), BF16_NAN, dtype=np.uint16)
    for b in range(B):
        end = int(pos[b]) + T
        js = np.arange(max(0, end - S), end)
        kr[b][:, js % S] = normal_bf16(rng, (Hkv, len(js), d))
        vr[b][:, js % S] = normal_bf16(rng, (Hkv, len(js), d))
    return WindowInputs(q, kr, vr, pos)


# --------------------------------------------------------------------------- draft trees

def token_stream(n: int, vocab: int, rng: np.random.Generator, copy_p: float = 0.6) -> np.ndarray:
    """A token stream with the repetition that retrieval-based drafting relies
    on: with probability copy_p the next span (2 to 16 tokens) copies an
    earlier span of the stream, else one token is drawn uniformly."""
    out = np.empty(n, dtype=np.int32)
    fill = 0
    while fill < n:
        if fill > 8 and rng.random() < copy_p:
            a = int(rng.integers(0, fill - 1))
            ln = min(int(rng.integers(2, 17)), n - fill, fill - a)
            out[fill:fill + ln] = out[a:a + ln]
            fill += ln
        else:
            out[fill] = rng.integers(0, vocab)
            fill += 1
    return out


def lspec_inputs(B: int, V: int, Lh: int, lens, *, seed: int, vocab_used: int | None = None,
                 plant_m: int = 0, plant_guesses: int = 8):
    """Logits N(0, 1) [B][V] (float32) and token streams [B][Lh] (int32, zero
    past each length) with vocabulary vocab_used (default V).

    plant_m > 0 stands in for a target model that favours tokens seen in the
    context: the largest logit goes to a token that followed the stream's last
    plant_m - 1 tokens earlier in the stream, and the next plant_guesses
    logits to tokens that followed that token; the rest stay N(0, 1)."""
    rng = np.random.default_rng(np.random.SeedSequence([3000, seed]))
    lens = np.asarray(lens, dtype=np.int32).reshape(B)
    logits = rng.standard_normal((B, V), dtype=np.float32)
    hist = np.zeros((B, Lh), dtype=np.int32)
    for b in range(B):
        n = int(lens[b])
        h = token_stream(n, vocab_used or V, rng)
        hist[b, :n] = h
        if plant_m <= 1 or n < plant_m:
            continue
        tail = h[n - (plant_m - 1):]
        win = np.lib.stride_tricks.sliding_window_view(h[:n - 1], plant_m - 1)
        hits = np.nonzero((win == tail).all(axis=1))[0]
        hits = hits[hits + plant_m - 1 < n - 1]  # a token follows the earlier occurrence
        if hits.size == 0:
            continue
        x1 = int(h[hits[-1] + plant_m - 1])
        logits[b, x1] = 10.0
        after = h[1:n][h[:n - 1] == x1]  # tokens that followed x1
        seen = []
        for t in after[::-1]:
            if int(t) != x1 and int(t) not in seen:
                seen.append(int(t))
            if len(seen) == plant_guesses:
                break
        for r, t in enumerate(seen):
            logits[b, t] = 9.0 - 0.1 * r
    return logits, hist, lens

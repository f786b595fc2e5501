"""GPU parity of the draft model's two attention kinds ("LongSpec: Long-Context
Lossless Speculative Decoding with Efficient Drafting and Verification",
Korean summary 2.A, Dutch summary section 1):

* sliding-window self-attention (hta_window_attn) against oracle/window.py;
* cross-attention over the target's KV cache, which is prefix-only attention
  of the draft queries (hta_prefix_attn), against the monolithic oracle with
  an all-zero tree mask (no tree key visible).

Both are called through the C ABI; expected values come only from oracle/.
"""
import numpy as np
import pytest

from speculative_decoding_tree_hybrid_gb300 import workloads as wl

from _util import assert_close, to_device, to_torch_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle.window import window_attention  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import build as hbuild  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import hta  # noqa: E402

hbuild.build()
DEV = torch.device("cuda:0")


def run_window(inp, W, scale=0.0):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = hta.window_attn(to_torch_bf16(inp.q, DEV), to_torch_bf16(inp.k_ring, DEV),
                             to_torch_bf16(inp.v_ring, DEV), torch.from_numpy(inp.pos).to(DEV), W,
                             scale=scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return o, lse


# (B, T, Hq, Hkv, d, W, pos): the pages' window of 512 with positions before,
# at and far past one ring length; small windows with several tiles per query
# group; GQA, MHA and d = 64; T up to the tree size
CASES = [
    (2, 1, 32, 8, 128, 512, [0, 511]),
    (3, 1, 32, 8, 128, 512, [512, 1000, 70000]),
    (2, 5, 32, 8, 128, 512, [3, 4097]),
    (2, 16, 32, 8, 128, 512, [100, 2047]),
    (1, 64, 32, 8, 128, 512, [9000]),
    (2, 8, 8, 8, 128, 64, [0, 300]),
    (2, 7, 4, 1, 64, 100, [50, 1234]),
    (1, 3, 4, 2, 128, 1, [77]),
    (1, 33, 16, 4, 64, 200, [10]),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,d,W,pos", CASES)
def test_window_attention_matches_oracle(B, T, Hq, Hkv, d, W, pos):
    S = W + T - 1 + (T % 3)  # rings exactly long enough and a little longer
    inp = wl.window_inputs(B, T, Hq, Hkv, d, S, pos, seed=B * 1000 + T * 10 + W)
    o, lse = run_window(inp, W)
    ro, rl = window_attention(inp.q, inp.k_ring, inp.v_ring, inp.pos, W)
    assert_close(o, lse, ro, rl, f"window B={B} T={T} W={W} pos={pos}")


def test_window_attention_scale_and_determinism():
    inp = wl.window_inputs(2, 4, 32, 8, 128, 515, [600, 9], seed=5)
    o1, l1 = run_window(inp, 512, scale=0.05)
    o2, l2 = run_window(inp, 512, scale=0.05)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl = window_attention(inp.q, inp.k_ring, inp.v_ring, inp.pos, 512, scale=0.05)
    assert_close(o1, l1, ro, rl, "window scale 0.05")


def test_window_attention_rejects_short_ring():
    inp = wl.window_inputs(1, 4, 8, 8, 128, 10, [20], seed=1)
    with pytest.raises(hta.HtaError):
        run_window(inp, 8)  # needs 8 + 3 = 11 slots


def test_window_attention_flags_negative_position():
    inp = wl.window_inputs(1, 1, 8, 8, 128, 16, [0], seed=2)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    hta.window_attn(to_torch_bf16(inp.q, DEV), to_torch_bf16(inp.k_ring, DEV), to_torch_bf16(inp.v_ring, DEV),
                    torch.tensor([-3], dtype=torch.int32, device=DEV), 16, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & hta.DEVERR_CACHE_LEN


def _cross(oracle_mod, inp, rows=None):
    """Prefix-only attention: the oracle with an all-zero tree mask."""
    W = (inp.q.shape[1] + 31) // 32
    zero = np.zeros((inp.q.shape[0], inp.q.shape[1], W), np.uint32)
    return oracle_mod.attention(inp.q, inp.k_cache, inp.v_cache, inp.cache_lens, inp.k_spec, inp.v_spec, zero,
                                rows=rows)


@pytest.mark.parametrize("B,T,lens", [(1, 1, [32768]), (4, 1, [0, 1, 4097, 20000]), (2, 4, [777, 16384]),
                                      (32, 1, None)])
def test_cross_attention_is_prefix_attention(oracle_mod, B, T, lens):
    if lens is None:  # a ragged batch of 32 short contexts (full-length ones are measured by bench.py)
        lens = np.random.default_rng(32).integers(0, 3001, size=32)
    lens = np.asarray(lens, np.int32)
    inp = wl.random_inputs(B, T, 32, 8, 128, lens, seed=40 + B * 3 + T, Lmax=int(max(1, lens.max())))
    t = to_device(inp, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o_c, lse_c = hta.prefix_attn(t["q"], t["k_cache"], t["v_cache"], t["cache_lens"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    n = B * T * 32
    rng = np.random.default_rng(B * 7 + T)
    rows = np.unique(np.concatenate([rng.integers(0, n, size=min(n, 256)), [0, n - 1]])).astype(np.int64)
    ro, rl = _cross(oracle_mod, inp, rows)
    og = o_c.reshape(n, 128)[torch.from_numpy(rows).to(DEV)]
    lg = lse_c.reshape(n)[torch.from_numpy(rows).to(DEV)]
    assert_close(og, lg, ro, rl, f"cross B={B} T={T}")

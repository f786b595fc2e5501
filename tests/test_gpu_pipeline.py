"""One speculative decoding step end to end on the GPU, each stage fed by the
previous stage's device outputs and each checked against its oracle:

  LogitSpec draft tree ("LogitSpec: Accelerating Retrieval-based Speculative
  Decoding via Next Next Token Speculation", section 2)
    -> tree mask -> hybrid tree attention of one LLaMA-shaped layer ("LongSpec:
  Long-Context Lossless Speculative Decoding with Efficient Drafting and
  Verification", Korean summary 2.C) -> greedy accept walk + KV commit.
"""
import numpy as np
import pytest

from speculative_decoding_tree_hybrid_gb300 import workloads as wl

from _util import assert_close, to_torch_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle.accept import accept_commit as accept_ref  # noqa: E402
from oracle.logitspec import build_trees  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import build as hbuild  # noqa: E402
from speculative_decoding_tree_hybrid_gb300 import hta  # noqa: E402

hbuild.build()
DEV = torch.device("cuda:0")


def test_one_decoding_step(oracle_mod):
    B, V, Lh, T, k, m = 4, 5000, 3000, 64, 40, 3
    Hq, Hkv, d = 32, 8, 128
    keep = [12] + [max(1, 6 - r // 8) for r in range(1, k + 1)]
    logits, hist, lens = wl.lspec_inputs(B, V, Lh, [3000, 2500, 1800, 700], seed=21, vocab_used=300, plant_m=m)

    # 1. draft trees
    par, tok, nn, nxt = hta.logitspec_tree(torch.from_numpy(logits).to(DEV), torch.from_numpy(hist).to(DEV),
                                           torch.from_numpy(lens).to(DEV), k, m, keep, T)
    r_par, r_tok, r_nn, r_nxt = build_trees(logits, hist, lens, k, m, keep, T)
    assert np.array_equal(par.cpu().numpy(), r_par) and np.array_equal(tok.cpu().numpy(), r_tok)

    # 2. the mask of those trees
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mask = hta.build_mask(par, dev_err=err)
    r_mask, _ = oracle_mod.build_mask(r_par)
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), r_mask)

    # 3. one layer's verification: the cached part is the history, the tree part the T nodes
    rng = np.random.default_rng(5)
    q = wl.normal_bf16(rng, (B, T, Hq, d))
    kc = wl.normal_bf16(rng, (B, Hkv, Lh + T, d))
    vc = wl.normal_bf16(rng, (B, Hkv, Lh + T, d))
    ks = wl.normal_bf16(rng, (B, Hkv, T, d))
    vs = wl.normal_bf16(rng, (B, Hkv, T, d))
    for b in range(B):  # rows past each sequence's length are never read
        kc[b, :, lens[b]:] = wl.BF16_NAN
        vc[b, :, lens[b]:] = wl.BF16_NAN
    kc_d, vc_d = to_torch_bf16(kc, DEV), to_torch_bf16(vc, DEV)
    cl_d = torch.from_numpy(lens.astype(np.int32)).to(DEV)
    o, lse = hta.verify(to_torch_bf16(q, DEV), kc_d, vc_d, cl_d, to_torch_bf16(ks, DEV), to_torch_bf16(vs, DEV),
                        mask, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = np.unique(np.concatenate([rng.integers(0, B * T * Hq, size=256), [0, B * T * Hq - 1]])).astype(np.int64)
    ro, rl = oracle_mod.attention(q, kc, vc, lens, ks, vs, r_mask, rows=rows)
    sel = torch.from_numpy(rows).to(DEV)
    assert_close(o.reshape(-1, d)[sel], lse.reshape(-1)[sel], ro, rl, "pipeline verify")

    # 4. accept + commit: a target that follows the first child for a while, then diverges
    target = np.full((B, T), -7, np.int32)
    tok_np = r_tok
    for b in range(B):
        for p in range(int(r_nn[b])):
            kids = np.nonzero(r_par[b][:r_nn[b]] == p)[0]
            kids = kids[kids > 0]
            if len(kids) and rng.random() < 0.85:
                target[b, p] = tok_np[b, kids[0]]
    acc, n_acc, nxt_tok = hta.accept_commit(par, tok, torch.from_numpy(target).to(DEV), to_torch_bf16(ks, DEV),
                                            to_torch_bf16(vs, DEV), kc_d, vc_d, cl_d, dev_err=err)
    torch.cuda.synchronize()
    r_acc, r_n, r_next, r_kc, r_vc, r_lens, _ = accept_ref(r_par, r_tok, target, ks, vs, kc, vc, lens)
    assert np.array_equal(acc.cpu().numpy(), r_acc) and np.array_equal(n_acc.cpu().numpy(), r_n)
    assert np.array_equal(nxt_tok.cpu().numpy(), r_next) and np.array_equal(cl_d.cpu().numpy(), r_lens)
    got_kc = kc_d.cpu().view(torch.int16).numpy().view(np.uint16)
    for b in range(B):  # the appended rows (the rest of the cache is untouched)
        a, z = int(lens[b]), int(r_lens[b])
        assert np.array_equal(got_kc[b, :, a:z], r_kc[b, :, a:z])
        assert np.array_equal(got_kc[b, :, :a], kc[b, :, :a])
    assert (n_acc.cpu().numpy() >= 1).all()

"""Helpers shared by the tests: moving seeded inputs to the GPU and the
parity tolerances.

Tolerances: bf16 output max-abs error <= 2e-2 and LSE relative error <= 1e-3
(|dLSE| <= 1e-3 * max(1, |LSE|)), the mask bit-exact. These are the stated
acceptance bounds of the hot path; the fp32 partial outputs (cached part,
speculative part) use the same bounds.
"""
import numpy as np

O_ABS_TOL = 2e-2
LSE_REL_TOL = 1e-3


def to_torch_bf16(bits, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def to_device(inp, device="cuda"):
    import torch
    return dict(
        q=to_torch_bf16(inp.q, device),
        k_cache=to_torch_bf16(inp.k_cache, device),
        v_cache=to_torch_bf16(inp.v_cache, device),
        cache_lens=torch.from_numpy(np.ascontiguousarray(inp.cache_lens, np.int32)).to(device),
        k_spec=to_torch_bf16(inp.k_spec, device),
        v_spec=to_torch_bf16(inp.v_spec, device),
        parents=torch.from_numpy(np.ascontiguousarray(inp.parents, np.int32)).to(device),
    )


def mask_to_torch(mask_u32, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(mask_u32, np.uint32).view(np.int32)).to(device)


def errors(o_gpu, lse_gpu, o_ref, lse_ref):
    """(max-abs O error, max relative LSE error) between GPU tensors and fp64 refs."""
    o = o_gpu.float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    lse = lse_gpu.float().cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), "finite pattern of LSE differs"
    assert np.all(np.isneginf(lse[~fin]) == np.isneginf(lse_ref[~fin]))
    e_o = float(np.abs(o - o_ref).max()) if o.size else 0.0
    d = np.abs(lse[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
    e_l = float(d.max()) if d.size else 0.0
    if not np.all(np.isfinite(o)):
        e_o = float("inf")
    return e_o, e_l


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    e_o, e_l = errors(o_gpu, lse_gpu, o_ref, lse_ref)
    assert e_o <= O_ABS_TOL, f"{what}: O max-abs error {e_o:.3e} > {O_ABS_TOL}"
    assert e_l <= LSE_REL_TOL, f"{what}: LSE relative error {e_l:.3e} > {LSE_REL_TOL}"
    return e_o, e_l

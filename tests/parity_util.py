"""Shared helpers of the GPU parity tests: the tolerance check and the oracle
calls on the same seeded inputs the CUDA path consumes.

Tolerances (stated by the target of the path, applied to every comparison):
  latent output o_lat and projected output out: max |gpu - ref| <= 2e-2 and
  mean relative error sum|gpu - ref| / sum|ref| <= 5e-3;
  lse: |gpu - ref| <= 1e-3 where finite, identical -inf pattern.
Integer work (schedule, gather) is compared bit-exactly.
"""
import numpy as np
import torch

import oracle

O_MAX_ABS = 2e-2
O_MEAN_REL = 5e-3
LSE_ABS = 1e-3


def f32(t):
    return t.detach().float().cpu().numpy()


def o_errors(gpu, ref):
    g = f32(gpu).astype(np.float64) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    d = np.abs(g - ref)
    return float(d.max()) if d.size else 0.0, float(d.sum() / max(np.abs(ref).sum(), 1e-300))


def assert_o_close(gpu, ref, what="o"):
    g = f32(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    mx, mr = o_errors(gpu, ref)
    assert mx <= O_MAX_ABS and mr <= O_MEAN_REL, f"{what}: max abs {mx:.3e}, mean rel {mr:.3e}"
    return mx, mr


def assert_lse_close(gpu, ref, what="lse"):
    g = f32(gpu).astype(np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(g)), f"{what}: finite pattern differs"
    assert np.all(g[~fin] == -np.inf)
    err = float(np.abs(g[fin] - ref[fin]).max()) if fin.any() else 0.0
    assert err <= LSE_ABS, f"{what}: max abs {err:.3e}"
    return err


def oracle_decode(inp, q_abs_bf16):
    """Absorbed-form oracle on the bf16 absorbed query the GPU consumed."""
    return oracle.attend_absorbed(f32(q_abs_bf16), f32(inp.kv_cache), inp.block_table.cpu(), inp.seqlens.cpu(),
                                  inp.scale, inp.causal)


def oracle_end_to_end(inp):
    """Full fp64 chain from bf16 q, W_UK, W_UV: absorb -> attend -> out-proj."""
    qa = oracle.absorb_q(f32(inp.q), f32(inp.w_uk))
    o, lse = oracle.attend_absorbed(qa, f32(inp.kv_cache), inp.block_table.cpu(), inp.seqlens.cpu(), inp.scale,
                                    inp.causal)
    return qa, o, lse, oracle.out_proj(o, f32(inp.w_uv))

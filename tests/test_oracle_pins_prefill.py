"""Pins for the oracle's prefill in the naive (decompress) form
("DeepSeek-V3 MLA deep engineering", sec. 2.2 and 4.3: per-head K = W_UK c plus
the shared rope key, V = W_UV c, then ordinary causal attention; the SC11
article's opening contrasts this prefill stage with decode).

Pins that a transposed weight, a dropped rope term, a wrong causal offset or a
wrong normalisation fails:
  * the fp64 numpy brute force (explicit mask matrix) on whole-prompt and
    chunked-prompt shapes, causal and not;
  * the absorption identity: the absorbed chain (absorb, attend over the
    latent, out-project) gives the same output and lse;
  * causal row s of an s_q-token prefill equals a one-token decode over the
    first seqlen - s_q + s + 1 keys.
"""
import numpy as np
import pytest

import oracle
from mla_paged_kv_absorbed_gb300 import inputs as gen
from test_oracle_pins import absorbed_chain, brute_naive, f32, relmax


def prefill_inputs(B, s_q, H, seqlens, seed, causal=True):
    return gen.make_inputs(B, s_q, H, seqlens, seed, q_mode="q", causal=causal)


@pytest.mark.parametrize("B,s_q,H,seqlens,causal", [
    (2, 40, 2, [40, 40], True),        # whole prompts
    (2, 33, 3, [100, 33], True),       # a chunk after 67 earlier tokens, and a whole prompt
    (1, 70, 2, [130], False),
    (3, 5, 1, [1, 64, 65], True),      # rows with no visible key
])
def test_prefill_matches_bruteforce(B, s_q, H, seqlens, causal):
    inp = prefill_inputs(B, s_q, H, seqlens, seed=900 + B + s_q, causal=causal)
    out, lse = oracle.prefill_naive(f32(inp.q), f32(inp.kv_cache), inp.block_table, inp.seqlens, f32(inp.w_uk),
                                    f32(inp.w_uv), inp.scale, causal)
    ref, ref_lse = brute_naive(f32(inp.q), f32(inp.kv_cache), inp.block_table.numpy(), inp.seqlens.numpy(),
                               f32(inp.w_uk), f32(inp.w_uv), inp.scale, causal)
    assert relmax(out, ref) <= 1e-9
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-9


def test_prefill_equals_absorbed_chain():
    inp = prefill_inputs(2, 48, 4, [48, 200], seed=31)
    out, lse = oracle.prefill_naive(f32(inp.q), f32(inp.kv_cache), inp.block_table, inp.seqlens, f32(inp.w_uk),
                                    f32(inp.w_uv), inp.scale, True)
    out_a, lse_a, _ = absorbed_chain(inp)
    assert relmax(out, out_a) <= 1e-9
    assert np.abs(lse - lse_a).max() <= 1e-9


def test_prefill_causal_row_is_a_shorter_decode():
    inp = prefill_inputs(1, 20, 2, [90], seed=7)
    out, lse = oracle.prefill_naive(f32(inp.q), f32(inp.kv_cache), inp.block_table, inp.seqlens, f32(inp.w_uk),
                                    f32(inp.w_uv), inp.scale, True)
    for s in (0, 7, 19):
        n = 90 - 20 + s + 1
        o1, l1 = oracle.prefill_naive(f32(inp.q[:, s:s + 1]), f32(inp.kv_cache), inp.block_table,
                                      np.array([n], np.int32), f32(inp.w_uk), f32(inp.w_uv), inp.scale, True)
        assert relmax(out[:, s:s + 1], o1) <= 1e-12
        assert np.abs(lse[:, s:s + 1] - l1).max() <= 1e-12

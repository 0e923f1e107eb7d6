"""GPU unit tests of single building blocks, through the C ABI:
schedule (bit-exact vs the oracle), paged TMA gather (bit-exact vs a CPU
gather), one-tile tcgen05 products (vs fp64 products of the same bf16
values), the two projections (vs the oracle)."""
import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_absorbed_gb300 import inputs as gen
from parity_util import assert_o_close, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from mla_paged_kv_absorbed_gb300 import _build
    _build.build()
    from mla_paged_kv_absorbed_gb300 import api as a
    return a


# ---------------------------------------------------------------- schedule --

SCHEDULE_CASES = [
    ([37, 100], 4), ([37, 100], 76), ([512] * 128, 76), ([4096] * 132, 38), ([0, 130, 64, 1], 3),
    ([0] * 5, 7), ([1], 1), ([70000, 3, 5000, 0, 2049], 13),
]


@pytest.mark.parametrize("seqlens,num_parts", SCHEDULE_CASES)
def test_schedule_bit_exact(api, seqlens, num_parts):
    ovh, min_split = api.mla_schedule_constants()
    sl = torch.tensor(seqlens, dtype=torch.int32)
    tm, ns = api.mla_get_metadata(sl.cuda(), 1, 128, num_parts)
    ref_tm, ref_ns = oracle.metadata(sl.numpy(), num_parts, ovh, min_split)
    assert np.array_equal(tm.cpu().numpy(), ref_tm)
    assert np.array_equal(ns.cpu().numpy(), ref_ns)


@pytest.mark.parametrize("seed", range(6))
def test_schedule_bit_exact_random(api, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 3000))
    sl = rng.integers(0, 40000, B).astype(np.int32) if seed % 2 else rng.integers(1, 1200, B).astype(np.int32)
    ovh, min_split = api.mla_schedule_constants()
    for num_parts in (1, 38, 76, 1000):
        tm, ns = api.mla_get_metadata(torch.from_numpy(sl).cuda(), 1, 128, num_parts)
        ref_tm, ref_ns = oracle.metadata(sl, num_parts, ovh, min_split)
        assert np.array_equal(tm.cpu().numpy(), ref_tm)
        assert np.array_equal(ns.cpu().numpy(), ref_ns)


# ------------------------------------------------------------------ gather --

def test_paged_gather_bit_exact(api):
    inp = gen.make_inputs(5, 1, 16, [1, 64, 65, 130, 333], seed=3, q_mode="q_abs")
    max_tokens = 384
    out = api.mla_debug_gather(inp.kv_cache.cuda(), inp.block_table.cuda(), inp.seqlens.cuda(), max_tokens).cpu()
    kv = inp.kv_cache.view(-1, 576)
    for b in range(inp.B):
        n = int(inp.seqlens[b])
        idx = torch.tensor([int(inp.block_table[b, t // 64]) * 64 + t % 64 for t in range(n)])
        assert torch.equal(out[b, :n].view(torch.int16), kv[idx].view(torch.int16))
        assert torch.all(out[b, n:] == 0)


# ------------------------------------------------------------- tcgen05 tile --

@pytest.mark.parametrize("a_tmem", [0, 1, 2])
@pytest.mark.parametrize("K,N,kmajor", [(64, 64, True), (576, 64, True), (320, 64, True), (64, 256, False),
                                        (128, 128, False), (576, 256, True), (192, 64, False), (512, 128, True)])
def test_mma_tile(api, K, N, kmajor, a_tmem):
    g = torch.Generator().manual_seed(K * 1000 + N)
    a = torch.randn(128, K, generator=g).to(torch.bfloat16)
    b = torch.randn((N, K) if kmajor else (K, N), generator=g).to(torch.bfloat16)
    d = api.mla_debug_mma(a.cuda(), b.cuda(), kmajor, a_tmem).cpu().double()
    bm = b.double().T if kmajor else b.double()
    ref = a.double() @ bm
    err = (d - ref).abs().max().item()
    assert err <= 1e-3 * np.sqrt(K), err


# ------------------------------------------------------------- projections --

@pytest.mark.parametrize("B,s_q,H", [(2, 1, 16), (128, 1, 128), (132, 2, 128), (3, 2, 64), (130, 1, 32)])
def test_absorb_q(api, B, s_q, H):
    inp = gen.make_inputs(B, s_q, H, 64, seed=B + H, q_mode="q", garbage=False, decoy_frac=0.0)
    q_abs = api.mla_absorb_q(inp.q.cuda(), inp.w_uk.cuda()).cpu()
    ref = oracle.absorb_q(f32(inp.q), f32(inp.w_uk))
    assert_o_close(q_abs, ref, "q_abs")
    # the rope part is a plain copy
    assert torch.equal(q_abs[..., 512:].view(torch.int16), inp.q[..., 128:].view(torch.int16))


# rows per head: 1 tile (2, 128, 5), 3 tiles (264), 9 tiles looped in one CTA
# per head (1100), five 1-tile groups (600 rows, 16 heads), uneven groups of
# 2, 2, 1 tiles (600 rows, 32 heads)
@pytest.mark.parametrize("B,s_q,H", [(2, 1, 16), (128, 1, 128), (132, 2, 128), (5, 1, 64), (1100, 1, 128),
                                     (600, 1, 16), (300, 2, 32)])
def test_out_proj(api, B, s_q, H):
    g = torch.Generator().manual_seed(B * 7 + H)
    o = (torch.randn(B, s_q, H, 512, generator=g) * 0.2).to(torch.bfloat16)
    w = (torch.randn(H, 512, 128, generator=g) / np.sqrt(512)).to(torch.bfloat16)
    out = api.mla_out_proj(o.cuda(), w.cuda()).cpu()
    ref = oracle.out_proj(f32(o), f32(w))
    assert_o_close(out, ref, "out")

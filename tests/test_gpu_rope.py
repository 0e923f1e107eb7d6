"""GPU parity of mla_rope_append (rotary encoding of the rope parts and the
append of the new tokens to the paged cache) through the C ABI against the
CPU oracle (oracle.rope, oracle.cache_append).

Byte work is compared bit-exactly: the latent copied into its slot, every
other slot of the cache, the nope part of q. The rotated values are compared
with the oracle's fp64 rotation within the bound of the arithmetic: one bf16
rounding of the result (half an ulp, at most 2^-8 of its magnitude) plus the
fp32 rotation's own error (a few float ulps of the inputs)."""
import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_absorbed_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

BASE = 10000.0


@pytest.fixture(scope="module")
def api():
    from mla_paged_kv_absorbed_gb300 import _build
    _build.build()
    from mla_paged_kv_absorbed_gb300 import api as a
    return a


def f64(t):
    return t.detach().cpu().double().numpy()


def assert_rotated_close(gpu, ref, x):
    """|gpu - ref| <= 2^-8 |ref| + 1e-6 * max |x| elementwise (x: the un-rotated input)."""
    bound = 2.0 ** -8 * np.abs(ref) + 1e-6 * (np.abs(x).max() if x.size else 0.0)
    err = np.abs(gpu - ref)
    assert np.all(err <= bound), f"max excess {float((err - bound).max()):.3e}"


def positions(seqlens, s_q):
    return (seqlens.long()[:, None] - s_q + torch.arange(s_q)[None, :]).numpy()  # [B, s_q]


CASES = [
    (2, 1, 16, [37, 100]),
    (3, 2, 64, [1, 5, 300]),                 # sequence 0: its first new token would sit at t = -1
    (132, 2, 128, 4096),
    (16, 1, 128, (16384, 32768)),            # positions of tens of thousands of radians
    (64, 1, 128, (129, 1152)),
]


@pytest.mark.parametrize("B,s_q,H,seqlens", CASES)
def test_rope_append_parity(api, B, s_q, H, seqlens):
    inp = gen.make_inputs(B, s_q, H, seqlens, seed=500 + B + s_q, q_mode="q", weights=False)
    g = torch.Generator().manual_seed(B * 11 + s_q)
    kv_new = torch.randn(B, s_q, 576, generator=g).to(torch.bfloat16)
    q0, kv0 = inp.q.clone(), inp.kv_cache.clone()
    d = inp.to("cuda")
    api.mla_rope_append(d.q, kv_new.cuda(), d.seqlens, d.block_table, d.kv_cache, BASE)
    assert api.mla_read_device_error() == 0
    q_gpu, kv_gpu = d.q.cpu(), d.kv_cache.cpu()

    # the query: nope part untouched, rope part rotated at the token's position
    assert torch.equal(q_gpu[..., :128].view(torch.int16), q0[..., :128].view(torch.int16))
    pos = positions(inp.seqlens, s_q)
    valid = pos >= 0
    x = f64(q0[..., 128:])
    ref = oracle.rope(q0[..., 128:].float().numpy(), np.broadcast_to(pos[:, :, None], (B, s_q, H)), BASE)
    assert_rotated_close(f64(q_gpu[..., 128:])[valid], ref[valid], x[valid])
    assert torch.equal(q_gpu[~torch.from_numpy(valid)].view(torch.int16), q0[~torch.from_numpy(valid)].view(torch.int16))

    # the cache: every slot but the new tokens' bit-identical, latent copied, rope rotated
    kv_ref = oracle.cache_append(kv0.float().numpy(), kv_new.float().numpy(), inp.block_table, inp.seqlens, BASE)
    kv_g = f64(kv_gpu)
    touched = np.zeros(kv_ref.shape[:2], bool)
    for b in range(B):
        for s in range(s_q):
            t = int(pos[b, s])
            if t >= 0:
                touched[int(inp.block_table[b, t // 64]), t % 64] = True
    assert np.array_equal(kv_g[~touched], kv_ref[~touched])
    assert np.array_equal(kv_g[touched][:, :512], kv_ref[touched][:, :512])
    xs = np.stack([f64(kv_new)[b, s, 512:] for b in range(B) for s in range(s_q) if pos[b, s] >= 0])
    assert_rotated_close(kv_g[touched][:, 512:], kv_ref[touched][:, 512:], xs)


def test_rope_append_then_decode_sees_the_new_tokens(api):
    """The appended rows are what the decode reads: after the append, the
    absorbed query carries the rotated rope part bit-exactly, and the decode
    matches the oracle on the cache and query the GPU holds (whose appended
    rows the parity test above ties to the oracle's append)."""
    from parity_util import assert_lse_close, assert_o_close
    inp = gen.make_inputs(4, 2, 128, [65, 130, 2, 700], seed=77, q_mode="q")
    g = torch.Generator().manual_seed(5)
    kv_new = torch.randn(4, 2, 576, generator=g).to(torch.bfloat16)
    kv0 = inp.kv_cache.clone()
    d = inp.to("cuda")
    api.mla_rope_append(d.q, kv_new.cuda(), d.seqlens, d.block_table, d.kv_cache, BASE)
    tm, ns = api.mla_get_metadata(d.seqlens, 2, 128, 6)
    q_abs = api.mla_absorb_q(d.q, d.w_uk)
    o, lse = api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, True)
    assert api.mla_read_device_error() == 0
    assert torch.equal(q_abs[..., 512:].cpu().view(torch.int16), d.q[..., 128:].cpu().view(torch.int16))
    kv_gpu = d.kv_cache.cpu()
    assert not torch.equal(kv_gpu.view(torch.int16), kv0.view(torch.int16))
    o_ref, lse_ref = oracle.attend_absorbed(q_abs.cpu().float().numpy(), kv_gpu.float().numpy(), inp.block_table,
                                            inp.seqlens, inp.scale, True)
    assert_o_close(o.cpu(), o_ref, "o_lat after append")
    assert_lse_close(lse.cpu(), lse_ref, "lse after append")


def test_rope_append_reports_a_position_past_the_table(api):
    inp = gen.make_inputs(2, 1, 16, [64, 10], seed=3, q_mode="q", weights=False)
    sl = inp.seqlens.clone()
    sl[0] = 65  # token at t = 64 needs a second page the table row does not have
    kv0 = inp.kv_cache.clone()
    d = inp.to("cuda")
    kv_new = torch.randn(2, 1, 576).to(torch.bfloat16).cuda()
    api.mla_rope_append(d.q, kv_new, sl.cuda(), d.block_table, d.kv_cache, BASE)
    assert api.mla_read_device_error() == api.MLA_ERR_BAD_BLOCK
    kv = d.kv_cache.cpu()
    # sequence 1 was appended, sequence 0's missing slot wrote nothing
    t1 = 9
    blk1 = int(inp.block_table[1, 0])
    assert torch.equal(kv[blk1, t1, :512].view(torch.int16), kv_new[1, 0, :512].cpu().view(torch.int16))
    changed = (kv.view(torch.int16) != kv0.view(torch.int16)).any(-1)
    assert int(changed.sum()) == 1

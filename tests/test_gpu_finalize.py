"""GPU parity of the fused finalize path (mla_decode_out_proj: the decode, then
one kernel that merges the split pieces of each row straight into the output
projection) against the oracle: every projected output and every lse, on small
edge cases (empty sequences, many pieces per row, head counts below 128, ragged
row tiles), forced split counts and the named workloads at full size, two
seeds. The fused output is also held to the unfused path (mla_decode_paged +
mla_out_proj on the same inputs): both round the attention output to bf16
before the projection, so they differ only by the fp32 merge's rounding.

Sources: "DeepSeek-V3 MLA deep engineering" (ybb.press) sec. 2.2 (the value
up-projection on the latent side); "MLA decode fused operator" (cshb120.cn,
SC11 article) Fig. 1 text (projection fused with attention); "FlashMLA"
(wuwenjie.xyz) usage example (num_splits, lse)."""
import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_absorbed_gb300 import inputs as gen
from parity_util import assert_lse_close, assert_o_close, f32, o_errors, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from mla_paged_kv_absorbed_gb300 import _build
    _build.build()
    from mla_paged_kv_absorbed_gb300 import api as a
    return a


def run_both(api, inp, num_parts=None):
    d = inp.to("cuda")
    w_uv = d.w_uv if d.w_uv is not None else gen.draw_w_uv(d.H, inp.seed).to("cuda")
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H, num_parts)
    q_abs = d.q_abs if d.q is None else api.mla_absorb_q(d.q, d.w_uk)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    out, lse = api.mla_decode_out_proj(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                       w_uv, workspace=ws)
    status = api.mla_read_device_error(ws)
    o_u, lse_u = api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                      workspace=ws)
    out_u = api.mla_out_proj(o_u, w_uv)
    torch.cuda.synchronize()
    return {"q_abs": q_abs.cpu(), "out": out.cpu(), "lse": lse.cpu(), "out_u": out_u.cpu(), "lse_u": lse_u.cpu(),
            "w_uv": w_uv.cpu(), "status": status, "ns": ns.cpu()}


def check(inp, r):
    assert r["status"] == 0, f"device status {r['status']}"
    o_ref, lse_ref = oracle_decode(inp, r["q_abs"])
    out_ref = oracle.out_proj(o_ref, f32(r["w_uv"]))
    assert_o_close(r["out"], out_ref, "out")
    assert_lse_close(r["lse"], lse_ref)
    # against the unfused path: the same bf16 rounding of o before the product
    mx, mr = o_errors(r["out"], f32(r["out_u"]))
    assert mx <= 8e-3 and mr <= 1e-3, f"fused vs unfused out: max abs {mx:.3e}, mean rel {mr:.3e}"
    lf, lu = r["lse"].numpy(), r["lse_u"].numpy()
    assert np.array_equal(np.isneginf(lf), np.isneginf(lu))
    fin = np.isfinite(lu)
    assert np.all(np.abs(lf[fin] - lu[fin]) <= 1e-5), "fused vs unfused lse"


SMALL = [
    (3, 1, 128, [1, 64, 65]),
    (4, 2, 128, [2, 63, 64, 129]),
    (2, 1, 16, [37, 100]),
    (3, 2, 64, [0, 5, 300]),          # an empty sequence
    (5, 1, 32, [200, 0, 77, 128, 513]),
    (70, 2, 16, (1, 700)),            # 140 rows: a ragged second tile
    (130, 1, 128, (1, 300)),          # 130 rows
]


@pytest.mark.parametrize("B,s_q,H,seqlens", SMALL)
@pytest.mark.parametrize("num_parts", [None, 1, 7, 40])
def test_small_full_parity(api, B, s_q, H, seqlens, num_parts):
    inp = gen.make_inputs(B, s_q, H, seqlens, seed=B * 31 + s_q * 7 + H, q_mode="q")
    check(inp, run_both(api, inp, num_parts))


def test_many_pieces_per_row(api):
    """Long sequences cut into many pieces: rows merge more than four pieces
    (the merge's first batch of loads covers four)."""
    inp = gen.make_inputs(3, 2, 64, [3000, 2500, 40], seed=77, q_mode="q")
    r = run_both(api, inp, 60)
    ns = r["ns"].numpy()
    assert int(np.max(np.diff(ns))) > 4, "the schedule should split a sequence into more than four pieces"
    check(inp, r)


NAMED = ["dsv3", "varlen", "long", "spec"]


@pytest.mark.parametrize("rep", [0, 1])
@pytest.mark.parametrize("name", NAMED)
def test_named_workload_full_parity(api, name, rep):
    """Each named workload at full size in the default launch configuration."""
    inp = gen.make_workload(name, rep=rep)
    check(inp, run_both(api, inp))


def test_repeated_calls_deterministic(api):
    inp = gen.make_workload("spec")
    d = inp.to("cuda")
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H)
    q_abs = api.mla_absorb_q(d.q, d.w_uk)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    out0, lse0 = api.mla_decode_out_proj(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                         d.w_uv, workspace=ws)
    out, lse = torch.empty_like(out0), torch.empty_like(lse0)
    api.mla_set_wait_limit_ns(250_000_000)
    try:
        for i in range(60):
            api.mla_decode_out_proj(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal, d.w_uv,
                                    out=out, lse=lse, workspace=ws)
            if i % 20 == 19:
                assert api.mla_read_device_error(ws) == 0
                assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
                assert torch.equal(lse, lse0)
    finally:
        api.mla_set_wait_limit_ns(0)

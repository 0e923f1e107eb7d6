"""GPU parity of the INT8 latent cache path through the C ABI against the
oracle: the quantiser and the append into the INT8 cache bit for bit, and the
decode over INT8 records on every output, against the oracle's attention over
the cache the records stand for (same tolerances as the bf16 decode). Because
the power-of-two scales make every dequantised value exact in bf16, the INT8
decode must also equal the bf16 decode over the dequantised cache bit for bit.

Sources: "DeepSeek-V3 MLA deep engineering" (ybb.press) sec. 7.2; "DeepSeek
tech explainer (1)" (sunshychen.top) sec. 3.1."""
import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_absorbed_gb300 import inputs as gen
from parity_util import assert_lse_close, assert_o_close, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from mla_paged_kv_absorbed_gb300 import _build
    _build.build()
    from mla_paged_kv_absorbed_gb300 import api as a
    return a


def quantise(api, kv_dev):
    kv8, sc = api.mla_quantize_cache(kv_dev)
    torch.cuda.synchronize()
    return kv8, sc


def run_q8(api, inp, num_parts=None, kv8=None, sc=None):
    d = inp.to("cuda")
    if kv8 is None:
        kv8, sc = quantise(api, d.kv_cache)
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H, num_parts)
    q_abs = d.q_abs if d.q is None else api.mla_absorb_q(d.q, d.w_uk)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    o, lse = api.mla_decode_paged_q8(q_abs, kv8, sc, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                     workspace=ws)
    status = api.mla_read_device_error(ws)
    return {"q_abs": q_abs, "o": o, "lse": lse, "status": status, "kv8": kv8, "sc": sc, "tm": tm, "ns": ns,
            "ws": ws, "d": d}


def check_q8(inp, r):
    assert r["status"] == 0, f"device status {r['status']}"
    o_ref, lse_ref = oracle.attend_absorbed_q8(f32(r["q_abs"]), r["kv8"].cpu().numpy(), r["sc"].cpu().numpy(),
                                               inp.block_table, inp.seqlens, inp.scale, inp.causal)
    assert_o_close(r["o"].cpu(), o_ref, "o_lat")
    assert_lse_close(r["lse"].cpu(), lse_ref)


# ---------------------------------------------------------------- quantiser --

def test_quantiser_bit_exact(api):
    g = torch.Generator().manual_seed(3)
    rows = torch.randn((4096, 576), generator=g) * torch.exp(torch.empty((4096, 1)).uniform_(-10, 10, generator=g))
    rows[0] = 0
    rows[1, :512] = 0
    rows[2, 5] = 127.0 / 64     # the largest code at the power-of-two boundary
    rows[3, :512] = torch.linspace(-3, 3, 512)
    kv = rows.to(torch.bfloat16)
    kv8, sc = quantise(api, kv.cuda())
    rec, scale = oracle.quantize_cache(kv.float().numpy())
    np.testing.assert_array_equal(kv8.cpu().numpy(), rec)
    np.testing.assert_array_equal(sc.cpu().numpy(), scale)


def test_quantiser_golden_rows(api):
    from test_oracle_pins_q8 import read_golden
    cases = read_golden()
    kv = torch.zeros((len(cases), 576))
    for i, c in enumerate(cases):
        kv[i, :512] = torch.from_numpy(c["x"])
    kv8, sc = quantise(api, kv.to(torch.bfloat16).cuda())
    for i, c in enumerate(cases):
        assert float(sc[i]) == c["scale"], c["name"]
        np.testing.assert_array_equal(kv8[i, :512].cpu().numpy().view(np.int8), c["codes"], err_msg=c["name"])


@pytest.mark.parametrize("name", ["tiny", "dsv3"])
def test_quantiser_whole_cache(api, name):
    inp = gen.make_workload(name)
    kv8, sc = quantise(api, inp.kv_cache.cuda())
    rec, scale = oracle.quantize_cache(inp.kv_cache.float().numpy())
    np.testing.assert_array_equal(kv8.cpu().numpy(), rec)
    np.testing.assert_array_equal(sc.cpu().numpy(), scale)


def test_append_into_int8_cache(api):
    """The INT8 append writes the record of the token the bf16 append writes:
    the quantised latent and the same rotated rope bytes; q is rotated alike."""
    B, s_q, H = 3, 2, 32
    inp = gen.make_inputs(B, s_q, H, [5, 64, 130], seed=21, q_mode="q")
    g = torch.Generator().manual_seed(22)
    kv_new = torch.randn((B, s_q, 576), generator=g).to(torch.bfloat16)
    d = inp.to("cuda")
    kv_bf16 = d.kv_cache.clone()
    q1 = d.q.clone()
    api.mla_rope_append(q1, kv_new.cuda(), d.seqlens, d.block_table, kv_bf16)
    kv8, sc = quantise(api, d.kv_cache)
    q2 = d.q.clone()
    api.mla_rope_append_q8(q2, kv_new.cuda(), d.seqlens, d.block_table, kv8, sc)
    torch.cuda.synchronize()
    assert api.mla_read_device_error() == 0
    assert torch.equal(q1.view(torch.int16), q2.view(torch.int16))
    rec_ref, sc_ref = oracle.quantize_cache(kv_bf16.float().cpu().numpy())
    np.testing.assert_array_equal(kv8.cpu().numpy(), rec_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)


# ------------------------------------------------------------------- decode --

SMALL = [
    (3, 1, 128, [1, 64, 65]),
    (4, 2, 128, [2, 63, 64, 129]),
    (2, 1, 16, [37, 100]),
    (3, 2, 64, [1, 5, 300]),
    (5, 1, 32, [200, 1, 77, 128, 513]),
]


@pytest.mark.parametrize("B,s_q,H,seqlens", SMALL)
@pytest.mark.parametrize("num_parts", [None, 1, 7])
def test_q8_small_full_parity(api, B, s_q, H, seqlens, num_parts):
    inp = gen.make_inputs(B, s_q, H, seqlens, seed=B * 37 + s_q * 5 + H, q_mode="q_abs")
    check_q8(inp, run_q8(api, inp, num_parts))


@pytest.mark.parametrize("s_q", [1, 2])
@pytest.mark.parametrize("num_parts", [1, 13, 40])
def test_q8_split_kv(api, s_q, num_parts):
    inp = gen.make_inputs(3, s_q, 128, [2100, 3000, 4095], seed=87 + s_q, q_mode="q_abs")
    r = run_q8(api, inp, num_parts)
    if num_parts >= 13:
        assert int(r["ns"][-1].cpu()) > 3
    check_q8(inp, r)


@pytest.mark.parametrize("case", [(4, 2, 128, [2, 63, 64, 129], None), (5, 1, 32, [200, 1, 77, 128, 513], 7),
                                  (3, 1, 128, [2100, 3000, 4095], 13)])
def test_q8_equals_bf16_decode_of_dequantised_cache(api, case):
    B, s_q, H, seqlens, parts = case
    inp = gen.make_inputs(B, s_q, H, seqlens, seed=5 + B, q_mode="q_abs")
    r = run_q8(api, inp, parts)
    assert r["status"] == 0
    deq = oracle.dequantize_cache(r["kv8"].cpu().numpy(), r["sc"].cpu().numpy())
    kv_deq = torch.from_numpy(deq).to(torch.bfloat16)
    assert torch.equal(kv_deq.float(), torch.from_numpy(deq))  # every dequantised value is exact in bf16
    d = r["d"]
    ws = api.make_workspace(d.B, d.s_q, d.H, r["tm"].shape[0])
    o, lse = api.mla_decode_paged(r["q_abs"], kv_deq.cuda(), d.block_table, d.seqlens, r["tm"], r["ns"], d.scale,
                                  d.causal, workspace=ws)
    assert api.mla_read_device_error(ws) == 0
    # rows past each sequence hold different bytes in the two caches but never contribute
    assert torch.equal(o.view(torch.int16), r["o"].view(torch.int16))
    assert torch.equal(lse, r["lse"])


def test_q8_page_permutation_bit_identical(api):
    inp = gen.make_inputs(3, 1, 128, [70, 300, 1000], seed=19, q_mode="q_abs")
    r1 = run_q8(api, inp)
    perm = torch.randperm(inp.num_blocks, generator=torch.Generator().manual_seed(4)).cuda()
    kv8 = torch.empty_like(r1["kv8"])
    kv8[perm] = r1["kv8"]
    sc = torch.empty_like(r1["sc"])
    sc[perm] = r1["sc"]
    table = inp.block_table.clone().cuda()
    valid = table >= 0
    table[valid] = perm[table[valid].long()].to(torch.int32)
    d = r1["d"]
    ws = api.make_workspace(d.B, d.s_q, d.H, r1["tm"].shape[0])
    o, lse = api.mla_decode_paged_q8(d.q_abs, kv8, sc, table, d.seqlens, r1["tm"], r1["ns"], d.scale, True,
                                     workspace=ws)
    assert api.mla_read_device_error(ws) == 0
    assert torch.equal(o.view(torch.int16), r1["o"].view(torch.int16))
    assert torch.equal(lse, r1["lse"])


def test_q8_empty_and_nan_tails(api):
    """A sequence of length 0 gives o = 0, lse = -inf; the records and scales
    past each sequence's last token may hold anything (here NaN scales and
    arbitrary codes) without reaching the outputs."""
    inp = gen.make_inputs(4, 1, 64, [0, 1, 65, 130], seed=31, q_mode="q_abs")
    d = inp.to("cuda")
    kv8, sc = quantise(api, d.kv_cache)
    ref = run_q8(api, inp, kv8=kv8.clone(), sc=sc.clone())
    for b in range(inp.B):
        L = int(inp.seqlens[b])
        n = (L + 63) // 64
        if n and L % 64:
            blk = int(inp.block_table[b, n - 1])
            sc[blk, L % 64:] = float("nan")
            kv8[blk, L % 64:] = 0x7F
    r = run_q8(api, inp, kv8=kv8, sc=sc)
    assert r["status"] == 0
    assert torch.equal(r["o"].view(torch.int16), ref["o"].view(torch.int16))
    assert torch.equal(r["lse"], ref["lse"])
    assert torch.all(r["o"][0] == 0) and torch.all(torch.isneginf(r["lse"][0]))
    check_q8(inp, ref)


@pytest.mark.parametrize("seqlens,num_parts", [([0, 5, 0, 70, 0], None), ([0, 0], 3), ([0, 2100, 0, 0], 13)])
def test_q8_empty_sequences_written_everywhere(api, seqlens, num_parts):
    """As for the bf16 cache: outputs start as NaN, and the rows of empty
    sequences must read o = 0, lse = -inf wherever they sit, with and without
    a split sequence (and so with and without the merge launch)."""
    B = len(seqlens)
    inp = gen.make_inputs(B, 1, 64, seqlens, seed=41 + B, q_mode="q_abs")
    d = inp.to("cuda")
    kv8, sc = quantise(api, d.kv_cache)
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H, num_parts)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    o = torch.full((B, 1, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, 1, 64), float("nan"), dtype=torch.float32, device="cuda")
    api.mla_decode_paged_q8(d.q_abs, kv8, sc, d.block_table, d.seqlens, tm, ns, d.scale, d.causal, o_lat=o, lse=lse,
                            workspace=ws)
    r = {"q_abs": d.q_abs, "o": o, "lse": lse, "status": api.mla_read_device_error(ws), "kv8": kv8, "sc": sc}
    check_q8(inp, r)
    for b, L in enumerate(seqlens):
        if L == 0:
            assert torch.all(o[b] == 0) and torch.all(torch.isneginf(lse[b])), f"batch {b}"


NAMED = ["dsv3", "varlen", "long", "spec"]


@pytest.mark.parametrize("name", NAMED)
def test_q8_named_workload_full_parity(api, name):
    inp = gen.make_workload(name, rep=0)
    check_q8(inp, run_q8(api, inp))


@pytest.mark.parametrize("name,calls", [("long", 120), ("spec", 60), ("varlen", 200)])
def test_q8_repeated_calls_no_device_error(api, name, calls):
    """Back-to-back INT8 decode calls: the in-place expansion lengthens the
    score side's per-page chain, so the cross-warp handshakes (the reference
    max passed between the two softmax groups above all) meet timings the bf16
    path rarely produces. The device error word stays clear and every call
    returns the first call's bytes."""
    d = gen.make_workload(name).to("cuda")
    kv8, sc = quantise(api, d.kv_cache)
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H)
    q_abs = d.q_abs if d.q is None else api.mla_absorb_q(d.q, d.w_uk)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    o0, lse0 = api.mla_decode_paged_q8(q_abs, kv8, sc, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                       workspace=ws)
    assert api.mla_read_device_error(ws) == 0
    o, lse = torch.empty_like(o0), torch.empty_like(lse0)
    api.mla_set_wait_limit_ns(250_000_000)  # a lost wakeup shows up in a quarter second
    try:
        for i in range(calls):
            api.mla_decode_paged_q8(q_abs, kv8, sc, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                    o_lat=o, lse=lse, workspace=ws)
            if i % 20 == 19 or i == calls - 1:
                assert api.mla_read_device_error(ws) == 0, f"device status after call {i}"
                assert torch.equal(o.view(torch.int16), o0.view(torch.int16))
                assert torch.equal(lse, lse0)
    finally:
        api.mla_set_wait_limit_ns(0)

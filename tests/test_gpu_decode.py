"""GPU parity of the decode path through the C ABI against the CPU oracle.

Every comparison covers every output: small edge cases, forced split counts,
and the five named workloads at full size in the launch configuration the
benchmark times (default number of schedule parts), two seeds each. Device
failure handling is exercised without any fault: a bounded wait made to run
out, a block id outside the pool, and a schedule built from other lengths."""
import time

import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_absorbed_gb300 import inputs as gen
from parity_util import assert_lse_close, assert_o_close, f32, oracle_decode, oracle_end_to_end

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from mla_paged_kv_absorbed_gb300 import _build
    _build.build()
    from mla_paged_kv_absorbed_gb300 import api as a
    return a


def run(api, inp, num_parts=None):
    d = inp.to("cuda")
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H, num_parts)
    q_abs = d.q_abs if d.q is None else api.mla_absorb_q(d.q, d.w_uk)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    o, lse = api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                  workspace=ws)
    out = api.mla_out_proj(o, d.w_uv) if d.w_uv is not None else None
    status = api.mla_read_device_error(ws)
    return {"q_abs": q_abs.cpu(), "o": o.cpu(), "lse": lse.cpu(), "out": None if out is None else out.cpu(),
            "status": status, "tm": tm.cpu(), "ns": ns.cpu()}


def check_decode(inp, r):
    assert r["status"] == 0, f"device status {r['status']}"
    o_ref, lse_ref = oracle_decode(inp, r["q_abs"])
    assert_o_close(r["o"], o_ref, "o_lat")
    assert_lse_close(r["lse"], lse_ref)


# -------------------------------------------------------------- small, full --

SMALL = [
    (3, 1, 128, [1, 64, 65]),
    (4, 2, 128, [2, 63, 64, 129]),
    (2, 1, 16, [37, 100]),
    (3, 2, 64, [1, 5, 300]),
    (5, 1, 32, [200, 1, 77, 128, 513]),
    (2, 2, 16, [64, 65]),
]


@pytest.mark.parametrize("B,s_q,H,seqlens", SMALL)
@pytest.mark.parametrize("num_parts", [None, 1, 7])
def test_small_full_parity(api, B, s_q, H, seqlens, num_parts):
    inp = gen.make_inputs(B, s_q, H, seqlens, seed=B * 31 + s_q * 7 + H, q_mode="q_abs")
    check_decode(inp, run(api, inp, num_parts))


@pytest.mark.parametrize("s_q", [1, 2])
@pytest.mark.parametrize("num_parts", [1, 5, 13, 40])
def test_split_kv_and_combine(api, s_q, num_parts):
    inp = gen.make_inputs(3, s_q, 128, [2100, 3000, 4095], seed=77 + s_q, q_mode="q_abs")
    r = run(api, inp, num_parts)
    if num_parts >= 5:
        assert int(r["ns"][-1]) > 3  # the schedule really split something
    check_decode(inp, r)


def qabs_rounding_bound(inp, qa_exact, qa_gpu):
    """Per query row, a bound on how far the scores (hence lse, which moves by
    at most the largest score change) can move because the path rounds the
    absorbed query to bf16: scale * sum_c |qa_exact - qa_gpu|[c] * max_t |kv_t[c]|
    over the row's visible keys."""
    kv = inp.kv_cache.float().numpy().astype(np.float64)
    dq = np.abs(qa_exact - f32(qa_gpu).astype(np.float64))
    B, s_q, H, _ = dq.shape
    bound = np.zeros((B, s_q, H))
    for b in range(B):
        L = int(inp.seqlens[b])
        for s in range(s_q):
            n = max(0, min(L, L - s_q + s + 1)) if inp.causal else L
            if n == 0:
                continue
            rows = [int(inp.block_table[b, t // 64]) * 64 + t % 64 for t in range(n)]
            kmax = np.abs(kv.reshape(-1, 576)[rows]).max(0)
            bound[b, s] = inp.scale * (dq[b, s] * kmax).sum(-1)
    return bound


def test_tiny_end_to_end(api):
    """End to end from q, W_UK and W_UV: q_abs and the projected output within
    the stated tolerances of the oracle's unrounded fp64 chain; lse within the
    decode tolerance plus the movement the bf16 absorbed query alone allows
    (the tolerance applies to the decode's lse, which check_decode holds to
    1e-3 on the query the decode consumed)."""
    inp = gen.make_workload("tiny")
    r = run(api, inp)
    check_decode(inp, r)
    qa, o, lse, out = oracle_end_to_end(inp)
    assert_o_close(r["q_abs"], qa, "q_abs")
    assert_o_close(r["out"], out, "out")
    bound = qabs_rounding_bound(inp, qa, r["q_abs"]) + 1e-3
    err = np.abs(f32(r["lse"]).astype(np.float64) - lse)
    assert np.all(err <= bound), f"lse (end to end): max excess {float((err - bound).max()):.3e}"


def test_empty_and_fully_masked_rows(api):
    inp = gen.make_inputs(4, 2, 128, [0, 1, 64, 65], seed=5, q_mode="q_abs")
    r = run(api, inp, 3)
    check_decode(inp, r)
    assert torch.all(r["o"][0] == 0) and torch.all(r["lse"][0] == -np.inf)
    assert torch.all(r["o"][1, 0] == 0) and torch.all(r["lse"][1, 0] == -np.inf)


EMPTY_MIXES = [
    (1, [0, 5, 0, 0, 70, 0]),  # leading, inner and trailing empty sequences, no split possible
    (2, [0, 0, 0]),  # every sequence empty
    (1, [0, 2100, 0, 3000, 0, 0]),  # empty sequences around split ones
    (2, [100, 0, 0, 0, 1]),
]


@pytest.mark.parametrize("s_q,seqlens", EMPTY_MIXES)
@pytest.mark.parametrize("num_parts", [None, 1, 3, 13])
def test_empty_sequences_written_once_everywhere(api, s_q, seqlens, num_parts):
    """Outputs start as NaN, so a row of an empty sequence that nothing writes
    (or a part that writes one it does not own) shows; such rows must read
    o = 0 and lse = -inf wherever they sit in the batch."""
    B = len(seqlens)
    inp = gen.make_inputs(B, s_q, 64, seqlens, seed=sum(seqlens) + s_q, q_mode="q_abs")
    d = inp.to("cuda")
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H, num_parts)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    o = torch.full((B, s_q, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, s_q, 64), float("nan"), dtype=torch.float32, device="cuda")
    api.mla_decode_paged(d.q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal, o_lat=o, lse=lse,
                         workspace=ws)
    r = {"q_abs": d.q_abs.cpu(), "o": o.cpu(), "lse": lse.cpu(), "status": api.mla_read_device_error(ws)}
    check_decode(inp, r)
    for b, L in enumerate(seqlens):
        if L == 0:
            assert torch.all(r["o"][b] == 0) and torch.all(r["lse"][b] == -np.inf), f"batch {b}"


def test_nan_and_inf_in_tail_rows_do_not_leak(api):
    inp = gen.make_inputs(3, 1, 128, [3, 70, 200], seed=9, q_mode="q_abs", tail_fill=float("nan"))
    check_decode(inp, run(api, inp))
    inp = gen.make_inputs(3, 2, 128, [3, 70, 200], seed=10, q_mode="q_abs", tail_fill=float("inf"))
    check_decode(inp, run(api, inp))


def test_page_permutation_bit_identical(api):
    inp = gen.make_inputs(4, 2, 128, [100, 640, 64, 3000], seed=12, q_mode="q_abs")
    r1 = run(api, inp, 9)
    g = torch.Generator().manual_seed(1)
    perm = torch.randperm(inp.num_blocks, generator=g)
    kv2 = torch.empty_like(inp.kv_cache)
    kv2[perm] = inp.kv_cache
    table = inp.block_table.clone()
    valid = table >= 0
    table[valid] = perm[table[valid].long()].to(torch.int32)
    inp2 = gen.MLAInputs(inp.B, inp.s_q, inp.H, inp.scale, inp.causal, inp.seqlens, table, kv2, None, inp.q_abs,
                         None, None)
    r2 = run(api, inp2, 9)
    assert torch.equal(r1["o"].view(torch.int16), r2["o"].view(torch.int16))
    assert torch.equal(r1["lse"], r2["lse"])


def test_non_causal_multi_token(api):
    inp = gen.make_inputs(3, 2, 128, [65, 129, 1], seed=14, q_mode="q_abs", causal=False)
    check_decode(inp, run(api, inp))


# ------------------------------------------- named workloads, every output --

NAMED = [("tiny", True), ("dsv3", True), ("varlen", False), ("long", False), ("spec", True)]


@pytest.mark.parametrize("rep", [0, 1])
@pytest.mark.parametrize("name,end_to_end", NAMED)
def test_named_workload_full_parity(api, name, end_to_end, rep):
    """Each named workload at full size, in the launch configuration the
    benchmark times (default number of schedule parts), two seeds: the schedule
    bit-exact, every (b, s, h) of o_lat and lse against the oracle on the GPU's
    absorbed query, and for the end-to-end workloads q_abs and the projected
    output against the oracle's full fp64 chain from q, W_UK and W_UV."""
    inp = gen.make_workload(name, rep=rep)
    r = run(api, inp)
    ovh, min_split = api.mla_schedule_constants()
    ref_tm, ref_ns = oracle.metadata(inp.seqlens.numpy(), r["tm"].shape[0], ovh, min_split)
    assert np.array_equal(r["tm"].numpy(), ref_tm) and np.array_equal(r["ns"].numpy(), ref_ns)
    check_decode(inp, r)
    if end_to_end:
        qa, _, _, out = oracle_end_to_end(inp)
        assert_o_close(r["q_abs"], qa, f"{name} q_abs")
        assert_o_close(r["out"], out, f"{name} out")


# ------------------------------------------------------ repeated launches --

@pytest.mark.parametrize("name,calls", [("dsv3", 400), ("varlen", 300), ("spec", 60), ("long", 100)])
def test_repeated_calls_no_device_error(api, name, calls):
    """Hundreds of back-to-back calls, so that the cross-CTA handshakes of the
    decode kernel meet many different timings: the device error word stays
    clear (a lost wakeup would end in MLA_ERR_TIMEOUT) and every call returns
    the first call's bytes (the kernel is deterministic)."""
    d = gen.make_workload(name).to("cuda")
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H)
    q_abs = d.q_abs if d.q is None else api.mla_absorb_q(d.q, d.w_uk)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    o0, lse0 = api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                    workspace=ws)
    assert api.mla_read_device_error(ws) == 0
    o, lse = torch.empty_like(o0), torch.empty_like(lse0)
    api.mla_set_wait_limit_ns(250_000_000)  # a lost wakeup shows up in a quarter second, not four
    try:
        for i in range(calls):
            api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                 o_lat=o, lse=lse, workspace=ws)
            if i % 50 == 49 or i == calls - 1:
                assert api.mla_read_device_error(ws) == 0, f"device status after call {i}"
                assert torch.equal(o.view(torch.int16), o0.view(torch.int16))
                assert torch.equal(lse, lse0)
    finally:
        api.mla_set_wait_limit_ns(0)


# ------------------------------------------------------------------ errors --

def test_bad_block_is_reported(api):
    inp = gen.make_inputs(2, 1, 128, [100, 100], seed=21, q_mode="q_abs")
    inp.block_table[1, 1] = inp.num_blocks + 5
    r = run(api, inp)
    assert r["status"] == api.MLA_ERR_BAD_BLOCK
    # the healthy sequence is still right
    o_ref, lse_ref = oracle.attend_absorbed(f32(r["q_abs"][:1]), f32(inp.kv_cache), inp.block_table[:1],
                                            inp.seqlens[:1], inp.scale, True)
    assert_o_close(r["o"][:1], o_ref)


def test_host_rejects_bad_shapes(api):
    d = gen.make_inputs(2, 1, 128, [10, 10], seed=1, q_mode="q_abs").to("cuda")
    tm, ns = api.mla_get_metadata(d.seqlens, 1, 128, 4)
    with pytest.raises(api.MLAError) as e:
        api.mla_get_metadata(d.seqlens, 3, 128, 4)
    assert e.value.status == api.MLA_ERR_INVALID_ARG
    ws = api.make_workspace(2, 1, 128, 4)
    small_ws = ws[: ws.numel() // 2]
    with pytest.raises(api.MLAError) as e:
        api.mla_decode_paged(d.q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, True, workspace=small_ws)
    assert e.value.status == api.MLA_ERR_INVALID_ARG
    # a misaligned q_abs view
    flat = torch.zeros(d.q_abs.numel() + 8, dtype=torch.bfloat16, device="cuda")
    mis = flat[1:1 + d.q_abs.numel()].view_as(d.q_abs)
    with pytest.raises(api.MLAError) as e:
        api.mla_decode_paged(mis, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, True, workspace=ws)
    assert e.value.status == api.MLA_ERR_INVALID_ARG


def test_mispaired_schedule_reports_bad_block_promptly(api):
    """A schedule built from other sequence lengths walks table entries past
    the sequences' pages: the device records MLA_ERR_BAD_BLOCK and both CTAs
    of every cluster that met it leave at once, instead of waiting out the
    default four-second limit."""
    inp = gen.make_workload("tiny")
    check_decode(inp, run(api, inp, 4))  # module loaded and warm
    d = inp.to("cuda")
    q_abs = api.mla_absorb_q(d.q, d.w_uk)
    other = torch.tensor([1000, 2000], dtype=torch.int32, device="cuda")
    tm, ns = api.mla_get_metadata(other, d.s_q, d.H, 4)
    ws = api.make_workspace(d.B, d.s_q, d.H, 4)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal, workspace=ws)
    status = api.mla_read_device_error(ws)
    dt = time.perf_counter() - t0
    assert status == api.MLA_ERR_BAD_BLOCK
    assert dt < 0.5, f"took {dt:.3f} s"
    # the context is still usable
    check_decode(inp, run(api, inp, 4))


@pytest.mark.parametrize("name", ["tiny", "dsv3"])
def test_bounded_wait_expiry_returns_timeout(api, name):
    """A wait that nothing will ever satisfy runs out: with the value CTA's
    first page load withheld (a test hook; no fault, nothing out of bounds), the
    P.V warp's wait expires after the limit, the kernel records
    MLA_ERR_TIMEOUT, aborts both CTAs of every cluster with work, drains its
    copies and MMAs, frees its tensor memory and returns. Afterwards, with the
    default limit and the hook off, the same call matches the oracle."""
    inp = gen.make_workload(name)
    d = inp.to("cuda")
    tm, ns = api.mla_get_metadata(d.seqlens, d.s_q, d.H)
    q_abs = api.mla_absorb_q(d.q, d.w_uk)
    ws = api.make_workspace(d.B, d.s_q, d.H, tm.shape[0])
    api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal, workspace=ws)
    assert api.mla_read_device_error(ws) == 0
    api.mla_set_wait_limit_ns(20_000_000)  # 20 ms
    api.mla_debug_withhold_value_load(True)
    try:
        t0 = time.perf_counter()
        api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal, workspace=ws)
        status = api.mla_read_device_error(ws)
        dt = time.perf_counter() - t0
    finally:
        api.mla_debug_withhold_value_load(False)
        api.mla_set_wait_limit_ns(0)
    assert status == api.MLA_ERR_TIMEOUT
    assert dt < 1.0, f"took {dt:.3f} s"
    for _ in range(2):
        o, lse = api.mla_decode_paged(q_abs, d.kv_cache, d.block_table, d.seqlens, tm, ns, d.scale, d.causal,
                                      workspace=ws)
        assert api.mla_read_device_error(ws) == 0
        check_decode(inp, {"q_abs": q_abs.cpu(), "o": o.cpu(), "lse": lse.cpu(), "status": 0})

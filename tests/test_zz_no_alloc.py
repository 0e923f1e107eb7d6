"""The no-allocation decode entry point (mla_decode_paged_noalloc) against the
regular one (mla_decode_paged), through the C ABI.

Callers such as engine plugins that are handed only their input and output
buffers cannot call cudaMalloc; this entry point takes its scratch from an
array inside the library instead. The test runs it twice in a row (the scratch
is shared and keeps the previous call's contents) and compares both results
with the regular entry point's within the parity tolerances of the other GPU
tests. The file is named so that pytest collects it last."""
import pytest
import torch

from mla_paged_kv_absorbed_gb300 import inputs as gen
from parity_util import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from mla_paged_kv_absorbed_gb300 import _build
    _build.build()
    from mla_paged_kv_absorbed_gb300 import api as a
    return a


@pytest.mark.parametrize("s_q,seqlens,num_parts", [
    (1, [5000, 64, 3000, 1, 700, 2500, 129, 4096], None),   # long sequences split -> partials in the scratch
    (2, [4096, 65, 2049, 300], 13),
])
def test_noalloc_matches_regular_entry_twice(api, s_q, seqlens, num_parts):
    inp = gen.make_inputs(len(seqlens), s_q, 128, seqlens, seed=404 + s_q, q_mode="q_abs").to("cuda")
    tm, ns = api.mla_get_metadata(inp.seqlens, s_q, 128, num_parts)
    assert int(ns[-1]) > inp.B, "the schedule should split some sequences"
    ref_o, ref_lse = api.mla_decode_paged(inp.q_abs, inp.kv_cache, inp.block_table, inp.seqlens, tm, ns, inp.scale,
                                          inp.causal)
    ref_o, ref_lse = ref_o.cpu().double().numpy(), ref_lse.cpu().double().numpy()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    outs = [(torch.empty((inp.B, s_q, 128, 512), dtype=torch.bfloat16, device="cuda"),
             torch.empty((inp.B, s_q, 128), dtype=torch.float32, device="cuda")) for _ in range(2)]
    free_before = None
    for call, (o, lse) in enumerate(outs):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize()
        if call == 1:
            free_before = torch.cuda.mem_get_info()[0]
        api.mla_decode_paged_noalloc(inp.q_abs, inp.kv_cache, inp.block_table, inp.seqlens, tm, ns, inp.scale,
                                     inp.causal, o, lse, device_status=status)
        torch.cuda.synchronize()
        if call == 1:
            # after the first call (which may load the module and reserve the
            # scratch array), a call takes no device memory at all
            assert torch.cuda.mem_get_info()[0] == free_before
        assert int(status.item()) == 0
        assert_o_close(o.cpu(), ref_o, "o_lat (no-alloc vs regular)")
        assert_lse_close(lse.cpu(), ref_lse, "lse (no-alloc vs regular)")


def test_noalloc_rejects_shapes_beyond_its_scratch(api):
    B = 300  # (300 + 76) * 1 * 128 rows > 32768
    inp = gen.make_inputs(B, 1, 128, 64, seed=1, q_mode="q_abs", garbage=False, decoy_frac=0.0).to("cuda")
    tm, ns = api.mla_get_metadata(inp.seqlens, 1, 128, 76)
    o = torch.empty((B, 1, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, 1, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(api.MLAError) as e:
        api.mla_decode_paged_noalloc(inp.q_abs, inp.kv_cache, inp.block_table, inp.seqlens, tm, ns, inp.scale, True,
                                     o, lse)
    assert e.value.status == api.MLA_ERR_INVALID_ARG

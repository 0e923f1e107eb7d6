"""Pins of the oracle's quantised latent cache (oracle.quantize_latent,
quantize_cache, dequantize_cache, attend_absorbed_q8) against values that do
not come from the oracle itself: hand-derived codes and scales
(tests/golden/q8_quantize.txt), the record's byte layout, the bounds the
power-of-two reading implies, lossless round trips of latents that are already
codes times a power of two, and attention over a losslessly quantised cache,
which must equal attention over the original cache.

Source: "DeepSeek-V3 MLA deep engineering" (ybb.press) sec. 7.2 (the latent
quantised to 8 bits); "DeepSeek tech explainer (1)" (sunshychen.top) sec. 3.1."""
import os

import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_absorbed_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q8_quantize.txt")


def read_golden():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest, "x": np.zeros(512, np.float32), "codes": np.zeros(512, np.int8)}
            cases.append(cur)
        elif key == "x":
            for kv in rest.split():
                i, v = kv.split("=")
                cur["x"][int(i)] = float(v)
        elif key == "scale":
            cur["scale"] = float(rest)
        elif key == "codes":
            for kv in rest.split():
                i, v = kv.split("=")
                cur["codes"][int(i)] = int(v)
    return cases


@pytest.mark.parametrize("case", read_golden(), ids=lambda c: c["name"])
def test_golden_codes_and_scale(case):
    codes, scale = oracle.quantize_latent(case["x"][None])
    assert float(scale[0]) == case["scale"]
    np.testing.assert_array_equal(codes[0], case["codes"])


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def test_bounds_random_rows():
    g = np.random.default_rng(5)
    x = _bf16(g.standard_normal((300, 512)) * np.exp(g.uniform(-8, 8, (300, 1))))
    codes, scale = oracle.quantize_latent(x)
    amax = np.abs(x).max(axis=1)
    # the scale is a power of two and the smallest with 127 s >= amax
    m, _ = np.frexp(scale)
    assert np.all(m == 0.5)
    assert np.all(127.0 * scale.astype(np.float64) >= amax)
    assert np.all(63.5 * scale.astype(np.float64) < amax)
    assert codes.min() >= -127 and codes.max() <= 127
    # the largest code of a row reaches at least 64 (the row uses the upper half of the range)
    assert np.all(np.abs(codes.astype(np.int32)).max(axis=1) >= 64)
    err = np.abs(codes.astype(np.float64) * scale[:, None] - x)
    assert np.all(err <= scale[:, None].astype(np.float64) / 2)


def test_lossless_when_already_quantised():
    g = np.random.default_rng(6)
    codes = g.integers(-127, 128, (50, 512)).astype(np.int8)
    codes[:, 7] = g.choice([-1, 1], 50) * g.integers(64, 128, 50)  # the row maximum sets the scale
    codes = np.where(np.abs(codes.astype(np.int32)) > np.abs(codes[:, 7:8].astype(np.int32)), 0, codes).astype(np.int8)
    e = g.integers(-20, 10, 50)
    x = codes.astype(np.float64) * np.ldexp(1.0, e)[:, None]
    c2, s2 = oracle.quantize_latent(x.astype(np.float32))
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2, np.ldexp(1.0, e).astype(np.float32))


def test_record_layout_and_round_trip():
    kv = np.zeros((2, 576), np.float32)
    kv[0, 0] = 3.0
    kv[0, 1] = -1.0
    kv[0, 512] = 1.0      # bf16 0x3F80 -> bytes 0x80, 0x3F
    kv[0, 575] = -2.0     # bf16 0xC000 -> bytes 0x00, 0xC0
    kv[1, 100] = -0.25
    rec, scale = oracle.quantize_cache(kv)
    assert rec.shape == (2, 640) and scale.shape == (2,)
    assert scale[0] == 1.0 / 32 and rec[0, 0] == 96 and rec[0, 1] == (256 - 32) and rec[0, 2] == 0
    assert rec[0, 512] == 0x80 and rec[0, 513] == 0x3F and rec[0, 638] == 0x00 and rec[0, 639] == 0xC0
    # -0.25 = 0.5 * 2^-1: s = 2^-8, code -64
    assert scale[1] == 2.0 ** -8 and rec[1, 100] == 256 - 64
    back = oracle.dequantize_cache(rec, scale)
    np.testing.assert_array_equal(back, kv)


def test_rope_part_copied_bit_for_bit():
    g = np.random.default_rng(7)
    kv = _bf16(g.standard_normal((3, 64, 576)))
    rec, scale = oracle.quantize_cache(kv)
    back = oracle.dequantize_cache(rec, scale)
    np.testing.assert_array_equal(back[..., 512:], kv[..., 512:])
    err = np.abs(back[..., :512].astype(np.float64) - kv[..., :512])
    assert np.all(err <= scale[..., None] / 2)


def _lossless_cache(inp, g):
    """inp's cache with every latent row replaced by codes x 2^e (quantisation is lossless on it)."""
    kv = inp.kv_cache.float().numpy().copy()
    n = kv.shape[0] * kv.shape[1]
    codes = g.integers(-127, 128, (n, 512)).astype(np.float64)
    codes[:, 0] = 127.0
    e = g.integers(-9, -4, n)
    kv.reshape(n, 576)[:, :512] = (codes * np.ldexp(1.0, e)[:, None]).astype(np.float32)
    return kv


@pytest.mark.parametrize("causal,s_q", [(True, 1), (True, 2), (False, 1)])
def test_attention_over_lossless_cache_equals_bf16_attention(causal, s_q):
    inp = gen.make_inputs(3, s_q, 16, [1, 100, 190], seed=71 + s_q, q_mode="q_abs", causal=causal, garbage=False)
    kv = _lossless_cache(inp, np.random.default_rng(8))
    rec, scale = oracle.quantize_cache(kv)
    qa = inp.q_abs.float().numpy()
    o8, l8 = oracle.attend_absorbed_q8(qa, rec, scale, inp.block_table, inp.seqlens, inp.scale, causal)
    o, lse = oracle.attend_absorbed(qa, kv, inp.block_table, inp.seqlens, inp.scale, causal)
    np.testing.assert_array_equal(o8, o)
    np.testing.assert_array_equal(l8, lse)


def test_attention_over_quantised_cache_moves_within_the_quantisation_error():
    """A general cache: every score moves by at most scale * sum_c |q_c| s_t / 2,
    so lse moves by at most the largest such move."""
    inp = gen.make_inputs(2, 1, 16, [70, 130], seed=91, q_mode="q_abs", garbage=False)
    kv = inp.kv_cache.float().numpy()
    rec, scale = oracle.quantize_cache(kv)
    qa = inp.q_abs.float().numpy()
    o8, l8 = oracle.attend_absorbed_q8(qa, rec, scale, inp.block_table, inp.seqlens, inp.scale, True)
    o, lse = oracle.attend_absorbed(qa, kv, inp.block_table, inp.seqlens, inp.scale, True)
    smax = float(scale.max())
    bound = inp.scale * np.abs(qa[..., :512]).sum(-1) * smax / 2
    assert np.all(np.abs(l8 - lse) <= bound + 1e-12)
    assert np.abs(o8 - o).max() < 0.05

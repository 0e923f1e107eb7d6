"""CPU oracle for paged, absorbed MLA decode.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s ``cpu_baseline`` / ``--impl reference`` leg may import this
package. The CUDA library never calls it, and the two share no source.

The arithmetic lives in ``mla_oracle.c`` (plain C, double precision, scalar
loops); this module only builds that file with gcc and marshals numpy arrays
through ctypes. Every function documents the page passage it follows in the C
source. Inputs are float32 arrays holding the exact widening of the bf16 values
the GPU sees; outputs are float64.

Parity status per function (how each is pinned, see tests/test_oracle_pins.py):
  absorb_q, attend_absorbed, attend_naive, out_proj  - pinned (identity, closed
      forms, textbook special case, fp64 brute force)
  attend_streaming                                   - pinned (equals two-pass)
  combine, attend_split                              - pinned (split == single pass)
  metadata                                           - pinned by invariants and a
      hand-derived example; the pages print no schedule values.
  prefill_naive                                      - pinned (equals the
      absorbed form and the fp64 numpy brute force; causal row s equals a
      decode of the first seqlen - s_q + s + 1 keys)
  rope, cache_append                                 - pinned (identity at
      position 0, exact quarter and half turns, norm preservation, relative
      position, composition; bit-exact latent copy into the table's slot)
  quantize_latent, quantize_cache, dequantize_cache,
  attend_absorbed_q8                                 - pinned (hand-derived
      codes and scales incl. ties and the power-of-two boundary, the record
      bytes, round-trip bounds, lossless round trip of exactly representable
      latents, attention over a losslessly quantised cache == bf16 attention)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PAGE = 64
D_LATENT = 512
D_ROPE = 64
D_QK = 576
D_NOPE = 128
D_Q = 192
D_V = 128


def build(force: bool = False) -> str:
    """Compile mla_oracle.c into liboracle.so next to it (gcc, OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        D = ctypes.c_double
        lib.orc_absorb_q.argtypes = [P, P, I64, I, P]
        lib.orc_attend_absorbed.argtypes = [P, P, P, I, P, I, I, I, D, I, P, P]
        lib.orc_attend_naive.argtypes = [P, P, P, I, P, I, I, I, P, P, D, I, P, P]
        lib.orc_out_proj.argtypes = [P, P, I64, I, P]
        lib.orc_attend_streaming.argtypes = [P, P, P, I, P, I, I, I, D, I, P, P]
        lib.orc_combine.argtypes = [P, P, I, P, P]
        lib.orc_metadata.argtypes = [P, I, I, I, I, P, P]
        lib.orc_metadata.restype = I
        lib.orc_attend_split.argtypes = [P, P, P, I, P, I, I, I, D, I, P, I, P, P, P, P, P]
        lib.orc_num_threads.restype = I
        lib.orc_rope.argtypes = [P, I64, I, P, D, P]
        lib.orc_prefill_naive.argtypes = [P, P, P, I, P, I, I, I, P, P, D, I, P, P]
        lib.orc_cache_append.argtypes = [P, P, I, P, I, I, D, P]
        lib.orc_quantize_latent.argtypes = [P, I64, P, P]
        lib.orc_quantize_cache.argtypes = [P, I64, P, P]
        lib.orc_dequantize_cache.argtypes = [P, P, I64, P]
        _lib = lib
        return lib


def _arr(x, dtype):
    """Contiguous numpy array of `dtype` from a numpy array or a CPU torch tensor."""
    if hasattr(x, "detach") and hasattr(x, "numpy"):
        x = x.detach().cpu()
        if dtype == np.float32 or dtype == np.float64:
            x = x.double() if dtype == np.float64 else x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def absorb_q(q, w_uk) -> np.ndarray:
    """q [R?, ..., H, 192] (any leading dims), w_uk [H, 128, 512] -> q_abs [..., H, 576] float64."""
    q = _arr(q, np.float32)
    w = _arr(w_uk, np.float32)
    H = w.shape[0]
    assert q.shape[-1] == D_Q and q.shape[-2] == H and w.shape[1:] == (D_NOPE, D_LATENT)
    R = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    out = np.empty(q.shape[:-1] + (D_QK,), np.float64)
    _load().orc_absorb_q(_ptr(q), _ptr(w), R, H, _ptr(out))
    return out


def _attend_args(kv, block_table, seqlens):
    kv = _arr(kv, np.float32)
    bt = _arr(block_table, np.int32)
    sl = _arr(seqlens, np.int32)
    assert kv.ndim == 3 and kv.shape[1:] == (PAGE, D_QK)
    assert bt.ndim == 2 and sl.ndim == 1 and bt.shape[0] == sl.shape[0]
    return kv, bt, sl


def attend_absorbed(q_abs, kv, block_table, seqlens, scale: float, causal: bool = True):
    """q_abs [B, s_q, H, 576] -> (o_lat [B, s_q, H, 512], lse [B, s_q, H]) float64."""
    qa = _arr(q_abs, np.float64)
    kv, bt, sl = _attend_args(kv, block_table, seqlens)
    B, s_q, H, _ = qa.shape
    o = np.empty((B, s_q, H, D_LATENT), np.float64)
    lse = np.empty((B, s_q, H), np.float64)
    _load().orc_attend_absorbed(_ptr(qa), _ptr(kv), _ptr(bt), bt.shape[1], _ptr(sl), B, s_q, H,
                                float(scale), int(bool(causal)), _ptr(o), _ptr(lse))
    return o, lse


def attend_streaming(q_abs, kv, block_table, seqlens, scale: float, causal: bool = True):
    """The pages' one-key-at-a-time normalised recurrence; same shapes as attend_absorbed."""
    qa = _arr(q_abs, np.float64)
    kv, bt, sl = _attend_args(kv, block_table, seqlens)
    B, s_q, H, _ = qa.shape
    o = np.empty((B, s_q, H, D_LATENT), np.float64)
    lse = np.empty((B, s_q, H), np.float64)
    _load().orc_attend_streaming(_ptr(qa), _ptr(kv), _ptr(bt), bt.shape[1], _ptr(sl), B, s_q, H,
                                 float(scale), int(bool(causal)), _ptr(o), _ptr(lse))
    return o, lse


def attend_naive(q, kv, block_table, seqlens, w_uk, w_uv, scale: float, causal: bool = True):
    """Decompress form: q [B, s_q, H, 192] -> (out [B, s_q, H, 128], lse [B, s_q, H]) float64."""
    q = _arr(q, np.float32)
    kv, bt, sl = _attend_args(kv, block_table, seqlens)
    wk = _arr(w_uk, np.float32)
    wv = _arr(w_uv, np.float32)
    B, s_q, H, _ = q.shape
    assert wk.shape == (H, D_NOPE, D_LATENT) and wv.shape == (H, D_LATENT, D_V)
    out = np.empty((B, s_q, H, D_V), np.float64)
    lse = np.empty((B, s_q, H), np.float64)
    _load().orc_attend_naive(_ptr(q), _ptr(kv), _ptr(bt), bt.shape[1], _ptr(sl), B, s_q, H, _ptr(wk), _ptr(wv),
                             float(scale), int(bool(causal)), _ptr(out), _ptr(lse))
    return out, lse


def out_proj(o_lat, w_uv) -> np.ndarray:
    """o_lat [..., H, 512], w_uv [H, 512, 128] -> out [..., H, 128] float64."""
    o = _arr(o_lat, np.float64)
    w = _arr(w_uv, np.float32)
    H = w.shape[0]
    assert o.shape[-1] == D_LATENT and o.shape[-2] == H and w.shape[1:] == (D_LATENT, D_V)
    R = int(np.prod(o.shape[:-2])) if o.ndim > 2 else 1
    out = np.empty(o.shape[:-1] + (D_V,), np.float64)
    _load().orc_out_proj(_ptr(o), _ptr(w), R, H, _ptr(out))
    return out


def combine(o_parts, lse_parts):
    """o_parts [n, 512], lse_parts [n] -> (o [512], lse) float64."""
    o_parts = _arr(o_parts, np.float64)
    lse_parts = _arr(lse_parts, np.float64)
    n = lse_parts.shape[0]
    assert o_parts.shape == (n, D_LATENT)
    o = np.empty(D_LATENT, np.float64)
    lse = np.empty(1, np.float64)
    _load().orc_combine(_ptr(o_parts), _ptr(lse_parts), n, _ptr(o), _ptr(lse))
    return o, float(lse[0])


def metadata(seqlens, num_parts: int, ovh: int, min_split: int):
    """-> (tile_meta int32 [num_parts, 8], num_splits int32 [B + 1])."""
    sl = _arr(seqlens, np.int32)
    B = sl.shape[0]
    tm = np.zeros((num_parts, 8), np.int32)
    ns = np.zeros(B + 1, np.int32)
    rc = _load().orc_metadata(_ptr(sl), B, int(num_parts), int(ovh), int(min_split), _ptr(tm), _ptr(ns))
    if rc != 0:
        raise ValueError("orc_metadata: bad arguments")
    return tm, ns


def attend_split(q_abs, kv, block_table, seqlens, scale: float, causal: bool, tile_meta, num_splits):
    """Split-KV through a schedule, pieces combined with `combine`.

    -> (o_lat [B, s_q, H, 512], lse [B, s_q, H], o_parts [P, s_q, H, 512], lse_parts [P, s_q, H]).
    """
    qa = _arr(q_abs, np.float64)
    kv, bt, sl = _attend_args(kv, block_table, seqlens)
    tm = _arr(tile_meta, np.int32)
    ns = _arr(num_splits, np.int32)
    B, s_q, H, _ = qa.shape
    P = int(ns[B])
    o = np.empty((B, s_q, H, D_LATENT), np.float64)
    lse = np.empty((B, s_q, H), np.float64)
    op = np.empty((max(P, 1), s_q, H, D_LATENT), np.float64)
    lp = np.empty((max(P, 1), s_q, H), np.float64)
    _load().orc_attend_split(_ptr(qa), _ptr(kv), _ptr(bt), bt.shape[1], _ptr(sl), B, s_q, H, float(scale),
                             int(bool(causal)), _ptr(tm), tm.shape[0], _ptr(ns), _ptr(o), _ptr(lse),
                             _ptr(op), _ptr(lp))
    return o, lse, op[:P], lp[:P]


def rope(x, pos, base: float = 10000.0) -> np.ndarray:
    """Rotary encoding of x [..., d] at positions pos [...] (broadcast over the last dim) -> float64."""
    x = _arr(x, np.float32)
    d = x.shape[-1]
    assert d % 2 == 0
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, np.int64), x.shape[:-1]).reshape(rows))
    y = np.empty(x.shape, np.float64)
    _load().orc_rope(_ptr(x), rows, d, _ptr(p), float(base), _ptr(y))
    return y


def cache_append(kv, kv_new, block_table, seqlens, base: float = 10000.0) -> np.ndarray:
    """A copy of kv [num_blocks, 64, 576] (float64) with each sequence's s_q new
    tokens kv_new [B, s_q, 576] written to their slots (latent copied, rope part
    rotary-encoded at the token's position seqlen - s_q + s)."""
    out = np.array(_arr(kv, np.float64), copy=True)
    new = _arr(kv_new, np.float32)
    bt = _arr(block_table, np.int32)
    sl = _arr(seqlens, np.int32)
    B, s_q, d = new.shape
    assert d == D_QK and bt.shape[0] == B and sl.shape[0] == B and out.shape[1:] == (PAGE, D_QK)
    _load().orc_cache_append(_ptr(new), _ptr(bt), bt.shape[1], _ptr(sl), B, s_q, float(base), _ptr(out))
    return out


def prefill_naive(q, kv, block_table, seqlens, w_uk, w_uv, scale: float, causal: bool = True):
    """Prefill, naive form (per-head K and V materialised once per token):
    q [B, s_q, H, 192] -> (out [B, s_q, H, 128], lse [B, s_q, H]) float64."""
    q = _arr(q, np.float32)
    kv, bt, sl = _attend_args(kv, block_table, seqlens)
    wk = _arr(w_uk, np.float32)
    wv = _arr(w_uv, np.float32)
    B, s_q, H, _ = q.shape
    assert wk.shape == (H, D_NOPE, D_LATENT) and wv.shape == (H, D_LATENT, D_V)
    out = np.empty((B, s_q, H, D_V), np.float64)
    lse = np.empty((B, s_q, H), np.float64)
    _load().orc_prefill_naive(_ptr(q), _ptr(kv), _ptr(bt), bt.shape[1], _ptr(sl), B, s_q, H, _ptr(wk), _ptr(wv),
                              float(scale), int(bool(causal)), _ptr(out), _ptr(lse))
    return out, lse


def quantize_latent(x):
    """Per-token INT8 quantisation of latents x [..., 512] -> (codes int8 [..., 512],
    scale float32 [...]), scale a power of two (see mla_oracle.c)."""
    x = _arr(x, np.float32)
    assert x.shape[-1] == D_LATENT
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    codes = np.empty(x.shape, np.int8)
    scale = np.empty(x.shape[:-1], np.float32)
    _load().orc_quantize_latent(_ptr(x), rows, _ptr(codes), _ptr(scale))
    return codes, scale


def quantize_cache(kv):
    """kv [..., 576] (bf16 values as float32) -> (records uint8 [..., 640], scale float32 [...]):
    record = [512 INT8 codes | 64 bf16 rope values, little-endian]."""
    kv = _arr(kv, np.float32)
    assert kv.shape[-1] == D_QK
    bits = kv.view(np.uint32)
    assert not np.any(bits[..., D_LATENT:] & 0xFFFF), "rope values must be exact bf16"
    tokens = int(np.prod(kv.shape[:-1]))
    rec = np.empty(kv.shape[:-1] + (640,), np.uint8)
    scale = np.empty(kv.shape[:-1], np.float32)
    _load().orc_quantize_cache(_ptr(kv), tokens, _ptr(rec), _ptr(scale))
    return rec, scale


def dequantize_cache(rec, scale):
    """records [..., 640] uint8 + scale [...] -> the cache they stand for, float32 [..., 576]."""
    rec = _arr(rec, np.uint8)
    scale = _arr(scale, np.float32)
    assert rec.shape[-1] == 640 and rec.shape[:-1] == scale.shape
    tokens = int(np.prod(rec.shape[:-1]))
    kv = np.empty(rec.shape[:-1] + (D_QK,), np.float32)
    _load().orc_dequantize_cache(_ptr(rec), _ptr(scale), tokens, _ptr(kv))
    return kv


def attend_absorbed_q8(q_abs, rec, scale, block_table, seqlens, softmax_scale: float, causal: bool = True):
    """Decode over a quantised cache (records [num_blocks, 64, 640], scale [num_blocks, 64]):
    the absorbed-form attention over the cache the records stand for."""
    return attend_absorbed(q_abs, dequantize_cache(rec, scale), block_table, seqlens, softmax_scale, causal)

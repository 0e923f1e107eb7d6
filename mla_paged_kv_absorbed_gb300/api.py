"""ctypes binding of libmla (include/mla.h) over torch tensors.

Argument marshalling only: every function checks dtypes, devices and
contiguity, allocates missing outputs with torch (device memory is torch's
job), passes raw pointers and the current CUDA stream, and raises MLAError on
a non-zero status. All arithmetic runs in the library's CUDA kernels; there is
no fallback: if libmla.so is missing or cannot load, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_CUDA = 3
MLA_ERR_TIMEOUT = 4
MLA_ERR_BAD_BLOCK = 5

PAGE = 64
D_QK = 576
D_LATENT = 512
D_Q = 192
Q8_RECORD = 640  # bytes per token of the INT8 cache: 512 codes + 64 bf16 rope values
D_V = 128

_lock = threading.Lock()
_lib = None


class MLAError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded libmla.so. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmla.so not found at {LIB_PATH}: build it with "
                               "`python -m mla_paged_kv_absorbed_gb300._build` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, SZ, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_longlong
        L.mla_status_string.argtypes = [I]
        L.mla_status_string.restype = ctypes.c_char_p
        L.mla_version.restype = I
        L.mla_schedule_constants.argtypes = [ctypes.POINTER(I), ctypes.POINTER(I)]
        L.mla_default_num_parts.argtypes = [I, I]
        L.mla_default_num_parts.restype = I
        L.mla_workspace_size.argtypes = [I, I, I, I]
        L.mla_workspace_size.restype = SZ
        L.mla_set_wait_limit_ns.argtypes = [LL]
        L.mla_get_metadata.argtypes = [P, I, I, I, I, I, P, P, P]
        L.mla_get_metadata.restype = I
        L.mla_absorb_q.argtypes = [P, P, P, I, I, I, P]
        L.mla_absorb_q.restype = I
        L.mla_decode_paged.argtypes = [P, P, I, P, I, P, I, I, I, P, P, I, F, I, P, P, P, SZ, P]
        L.mla_decode_paged.restype = I
        L.mla_decode_out_proj.argtypes = [P, P, I, P, I, P, I, I, I, P, P, I, F, I, P, P, P, P, P, SZ, P]
        L.mla_decode_out_proj.restype = I
        L.mla_out_proj.argtypes = [P, P, P, I, I, I, P]
        L.mla_out_proj.restype = I
        L.mla_read_device_error.argtypes = [P, P]
        L.mla_read_device_error.restype = I
        L.mla_debug_gather.argtypes = [P, I, P, I, P, I, I, P, P]
        L.mla_debug_gather.restype = I
        L.mla_debug_mma.argtypes = [P, P, I, I, I, I, P, P]
        L.mla_debug_mma.restype = I
        L.mla_debug_withhold_value_load.argtypes = [I]
        L.mla_prefill_workspace_size.argtypes = [I, I, I]
        L.mla_prefill_workspace_size.restype = SZ
        L.mla_prefill_paged.argtypes = [P, P, I, P, I, P, I, I, I, P, P, F, I, P, P, P, SZ, P]
        L.mla_prefill_paged.restype = I
        L.mla_rope_append.argtypes = [P, P, P, P, I, P, I, I, I, I, F, P]
        L.mla_rope_append.restype = I
        L.mla_quantize_cache.argtypes = [P, LL, P, P, P]
        L.mla_quantize_cache.restype = I
        L.mla_rope_append_q8.argtypes = [P, P, P, P, I, P, P, I, I, I, I, F, P]
        L.mla_rope_append_q8.restype = I
        L.mla_decode_paged_q8.argtypes = [P, P, P, I, P, I, P, I, I, I, P, P, I, F, I, P, P, P, SZ, P]
        L.mla_decode_paged_q8.restype = I
        _lib = L
        return L


def status_string(status: int) -> str:
    """Human-readable name of a status code (mla_status_string)."""
    try:
        return lib().mla_status_string(int(status)).decode()
    except Exception:
        return f"status {status}"


def _check(call: str, status: int):
    if status != MLA_OK:
        raise MLAError(call, status)


def _p(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype, ndim: Optional[int] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")


# ------------------------------------------------------------------ queries --

def mla_version() -> int:
    """Library ABI version, major * 100 + minor."""
    return int(lib().mla_version())


def mla_schedule_constants() -> Tuple[int, int]:
    """(piece overhead in page-equivalents, minimum pages of a split sequence)
    compiled into the schedule."""
    a, b = ctypes.c_int(), ctypes.c_int()
    lib().mla_schedule_constants(ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def mla_default_num_parts(device: Optional[int] = None, s_q: int = 1) -> int:
    """Schedule parts for `device` (default: the current one): one per pair of
    SMs for each query token, floor(SM count / (2 s_q))."""
    dev = torch.cuda.current_device() if device is None else int(device)
    n = int(lib().mla_default_num_parts(dev, int(s_q)))
    if n <= 0:
        raise MLAError("mla_default_num_parts", -n)
    return n


def mla_workspace_size(B: int, s_q: int, H: int, num_parts: int) -> int:
    """Device workspace bytes mla_decode_paged needs for this shape (0 for bad
    arguments); make_workspace allocates and zero-fills one."""
    return int(lib().mla_workspace_size(int(B), int(s_q), int(H), int(num_parts)))


def mla_set_wait_limit_ns(ns: int):
    """Limit of every bounded wait inside the kernels, in nanoseconds (<= 0
    restores the default of four seconds); a wait that runs out records
    MLA_ERR_TIMEOUT. Process-wide, for launches made afterwards."""
    lib().mla_set_wait_limit_ns(int(ns))


def mla_debug_withhold_value_load(enable: bool):
    """Test hook: later decode launches never issue the value CTA's first page
    load, so a bounded wait runs out (see include/mla.h)."""
    lib().mla_debug_withhold_value_load(int(bool(enable)))


def make_workspace(B: int, s_q: int, H: int, num_parts: int, device=None) -> torch.Tensor:
    """Zero-filled device workspace of mla_workspace_size bytes (256-byte aligned by torch)."""
    n = mla_workspace_size(B, s_q, H, num_parts)
    if n == 0:
        raise MLAError("mla_workspace_size", MLA_ERR_INVALID_ARG)
    return torch.zeros(n, dtype=torch.uint8, device=device if device is not None else "cuda")


# ---------------------------------------------------------------- hot path --

def mla_get_metadata(cache_seqlens: torch.Tensor, s_q: int, H: int, num_parts: Optional[int] = None, h_kv: int = 1,
                     tile_meta: Optional[torch.Tensor] = None, num_splits: Optional[torch.Tensor] = None,
                     stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split/tile schedule of one decode step from cache_seqlens int32 [B]:
    (tile_meta int32 [num_parts, 8], num_splits int32 [B + 1]), computed once per
    step and shared by the layers. See include/mla.h."""
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    B = cache_seqlens.shape[0]
    if num_parts is None:
        num_parts = mla_default_num_parts(cache_seqlens.device.index, s_q)
    if tile_meta is None:
        tile_meta = torch.empty((num_parts, 8), dtype=torch.int32, device=cache_seqlens.device)
    if num_splits is None:
        num_splits = torch.empty((B + 1,), dtype=torch.int32, device=cache_seqlens.device)
    _need(tile_meta, "tile_meta", torch.int32, 2)
    _need(num_splits, "num_splits", torch.int32, 1)
    if tile_meta.shape != (num_parts, 8) or num_splits.shape[0] != B + 1:
        raise ValueError("tile_meta must be [num_parts, 8] and num_splits [B + 1]")
    _check("mla_get_metadata", lib().mla_get_metadata(_p(cache_seqlens), B, int(s_q), int(H), int(h_kv),
                                                      int(num_parts), _p(tile_meta), _p(num_splits), _stream(stream)))
    return tile_meta, num_splits


def mla_absorb_q(q: torch.Tensor, w_uk: torch.Tensor, q_abs: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """q' = [W_UK^T q_nope | q_rope]: q bf16 [B, s_q, H, 192], w_uk bf16
    [H, 128, 512] -> q_abs bf16 [B, s_q, H, 576]. See include/mla.h."""
    _need(q, "q", torch.bfloat16, 4)
    _need(w_uk, "w_uk", torch.bfloat16, 3)
    B, s_q, H, dq = q.shape
    if dq != D_Q or tuple(w_uk.shape) != (H, 128, D_LATENT):
        raise ValueError("q must be [B, s_q, H, 192] and w_uk [H, 128, 512]")
    if q_abs is None:
        q_abs = torch.empty((B, s_q, H, D_QK), dtype=torch.bfloat16, device=q.device)
    _need(q_abs, "q_abs", torch.bfloat16, 4)
    if tuple(q_abs.shape) != (B, s_q, H, D_QK):
        raise ValueError(f"q_abs must be [{B}, {s_q}, {H}, 576]")
    _check("mla_absorb_q", lib().mla_absorb_q(_p(q), _p(w_uk), _p(q_abs), B, s_q, H, _stream(stream)))
    return q_abs


def _check_decode_inputs(q_abs, kv_cache, block_table, cache_seqlens, tile_meta, num_splits, kv_scale=None):
    """dtype, device, contiguity and shape checks shared by the decode entry
    points (the C ABI sees only pointers, so a shape mismatch would make the
    kernels read or write out of bounds). kv_scale given: kv_cache is the INT8
    cache (uint8 [num_blocks, 64, 640], scales fp32 [num_blocks, 64]).
    Returns (B, s_q, H)."""
    _need(q_abs, "q_abs", torch.bfloat16, 4)
    if kv_scale is None:
        _need(kv_cache, "kv_cache", torch.bfloat16, 3)
    else:
        _need(kv_cache, "kv8", torch.uint8, 3)
        _need(kv_scale, "kv_scale", torch.float32, 2)
        if tuple(kv_cache.shape[1:]) != (PAGE, Q8_RECORD) or tuple(kv_scale.shape) != (kv_cache.shape[0], PAGE):
            raise ValueError("kv8 must be [num_blocks, 64, 640] and kv_scale [num_blocks, 64]")
    _need(block_table, "block_table", torch.int32, 2)
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    _need(tile_meta, "tile_meta", torch.int32, 2)
    _need(num_splits, "num_splits", torch.int32, 1)
    B, s_q, H, d = q_abs.shape
    if d != D_QK or (kv_scale is None and tuple(kv_cache.shape[1:]) != (PAGE, D_QK)):
        raise ValueError("q_abs must be [B, s_q, H, 576] and kv_cache [num_blocks, 64, 576]")
    if block_table.shape[0] != B or cache_seqlens.shape[0] != B or num_splits.shape[0] != B + 1:
        raise ValueError("block_table, cache_seqlens and num_splits must match the batch of q_abs")
    if tile_meta.shape[1] != 8:
        raise ValueError("tile_meta must be [num_parts, 8]")
    return B, s_q, H


def _check_decode_outputs(o_lat, lse, B, s_q, H):
    _need(o_lat, "o_lat", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    if tuple(o_lat.shape) != (B, s_q, H, D_LATENT) or tuple(lse.shape) != (B, s_q, H):
        raise ValueError(f"o_lat must be [{B}, {s_q}, {H}, 512] and lse [{B}, {s_q}, {H}]")


def mla_decode_paged(q_abs: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                     cache_seqlens: torch.Tensor, tile_meta: torch.Tensor, num_splits: torch.Tensor,
                     softmax_scale: float, causal: bool = True, o_lat: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Absorbed attention over the paged latent cache: q_abs bf16 [B, s_q, H, 576],
    kv_cache bf16 [num_blocks, 64, 576], block_table int32 [B, max_blocks],
    cache_seqlens int32 [B] and the schedule of mla_get_metadata -> (o_lat bf16
    [B, s_q, H, 512], lse fp32 [B, s_q, H]). See include/mla.h."""
    B, s_q, H = _check_decode_inputs(q_abs, kv_cache, block_table, cache_seqlens, tile_meta, num_splits)
    num_parts = tile_meta.shape[0]
    if o_lat is None:
        o_lat = torch.empty((B, s_q, H, D_LATENT), dtype=torch.bfloat16, device=q_abs.device)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=q_abs.device)
    if workspace is None:
        workspace = make_workspace(B, s_q, H, num_parts, q_abs.device)
    _check_decode_outputs(o_lat, lse, B, s_q, H)
    _need(workspace, "workspace", torch.uint8, 1)
    _check("mla_decode_paged", lib().mla_decode_paged(
        _p(q_abs), _p(kv_cache), kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(cache_seqlens),
        B, s_q, H, _p(tile_meta), _p(num_splits), num_parts, float(softmax_scale), int(bool(causal)),
        _p(o_lat), _p(lse), _p(workspace), workspace.numel(), _stream(stream)))
    return o_lat, lse


def mla_decode_out_proj(q_abs: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                        cache_seqlens: torch.Tensor, tile_meta: torch.Tensor, num_splits: torch.Tensor,
                        softmax_scale: float, causal: bool, w_uv: torch.Tensor, out: Optional[torch.Tensor] = None,
                        lse: Optional[torch.Tensor] = None, o_lat: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """mla_decode_paged followed by the output projection, the split merge and
    the projection fused (w_uv bf16 [H, 512, 128] -> out bf16 [B, s_q, H, 128]).
    o_lat is scratch (rows of unsplit sequences only). See include/mla.h."""
    B, s_q, H = _check_decode_inputs(q_abs, kv_cache, block_table, cache_seqlens, tile_meta, num_splits)
    num_parts = tile_meta.shape[0]
    _need(w_uv, "w_uv", torch.bfloat16, 3)
    if tuple(w_uv.shape) != (H, D_LATENT, D_V) or w_uv.device != q_abs.device:
        raise ValueError(f"w_uv must be [{H}, {D_LATENT}, {D_V}] on the query's device")
    dev = q_abs.device
    if out is None:
        out = torch.empty((B, s_q, H, D_V), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=dev)
    if o_lat is None:
        o_lat = torch.empty((B, s_q, H, D_LATENT), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = make_workspace(B, s_q, H, num_parts, dev)
    _check_decode_outputs(o_lat, lse, B, s_q, H)
    _need(out, "out", torch.bfloat16, 4)
    if tuple(out.shape) != (B, s_q, H, D_V) or out.device != dev:
        raise ValueError(f"out must be [{B}, {s_q}, {H}, {D_V}] on the query's device")
    _need(workspace, "workspace", torch.uint8, 1)
    _check("mla_decode_out_proj", lib().mla_decode_out_proj(
        _p(q_abs), _p(kv_cache), kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(cache_seqlens),
        B, s_q, H, _p(tile_meta), _p(num_splits), num_parts, float(softmax_scale), int(bool(causal)),
        _p(w_uv), _p(o_lat), _p(out), _p(lse), _p(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def mla_decode_paged_q8(q_abs: torch.Tensor, kv8: torch.Tensor, kv_scale: torch.Tensor, block_table: torch.Tensor,
                        cache_seqlens: torch.Tensor, tile_meta: torch.Tensor, num_splits: torch.Tensor,
                        softmax_scale: float, causal: bool = True, o_lat: Optional[torch.Tensor] = None,
                        lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """mla_decode_paged over the INT8 cache (kv8 uint8 [num_blocks, 64, 640],
    kv_scale fp32 [num_blocks, 64]). See include/mla.h."""
    B, s_q, H = _check_decode_inputs(q_abs, kv8, block_table, cache_seqlens, tile_meta, num_splits, kv_scale)
    num_parts = tile_meta.shape[0]
    if o_lat is None:
        o_lat = torch.empty((B, s_q, H, D_LATENT), dtype=torch.bfloat16, device=q_abs.device)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=q_abs.device)
    if workspace is None:
        workspace = make_workspace(B, s_q, H, num_parts, q_abs.device)
    _check_decode_outputs(o_lat, lse, B, s_q, H)
    _need(workspace, "workspace", torch.uint8, 1)
    _check("mla_decode_paged_q8", lib().mla_decode_paged_q8(
        _p(q_abs), _p(kv8), _p(kv_scale), kv8.shape[0], _p(block_table), block_table.shape[1], _p(cache_seqlens),
        B, s_q, H, _p(tile_meta), _p(num_splits), num_parts, float(softmax_scale), int(bool(causal)),
        _p(o_lat), _p(lse), _p(workspace), workspace.numel(), _stream(stream)))
    return o_lat, lse


def mla_quantize_cache(kv: torch.Tensor, kv8: Optional[torch.Tensor] = None, kv_scale: Optional[torch.Tensor] = None,
                       stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """bf16 cache rows kv [..., 576] -> (kv8 uint8 [..., 640], kv_scale fp32 [...]). See include/mla.h."""
    _need(kv, "kv", torch.bfloat16)
    if kv.shape[-1] != D_QK:
        raise ValueError("kv must be [..., 576]")
    lead = tuple(kv.shape[:-1])
    tokens = kv.numel() // D_QK
    if kv8 is None:
        kv8 = torch.empty(lead + (Q8_RECORD,), dtype=torch.uint8, device=kv.device)
    if kv_scale is None:
        kv_scale = torch.empty(lead, dtype=torch.float32, device=kv.device)
    _need(kv8, "kv8", torch.uint8)
    _need(kv_scale, "kv_scale", torch.float32)
    if kv8.numel() != tokens * Q8_RECORD or kv_scale.numel() != tokens:
        raise ValueError("kv8 must hold 640 bytes and kv_scale one float per row of kv")
    _check("mla_quantize_cache", lib().mla_quantize_cache(_p(kv), tokens, _p(kv8), _p(kv_scale), _stream(stream)))
    return kv8, kv_scale


def mla_rope_append_q8(q: torch.Tensor, kv_new: torch.Tensor, cache_seqlens: torch.Tensor, block_table: torch.Tensor,
                       kv8: torch.Tensor, kv_scale: torch.Tensor, rope_base: float = 10000.0, stream=None):
    """mla_rope_append into the INT8 cache (q's rope parts rotated in place; the
    new tokens' records and scales written). See include/mla.h."""
    _need(q, "q", torch.bfloat16, 4)
    _need(kv_new, "kv_new", torch.bfloat16, 3)
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    _need(kv8, "kv8", torch.uint8, 3)
    _need(kv_scale, "kv_scale", torch.float32, 2)
    B, s_q, H, dq = q.shape
    if dq != D_Q or tuple(kv_new.shape) != (B, s_q, D_QK) or tuple(kv8.shape[1:]) != (PAGE, Q8_RECORD):
        raise ValueError("q must be [B, s_q, H, 192], kv_new [B, s_q, 576] and kv8 [num_blocks, 64, 640]")
    if tuple(kv_scale.shape) != (kv8.shape[0], PAGE):
        raise ValueError("kv_scale must be [num_blocks, 64]")
    if block_table.shape[0] != B or cache_seqlens.shape[0] != B:
        raise ValueError("block_table and cache_seqlens must match the batch of q")
    _check("mla_rope_append_q8", lib().mla_rope_append_q8(
        _p(q), _p(kv_new), _p(cache_seqlens), _p(block_table), block_table.shape[1], _p(kv8), _p(kv_scale),
        kv8.shape[0], B, s_q, H, float(rope_base), _stream(stream)))


def mla_out_proj(o_lat: torch.Tensor, w_uv: torch.Tensor, out: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """out = W_UV^T o_lat per head: o_lat bf16 [B, s_q, H, 512], w_uv bf16
    [H, 512, 128] -> out bf16 [B, s_q, H, 128]. See include/mla.h."""
    _need(o_lat, "o_lat", torch.bfloat16, 4)
    _need(w_uv, "w_uv", torch.bfloat16, 3)
    B, s_q, H, d = o_lat.shape
    if d != D_LATENT or tuple(w_uv.shape) != (H, D_LATENT, D_V):
        raise ValueError("o_lat must be [B, s_q, H, 512] and w_uv [H, 512, 128]")
    if out is None:
        out = torch.empty((B, s_q, H, D_V), dtype=torch.bfloat16, device=o_lat.device)
    _need(out, "out", torch.bfloat16, 4)
    if tuple(out.shape) != (B, s_q, H, D_V):
        raise ValueError(f"out must be [{B}, {s_q}, {H}, 128]")
    _check("mla_out_proj", lib().mla_out_proj(_p(o_lat), _p(w_uv), _p(out), B, s_q, H, _stream(stream)))
    return out


def mla_read_device_error(workspace: Optional[torch.Tensor] = None, stream=None) -> int:
    """Device-recorded status since the last read (synchronises the stream):
    the workspace's error word (if given) and the library's own word."""
    return int(lib().mla_read_device_error(_p(workspace), _stream(stream)))


def mla_rope_append(q: torch.Tensor, kv_new: torch.Tensor, cache_seqlens: torch.Tensor, block_table: torch.Tensor,
                    kv_cache: torch.Tensor, rope_base: float = 10000.0, stream=None) -> None:
    """Rotary-encodes the rope part of q [B, s_q, H, 192] in place and writes
    each new token [c_KV | RoPE(k_rope)] from kv_new [B, s_q, 576] into its
    cache slot (position cache_seqlens[b] - s_q + s). See include/mla.h."""
    _need(q, "q", torch.bfloat16, 4)
    _need(kv_new, "kv_new", torch.bfloat16, 3)
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    _need(kv_cache, "kv_cache", torch.bfloat16, 3)
    B, s_q, H, dq = q.shape
    if dq != D_Q or tuple(kv_new.shape) != (B, s_q, D_QK) or tuple(kv_cache.shape[1:]) != (PAGE, D_QK):
        raise ValueError("q must be [B, s_q, H, 192], kv_new [B, s_q, 576] and kv_cache [num_blocks, 64, 576]")
    if cache_seqlens.shape[0] != B or block_table.shape[0] != B:
        raise ValueError("cache_seqlens and block_table must match the batch of q")
    _check("mla_rope_append", lib().mla_rope_append(_p(q), _p(kv_new), _p(cache_seqlens), _p(block_table),
                                                    block_table.shape[1], _p(kv_cache), kv_cache.shape[0], B, s_q, H,
                                                    float(rope_base), _stream(stream)))


# -------------------------------------------------------------- test hooks --

def mla_debug_gather(kv_cache: torch.Tensor, block_table: torch.Tensor, cache_seqlens: torch.Tensor,
                     max_tokens: int, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Test hook: rows t < min(seqlen_b, max_tokens) of each sequence b, gathered
    through the block table by TMA into out bf16 [B, max_tokens, 576] (other rows
    untouched; zeros when out is allocated here). Bit-exact copy."""
    _need(kv_cache, "kv_cache", torch.bfloat16, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    B = block_table.shape[0]
    if out is None:
        out = torch.zeros((B, max_tokens, D_QK), dtype=torch.bfloat16, device=kv_cache.device)
    _check("mla_debug_gather", lib().mla_debug_gather(_p(kv_cache), kv_cache.shape[0], _p(block_table),
                                                      block_table.shape[1], _p(cache_seqlens), B, int(max_tokens),
                                                      _p(out), _stream(stream)))
    return out


def mla_debug_mma(a: torch.Tensor, b: torch.Tensor, b_kmajor: bool, a_tmem: int = 0,
                  stream=None) -> torch.Tensor:
    """a [128, K]; b [N, K] if b_kmajor else [K, N]; returns fp32 [128, N] = a . B
    (A from shared memory for a_tmem = 0, from tensor memory written by thread
    stores for 1, or copied in by tcgen05.cp for 2)."""
    _need(a, "a", torch.bfloat16, 2)
    _need(b, "b", torch.bfloat16, 2)
    K = a.shape[1]
    N = b.shape[0] if b_kmajor else b.shape[1]
    d = torch.empty((128, N), dtype=torch.float32, device=a.device)
    _check("mla_debug_mma", lib().mla_debug_mma(_p(a), _p(b), K, N, int(bool(b_kmajor)), int(a_tmem), _p(d),
                                                _stream(stream)))
    return d


# ------------------------------------------------------------- convenience --

def decode_step(inputs, num_parts: Optional[int] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """One pass of the path on device-resident inputs (an inputs.MLAInputs on cuda):
    metadata -> absorb (when q is given) -> decode (+ combine) -> out-projection.
    Returns dict(o_lat, lse, out, q_abs, tile_meta, num_splits)."""
    s_q, H = inputs.s_q, inputs.H
    tm, ns = mla_get_metadata(inputs.seqlens, s_q, H, num_parts, stream=stream)
    q_abs = inputs.q_abs if inputs.q is None else mla_absorb_q(inputs.q, inputs.w_uk, stream=stream)
    o_lat, lse = mla_decode_paged(q_abs, inputs.kv_cache, inputs.block_table, inputs.seqlens, tm, ns, inputs.scale,
                                  inputs.causal, workspace=workspace, stream=stream)
    out = mla_out_proj(o_lat, inputs.w_uv, stream=stream) if inputs.w_uv is not None else None
    return {"o_lat": o_lat, "lse": lse, "out": out, "q_abs": q_abs, "tile_meta": tm, "num_splits": ns}


# ------------------------------------------------------- no-allocation entry --

def mla_decode_paged_noalloc(q_abs: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                             cache_seqlens: torch.Tensor, tile_meta: torch.Tensor, num_splits: torch.Tensor,
                             softmax_scale: float, causal: bool, o_lat: torch.Tensor, lse: torch.Tensor,
                             device_status: Optional[torch.Tensor] = None, stream=None):
    """mla_decode_paged for callers that must not allocate device memory: the
    scratch comes from an array inside the library, the caller passes every
    input and output (this wrapper allocates nothing either). See include/mla.h."""
    L = lib()
    fn = L.mla_decode_paged_noalloc
    if fn.restype is not ctypes.c_int or fn.argtypes is None:
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fn.argtypes = [P, P, I, P, I, P, I, I, I, P, P, I, F, I, P, P, P, P]
        fn.restype = I
    B, s_q, H = _check_decode_inputs(q_abs, kv_cache, block_table, cache_seqlens, tile_meta, num_splits)
    _check_decode_outputs(o_lat, lse, B, s_q, H)
    if device_status is not None:
        _need(device_status, "device_status", torch.int32)
    _check("mla_decode_paged_noalloc", fn(
        _p(q_abs), _p(kv_cache), kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(cache_seqlens),
        B, s_q, H, _p(tile_meta), _p(num_splits), tile_meta.shape[0], float(softmax_scale), int(bool(causal)),
        _p(o_lat), _p(lse), _p(device_status), _stream(stream)))
    return o_lat, lse


# ------------------------------------------------------------------ prefill --

def mla_prefill_workspace_size(B: int, H: int, max_blocks_per_seq: int) -> int:
    """Device workspace bytes mla_prefill_paged needs (gathered latent and the
    decompressed K and V, padded to max_blocks_per_seq pages)."""
    return int(lib().mla_prefill_workspace_size(int(B), int(H), int(max_blocks_per_seq)))


def mla_prefill_paged(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor, cache_seqlens: torch.Tensor,
                      w_uk: torch.Tensor, w_uv: torch.Tensor, softmax_scale: float, causal: bool = True,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Prefill in the naive form over the paged cache: q [B, s_q, H, 192] (the
    last s_q positions of each sequence) -> (out [B, s_q, H, 128], lse [B, s_q, H]).
    See include/mla.h."""
    _need(q, "q", torch.bfloat16, 4)
    _need(kv_cache, "kv_cache", torch.bfloat16, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    _need(w_uk, "w_uk", torch.bfloat16, 3)
    _need(w_uv, "w_uv", torch.bfloat16, 3)
    B, s_q, H, dq = q.shape
    if dq != D_Q or tuple(kv_cache.shape[1:]) != (PAGE, D_QK):
        raise ValueError("q must be [B, s_q, H, 192] and kv_cache [num_blocks, 64, 576]")
    if tuple(w_uk.shape) != (H, 128, D_LATENT) or tuple(w_uv.shape) != (H, D_LATENT, D_V):
        raise ValueError("w_uk must be [H, 128, 512] and w_uv [H, 512, 128]")
    if block_table.shape[0] != B or cache_seqlens.shape[0] != B:
        raise ValueError("block_table and cache_seqlens must match the batch of q")
    mbps = block_table.shape[1]
    if out is None:
        out = torch.empty((B, s_q, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    if tuple(out.shape) != (B, s_q, H, D_V) or tuple(lse.shape) != (B, s_q, H):
        raise ValueError(f"out must be [{B}, {s_q}, {H}, 128] and lse [{B}, {s_q}, {H}]")
    if workspace is None:
        n = mla_prefill_workspace_size(B, H, mbps)
        if n == 0:
            raise MLAError("mla_prefill_workspace_size", MLA_ERR_INVALID_ARG)
        workspace = torch.empty(n + 1024, dtype=torch.uint8, device=q.device)
        off = (-workspace.data_ptr()) % 1024
        workspace = workspace[off:off + n]
    _need(workspace, "workspace", torch.uint8, 1)
    _check("mla_prefill_paged", lib().mla_prefill_paged(
        _p(q), _p(kv_cache), kv_cache.shape[0], _p(block_table), mbps, _p(cache_seqlens), B, s_q, H, _p(w_uk),
        _p(w_uv), float(softmax_scale), int(bool(causal)), _p(out), _p(lse), _p(workspace), workspace.numel(),
        _stream(stream)))
    return out, lse

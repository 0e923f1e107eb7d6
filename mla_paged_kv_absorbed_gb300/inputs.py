"""Seeded synthetic inputs for paged MLA decode.

This module draws random tensors and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle may consume what
it produces.

Recipe (one ``torch.Generator('cpu')`` per call, seeded with ``seed``):
  * q [B, s_q, H, 192] = [q_nope 128 | q_rope 64] ~ N(0, 1) -> bf16 (RNE);
    the decode-only workloads draw q_abs [B, s_q, H, 576] ~ N(0, 1) directly.
  * W_UK [H, 128, 512] and W_UV [H, 512, 128] ~ N(0, 1/512) -> bf16.
  * Every visible cache row [c_KV 512 | k_rope 64] ~ N(0, 1) -> bf16.
  * Pages: pool = sum of pages + ceil(10 %) decoy blocks; physical blocks are
    a random permutation of the pool. Decoy blocks and the rows past seqlen in
    each last page hold finite garbage, N(0, 1) x 1e4 -> bf16.
  * Block-table entries past a sequence's last page are -1.

Workloads named after what they are (DeepSeek-V3 decode shapes: 128 heads,
d_c = 512, rope 64, 64-token bf16 pages, softmax scale 1/sqrt(192)):
  tiny      B=2,   s_q=1, H=16,  seqlens {37, 100}
  dsv3      B=128, s_q=1, H=128, seqlen 512
  varlen    B=64,  s_q=1, H=128, seqlen ~ U[129, 1152]      (q_abs drawn directly)
  long      B=16,  s_q=1, H=128, seqlen ~ U[16384, 32768]   (q_abs drawn directly)
  spec      B=132, s_q=2, H=128, seqlen 4096, causal        (end to end)
  prefill   B=8, whole prompts of 2048 tokens (s_q = seqlen = 2048), H=128,
            causal; for the naive-form prefill over the same paged cache
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

PAGE = 64
D_LATENT = 512
D_ROPE = 64
D_QK = 576
D_NOPE = 128
D_Q = 192
D_V = 128
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)

WORKLOADS = {
    "tiny": dict(B=2, s_q=1, H=16, seqlens=[37, 100], q_mode="q", causal=True),
    "dsv3": dict(B=128, s_q=1, H=128, seqlens=512, q_mode="q", causal=True),
    "varlen": dict(B=64, s_q=1, H=128, seqlens=(129, 1152), q_mode="q_abs", causal=True),
    "long": dict(B=16, s_q=1, H=128, seqlens=(16384, 32768), q_mode="q_abs", causal=True),
    "spec": dict(B=132, s_q=2, H=128, seqlens=4096, q_mode="q", causal=True),
    "prefill": dict(B=8, s_q=2048, H=128, seqlens=2048, q_mode="q", causal=True),
}
WORKLOAD_ORDER = ["tiny", "dsv3", "varlen", "long", "spec", "prefill"]


@dataclass
class MLAInputs:
    B: int
    s_q: int
    H: int
    scale: float
    causal: bool
    seqlens: torch.Tensor            # int32 [B]
    block_table: torch.Tensor        # int32 [B, max_blocks_per_seq]
    kv_cache: torch.Tensor           # bf16 [num_blocks, 64, 576]
    q: Optional[torch.Tensor]        # bf16 [B, s_q, H, 192] (None when q_abs is drawn directly)
    q_abs: Optional[torch.Tensor]    # bf16 [B, s_q, H, 576] (None when q is drawn)
    w_uk: Optional[torch.Tensor]     # bf16 [H, 128, 512]
    w_uv: Optional[torch.Tensor]     # bf16 [H, 512, 128]
    seed: int = 0
    name: str = "custom"
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def kv_bytes(self) -> int:
        """Latent-cache bytes a decode call must read: sum of seqlen x 576 x 2."""
        return int(self.seqlens.clamp(min=0).sum().item()) * D_QK * 2

    def to(self, device) -> "MLAInputs":
        def mv(t):
            return None if t is None else t.to(device)
        return MLAInputs(self.B, self.s_q, self.H, self.scale, self.causal, mv(self.seqlens), mv(self.block_table),
                         mv(self.kv_cache), mv(self.q), mv(self.q_abs), mv(self.w_uk), mv(self.w_uv), self.seed,
                         self.name, dict(self.meta))


def _randn(g, shape, std=1.0):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def _garbage(g, shape, amp=1.0e4):
    # normal rather than uniform: torch.rand with a generator is several times
    # slower, and only the magnitude matters (finite values far from the data)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * amp).to(torch.bfloat16)


def make_inputs(B: int, s_q: int, H: int, seqlens, seed: int, *, q_mode: str = "q", causal: bool = True,
                scale: float = DEFAULT_SCALE, decoy_frac: float = 0.10, garbage: bool = True,
                max_blocks_per_seq: Optional[int] = None, name: str = "custom",
                tail_fill: Optional[float] = None, weights: bool = True) -> MLAInputs:
    """Draw one workload.

    seqlens: an int (all equal), a (lo, hi) tuple (uniform integers, inclusive), or
    a list of B ints. q_mode: "q" draws q [B, s_q, H, 192] (and the weights);
    "q_abs" draws the absorbed query [B, s_q, H, 576] directly. tail_fill
    replaces the garbage of the rows past seqlen by a constant (e.g. nan).
    """
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    if isinstance(seqlens, int):
        sl = torch.full((B,), seqlens, dtype=torch.int32)
    elif isinstance(seqlens, tuple):
        lo, hi = seqlens
        sl = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32)
    else:
        sl = torch.tensor(list(seqlens), dtype=torch.int32)
        assert sl.numel() == B
    nblk = [(max(int(s), 0) + PAGE - 1) // PAGE for s in sl.tolist()]
    used = sum(nblk)
    pool = used + int(math.ceil(decoy_frac * used)) if decoy_frac > 0 else used
    pool = max(pool, 1)
    mbps = max_blocks_per_seq if max_blocks_per_seq is not None else max(max(nblk) if nblk else 1, 1)
    assert mbps >= max(nblk + [0])
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    table = torch.full((B, mbps), -1, dtype=torch.int32)
    if garbage:
        # every block is overwritten below except the decoys: draw garbage for those only
        kv = torch.empty((pool, PAGE, D_QK), dtype=torch.bfloat16)
        decoys = perm[used:].long()
        if decoys.numel():
            kv[decoys] = _garbage(g, (decoys.numel(), PAGE, D_QK))
    else:
        kv = torch.zeros((pool, PAGE, D_QK), dtype=torch.bfloat16)
    k = 0
    for b in range(B):
        n = nblk[b]
        if n == 0:
            continue
        blocks = perm[k:k + n]
        k += n
        table[b, :n] = blocks
        L = int(sl[b])
        vals = _randn(g, (n * PAGE, D_QK))
        vals = vals.view(n, PAGE, D_QK)
        tail = n * PAGE - L
        if tail > 0:
            # rows past seqlen hold garbage (or the requested fill)
            if tail_fill is not None:
                vals[-1, PAGE - tail:] = tail_fill
            elif garbage:
                vals[-1, PAGE - tail:] = _garbage(g, (tail, D_QK))
            else:
                vals[-1, PAGE - tail:] = 0
        kv[blocks.long()] = vals
    q = q_abs = w_uk = w_uv = None
    if q_mode == "q":
        q = _randn(g, (B, s_q, H, D_Q))
        if weights:
            w_uk = _randn(g, (H, D_NOPE, D_LATENT), std=1.0 / math.sqrt(D_LATENT))
            w_uv = _randn(g, (H, D_LATENT, D_V), std=1.0 / math.sqrt(D_LATENT))
    elif q_mode == "q_abs":
        q_abs = _randn(g, (B, s_q, H, D_QK))
    else:
        raise ValueError(q_mode)
    return MLAInputs(B, s_q, H, float(scale), bool(causal), sl, table, kv, q, q_abs, w_uk, w_uv, int(seed), name,
                     {"pool": pool, "used_blocks": used})


def draw_w_uv(H: int, seed: int) -> torch.Tensor:
    """A seeded W_UV [H, 512, 128] (bf16, N(0, 1/512)) for workloads drawn with
    the absorbed query directly, which carry no weights."""
    g = torch.Generator("cpu")
    g.manual_seed(int(seed) + 7919)
    return _randn(g, (H, D_LATENT, D_V), std=1.0 / math.sqrt(D_LATENT))


def workload_seed(name: str, rep: int = 0) -> int:
    """seed = 1000 x (1-based workload index) + rep."""
    return 1000 * (WORKLOAD_ORDER.index(name) + 1) + int(rep)


def make_workload(name: str, rep: int = 0, **overrides) -> MLAInputs:
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    seqlens = cfg.pop("seqlens")
    B = cfg.pop("B")
    s_q = cfg.pop("s_q")
    H = cfg.pop("H")
    if isinstance(seqlens, list):
        seqlens = list(seqlens)
    return make_inputs(B, s_q, H, seqlens, workload_seed(name, rep), name=name, **cfg)


def sample_batches(inp: MLAInputs, batches: Sequence[int]) -> MLAInputs:
    """The sub-workload of the listed sequences, with a compact page pool.

    The returned cache holds only the pages those sequences use (in the same
    order as their table rows), so the oracle can evaluate them one by one at
    full sequence length without touching the whole pool.
    """
    idx = torch.tensor(list(batches), dtype=torch.long)
    sl = inp.seqlens[idx].clone()
    nblk = [(max(int(s), 0) + PAGE - 1) // PAGE for s in sl.tolist()]
    mbps = max(max(nblk) if nblk else 1, 1)
    table = torch.full((len(batches), mbps), -1, dtype=torch.int32)
    pages = []
    k = 0
    for i, b in enumerate(batches):
        n = nblk[i]
        if n:
            pages.append(inp.kv_cache[inp.block_table[b, :n].long()])
            table[i, :n] = torch.arange(k, k + n, dtype=torch.int32)
            k += n
    kv = torch.cat(pages, 0) if pages else torch.zeros((1, PAGE, D_QK), dtype=torch.bfloat16)

    def sel(t):
        return None if t is None else t[idx].clone()
    return MLAInputs(len(batches), inp.s_q, inp.H, inp.scale, inp.causal, sl, table, kv, sel(inp.q), sel(inp.q_abs),
                     inp.w_uk, inp.w_uv, inp.seed, inp.name + "[sample]", {"batches": list(batches)})

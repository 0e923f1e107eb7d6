"""Pins for the CPU oracle: checks against what the pages and plain mathematics
fix, never against the oracle's own formula retyped.

Pins used (each chosen so that a plausible mistake fails one of them):
  * absorption identity q^T (W_UK c) = (W_UK^T q)^T c between the naive
    (decompress) and absorbed forms ("DeepSeek-V3 MLA deep engineering",
    sec. 2.4) - catches a transposed W_UK, a dropped rope term in one form, a
    wrong W_UV orientation;
  * a fp64 brute force of the naive form built from numpy matmuls and an
    explicit mask (tiny shapes) - catches scale, sign and mask errors;
  * a textbook single-head case against scipy.special.softmax;
  * closed forms: constant latent rows give o = 1 (rows of p sum to 1);
    one key gives o = c_0 and lse = score_0; identical keys give the mean
    and lse = s + ln n; a hand-derived two-key example (tests/golden);
  * exp(lse) = sum exp(score) against scipy.special.logsumexp;
  * invariances: physical page permutation (bit-identical); causal row s of
    s_q equals a single-query decode on the first seqlen - s_q + s + 1 keys;
  * the pages' streaming recurrence ("DeepSeek-V3 MLA deep engineering",
    sec. 4.1) equals the two-pass softmax; every split schedule equals the
    single pass; the combine weights of a closed-form example;
  * schedule: hand-derived examples (tests/golden) and invariants.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from mla_paged_kv_absorbed_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SCALE = 1.0 / math.sqrt(192.0)


def f32(t):
    return t.float().numpy()


def small(B=2, s_q=1, H=4, seqlens=(65, 130), seed=7, q_mode="q", **kw):
    return gen.make_inputs(B, s_q, H, list(seqlens) if not isinstance(seqlens, int) else seqlens, seed,
                           q_mode=q_mode, **kw)


def gather_keys(kv, table_row, n):
    """Rows of the logical sequence through its block table (a plain gather)."""
    idx = [int(table_row[t // 64]) * 64 + t % 64 for t in range(n)]
    flat = kv.reshape(-1, kv.shape[-1])
    return flat[idx]


def brute_naive(q, kv, table, seqlens, w_uk, w_uv, scale, causal):
    """fp64 naive form: decompress K and V per head with numpy matmuls, explicit
    causal mask matrix, softmax with explicit exp; independent of the C code."""
    q = q.astype(np.float64)
    kv = kv.astype(np.float64)
    w_uk = w_uk.astype(np.float64)
    w_uv = w_uv.astype(np.float64)
    B, s_q, H, _ = q.shape
    out = np.zeros((B, s_q, H, 128))
    lse = np.full((B, s_q, H), -np.inf)
    for b in range(B):
        L = int(seqlens[b])
        if L <= 0:
            continue
        C = gather_keys(kv, table[b], L)                # [L, 576]
        for h in range(H):
            K = np.concatenate([C[:, :512] @ w_uk[h].T, C[:, 512:]], axis=1)   # [L, 192]
            V = C[:, :512] @ w_uv[h]                                          # [L, 128]
            S = (q[b, :, h, :] @ K.T) * scale                                # [s_q, L]
            # bottom-right aligned lower-triangular mask
            mask = np.ones((s_q, L), bool)
            if causal:
                for s in range(s_q):
                    for t in range(L):
                        mask[s, t] = t <= L - s_q + s
            for s in range(s_q):
                if not mask[s].any():
                    continue
                sc = S[s][mask[s]]
                mx = sc.max()
                e = np.exp(sc - mx)
                out[b, s, h] = (e[:, None] * V[mask[s]]).sum(0) / e.sum()
                lse[b, s, h] = mx + math.log(e.sum())
    return out, lse


def absorbed_chain(inp, causal=None):
    causal = inp.causal if causal is None else causal
    qa = oracle.absorb_q(f32(inp.q), f32(inp.w_uk))
    o, lse = oracle.attend_absorbed(qa, f32(inp.kv_cache), inp.block_table, inp.seqlens, inp.scale, causal)
    return oracle.out_proj(o, f32(inp.w_uv)), lse, o


def relmax(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


# ----------------------------------------------------------------- identity --

@pytest.mark.parametrize("s_q,seqlens", [(1, (1, 65, 130)), (2, (2, 64, 129)), (2, (1, 3, 200))])
def test_absorption_identity_naive_equals_absorbed(s_q, seqlens):
    inp = small(B=len(seqlens), s_q=s_q, H=3, seqlens=seqlens, seed=11)
    out_n, lse_n = oracle.attend_naive(f32(inp.q), f32(inp.kv_cache), inp.block_table, inp.seqlens,
                                       f32(inp.w_uk), f32(inp.w_uv), inp.scale, True)
    out_a, lse_a, _ = absorbed_chain(inp)
    fin = np.isfinite(lse_n)
    assert np.array_equal(fin, np.isfinite(lse_a))
    assert relmax(out_a, out_n) <= 1e-5
    assert np.abs(lse_a[fin] - lse_n[fin]).max() <= 1e-9


@pytest.mark.parametrize("s_q,causal", [(1, True), (2, True), (2, False)])
def test_bruteforce_fp64_tiny(s_q, causal):
    inp = small(B=3, s_q=s_q, H=2, seqlens=(1, 63, 129), seed=21)
    ref_out, ref_lse = brute_naive(f32(inp.q), f32(inp.kv_cache), inp.block_table.numpy(), inp.seqlens.numpy(),
                                   f32(inp.w_uk), f32(inp.w_uv), inp.scale, causal)
    out_n, lse_n = oracle.attend_naive(f32(inp.q), f32(inp.kv_cache), inp.block_table, inp.seqlens,
                                       f32(inp.w_uk), f32(inp.w_uv), inp.scale, causal)
    out_a, lse_a, _ = absorbed_chain(inp, causal)
    for out, lse in ((out_n, lse_n), (out_a, lse_a)):
        assert relmax(out, ref_out) <= 1e-10
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-10


def test_bruteforce_tiny_workload_in_full():
    inp = gen.make_workload("tiny")
    ref_out, ref_lse = brute_naive(f32(inp.q), f32(inp.kv_cache), inp.block_table.numpy(), inp.seqlens.numpy(),
                                   f32(inp.w_uk), f32(inp.w_uv), inp.scale, True)
    out_a, lse_a, _ = absorbed_chain(inp)
    assert relmax(out_a, ref_out) <= 1e-10
    assert np.abs(lse_a - ref_lse).max() <= 1e-10


# ------------------------------------------------------------ closed forms --

def test_textbook_single_head_contiguous_pages():
    """H = 1, s_q = 1, identity block table: ordinary softmax(Q K^T * scale) V."""
    inp = small(B=1, s_q=1, H=1, seqlens=(150,), seed=5, q_mode="q_abs", decoy_frac=0.0)
    n = int(inp.seqlens[0])
    # rebuild the cache so that logical page j is physical block j
    kv_logical = gather_keys(f32(inp.kv_cache), inp.block_table[0].numpy(), n)
    pages = (n + 63) // 64
    kv = np.zeros((pages, 64, 576), np.float32)
    kv.reshape(-1, 576)[:n] = kv_logical
    table = np.arange(pages, dtype=np.int32)[None]
    qa = f32(inp.q_abs).astype(np.float64)
    o, lse = oracle.attend_absorbed(qa, kv, table, inp.seqlens, inp.scale, True)
    K = kv_logical.astype(np.float64)
    scores = (K @ qa[0, 0, 0]) * inp.scale
    p = scipy.special.softmax(scores)
    assert np.abs(o[0, 0, 0] - p @ K[:, :512]).max() <= 1e-12
    assert abs(lse[0, 0, 0] - scipy.special.logsumexp(scores)) <= 1e-12


def test_constant_latent_rows_give_ones():
    """If every visible c_KV row is all ones, o = sum_t p_t * 1 = 1 iff p sums to 1."""
    inp = small(B=2, s_q=2, H=5, seqlens=(70, 191), seed=9, q_mode="q_abs")
    kv = f32(inp.kv_cache).copy()
    for b in range(inp.B):
        n = int(inp.seqlens[b])
        for t in range(n):
            blk = int(inp.block_table[b, t // 64])
            kv[blk, t % 64, :512] = 1.0
    o, lse = oracle.attend_absorbed(f32(inp.q_abs), kv, inp.block_table, inp.seqlens, inp.scale, True)
    assert np.abs(o - 1.0).max() <= 1e-12


def test_lse_is_logsumexp_of_scores():
    inp = small(B=2, s_q=1, H=3, seqlens=(33, 257), seed=13, q_mode="q_abs")
    kv = f32(inp.kv_cache)
    qa = f32(inp.q_abs).astype(np.float64)
    _, lse = oracle.attend_absorbed(qa, kv, inp.block_table, inp.seqlens, inp.scale, True)
    for b in range(inp.B):
        K = gather_keys(kv, inp.block_table[b].numpy(), int(inp.seqlens[b])).astype(np.float64)
        for h in range(inp.H):
            s = (K @ qa[b, 0, h]) * inp.scale
            assert abs(lse[b, 0, h] - scipy.special.logsumexp(s)) <= 1e-12


def test_single_key_returns_its_latent():
    inp = small(B=3, s_q=1, H=4, seqlens=(1, 1, 1), seed=17, q_mode="q_abs")
    kv = f32(inp.kv_cache)
    qa = f32(inp.q_abs).astype(np.float64)
    o, lse = oracle.attend_absorbed(qa, kv, inp.block_table, inp.seqlens, inp.scale, True)
    for b in range(3):
        c0 = kv[int(inp.block_table[b, 0]), 0].astype(np.float64)
        for h in range(4):
            assert np.array_equal(o[b, 0, h], c0[:512])
            assert abs(lse[b, 0, h] - inp.scale * float(qa[b, 0, h] @ c0)) <= 1e-12


def test_identical_keys_give_mean_and_log_n():
    inp = small(B=1, s_q=1, H=2, seqlens=(77,), seed=19, q_mode="q_abs")
    kv = f32(inp.kv_cache).copy()
    row = np.random.default_rng(0).standard_normal(576).astype(np.float32)
    for t in range(77):
        kv[int(inp.block_table[0, t // 64]), t % 64] = row
    qa = f32(inp.q_abs).astype(np.float64)
    o, lse = oracle.attend_absorbed(qa, kv, inp.block_table, inp.seqlens, inp.scale, True)
    for h in range(2):
        s = inp.scale * float(qa[0, 0, h] @ row.astype(np.float64))
        assert np.abs(o[0, 0, h] - row[:512]).max() <= 1e-12
        assert abs(lse[0, 0, h] - (s + math.log(77))) <= 1e-12


def _read_golden_kv(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = [x.strip() for x in line.split("=", 1)]
            vals[k] = v
    return vals


def _num(s):
    named = {"ln2": math.log(2.0), "ln3": math.log(3.0), "2/3": 2.0 / 3.0}
    return named[s] if s in named else float(s)


def test_golden_two_keys():
    g = _read_golden_kv(os.path.join(GOLDEN, "two_keys_attention.txt"))
    kv = np.zeros((2, 64, 576), np.float32)
    for t, key in enumerate(("key0", "key1")):
        for item in g[key].split():
            d, v = item.split(":")
            kv[1, t, int(d)] = float(v)
    qa = np.zeros((1, 1, 1, 576))
    qa[0, 0, 0, 0] = float(g["q_abs_dim0"])
    table = np.array([[1]], np.int32)
    seqlens = np.array([int(g["seqlen"])], np.int32)
    o, lse = oracle.attend_absorbed(qa, kv, table, seqlens, _num(g["scale"]), True)
    assert abs(o[0, 0, 0, 0] - _num(g["expect_o0"])) <= 1e-12
    assert abs(o[0, 0, 0, 1] - _num(g["expect_o1"])) <= 1e-12
    assert np.abs(o[0, 0, 0, 2:]).max() == _num(g["expect_o_rest"])
    assert abs(lse[0, 0, 0] - _num(g["expect_lse"])) <= 1e-12


def test_combine_closed_form():
    o1 = np.full((1, 512), 2.0)
    o2 = np.full((1, 512), -1.0)
    # lse = (ln 1, ln 3): weights 1/4 and 3/4, total lse ln 4
    o, lse = oracle.combine(np.concatenate([o1, o2]), np.array([0.0, math.log(3.0)]))
    assert abs(lse - math.log(4.0)) <= 1e-15
    assert np.abs(o - (0.25 * 2.0 + 0.75 * -1.0)).max() <= 1e-15
    o, lse = oracle.combine(np.zeros((2, 512)) + 5.0, np.array([-np.inf, 1.5]))
    assert lse == 1.5 and np.abs(o - 5.0).max() == 0.0
    o, lse = oracle.combine(np.ones((2, 512)), np.array([-np.inf, -np.inf]))
    assert lse == -np.inf and np.abs(o).max() == 0.0


# ------------------------------------------------------------- invariances --

def test_page_permutation_invariance_bit_identical():
    inp = small(B=3, s_q=2, H=4, seqlens=(64, 100, 300), seed=23, q_mode="q_abs")
    kv = f32(inp.kv_cache)
    o1, l1 = oracle.attend_absorbed(f32(inp.q_abs), kv, inp.block_table, inp.seqlens, inp.scale, True)
    rng = np.random.default_rng(1)
    perm = rng.permutation(kv.shape[0])           # new position of old block i is perm[i]
    kv2 = np.empty_like(kv)
    kv2[perm] = kv
    table = inp.block_table.numpy().copy()
    valid = table >= 0
    table[valid] = perm[table[valid]]
    o2, l2 = oracle.attend_absorbed(f32(inp.q_abs), kv2, table, inp.seqlens, inp.scale, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_causal_row_equals_shorter_decode():
    inp = small(B=2, s_q=2, H=3, seqlens=(65, 129), seed=29, q_mode="q_abs")
    kv = f32(inp.kv_cache)
    qa = f32(inp.q_abs).astype(np.float64)
    o, lse = oracle.attend_absorbed(qa, kv, inp.block_table, inp.seqlens, inp.scale, True)
    for s in range(2):
        sl = inp.seqlens.numpy() - 2 + s + 1
        o1, l1 = oracle.attend_absorbed(qa[:, s:s + 1], kv, inp.block_table, sl, inp.scale, True)
        assert np.abs(o1[:, 0] - o[:, s]).max() <= 1e-13
        assert np.abs(l1[:, 0] - lse[:, s]).max() <= 1e-13


def test_empty_and_fully_masked_rows():
    inp = small(B=3, s_q=2, H=2, seqlens=(0, 1, 5), seed=31, q_mode="q_abs")
    o, lse = oracle.attend_absorbed(f32(inp.q_abs), f32(inp.kv_cache), inp.block_table, inp.seqlens, inp.scale, True)
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf)        # seqlen 0
    assert np.all(o[1, 0] == 0) and np.all(lse[1, 0] == -np.inf)  # query 0 of 2 sees no key
    assert np.all(np.isfinite(lse[1, 1])) and np.all(np.isfinite(lse[2]))


def test_streaming_recurrence_equals_two_pass():
    inp = small(B=2, s_q=2, H=3, seqlens=(1, 300), seed=37, q_mode="q_abs")
    args = (f32(inp.q_abs), f32(inp.kv_cache), inp.block_table, inp.seqlens, inp.scale, True)
    o1, l1 = oracle.attend_absorbed(*args)
    o2, l2 = oracle.attend_streaming(*args)
    assert np.abs(o1 - o2).max() <= 1e-12
    fin = np.isfinite(l1)
    assert np.array_equal(fin, np.isfinite(l2))
    assert np.abs(l1[fin] - l2[fin]).max() <= 1e-12


@pytest.mark.parametrize("num_parts,ovh,min_split", [(1, 7, 32), (2, 7, 1), (3, 0, 1), (7, 7, 1), (64, 2, 1),
                                                      (5, 7, 32), (200, 1, 1)])
def test_split_equals_single_pass(num_parts, ovh, min_split):
    inp = small(B=4, s_q=2, H=2, seqlens=(1, 200, 640, 65), seed=41, q_mode="q_abs")
    tm, ns = oracle.metadata(inp.seqlens, num_parts, ovh, min_split)
    args = (f32(inp.q_abs), f32(inp.kv_cache), inp.block_table, inp.seqlens, inp.scale, True)
    o1, l1 = oracle.attend_absorbed(*args)
    o2, l2, op, lp = oracle.attend_split(*args, tm, ns)
    assert op.shape[0] == ns[-1]
    assert np.abs(o1 - o2).max() <= 1e-12
    fin = np.isfinite(l1)
    assert np.array_equal(fin, np.isfinite(l2))
    assert np.abs(l1[fin] - l2[fin]).max() <= 1e-12


# -------------------------------------------------------------- schedule --

def _golden_schedules():
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, "schedule_examples.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = {"name": tok[1], "parts": []}
            elif tok[0] == "end":
                cases.append(cur)
            elif tok[0] == "part":
                cur["parts"].append([int(x) for x in tok[1:]])
            elif tok[0] in ("seqlens", "splits"):
                cur[tok[0]] = [int(x) for x in tok[1:]]
            else:
                cur[tok[0]] = int(tok[1])
    return cases


@pytest.mark.parametrize("case", _golden_schedules(), ids=lambda c: c["name"])
def test_schedule_golden(case):
    tm, ns = oracle.metadata(np.array(case["seqlens"], np.int32), case["num_parts"], case["ovh"], case["min_split"])
    assert tm.tolist() == case["parts"]
    assert ns.tolist() == case["splits"]


def check_schedule_invariants(seqlens, tm, ns, num_parts, ovh, min_split):
    seqlens = np.asarray(seqlens)
    B = len(seqlens)
    nblk = [(max(int(s), 0) + 63) // 64 for s in seqlens]
    covered = [np.zeros(n, int) for n in nblk]
    pieces_seen = 0
    total = sum(n + ovh for n in nblk if n > 0)
    quota = max(1, -(-total // num_parts))
    prev_end = (-1, 0)
    piece_batches = []
    for p in range(num_parts):
        row = tm[p]
        if row[5] == 0:
            assert list(row) == [0] * 8
            continue
        assert row[4] == pieces_seen
        b0, j0, b1, j1 = row[:4]
        assert (b0, j0) >= prev_end          # parts are in walk order
        cost = 0
        touched = 0
        for b in range(b0, b1 + 1):
            if nblk[b] == 0:
                continue
            lo = j0 if b == b0 else 0
            hi = j1 if b == b1 else nblk[b]
            assert 0 <= lo < hi <= nblk[b]
            covered[b][lo:hi] += 1
            touched += 1
            piece_batches.append(b)
            cost += (hi - lo) + (ovh if lo == 0 else 0)
        assert touched == row[5]
        # a part never holds more than its quota plus one short batch (or one
        # page of a long one) beyond it
        longest_short = max([n + ovh for n in nblk if 0 < n < min_split] + [ovh + 1])
        assert cost <= quota + longest_short
        pieces_seen += touched
        prev_end = (b1, j1)
    for b in range(B):
        assert np.all(covered[b] == 1), f"batch {b} pages covered {covered[b]}"
        if 0 < nblk[b] < min_split:
            assert ns[b + 1] - ns[b] == 1       # short batches are never split
    assert ns[0] == 0 and ns[B] == pieces_seen and np.all(np.diff(ns) >= 0)
    assert pieces_seen <= B + num_parts
    # pieces are numbered in order and each batch's pieces are consecutive
    for b in range(B):
        assert piece_batches[ns[b]:ns[b + 1]] == [b] * (ns[b + 1] - ns[b])


@pytest.mark.parametrize("seed", range(12))
def test_schedule_invariants_random(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    kind = seed % 4
    if kind == 0:
        seqlens = rng.integers(0, 3000, B)
    elif kind == 1:
        seqlens = np.full(B, int(rng.integers(1, 1000)))
    elif kind == 2:
        seqlens = rng.integers(16384, 32769, B)
    else:
        seqlens = np.where(rng.random(B) < 0.3, 0, rng.integers(1, 200, B))
    for num_parts in (1, 3, 38, 76, 1000):
        for ovh, min_split in ((7, 32), (0, 1), (3, 2)):
            tm, ns = oracle.metadata(seqlens.astype(np.int32), num_parts, ovh, min_split)
            check_schedule_invariants(seqlens, tm, ns, num_parts, ovh, min_split)


def test_schedule_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.metadata(np.array([10], np.int32), 0, 7, 32)

"""Host-side check of the rule by which the decode kernel, when no merge kernel
follows it, gives the rows of empty sequences o = 0 and lse = -inf: every empty
sequence must be written by exactly one schedule part, and no part may write a
sequence that has keys. The rule is restated here from its description in the
decode kernel (an empty batch belongs to the part holding page 0 of the next
non-empty batch; trailing empty batches to the part holding the last page of
the last non-empty one; with every sequence empty, all batches to part 0) and
run over schedules from the oracle's metadata on random length mixes with many
empty sequences, including part counts that leave parts without work."""
import numpy as np
import pytest

import oracle

PAGE = 64


def items_of_part(row, pages):
    """The part's work items (b, lo, hi), walking its schedule row the way the
    decode kernel does: batches begin_b .. end_b, empty ones skipped."""
    if row[5] == 0:
        return []
    out = []
    for b in range(row[0], row[2] + 1):
        n = pages[b]
        if n == 0:
            continue
        lo = row[1] if b == row[0] else 0
        hi = row[3] if b == row[2] else n
        out.append((b, lo, hi))
    return out


def writers_of_empty_rows(tile_meta, pages):
    B = len(pages)
    writes = np.zeros(B, np.int64)
    for p, row in enumerate(tile_meta):
        items = items_of_part(row, pages)
        if not items:
            if p == 0:
                writes[:] += 1  # only when no part has work: every sequence is empty
            continue
        for b, lo, _ in items:
            if lo == 0:
                e = b - 1
                while e >= 0 and pages[e] == 0:
                    writes[e] += 1
                    e -= 1
        b, _, hi = items[-1]
        if hi == pages[b] and all(pages[e] == 0 for e in range(b + 1, B)):
            writes[b + 1:] += 1
    return writes


def mixes():
    rng = np.random.default_rng(2024)
    out = [[0], [0, 0, 0], [5], [0, 5, 0], [0, 2100, 0, 3000, 0, 0], [100, 0, 0, 0, 1]]
    for _ in range(60):
        B = int(rng.integers(1, 200))
        L = rng.integers(1, 40 * PAGE, size=B)
        L[rng.random(B) < rng.uniform(0.0, 0.9)] = 0
        out.append(L.tolist())
    return out


@pytest.mark.parametrize("num_parts", [1, 3, 7, 38, 76, 152])
def test_each_empty_sequence_has_exactly_one_writer(num_parts):
    for seqlens in mixes():
        sl = np.asarray(seqlens, np.int32)
        pages = [(int(x) + PAGE - 1) // PAGE if x > 0 else 0 for x in sl]
        tm, ns = oracle.metadata(sl, num_parts, 7, 32)
        writes = writers_of_empty_rows(tm, pages)
        empty = np.array([n == 0 for n in pages])
        assert np.all(writes[empty] == 1), (seqlens, num_parts, writes.tolist())
        assert np.all(writes[~empty] == 0), (seqlens, num_parts, writes.tolist())

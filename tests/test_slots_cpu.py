"""Host-side invariants of the chunk-slot numbering the tensor-core prefill
relies on: chunk j of sequence n occupies slot cu[n] // 64 + n + j.  The
workspace holds ntok // 64 + N + 1 slots per head, the intra-chunk kernel
finds a slot's sequence as the last n with cu[n] // 64 + n <= slot, and the
recurrence kernel reads a sequence's records from its first slot on.  These
checks run the numbering over random ragged batches (empty and one-token
sequences included) and fail if two chunks could share a slot, a slot could
fall outside the workspace, or the search could name the wrong sequence."""
import bisect

import numpy as np
import pytest

C = 64


def slots_of(cu):
    out = {}
    for n in range(len(cu) - 1):
        first = cu[n] // C + n
        nc = -(-(cu[n + 1] - cu[n]) // C)
        for j in range(nc):
            out[first + j] = (n, j)
    return out


def search(cu, slot):
    """The last n with cu[n] // 64 + n <= slot, or None (before the first)."""
    keys = [cu[n] // C + n for n in range(len(cu) - 1)]
    i = bisect.bisect_right(keys, slot) - 1
    return None if i < 0 else i


@pytest.mark.parametrize("seed", range(40))
def test_slot_numbering(seed):
    rs = np.random.default_rng(seed)
    N = int(rs.integers(1, 40))
    kind = seed % 4
    if kind == 0:
        lens = rs.integers(0, 3 * C, N)
    elif kind == 1:
        lens = rs.integers(0, 3, N)           # empty and one-token sequences
    elif kind == 2:
        lens = rs.choice([0, 1, C - 1, C, C + 1, 2 * C], N)
    else:
        lens = rs.integers(C * 10, C * 40, N)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64).tolist()
    ntok = cu[-1] + int(rs.integers(0, 100))  # tokens after the last sequence too
    table = slots_of(cu)
    n_slots = ntok // C + N + 1
    # every chunk has its own slot, inside the workspace
    assert len(table) == sum(-(-(cu[n + 1] - cu[n]) // C) for n in range(N))
    assert all(0 <= s < n_slots for s in table)
    # the search names the owner of every occupied slot, and every free slot
    # resolves to a sequence whose chunks end before it (so it is skipped)
    for s in range(n_slots):
        n = search(cu, s)
        if s in table:
            assert n == table[s][0]
            assert s - (cu[n] // C + n) == table[s][1]
        elif n is not None:
            nc = -(-(cu[n + 1] - cu[n]) // C)
            assert s - (cu[n] // C + n) >= nc

"""The work split of the attention kernels, restated on the host and checked on random
batches (no GPU).

Decode/verify: all sequences lie end to end on a cost axis (UNIT_COST units of fixed cost,
then the sequence's 128-key blocks) cut into one contiguous range per CTA; each CTA forms one
unit per sequence whose blocks its range reaches; a unit that holds part of a sequence
writes a partial into slot 2c (the CTA's first unit) or 2c + 1 (a unit that begins inside
the range), and the merge kernel finds a split sequence's pieces from the lengths alone.
Prefill: blocks of P positions go out a round at a time, longest first; the units of an
incomplete last round, when their halves fit in one round, run as two key halves each and
are merged in pairs. The checks: every key of every sequence (every position block) is
covered exactly once, a sequence is written directly if and only if one unit holds it all,
and the slots the merge reads are exactly the ones the pieces wrote.

The arithmetic restates the kernels' (mla_attention_tc.cu: the split plan, unit_info and
launch_prefill_tc; mla_merge.cu: merge_split_kernel and merge_prefill_kernel); the CUDA
path itself is checked against the oracle by the GPU tests.
"""
import random

import pytest

KEY_BLOCK = 128
UNIT_COST = 5


def blocks_of(L):
    return (L + KEY_BLOCK - 1) // KEY_BLOCK


def range_lo(c, total, n):
    return c * total // n


def range_of(x, total, n):
    return ((x + 1) * n + total - 1) // total - 1


def decode_units(lens, n):
    """Units per CTA: (b, key_lo, key_hi, final, slot)."""
    spans, x = [], 0
    for b, L in enumerate(lens):
        nb = blocks_of(L)
        if nb > 0:
            spans.append((b, x + UNIT_COST, nb))
            x += UNIT_COST + nb
    total = x
    out = []
    for c in range(n):
        x0 = range_lo(c, total, n) if total else 0
        x1 = range_lo(c + 1, total, n) if total else 0
        mine = []
        for b, first, nb in spans:
            blo, bhi = max(x0, first), min(x1, first + nb)
            if bhi <= blo:
                continue
            L = lens[b]
            final = blo == first and bhi == first + nb
            slot = 2 * c + (0 if first - UNIT_COST <= x0 else 1)
            mine.append((b, (blo - first) * KEY_BLOCK, min(L, (bhi - first) * KEY_BLOCK), final, slot))
        out.append(mine)
    return out, spans, total


def merge_pieces(first, nb, total, n):
    """The merge kernel's view of a sequence: its pieces' partial slots."""
    c0 = range_of(first, total, n)
    count = (range_of(first + nb - 1, total, n) - c0 + 1) if total >= n else nb
    first_odd = 1 if range_lo(c0, total, n) < first - UNIT_COST else 0

    def slot_of(i):
        if i == 0:
            return 2 * c0 + first_odd
        return 2 * ((c0 + i) if total >= n else range_of(first + i, total, n))

    return [slot_of(i) for i in range(count)]


def check_decode(lens, n):
    units, spans, total = decode_units(lens, n)
    per_seq = {b: [] for b in range(len(lens))}
    for c, mine in enumerate(units):
        partial = [u for u in mine if not u[3]]
        # only the first and the last unit of a range can hold part of a sequence
        assert len(partial) <= 2
        assert len({u[4] for u in partial}) == len(partial)
        for u in mine:
            assert u[2] > u[1]
            per_seq[u[0]].append((c, u))
    for b, first, nb in spans:
        got = sorted(per_seq[b], key=lambda cu: cu[1][1])
        pos = 0
        for _, u in got:
            assert u[1] == pos
            pos = u[2]
        assert pos == lens[b]
        slots = merge_pieces(first, nb, total, n)
        if len(slots) == 1:
            assert len(got) == 1 and got[0][1][3]
        else:
            assert all(not u[3] for _, u in got)
            assert sorted(slots) == sorted(u[4] for _, u in got)
            assert all(0 <= s < 2 * n for s in slots)
    for b, L in enumerate(lens):
        if blocks_of(L) == 0:
            assert per_seq[b] == []


@pytest.mark.parametrize("seed", range(6))
def test_decode_split_covers_every_key_once(seed):
    rng = random.Random(seed)
    for _ in range(300):
        n = rng.choice([1, 2, 3, 7, 16, 76, 148, 152, 160, 300])
        B = rng.choice([1, 2, 3, 8, 32, 100, 500])
        mode = rng.random()
        if mode < 0.3:
            lens = [rng.randint(0, 2000) for _ in range(B)]
        elif mode < 0.6:
            lens = [rng.randint(0, 40000) for _ in range(B)]
        elif mode < 0.8:
            lens = [rng.choice([0, 1, 127, 128, 129, 32772, 142000]) for _ in range(B)]
        else:
            lens = [rng.randint(4096, 16384) for _ in range(B)]
        check_decode(lens, n)


def test_decode_split_named_workloads():
    # batched decode (lengths in [4096, 16384]), long history, speculative verify
    rng = random.Random(0)
    check_decode([rng.randint(4096, 16384) for _ in range(32)], 152)
    check_decode([142000], 152)
    check_decode([32772] * 8, 152)


def prefill_plan(T, H, L, sms):
    """(full units per CTA, pieces, merge pairs) as launch_prefill_tc forms them."""
    P = 48 // H
    num_units = (T + P - 1) // P
    grid = min(sms, num_units)
    left = num_units % grid
    split = left > 0 and 2 * left <= grid
    split_base = num_units - left
    unit_end = split_base if split else num_units

    def unit(v):
        pos0 = (num_units - 1 - v) * P
        npos = min(P, T - pos0)
        return pos0, npos, max(0, min(L, L - T + pos0 + npos))

    full = [[unit(u) for u in range(c, unit_end, grid)] for c in range(grid)]
    pieces = []
    if split:
        for q in range(2 * left):  # one half a CTA of the second launch
            pos0, npos, key_hi = unit(split_base + q // 2)
            mid = min(key_hi, ((key_hi + 2 * KEY_BLOCK - 1) // (2 * KEY_BLOCK)) * KEY_BLOCK)
            lo, hi = (0, mid) if q % 2 == 0 else (mid, key_hi)
            pieces.append((q, pos0, npos, lo, hi))
    pairs = [((left - 1 - v) * P, 2 * v, 2 * v + 1) for v in range(left)] if split else []
    return full, pieces, pairs, P, split


@pytest.mark.parametrize("T,H,prefix,sms", [(8192, 12, 32768, 152), (2048, 12, 32768, 152),
                                             (759, 12, 0, 152), (1139, 8, 500, 152),
                                             (485, 16, 2000, 152), (1, 12, 0, 152),
                                             (130, 16, 0, 152), (5000, 12, 100, 148),
                                             (7, 3, 5, 152)])
def test_prefill_split_covers_every_block_once(T, H, prefix, sms):
    L = prefix + T
    full, pieces, pairs, P, split = prefill_plan(T, H, L, sms)
    seen = {}
    for mine in full:
        for pos0, npos, key_hi in mine:
            assert pos0 not in seen
            seen[pos0] = [(0, key_hi)]
    halves = {}
    for q, pos0, npos, lo, hi in pieces:
        assert pos0 not in seen
        halves.setdefault(pos0, []).append((q, lo, hi))
        assert q < sms  # a partial slot per CTA in the workspace
    for pos0, hs in halves.items():
        assert len(hs) == 2
        (q0, lo0, hi0), (q1, lo1, hi1) = sorted(hs)
        assert q1 == q0 + 1 and q0 % 2 == 0 and lo0 == 0 and hi0 == lo1
        assert hi1 == max(0, min(L, L - T + pos0 + min(P, T - pos0)))
        assert hi0 % KEY_BLOCK == 0 or hi0 == hi1
    # the merge kernel's pairs are exactly the split units
    assert sorted(p[0] for p in pairs) == sorted(halves)
    for pos0, s0, s1 in pairs:
        assert sorted(q for q, _, _ in halves[pos0]) == [s0, s1]
    # every position block of the chunk, once
    assert sorted(list(seen) + list(halves)) == list(range(0, T, P))
    # the split happens exactly when the last round is incomplete and its halves fit
    units = (T + P - 1) // P
    grid = min(sms, units)
    assert split == (units % grid > 0 and 2 * (units % grid) <= grid)

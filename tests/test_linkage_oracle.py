"""Pins of the oracle's ratio-2 predecessor linkage ("[Feature][PCP] Add
DeepSeek-V4.1-Flash support", "Implementation" and "Rank-local Compressor
Revision"): hand-worked cases, and properties checked against the pinned
DualChunkSwap partition on random batches."""
import os

import numpy as np
import pytest

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ratio2_linkage.txt")
KEYS = ("first", "last", "pred", "pred_shard", "flags")


def _golden_cases():
    cases, cur = [], None
    for ln in open(GOLDEN):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        f = ln.split()
        if f[0] == "case":
            cur = dict(name=f[1], P=int(f[2]), cu=[int(x) for x in f[3].split(",")],
                       qs=[int(x) for x in f[4].split(",")],
                       dec=[int(x) for x in f[5].split(",")], rows=[])
            cases.append(cur)
        else:
            cur["rows"].append([int(x) for x in f])
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_linkage_matches_hand_worked_cases(case):
    got = orc.ratio2_linkage(case["P"], case["cu"], case["qs"], case["dec"])
    want = np.array(case["rows"], dtype=np.int64)
    assert len(got["first"]) == len(want)
    for col, key in enumerate(KEYS, start=3):
        assert np.array_equal(got[key], want[:, col]), (key, got[key], want[:, col])


def _random_batch(rng):
    P = int(rng.choice([1, 2, 3, 4, 5, 8]))
    B = int(rng.integers(1, 5))
    lens, qs, dec = [], [], []
    for _ in range(B):
        if rng.random() < 0.2:
            lens.append(1)
            qs.append(int(rng.integers(0, 100)))
            dec.append(1)
        else:
            lens.append(int(rng.integers(0, 41)))
            qs.append(int(rng.integers(0, 9)) if rng.random() < 0.4 else 0)
            dec.append(0)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return P, cu, np.array(qs, np.int32), np.array(dec, np.uint8)


@pytest.mark.parametrize("seed", range(40))
def test_linkage_properties_against_the_partition(seed):
    """For every prefill token at an odd position whose predecessor position
    was scheduled in this batch: if the partition puts the two tokens in
    different chunks, the token opens its chunk and the chunk's predecessor
    is that token, on the shard the partition gives it; only chunks' last
    rows are ever gathered; a predecessor never leaves its request."""
    rng = np.random.default_rng(seed)
    P, cu, qs, dec = _random_batch(rng)
    part = orc.partition(P, cu, qs, dec)
    lk = orc.ratio2_linkage(P, cu, qs, dec)
    B = len(cu) - 1
    n_prefill = int((dec == 0).sum())
    assert len(lk["first"]) == P * n_prefill * 2
    # the entries, in order, against the partition's shard rows: each shard's
    # prefill rows are its chunks' tokens, chunk r then chunk 2P-1-r
    e = 0
    for r in range(P):
        rows = part["rows"][part["shard_offsets"][r]:part["shard_offsets"][r + 1]]
        req = part["req"][part["shard_offsets"][r]:part["shard_offsets"][r + 1]]
        for b in range(B):
            if dec[b]:
                continue
            mine = rows[req == b]
            got = []
            for k in range(2):
                if lk["first"][e + k] >= 0:
                    got.extend(range(lk["first"][e + k], lk["last"][e + k] + 1))
            assert np.array_equal(np.array(got, dtype=np.int64), mine.astype(np.int64))
            e += 2
    # predecessor of every chunk start, from the partition's owner map
    req_of = np.repeat(np.arange(B), np.diff(cu))
    lasts = set(int(x) for x in lk["last"] if x >= 0)
    by_first = {int(f): i for i, f in enumerate(lk["first"]) if f >= 0}
    for g in range(int(cu[-1])):
        b = req_of[g]
        if dec[b]:
            continue
        local = g - cu[b]
        p = qs[b] + local
        starts_chunk = g in by_first
        if starts_chunk:
            i = by_first[g]
            assert bool(lk["flags"][i] & 1) == (p % 2 == 1)
            if p % 2 == 1 and local >= 1:
                assert lk["pred"][i] == g - 1 and req_of[g - 1] == b
                assert lk["pred_shard"][i] == part["owner_shard"][g - 1]
                assert lk["pred"][i] in lasts  # only last rows are gathered
                assert not lk["flags"][i] & 2
            elif p % 2 == 1:
                assert lk["pred"][i] == -1 and lk["flags"][i] & 2
            else:
                assert lk["pred"][i] == -1 and lk["pred_shard"][i] == -1
        elif p % 2 == 1 and local >= 1:
            # a pair inside one chunk needs no gathered row
            assert part["owner_shard"][g] == part["owner_shard"][g - 1]
    # open ends: a chunk whose last position is even; the request's last
    # token is its newest open ring row
    for i in range(len(lk["first"])):
        if lk["first"][i] < 0:
            assert lk["flags"][i] == 0 and lk["pred"][i] == -1
            continue
        g = int(lk["last"][i])
        b = req_of[g]
        p = qs[b] + g - cu[b]
        assert bool(lk["flags"][i] & 4) == (p % 2 == 0)
        assert bool(lk["flags"][i] & 8) == (p % 2 == 0 and g == cu[b + 1] - 1)

"""Pins for the fp64 CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's formulas: they use the pages' PCP=4
diagram, closed forms worked out by hand, special cases with known answers,
textbook softmax from scipy as an independent library routine, the E4M3 and
bf16 conversions of torch as library decoders, and exact invariants of the
partitioned method.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 1.0 / math.sqrt(192.0)


def bf16_bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def rand_bits(rng, shape):
    return bf16_bits(rng.standard_normal(shape).astype(np.float32))


def textbook(q, kv, scale, sink=None):
    """Independent softmax attention for one query row (all heads) over the
    given keys, via scipy: q [H, 576], kv [n, 576] float64."""
    s = scale * q @ kv.T
    if sink is None:
        return softmax(s, axis=1) @ kv[:, :512], logsumexp(s, axis=1)
    ext = np.concatenate([s, np.asarray(sink, np.float64)[:, None]], axis=1)
    p = softmax(ext, axis=1)[:, :-1]
    return p @ kv[:, :512], logsumexp(s, axis=1)


# ------------------------------------------------------------------ decoding

def test_bf16_decode_matches_torch():
    codes = np.arange(0, 65536, 97, dtype=np.uint16)
    ref = bits_to_f64(codes)
    got = orc.bf16_to_float64(codes)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = orc.e4m3_to_float64(codes)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_e4m3_known_values():
    # OCP 8-bit floating point spec, E4M3: max normal 448, min normal 2^-6,
    # min subnormal 2^-9, 1.0 = 0 0111 000, NaN = S 1111 111.
    got = orc.e4m3_to_float64(np.array([0x7E, 0x08, 0x01, 0x38, 0xB8, 0x00], np.uint8))
    assert list(got) == [448.0, 2.0 ** -6, 2.0 ** -9, 1.0, -1.0, 0.0]
    assert np.isnan(orc.e4m3_to_float64(np.array([0x7F, 0xFF], np.uint8))).all()


# ----------------------------------------------------------------- partition

def _read_pcp4():
    out = {}
    with open(os.path.join(GOLDEN, "dualchunkswap_pcp4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            r, chunks = line.split(":")
            out[int(r)] = [int(c) for c in chunks.split()]
    return out


@pytest.mark.parametrize("c", [1, 3, 64])
def test_partition_matches_pcp4_diagram(c):
    diagram = _read_pcp4()
    S, P = 8 * c, 4
    part = orc.partition(P, [0, S], [0], [0])
    so = part["shard_offsets"]
    for r in range(P):
        rows = part["rows"][so[r]:so[r + 1]]
        want = np.concatenate([np.arange(ch * c, (ch + 1) * c) for ch in diagram[r]])
        assert np.array_equal(rows, want)
        assert np.array_equal(part["pos"][so[r]:so[r + 1]], want)


def test_partition_p2():
    c = 5
    part = orc.partition(2, [0, 4 * c], [0], [0])
    so = part["shard_offsets"]
    r0 = part["rows"][so[0]:so[1]]
    r1 = part["rows"][so[1]:so[2]]
    assert np.array_equal(r0, np.r_[0:c, 3 * c:4 * c])
    assert np.array_equal(r1, np.r_[c:2 * c, 2 * c:3 * c])


def test_partition_ragged_and_empty_chunks():
    # S = 10, P = 4 -> 8 chunks of sizes 2,2,1,1,1,1,1,1 (reading: first S mod 2P chunks one larger)
    part = orc.partition(4, [0, 10], [0], [0])
    so = part["shard_offsets"]
    assert np.array_equal(part["rows"][so[0]:so[1]], [0, 1, 9])
    assert np.array_equal(part["rows"][so[1]:so[2]], [2, 3, 8])
    assert np.array_equal(part["rows"][so[2]:so[3]], [4, 7])
    assert np.array_equal(part["rows"][so[3]:so[4]], [5, 6])
    # S = 3 < 2P = 8: chunks 0..2 hold one token, the rest are empty
    part = orc.partition(4, [0, 3], [0], [0])
    so = part["shard_offsets"]
    assert [list(part["rows"][so[r]:so[r + 1]]) for r in range(4)] == [[0], [1], [2], []]


def test_partition_varlen_decode_replicated_and_owned_once():
    cu = [0, 7, 8, 20, 21]
    qs = [0, 99, 0, 4]
    dec = [0, 1, 0, 1]
    P = 3
    part = orc.partition(P, cu, qs, dec)
    so = part["shard_offsets"]
    for r in range(P):
        rows = part["rows"][so[r]:so[r + 1]]
        assert 7 in rows and 20 in rows        # decode rows on every shard
    # every global token owned exactly once; decode rows owned by shard 0
    T = cu[-1]
    assert sorted(part["rows"][part["owner_row"]].tolist()) == list(range(T))
    assert part["owner_shard"][7] == 0 and part["owner_shard"][20] == 0
    assert part["pos"][part["owner_row"][7]] == 99 and part["pos"][part["owner_row"][20]] == 4
    # prefills: each token once over all shards
    counts = np.bincount(part["rows"], minlength=T)
    assert all(counts[t] == (P if t in (7, 20) else 1) for t in range(T))
    # requests keep their input order inside a shard
    for r in range(P):
        req = part["req"][so[r]:so[r + 1]]
        assert np.all(np.diff(req) >= 0)


def test_partition_balance_closed_form():
    with open(os.path.join(GOLDEN, "dualchunkswap_balance.txt")) as f:
        cases = [tuple(int(x) for x in l.split()) for l in f if l.strip() and not l.startswith("#")]
    for S, P, want in cases:
        part = orc.partition(P, [0, S], [0], [0])
        so = part["shard_offsets"]
        for r in range(P):
            got = int((part["pos"][so[r]:so[r + 1]].astype(np.int64) + 1).sum())
            assert got == want, (S, P, r)


# ----------------------------------------------------------------- attention

def _dense_case(rng, S, H):
    q = rand_bits(rng, (S, H, 576))
    kv = rand_bits(rng, (S, 576))
    return q, kv


@pytest.mark.parametrize("S,H", [(1, 1), (5, 2), (16, 2)])
def test_dense_attention_matches_textbook_bruteforce(S, H):
    rng = np.random.default_rng(S * 10 + H)
    q, kv = _dense_case(rng, S, H)
    sink = rng.standard_normal(H).astype(np.float32)
    for with_sink in (False, True):
        o, lse = orc.attention(q, np.arange(S), np.zeros(S), kv_bf16=kv, scale=SCALE,
                               sink=sink if with_sink else None)
        qf, kf = bits_to_f64(q), bits_to_f64(kv)
        for t in range(S):
            ro, rl = textbook(qf[t], kf[:t + 1], SCALE, sink if with_sink else None)
            np.testing.assert_allclose(o[t], ro, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[t], rl, rtol=1e-12, atol=1e-13)


def test_sparse_attention_matches_textbook_bruteforce():
    rng = np.random.default_rng(7)
    S, H, k = 12, 2, 4
    q, kv = _dense_case(rng, S, H)
    idx = np.full((S, k), -1, np.int32)
    for t in range(S):
        sel = np.sort(rng.choice(t + 1, size=min(k, t + 1), replace=False))
        idx[t, :len(sel)] = sel
    o, lse = orc.attention(q, np.arange(S), np.zeros(S), kv_bf16=kv, topk=idx, scale=SCALE)
    qf, kf = bits_to_f64(q), bits_to_f64(kv)
    for t in range(S):
        keys = idx[t][idx[t] >= 0]
        ro, rl = textbook(qf[t], kf[keys], SCALE)
        np.testing.assert_allclose(o[t], ro, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[t], rl, rtol=1e-12)


def test_fp8_attention_matches_textbook_bruteforce():
    rng = np.random.default_rng(3)
    S, H = 9, 2
    q = rand_bits(rng, (S, H, 576))
    lat = torch.from_numpy(rng.standard_normal((S, 512)).astype(np.float32))
    codes = lat.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    scales = (rng.random((S, 4)) * 1.5 + 0.5).astype(np.float32)
    rope = rand_bits(rng, (S, 64))
    o, lse = orc.attention(q, np.arange(S), np.zeros(S), kv_fp8=codes, kv_scale=scales,
                           kv_rope=rope, scale=SCALE)
    # the key matrix built with torch's E4M3 decoder and numpy broadcasting
    latf = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    latf = latf * np.repeat(scales.astype(np.float64), 128, axis=1)
    kf = np.concatenate([latf, bits_to_f64(rope)], axis=1)
    qf = bits_to_f64(q)
    for t in range(S):
        ro, rl = textbook(qf[t], kf[:t + 1], SCALE)
        np.testing.assert_allclose(o[t], ro, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[t], rl, rtol=1e-12)


def test_first_token_sees_only_itself():
    rng = np.random.default_rng(11)
    q, kv = _dense_case(rng, 4, 3)
    o, lse = orc.attention(q[:1], [0], [0], kv_bf16=kv, scale=SCALE)
    kf, qf = bits_to_f64(kv), bits_to_f64(q)
    np.testing.assert_array_equal(o[0], np.broadcast_to(kf[0, :512], (3, 512)))
    for h in range(3):
        s00 = SCALE * math.fsum(qf[0, h] * kf[0])
        assert abs(lse[0, h] - s00) < 1e-12


def test_equal_scores_give_mean_of_values():
    rng = np.random.default_rng(5)
    S, H = 10, 2
    kv = rand_bits(rng, (S, 576))
    q = bf16_bits(np.zeros((1, H, 576), np.float32))
    o, lse = orc.attention(q, [S - 1], [0], kv_bf16=kv, scale=SCALE)
    mean = bits_to_f64(kv)[:, :512].mean(axis=0)
    np.testing.assert_allclose(o[0], np.broadcast_to(mean, (H, 512)), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(S), rtol=1e-14)


def test_sink_two_key_closed_form_and_limits():
    # q along e0 and keys a*e0, b*e0 (rest of v arbitrary): s_j = scale*x_j exactly.
    H = 1
    q = np.zeros((1, H, 576), np.float32)
    q[0, 0, 0] = 1.0
    kv = np.zeros((2, 576), np.float32)
    kv[0, 0], kv[1, 0] = 2.0, -1.0
    kv[0, 1], kv[1, 1] = 3.0, 5.0
    s0, s1 = 2.0 * SCALE, -1.0 * SCALE
    sink = np.array([0.75], np.float32)
    o, lse = orc.attention(bf16_bits(q), [1], [0], kv_bf16=bf16_bits(kv), scale=SCALE, sink=sink)
    den = math.exp(s0) + math.exp(s1) + math.exp(0.75)
    assert abs(o[0, 0, 0] - (2.0 * math.exp(s0) - 1.0 * math.exp(s1)) / den) < 1e-14
    assert abs(o[0, 0, 1] - (3.0 * math.exp(s0) + 5.0 * math.exp(s1)) / den) < 1e-14
    assert abs(lse[0, 0] - math.log(math.exp(s0) + math.exp(s1))) < 1e-14  # LSE excludes sink
    # sink -> -inf gives plain attention
    o2, _ = orc.attention(bf16_bits(q), [1], [0], kv_bf16=bf16_bits(kv), scale=SCALE,
                          sink=np.array([-np.inf], np.float32))
    o3, _ = orc.attention(bf16_bits(q), [1], [0], kv_bf16=bf16_bits(kv), scale=SCALE)
    np.testing.assert_array_equal(o2, o3)


def test_sparse_with_all_positions_equals_dense():
    rng = np.random.default_rng(9)
    S, H = 20, 2
    q, kv = _dense_case(rng, S, H)
    idx = np.full((S, S), -1, np.int32)
    for t in range(S):
        idx[t, :t + 1] = np.arange(t + 1)
    od, ld = orc.attention(q, np.arange(S), np.zeros(S), kv_bf16=kv, scale=SCALE)
    os_, ls = orc.attention(q, np.arange(S), np.zeros(S), kv_bf16=kv, topk=idx, scale=SCALE)
    np.testing.assert_array_equal(od, os_)
    np.testing.assert_array_equal(ld, ls)


def test_empty_key_set_gives_zero_and_minus_inf():
    rng = np.random.default_rng(1)
    q, kv = _dense_case(rng, 4, 2)
    o, lse = orc.attention(q[:1], [3], [0], kv_bf16=kv, kv_lo=[2], kv_hi=[1], scale=SCALE)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_out_of_prefix_index_is_rejected():
    rng = np.random.default_rng(2)
    q, kv = _dense_case(rng, 4, 1)
    with pytest.raises(ValueError):
        orc.attention(q[:1], [1], [0], kv_bf16=kv, topk=np.array([[0, 3]], np.int32), scale=SCALE)


# --------------------------------------------------------------------- merge

def test_merge_single_partial_is_sink_scaling():
    rng = np.random.default_rng(4)
    n, H = 6, 3
    op = rng.standard_normal((n, H, 512))
    lp = rng.standard_normal((n, H))
    sink = rng.standard_normal(H).astype(np.float32)
    perm = rng.permutation(n).astype(np.int32)
    o, l = orc.merge(op, lp, np.arange(n + 1), perm, sink=sink)
    for g in range(n):
        f = 1.0 / (1.0 + np.exp(sink.astype(np.float64) - lp[perm[g]]))
        np.testing.assert_allclose(o[g], op[perm[g]] * f[:, None], rtol=1e-14)
        np.testing.assert_array_equal(l[g], lp[perm[g]])


def test_merge_ignores_empty_partials():
    op = np.ones((2, 1, 512))
    op[1] = 7.0
    lp = np.array([[0.3], [-np.inf]])
    o, l = orc.merge(op, lp, [0, 2], [0, 1])
    np.testing.assert_allclose(o[0], 1.0, rtol=1e-15)
    assert l[0, 0] == 0.3


# ----------------------------------------------------------------- invariants

def _kv_split_partials(q, pos, kv_kw, P, S, topk=None):
    """Partials of every row over each of the 2P DualChunkSwap KV chunks
    (the page-1 reading of per-rank partial attention)."""
    rows_o, rows_l, off, contrib = [], [], [0], []
    n = 0
    bounds = []
    base, rem = divmod(S, 2 * P)
    st = 0
    for c in range(2 * P):
        ln = base + (1 if c < rem else 0)
        bounds.append((st, st + ln - 1))
        st += ln
    for lo, hi in bounds:
        o, l = orc.attention(q, pos, np.zeros(len(pos)), kv_lo=np.full(len(pos), lo),
                             kv_hi=np.full(len(pos), hi), topk=topk, scale=SCALE, **kv_kw)
        rows_o.append(o)
        rows_l.append(l)
    T = len(pos)
    for g in range(T):
        for c in range(2 * P):
            contrib.append(c * T + g)
        off.append(len(contrib))
    return np.concatenate(rows_o), np.concatenate(rows_l), np.array(off), np.array(contrib)


@pytest.mark.parametrize("S,H,P", [(37, 2, 2), (64, 4, 4), (23, 1, 3)])
def test_partitioned_equals_unpartitioned_dense(S, H, P):
    rng = np.random.default_rng(S + P)
    q, kv = _dense_case(rng, S, H)
    sink = rng.standard_normal(H).astype(np.float32)
    o_ref, l_ref = orc.attention(q, np.arange(S), np.zeros(S), kv_bf16=kv, scale=SCALE, sink=sink)
    o, l = orc.pcp_attention(P, [0, S], [0], [0], q, [0], scale=SCALE, sink=sink, kv_bf16=kv)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, rtol=0, atol=1e-12)
    # KV-split: merging the 2P chunk partials of every row is also exact
    op, lp, off, contrib = _kv_split_partials(q, np.arange(S), dict(kv_bf16=kv), P, S)
    o2, l2 = orc.merge(op, lp, off, contrib, sink=sink)
    np.testing.assert_allclose(o2, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l_ref, rtol=0, atol=1e-12)


def test_partitioned_equals_unpartitioned_varlen_sparse_with_decode():
    rng = np.random.default_rng(21)
    H, P, k = 2, 3, 6
    plens, dctx = [11, 4], [9, 15]
    qlens = plens + [1, 1]
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    qs = np.array([0, 0, dctx[0] - 1, dctx[1] - 1], np.int32)
    dec = np.array([0, 0, 1, 1], np.uint8)
    kvlens = plens + dctx
    kv_start = np.concatenate([[0], np.cumsum(kvlens)[:-1]]).astype(np.int64)
    T = int(cu[-1])
    q = rand_bits(rng, (T, H, 576))
    kv = rand_bits(rng, (sum(kvlens), 576))
    sink = rng.standard_normal(H).astype(np.float32)
    pos = np.concatenate([np.arange(qlens[b]) + qs[b] for b in range(4)]).astype(np.int32)
    req = np.repeat(np.arange(4), qlens)
    idx = np.full((T, k), -1, np.int32)
    for g in range(T):
        sel = np.sort(rng.choice(pos[g] + 1, size=min(k, pos[g] + 1), replace=False))
        idx[g, :len(sel)] = sel
    o_ref, l_ref = orc.attention(q, pos, kv_start[req], kv_bf16=kv, topk=idx, scale=SCALE, sink=sink)
    o, l = orc.pcp_attention(P, cu, qs, dec, q, kv_start, scale=SCALE, sink=sink, kv_bf16=kv,
                             topk=idx)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, rtol=0, atol=1e-12)
    # brute force for the decode rows
    qf, kf = bits_to_f64(q), bits_to_f64(kv)
    for g in (T - 2, T - 1):
        keys = kv_start[req[g]] + idx[g][idx[g] >= 0]
        ro, _ = textbook(qf[g], kf[keys], SCALE, sink)
        np.testing.assert_allclose(o[g], ro, rtol=1e-12, atol=1e-13)


def test_sink_per_shard_is_wrong_on_tiny_dense_workload():
    """The sink must be applied once after the merge ("[DeepSeekV4][PCP] ...",
    "Main challenges").  Applying it to every KV-split partial instead changes
    the output by more than the 1e-2 tolerance on the 256-token, 4-head case."""
    rng = np.random.default_rng(0)
    S, H, P = 256, 4, 2
    q, kv = _dense_case(rng, S, H)
    sink = rng.standard_normal(H).astype(np.float32)
    o_ref, _ = orc.attention(q, np.arange(S), np.zeros(S), kv_bf16=kv, scale=SCALE, sink=sink)
    op, lp, off, contrib = _kv_split_partials(q, np.arange(S), dict(kv_bf16=kv), P, S)
    # wrong: sink inside every partial, then merge without sink
    f = 1.0 / (1.0 + np.exp(sink[None, :].astype(np.float64) - lp))
    f = np.where(np.isfinite(lp), f, 0.0)
    o_bad, _ = orc.merge(op * f[..., None], lp, off, contrib)
    assert np.abs(o_bad - o_ref).max() > 1e-2
    o_ok, _ = orc.merge(op, lp, off, contrib, sink=sink)
    assert np.abs(o_ok - o_ref).max() < 1e-12

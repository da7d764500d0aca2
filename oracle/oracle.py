"""ctypes wrapper around the fp64 CPU oracle (``cpmla_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The product library never imports
it, and it imports nothing from the product package.

Each function states the passage it follows; the C file's header lists the
readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpmla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DQK, DV, DROPE, GROUP = 576, 512, 64, 128

_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, OpenMP, no SIMD intrinsics)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
            "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_e4m3_to_double.restype = ctypes.c_double
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_partition_rows.restype = ctypes.c_longlong
            lib.oracle_partition_rows.argtypes = [ctypes.c_int, ctypes.c_int, _P, _P]
            lib.oracle_partition.restype = ctypes.c_int
            lib.oracle_partition.argtypes = [ctypes.c_int, ctypes.c_int] + [_P] * 9
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = (
                [ctypes.c_int, ctypes.c_int, _P, _P, _P, ctypes.c_int, _P, _P, _P, _P,
                 _P, ctypes.c_int, _P, _P, ctypes.c_double, _P, _P, _P])
            lib.oracle_merge.restype = None
            lib.oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int] + [_P] * 7
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_kv_insert.restype = ctypes.c_int
            lib.oracle_kv_insert.argtypes = ([ctypes.c_int, _P, _P, ctypes.c_int,
                                              ctypes.c_longlong] + [_P] * 4)
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def bf16_to_float64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64, via the oracle's decoder."""
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_double(int(b)) for b in flat]).reshape(np.shape(bits))


def e4m3_to_float64(codes: np.ndarray) -> np.ndarray:
    """Decode OCP E4M3 bytes to float64 from the bit fields (oracle decoder)."""
    lib = _load()
    flat = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_to_double(int(b)) for b in flat]).reshape(np.shape(codes))


def partition(P: int, cu_seqlens, q_start_pos, is_decode):
    """DualChunkSwap partition ("[Core] Add MRV2 virtual-batch PCP for MLA",
    sections "PCP algorithm" and "DualChunkSwap partitioning").

    Returns a dict of int32 arrays: shard_offsets [P+1], rows/pos/req
    [n_rows], owner_shard/owner_row [T].
    """
    lib = _load()
    cu = _c(cu_seqlens, np.int32)
    qs = _c(q_start_pos, np.int32)
    dec = _c(is_decode, np.uint8)
    B = len(cu) - 1
    T = int(cu[-1]) if B >= 0 else 0
    n = lib.oracle_partition_rows(P, B, _ptr(cu), _ptr(dec))
    out = dict(
        shard_offsets=np.zeros(P + 1, np.int32), rows=np.zeros(n, np.int32),
        pos=np.zeros(n, np.int32), req=np.zeros(n, np.int32),
        owner_shard=np.full(T, -1, np.int32), owner_row=np.full(T, -1, np.int32))
    rc = lib.oracle_partition(P, B, _ptr(cu), _ptr(qs), _ptr(dec),
                              *[_ptr(out[k]) for k in ("shard_offsets", "rows", "pos", "req",
                                                       "owner_shard", "owner_row")])
    if rc != 0:
        raise ValueError("oracle_partition: bad arguments")
    return out


def ratio2_linkage(P: int, cu_seqlens, q_start_pos, is_decode):
    """Predecessor-row linkage of a ratio-2 compressor across DualChunkSwap
    chunks ("[Feature][PCP] Add DeepSeek-V4.1-Flash support", sections
    "Overview" and "Implementation": ratio-2 groups are compressed on each
    rank's local token rows, and the pairs split across PCP chunks are closed
    with gathered predecessor rows -- only the last row of each local chunk is
    gathered; "Rank-local Compressor Revision" names the cases: PCP2/4
    linkage, replicated short prefills, empty ranks, request isolation and
    the newest open ring rows).

    Readings where the page is silent: a ratio-2 group is the pair of request
    positions (2m, 2m+1); chunk sizes, chunk order and shard assignment are
    those of the partition (first S mod 2P chunks one token larger; shard r
    holds chunks r and 2P-1-r); decode requests (replicated, one row) have no
    chunks and no entries.

    One entry per (shard r, prefill request b in input order, local chunk k:
    k = 0 is chunk r, k = 1 is chunk 2P-1-r), shard-major.  For a chunk
    holding request positions p0 .. p1 (global tokens first .. last):
      first, last  its first and last global token (-1, -1 when empty)
      flags bit 0  p0 is odd: the pair (p0-1, p0) straddles the chunk's start
            bit 1  ... and position p0-1 was scheduled in an earlier step (the
                   request's open ring row), not in this batch
            bit 2  p1 is even: the pair (p1, p1+1) is open at the chunk's end
            bit 3  ... and p1 is the request's last scheduled token, so that
                   row is the request's newest open ring row
      pred         global token of position p0-1 when bit 0 is set and that
                   position is in this batch (the last token of the nearest
                   earlier non-empty chunk of the same request), else -1
      pred_shard   the shard whose local chunk holds pred, else -1
    Returns a dict of int32 arrays (first, last, pred, pred_shard, flags)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    qs = np.asarray(q_start_pos, dtype=np.int64)
    dec = np.asarray(is_decode, dtype=np.int64)
    B = len(cu) - 1
    nch = 2 * P

    def chunk(S, c):  # start and length of chunk c of an S-token request
        base, rem = divmod(S, nch)
        return c * base + min(c, rem), base + (1 if c < rem else 0)

    def shard_of(c):
        return c if c < P else nch - 1 - c

    out = {k: [] for k in ("first", "last", "pred", "pred_shard", "flags")}
    for r in range(P):
        for b in range(B):
            if dec[b]:
                continue
            g0, S, q0 = int(cu[b]), int(cu[b + 1] - cu[b]), int(qs[b])
            for c in (r, nch - 1 - r):
                st, ln = chunk(S, c)
                first = last = pred = pshard = -1
                flags = 0
                if ln > 0:
                    first, last = g0 + st, g0 + st + ln - 1
                    p0, p1 = q0 + st, q0 + st + ln - 1
                    if p0 % 2 == 1:
                        flags |= 1
                        if st >= 1:
                            # local index st-1 lies in the nearest earlier
                            # non-empty chunk of this request
                            cp = max(cc for cc in range(c) if chunk(S, cc)[1] > 0)
                            pred, pshard = g0 + st - 1, shard_of(cp)
                        else:
                            flags |= 2
                    if p1 % 2 == 0:
                        flags |= 4
                        if st + ln == S:
                            flags |= 8
                out["first"].append(first)
                out["last"].append(last)
                out["pred"].append(pred)
                out["pred_shard"].append(pshard)
                out["flags"].append(flags)
    return {k: np.asarray(v, dtype=np.int32) for k, v in out.items()}


def attention(q_bits, pos, kv_start, *, kv_bf16=None, kv_fp8=None, kv_scale=None,
              kv_rope=None, topk=None, kv_lo=None, kv_hi=None, scale, sink=None):
    """Plain definition of (partial) attention for n query rows, all heads
    ("[DeepSeekV4][PCP] ...", "Implementation summary"; the key set is the
    causal prefix, or the row's top-k list).

    q_bits: uint16 bf16 bits [n, H, 576]; pos/kv_start: per row.
    KV: either kv_bf16 (uint16 [S, 576]) or kv_fp8 (uint8 [S, 512]) + kv_scale
    (float32 [S, 4]) + kv_rope (uint16 [S, 64]).
    Returns (o [n, H, 512] float64, lse [n, H] float64).
    """
    lib = _load()
    q = _c(q_bits, np.uint16)
    n, H, d = q.shape
    assert d == DQK
    pos = _c(pos, np.int32)
    kvs = _c(kv_start, np.int64)
    fmt = 0 if kv_bf16 is not None else 1
    kvb = _c(kv_bf16, np.uint16)
    kv8 = _c(kv_fp8, np.uint8)
    ksc = _c(kv_scale, np.float32)
    krp = _c(kv_rope, np.uint16)
    tk = _c(topk, np.int32)
    k = 0 if tk is None else tk.shape[1]
    lo = _c(kv_lo, np.int32)
    hi = _c(kv_hi, np.int32)
    snk = _c(sink, np.float32)
    o = np.zeros((n, H, DV), np.float64)
    lse = np.zeros((n, H), np.float64)
    rc = lib.oracle_attention(n, H, _ptr(q), _ptr(pos), _ptr(kvs), fmt, _ptr(kvb), _ptr(kv8),
                              _ptr(ksc), _ptr(krp), _ptr(tk), k, _ptr(lo), _ptr(hi),
                              float(scale), _ptr(snk), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attention: a top-k index lies outside the causal prefix")
    return o, lse


def merge(o_part, lse_part, contrib_off, contrib_rows, sink=None):
    """Global LSE merge + sink once + global order ("[DeepSeekV4][PCP] ...",
    "Implementation summary" and "Main challenges"; restore order from
    "[Core] Add MRV2 virtual-batch PCP for MLA").

    o_part [n_part, H, 512], lse_part [n_part, H] (float64, no sink);
    CSR (contrib_off [T+1], contrib_rows) lists each global row's partials.
    Returns (o [T, H, 512], lse [T, H]) float64.
    """
    lib = _load()
    op = _c(o_part, np.float64)
    lp = _c(lse_part, np.float64)
    off = _c(contrib_off, np.int32)
    rows = _c(contrib_rows, np.int32)
    snk = _c(sink, np.float32)
    T = len(off) - 1
    H = lp.shape[1]
    o = np.zeros((T, H, DV), np.float64)
    lse = np.zeros((T, H), np.float64)
    lib.oracle_merge(T, H, _ptr(op), _ptr(lp), _ptr(off), _ptr(rows), _ptr(snk), _ptr(o), _ptr(lse))
    return o, lse


def pcp_attention(P, cu_seqlens, q_start_pos, is_decode, q_bits, kv_start_req, *, scale,
                  sink=None, **kv):
    """The partitioned path end to end, in fp64: partition -> per-shard
    partials (no sink) -> global merge with the sink once -> global order.

    q_bits is indexed by global token [T, H, 576]; kv_start_req [B] is the KV
    row of each request's position 0; ``topk`` (if given) is [T, k] indexed by
    global token.  Returns (o [T,H,512], lse [T,H]).
    """
    part = partition(P, cu_seqlens, q_start_pos, is_decode)
    rows, pos, req = part["rows"], part["pos"], part["req"]
    topk = kv.pop("topk", None)
    o_p, l_p = attention(np.asarray(q_bits)[rows], pos, np.asarray(kv_start_req, np.int64)[req],
                         topk=None if topk is None else np.asarray(topk)[rows], scale=scale,
                         sink=None, **kv)
    T = len(part["owner_row"])
    off = np.arange(T + 1, dtype=np.int32)
    return merge(o_p, l_p, off, part["owner_row"], sink=sink)


def e4m3_encode(values: np.ndarray) -> np.ndarray:
    """binary32 -> OCP E4M3 bytes, round to nearest even, saturating to
    +-448 (oracle encoder, from the format definition)."""
    lib = _load()
    flat = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in flat],
                    dtype=np.uint8).reshape(np.shape(values))


def kv_insert(kv_bits, slot, *, fmt, s_cache, cache=None):
    """Insert tokens' latent KV (bf16 bits [n, 576]) into cache rows slot[t]
    (-1 skips), bf16 (fmt 0) or fp8 (fmt 1; per-128-channel amax/448 scales,
    E4M3 codes), as "[Core] Add MRV2 virtual-batch PCP for MLA" inserts the
    all-gathered latent KV into the cache.  The pages give no quantisation
    rule; this one is the library's: per group scale = amax / 448 in
    binary32 (1 for an all-zero group), code = E4M3(x / scale) with the
    quotient in binary32, nearest-even, saturating at +-448.  `cache` (dict
    of numpy arrays) is updated in place and returned; fresh zero arrays if
    None."""
    lib = _load()
    kv = _c(kv_bits, np.uint16)
    n = kv.shape[0]
    sl = _c(slot, np.int64)
    if cache is None:
        cache = (dict(kv=np.zeros((s_cache, DQK), np.uint16)) if fmt == 0 else
                 dict(kv_fp8=np.zeros((s_cache, DV), np.uint8),
                      kv_scale=np.zeros((s_cache, DV // GROUP), np.float32),
                      kv_rope=np.zeros((s_cache, DROPE), np.uint16)))
    rc = lib.oracle_kv_insert(n, _ptr(kv), _ptr(sl), fmt, s_cache, _ptr(cache.get("kv")),
                              _ptr(cache.get("kv_fp8")), _ptr(cache.get("kv_scale")),
                              _ptr(cache.get("kv_rope")))
    if rc != 0:
        raise ValueError("oracle_kv_insert: a slot lies outside [-1, s_cache)")
    return cache


def topk_select(logits, row_len, k):
    """Top-k selection of an indexer's logits (the step "[Feat][NVIDIA]
    DeepSeek-V4.1: Prefill support CP with multistream forward prepare (4/N)"
    runs after mqa_logits, its topk_v2): for row i, among columns
    0 .. row_len[i]-1, the k largest values -- ties to the smaller column --
    returned as column indices in ascending order, -1 padded; a row with at
    most k candidates returns all of them.  Values are ordered by the IEEE
    total order of non-NaN binary32 (-0 below +0); the pages give no tie
    rule, so ties go to the smaller column, which makes the selected set
    unique.  logits: float32 [n_rows, >= max(row_len)].
    Returns int32 [n_rows, k]."""
    x = np.asarray(logits, dtype=np.float32)
    lens = np.asarray(row_len, dtype=np.int64)
    out = np.full((x.shape[0], k), -1, dtype=np.int32)
    for i in range(x.shape[0]):
        n = int(lens[i])
        if n <= k:
            out[i, :n] = np.arange(n, dtype=np.int32)
            continue
        bits = x[i, :n].view(np.uint32).astype(np.int64)
        # an order-preserving integer image of the floats (total order)
        key = np.where(bits >> 31 == 1, 0xFFFFFFFF - bits, bits + 0x80000000)
        order = np.lexsort((np.arange(n), -key))  # value descending, column ascending
        out[i] = np.sort(order[:k]).astype(np.int32)
    return out


"""Thin ctypes binding of ``libcpmla.so`` (C ABI in ``include/cpmla.h``).

Argument marshalling only: every step of the path runs in the library's
kernels (or, for the partition, its host C++).  Tensors are passed as raw
pointers; torch is used for device memory and streams.  If the library is
missing the import of a function fails loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpmla.so")

CPMLA_OK, CPMLA_ERR_ARG, CPMLA_ERR_CUDA, CPMLA_ERR_UNSUPPORTED = 0, -1, -2, -3
CPMLA_ERR_TIMEOUT, CPMLA_ERR_INDEX = -4, -5
CPMLA_KV_BF16, CPMLA_KV_FP8_E4M3_G128 = 0, 1
DQK, DV = 576, 512

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float

_SIGS = {
    "cpmla_last_error": (ctypes.c_char_p, []),
    "cpmla_version": (_I, []),
    "cpmla_device_status": (_I, [_P, _I]),
    "cpmla_selftest_wait_timeout": (_I, [ctypes.c_uint, _P]),
    "pcp_partition_size": (_I, [_I, _I, _P, _P, _P]),
    "pcp_dualchunk_partition": (_I, [_I, _I] + [_P] * 9),
    "mla_partial_attn_dense": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I,
                                    _P, _P, _F, _P, _P, _P]),
    "mla_partial_attn_sparse": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I,
                                     _P, _P, _P, _I, _F, _P, _P, _P]),
    "lse_merge_with_sink": (_I, [_P, _P, _I64, _I, _P, _P, _I, _P, _P, _P, _P]),
    "mla_attn_dense_merged": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I,
                                   _P, _P, _F, _P, _I, _P, _P, _P, _P]),
    "mla_attn_sparse_merged": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I,
                                    _P, _P, _P, _I, _F, _P, _I, _P, _P, _P, _P]),
    "mla_kv_cache_insert": (_I, [_P, _I64, _I, _P, _I, _P, _P, _P, _P, _I64, _P]),
    "mla_topk_select": (_I, [_P, _I64, _I, _P, _I, _I, _P, _P]),
    "pcp_ratio2_linkage_size": (_I, [_I, _I, _P, _P, _P]),
    "pcp_ratio2_linkage": (_I, [_I, _I] + [_P] * 8),
    "pcp_gather_rows_f32": (_I, [_P, _I64, _I64, _I, _I, _P, _P, _I64, _P]),
    "mla_attn_split_kv_workspace_size": (ctypes.c_size_t, [_I, _I, _I]),
    "mla_attn_split_kv": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I, _P,
                               _I, _I, _F, _P, _I, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_attn_split_kv_noalloc": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _I64, _P, _P, _P, _P,
                                       _I, _P, _I, _I, _F, _P, _I, _P, _P, _P]),
}

_lock = threading.Lock()
_lib = None


class CpmlaError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("cpmla error %d: %s" % (code, msg))
        self.code = code


def lib():
    """Open libcpmla.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libcpmla.so not built: run __graft_entry__.build() or "
                                   "python context_sparse_mla_gb300/build.py")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
    return _lib


def _check(rc):
    if rc != CPMLA_OK:
        raise CpmlaError(rc, lib().cpmla_last_error().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data_as(ctypes.c_void_p)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, dtype, name):
    if t is None:
        return None
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))
    return t


# ------------------------------------------------------------------ partition
def pcp_dualchunk_partition(P, cu_seqlens, q_start_pos, is_decode):
    """Host DualChunkSwap partition; returns a dict of int32 numpy arrays
    (shard_offsets [P+1], rows/pos/req [n_rows], owner_shard/owner_row [T])."""
    L = lib()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    qs = np.ascontiguousarray(np.asarray(q_start_pos, dtype=np.int32))
    dec = np.ascontiguousarray(np.asarray(is_decode, dtype=np.uint8))
    B = len(cu) - 1
    n = ctypes.c_int64(0)
    _check(L.pcp_partition_size(P, B, _ptr(cu), _ptr(dec), ctypes.byref(n)))
    T = int(cu[-1]) if B >= 0 else 0
    out = dict(shard_offsets=np.zeros(P + 1, np.int32), rows=np.zeros(n.value, np.int32),
               pos=np.zeros(n.value, np.int32), req=np.zeros(n.value, np.int32),
               owner_shard=np.zeros(T, np.int32), owner_row=np.zeros(T, np.int32))
    _check(L.pcp_dualchunk_partition(P, B, _ptr(cu), _ptr(qs), _ptr(dec),
                                     *[_ptr(out[k]) for k in ("shard_offsets", "rows", "pos",
                                                              "req", "owner_shard", "owner_row")]))
    return out


def pcp_ratio2_linkage(P, cu_seqlens, q_start_pos, is_decode):
    """Host ratio-2 linkage across DualChunkSwap chunks; returns a dict of
    int32 numpy arrays (first, last, pred, pred_shard, flags), one entry per
    (shard, prefill request, local chunk), shard-major."""
    L = lib()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    qs = np.ascontiguousarray(np.asarray(q_start_pos, dtype=np.int32))
    dec = np.ascontiguousarray(np.asarray(is_decode, dtype=np.uint8))
    B = len(cu) - 1
    n = ctypes.c_int64(0)
    _check(L.pcp_ratio2_linkage_size(P, B, _ptr(cu), _ptr(dec), ctypes.byref(n)))
    keys = ("first", "last", "pred", "pred_shard", "flags")
    out = {k: np.zeros(n.value, np.int32) for k in keys}
    _check(L.pcp_ratio2_linkage(P, B, _ptr(cu), _ptr(qs), _ptr(dec), *[_ptr(out[k]) for k in keys]))
    return out


def pcp_gather_rows_f32(src, idx, out=None, *, stream=None):
    """out[i] = src[idx[i]] (fp32 rows, zeros where idx[i] == -1) on the GPU."""
    _dev(src, torch.float32, "src")
    _dev(idx, torch.int32, "idx")
    n_src, D = src.shape
    if out is None:
        out = torch.empty((idx.numel(), D), dtype=torch.float32, device=src.device)
    _dev(out, torch.float32, "out")
    _check(lib().pcp_gather_rows_f32(_ptr(src), src.stride(0), n_src, D, idx.numel(), _ptr(idx),
                                     _ptr(out), out.stride(0), _stream(stream)))
    return out


# ------------------------------------------------------------------ attention
def _attn_common(q, kv, kv_fp8, kv_scale, kv_rope):
    _dev(q, torch.bfloat16, "q")
    if q.dim() != 3 or q.shape[2] != DQK:
        raise ValueError("q must be [T, H, 576]")
    if kv is not None:
        _dev(kv, torch.bfloat16, "kv")
        return CPMLA_KV_BF16, kv.shape[0]
    _dev(kv_fp8, torch.uint8, "kv_fp8")
    _dev(kv_scale, torch.float32, "kv_scale")
    _dev(kv_rope, torch.bfloat16, "kv_rope")
    return CPMLA_KV_FP8_E4M3_G128, kv_fp8.shape[0]


def mla_partial_attn_dense(q, kv_start, rows, pos, req, o_part, lse_part, *, softmax_scale,
                           kv=None, kv_fp8=None, kv_scale=None, kv_rope=None, kv_lo=None,
                           kv_hi=None, stream=None):
    """Partial dense-causal attention of shard rows (no sink); writes o_part
    [n_rows, H, 512] fp32 and lse_part [n_rows, H] fp32 in place."""
    fmt, s_kv = _attn_common(q, kv, kv_fp8, kv_scale, kv_rope)
    n = rows.numel()
    _check(lib().mla_partial_attn_dense(
        _ptr(q), q.stride(0), q.shape[1], fmt, _ptr(kv), _ptr(kv_fp8), _ptr(kv_scale),
        _ptr(kv_rope), s_kv, _ptr(_dev(kv_start, torch.int64, "kv_start")),
        _ptr(_dev(rows, torch.int32, "rows")), _ptr(_dev(pos, torch.int32, "pos")),
        _ptr(_dev(req, torch.int32, "req")), n, _ptr(_dev(kv_lo, torch.int32, "kv_lo")),
        _ptr(_dev(kv_hi, torch.int32, "kv_hi")), float(softmax_scale),
        _ptr(_dev(o_part, torch.float32, "o_part")), _ptr(_dev(lse_part, torch.float32, "lse_part")),
        _stream(stream)))


def mla_partial_attn_sparse(q, kv_start, rows, pos, req, topk_idx, o_part, lse_part, *,
                            softmax_scale, kv=None, kv_fp8=None, kv_scale=None, kv_rope=None,
                            kv_lo=None, kv_hi=None, stream=None):
    """Partial top-k sparse attention of shard rows (no sink); topk_idx is
    [T, k] int32 indexed by global token, -1 padded."""
    fmt, s_kv = _attn_common(q, kv, kv_fp8, kv_scale, kv_rope)
    n = rows.numel()
    _dev(topk_idx, torch.int32, "topk_idx")
    _check(lib().mla_partial_attn_sparse(
        _ptr(q), q.stride(0), q.shape[1], fmt, _ptr(kv), _ptr(kv_fp8), _ptr(kv_scale),
        _ptr(kv_rope), s_kv, _ptr(_dev(kv_start, torch.int64, "kv_start")),
        _ptr(_dev(rows, torch.int32, "rows")), _ptr(_dev(pos, torch.int32, "pos")),
        _ptr(_dev(req, torch.int32, "req")), n, _ptr(_dev(kv_lo, torch.int32, "kv_lo")),
        _ptr(_dev(kv_hi, torch.int32, "kv_hi")), _ptr(topk_idx), topk_idx.shape[1],
        float(softmax_scale), _ptr(_dev(o_part, torch.float32, "o_part")),
        _ptr(_dev(lse_part, torch.float32, "lse_part")), _stream(stream)))


def mla_attn_merged(q, kv_start, rows, pos, req, owner_row, o_out, lse_out, *, softmax_scale,
                    sink=None, topk_idx=None, kv=None, kv_fp8=None, kv_scale=None, kv_rope=None,
                    kv_lo=None, kv_hi=None, stream=None):
    """Attention of shard rows with the single-partial merge folded in: each
    token's owner row writes o_out [T, H, 512] bf16 and lse_out [T, H] (sink
    applied once to O).  Dense when topk_idx is None, else top-k sparse."""
    fmt, s_kv = _attn_common(q, kv, kv_fp8, kv_scale, kv_rope)
    n = rows.numel()
    T = lse_out.shape[0]
    common = (_ptr(q), q.stride(0), q.shape[1], fmt, _ptr(kv), _ptr(kv_fp8), _ptr(kv_scale),
              _ptr(kv_rope), s_kv, _ptr(_dev(kv_start, torch.int64, "kv_start")),
              _ptr(_dev(rows, torch.int32, "rows")), _ptr(_dev(pos, torch.int32, "pos")),
              _ptr(_dev(req, torch.int32, "req")), n, _ptr(_dev(kv_lo, torch.int32, "kv_lo")),
              _ptr(_dev(kv_hi, torch.int32, "kv_hi")))
    tail = (float(softmax_scale), _ptr(_dev(owner_row, torch.int32, "owner_row")), T,
            _ptr(_dev(sink, torch.float32, "sink")), _ptr(_dev(o_out, torch.bfloat16, "o_out")),
            _ptr(_dev(lse_out, torch.float32, "lse_out")), _stream(stream))
    if topk_idx is None:
        _check(lib().mla_attn_dense_merged(*common, *tail))
    else:
        _dev(topk_idx, torch.int32, "topk_idx")
        _check(lib().mla_attn_sparse_merged(*common, _ptr(topk_idx), topk_idx.shape[1], *tail))


def split_kv_workspace(H, n_tokens, n_split, device="cuda"):
    """A device buffer of the size mla_attn_split_kv needs (uint8, 256-byte
    aligned by the caching allocator)."""
    n = lib().mla_attn_split_kv_workspace_size(H, n_tokens, n_split)
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


def mla_attn_split_kv(q, kv_start, tokens, pos, req, o_out, lse_out, *, softmax_scale, n_split,
                      workspace, sink=None, topk_idx=None, kv=None, kv_fp8=None, kv_scale=None,
                      kv_rope=None, stream=None):
    """Attention of the listed tokens (int32 tokens/pos/req on the device),
    each token's keys split into n_split parts computed side by side and
    merged with the sink once; writes their rows of o_out [T, H, 512] bf16
    and lse_out [T, H].  Dense causal when topk_idx is None."""
    fmt, s_kv = _attn_common(q, kv, kv_fp8, kv_scale, kv_rope)
    T = lse_out.shape[0]
    k = 0
    if topk_idx is not None:
        _dev(topk_idx, torch.int32, "topk_idx")
        k = topk_idx.shape[1]
    _dev(workspace, torch.uint8, "workspace")
    _check(lib().mla_attn_split_kv(
        _ptr(q), q.stride(0), q.shape[1], fmt, _ptr(kv), _ptr(kv_fp8), _ptr(kv_scale),
        _ptr(kv_rope), s_kv, _ptr(_dev(kv_start, torch.int64, "kv_start")),
        _ptr(_dev(tokens, torch.int32, "tokens")), _ptr(_dev(pos, torch.int32, "pos")),
        _ptr(_dev(req, torch.int32, "req")), tokens.numel(), _ptr(topk_idx), k, int(n_split),
        float(softmax_scale), _ptr(_dev(sink, torch.float32, "sink")), T,
        _ptr(_dev(o_out, torch.bfloat16, "o_out")), _ptr(_dev(lse_out, torch.float32, "lse_out")),
        _ptr(workspace), workspace.numel(), _stream(stream)))


def mla_kv_cache_insert(kv, slot_mapping, *, cache=None, cache_fp8=None, cache_scale=None,
                        cache_rope=None, stream=None):
    """Write each token's latent KV row (kv [n, 576] bf16) to its cache row
    slot_mapping[t] (int64, -1 skips): a bf16 cache [S, 576], or the fp8 one
    (cache_fp8 [S, 512] E4M3, cache_scale [S, 4] fp32, cache_rope [S, 64])."""
    fmt = CPMLA_KV_BF16 if cache is not None else CPMLA_KV_FP8_E4M3_G128
    if fmt == CPMLA_KV_BF16:
        _dev(cache, torch.bfloat16, "cache")
        s_cache = cache.shape[0]
    else:
        _dev(cache_fp8, torch.uint8, "cache_fp8")
        _dev(cache_scale, torch.float32, "cache_scale")
        _dev(cache_rope, torch.bfloat16, "cache_rope")
        s_cache = cache_fp8.shape[0]
    _dev(kv, torch.bfloat16, "kv")
    _check(lib().mla_kv_cache_insert(
        _ptr(kv), kv.stride(0), kv.shape[0], _ptr(_dev(slot_mapping, torch.int64, "slot_mapping")),
        fmt, _ptr(cache), _ptr(cache_fp8), _ptr(cache_scale), _ptr(cache_rope), s_cache,
        _stream(stream)))


def mla_topk_select(logits, row_len, k, *, max_row_len=None, out=None, stream=None):
    """Per row i, the k columns of the largest logits[i, :row_len[i]] (IEEE
    total order, ties to the smaller column) in ascending order, -1 padded:
    logits fp32 [n_rows, L] (L a multiple of 4), row_len int32 [n_rows].
    Returns int32 [n_rows, k] (``out`` if given)."""
    _dev(logits, torch.float32, "logits")
    _dev(row_len, torch.int32, "row_len")
    n_rows, width = logits.shape
    if out is None:
        out = torch.empty((n_rows, k), dtype=torch.int32, device=logits.device)
    _dev(out, torch.int32, "out")
    if out.shape != (n_rows, k):
        raise ValueError("out must be [%d, %d]" % (n_rows, k))
    _check(lib().mla_topk_select(
        _ptr(logits), width, n_rows, _ptr(row_len), width if max_row_len is None else max_row_len,
        k, _ptr(out), _stream(stream)))
    return out


def lse_merge_with_sink(o_part, lse_part, contrib_rows, o_out, lse_out, *, contrib_off=None,
                        sink=None, stream=None):
    """Global LSE merge + sink once + global order; writes o_out [T, H, 512]
    bf16 and lse_out [T, H] fp32 in place."""
    T, H = lse_out.shape
    _check(lib().lse_merge_with_sink(
        _ptr(_dev(o_part, torch.float32, "o_part")), _ptr(_dev(lse_part, torch.float32, "lse_part")),
        lse_part.shape[0], H, _ptr(_dev(contrib_off, torch.int32, "contrib_off")),
        _ptr(_dev(contrib_rows, torch.int32, "contrib_rows")), T,
        _ptr(_dev(sink, torch.float32, "sink")), _ptr(_dev(o_out, torch.bfloat16, "o_out")),
        _ptr(_dev(lse_out, torch.float32, "lse_out")), _stream(stream)))


def device_status(clear=True):
    """The first in-kernel fault recorded on the current device (0 = none)."""
    v = ctypes.c_int(0)
    _check(lib().cpmla_device_status(ctypes.byref(v), 1 if clear else 0))
    return v.value


def selftest_wait_timeout(limit_ms=200, stream=None):
    """Run a kernel whose bounded wait must give up after limit_ms; returns
    the recorded device status (CPMLA_ERR_TIMEOUT when the machinery works)."""
    device_status(clear=True)
    _check(lib().cpmla_selftest_wait_timeout(int(limit_ms), _stream(stream)))
    return device_status(clear=True)


# ------------------------------------------------------------- the whole path
class PcpPrefill:
    """The path for one batch: DualChunkSwap partition (host, once), then per
    call the partial attention of all shards in one launch and the global merge
    in a second -- or, with merged=True, one launch whose epilogue does the
    single-partial merge.  Holds the device copies of the partition maps and
    the fp32 partial buffers."""

    def __init__(self, P, cu_seqlens, q_start_pos, is_decode, kv_start, H, *, device="cuda",
                 topk=0, merged=False, split_decode=False):
        self.merged = merged
        self.P, self.H, self.topk = P, H, topk
        part = pcp_dualchunk_partition(P, cu_seqlens, q_start_pos, is_decode)
        self.part = part
        dev = torch.device(device)
        t = lambda a: torch.from_numpy(a).to(dev)
        self.rows, self.pos, self.req = t(part["rows"]), t(part["pos"]), t(part["req"])
        owner = part["owner_row"]
        # split_decode (merged only): the decode rows leave the merged launch
        # (no row owns them there) and go through mla_attn_split_kv, each
        # row's keys in P parts -- one per shard that holds a replica
        self.split_decode = bool(split_decode and merged)
        self.dec = None
        if self.split_decode:
            dec_rows = owner[np.flatnonzero(np.repeat(np.asarray(is_decode, np.uint8),
                                                      np.diff(np.asarray(cu_seqlens))))]
            if len(dec_rows):
                self.dec = dict(tokens=t(part["rows"][dec_rows]), pos=t(part["pos"][dec_rows]),
                                req=t(part["req"][dec_rows]))
                owner = owner.copy()
                owner[part["rows"][dec_rows]] = -1
                self.dec_ws = split_kv_workspace(H, len(dec_rows), P, device=dev)
        self.owner_row = t(owner)
        self.kv_start = torch.as_tensor(np.asarray(kv_start, np.int64)).to(dev)
        self.n_rows = len(part["rows"])
        self.T = len(part["owner_row"])
        # the fp32 partials exist only for the two-launch path
        self.o_part = self.lse_part = None
        if not merged:
            self.o_part = torch.empty((self.n_rows, H, DV), dtype=torch.float32, device=dev)
            self.lse_part = torch.empty((self.n_rows, H), dtype=torch.float32, device=dev)

    def attention(self, q, *, softmax_scale, idx=None, stream=None, **kv):
        if self.topk:
            mla_partial_attn_sparse(q, self.kv_start, self.rows, self.pos, self.req, idx,
                                    self.o_part, self.lse_part, softmax_scale=softmax_scale,
                                    stream=stream, **kv)
        else:
            mla_partial_attn_dense(q, self.kv_start, self.rows, self.pos, self.req, self.o_part,
                                   self.lse_part, softmax_scale=softmax_scale, stream=stream, **kv)

    def decode(self, q, o_out, lse_out, *, softmax_scale, sink=None, idx=None, stream=None,
               **kv):
        """The decode rows through split-KV (split_decode plans only)."""
        mla_attn_split_kv(q, self.kv_start, self.dec["tokens"], self.dec["pos"], self.dec["req"],
                          o_out, lse_out, softmax_scale=softmax_scale, n_split=self.P,
                          workspace=self.dec_ws, sink=sink, topk_idx=idx if self.topk else None,
                          stream=stream, **kv)

    def merge(self, o_out, lse_out, sink=None, stream=None):
        lse_merge_with_sink(self.o_part, self.lse_part, self.owner_row, o_out, lse_out, sink=sink,
                            stream=stream)

    def __call__(self, q, *, softmax_scale, sink=None, idx=None, o_out=None, lse_out=None,
                 stream=None, **kv):
        if o_out is None:
            o_out = torch.empty((self.T, self.H, DV), dtype=torch.bfloat16, device=q.device)
        if lse_out is None:
            lse_out = torch.empty((self.T, self.H), dtype=torch.float32, device=q.device)
        if self.merged:
            mla_attn_merged(q, self.kv_start, self.rows, self.pos, self.req, self.owner_row,
                            o_out, lse_out, softmax_scale=softmax_scale, sink=sink,
                            topk_idx=idx if self.topk else None, stream=stream, **kv)
            if self.dec is not None:
                self.decode(q, o_out, lse_out, softmax_scale=softmax_scale, sink=sink, idx=idx,
                            stream=stream, **kv)
            return o_out, lse_out
        self.attention(q, softmax_scale=softmax_scale, idx=idx, stream=stream, **kv)
        self.merge(o_out, lse_out, sink=sink, stream=stream)
        return o_out, lse_out


def kv_kwargs(prob):
    """The KV tensors of a synth.Problem as keyword arguments."""
    if prob.kv is not None:
        return dict(kv=prob.kv)
    return dict(kv_fp8=prob.kv_fp8, kv_scale=prob.kv_scale, kv_rope=prob.kv_rope)


def plan_for(prob, device="cuda", merged=False, split_decode=False):
    return PcpPrefill(prob.P, prob.cu_seqlens.numpy(), prob.q_start_pos.numpy(),
                      prob.is_decode.numpy(), prob.kv_start.numpy(), prob.H, device=device,
                      topk=prob.topk, merged=merged, split_decode=split_decode)

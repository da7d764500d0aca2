"""mla_attn_split_kv_noalloc: the split-KV attention for callers that cannot
allocate device scratch (a host framework that owns all device memory, a
serving loop whose memory is fixed at start-up) -- the parts' partial
results go to the library's own fixed device array instead of a caller
workspace.  Called through the C ABI, its result must match the workspace
entry point's on two calls in a row (the array keeps the previous call's
contents).  The file name makes pytest collect it last."""
import ctypes

import numpy as np
import pytest
import torch

from context_sparse_mla_gb300 import build as cbuild
from context_sparse_mla_gb300 import cpmla, synth
from tests import parity_util as pu

STATIC_BYTES = 32 << 20  # CPMLA_SPLIT_KV_STATIC_BYTES


def _args(prob, tokens, o, lse, n_split):
    """The C arguments of mla_attn_split_kv_noalloc, as ctypes values."""
    fmt, s_kv = cpmla._attn_common(prob.q, *[cpmla.kv_kwargs(prob).get(k) for k in
                                             ("kv", "kv_fp8", "kv_scale", "kv_rope")])
    kvk = cpmla.kv_kwargs(prob)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    toks = d(tokens)
    pos = d(prob.token_pos().numpy()[tokens])
    req = d(prob.token_req().numpy()[tokens])
    keep = (toks, pos, req, prob.kv_start.cuda())
    k = prob.idx.shape[1] if prob.idx is not None else 0
    args = (cpmla._ptr(prob.q), prob.q.stride(0), prob.H, fmt, cpmla._ptr(kvk.get("kv")),
            cpmla._ptr(kvk.get("kv_fp8")), cpmla._ptr(kvk.get("kv_scale")),
            cpmla._ptr(kvk.get("kv_rope")), s_kv, cpmla._ptr(keep[3]), cpmla._ptr(toks),
            cpmla._ptr(pos), cpmla._ptr(req), len(tokens), cpmla._ptr(prob.idx), k, n_split,
            float(prob.scale), cpmla._ptr(prob.sink), prob.T, cpmla._ptr(o), cpmla._ptr(lse),
            cpmla._stream(None))
    return args, keep


def _assert_close(o, lse, o_ref, lse_ref):
    """The tolerance of the parity tests: |d| <= 1e-2 + 2^-8 |ref|, mean |d|
    <= 1e-3, LSE |d| <= 1e-3."""
    a = o.float().cpu().numpy().astype(np.float64)
    b = o_ref.float().cpu().numpy().astype(np.float64)
    d = np.abs(a - b)
    assert (d - pu.O_REL * np.abs(b)).max() <= pu.O_MAX and d.mean() <= pu.O_MEAN
    la, lb = lse.cpu().numpy(), lse_ref.cpu().numpy()
    assert np.array_equal(np.isfinite(la), np.isfinite(lb))
    fin = np.isfinite(lb)
    assert (np.abs(la[fin] - lb[fin]) <= pu.LSE_MAX).all()


@pytest.mark.gpu
@pytest.mark.parametrize("H,topk,ctx,n_split", [
    (64, 2048, [4096, 131072, 9000, 70000, 5000, 100000] * 4, 8),  # 24 top-k decode rows
    (16, 0, [4096, 131072, 33333], 16),                            # dense, 1024 key tiles
])
def test_no_alloc_matches_the_workspace_entry_point_twice(H, topk, ctx, n_split):
    cbuild.build()
    lib = cpmla.lib()
    cpmla.device_status(clear=True)
    prob = synth.make_problem("varlen_p8_h64", prefill_lens=[], decode_ctx=ctx, H=H, topk=topk,
                              device="cuda", seed=41)
    tokens = np.arange(prob.T, dtype=np.int32)
    assert lib.mla_attn_split_kv_workspace_size(H, len(tokens), n_split) <= STATIC_BYTES
    # the result of the entry point that takes a caller workspace
    o_ref = torch.zeros((prob.T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse_ref = torch.zeros((prob.T, H), dtype=torch.float32, device="cuda")
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    ws = cpmla.split_kv_workspace(H, len(tokens), n_split)
    cpmla.mla_attn_split_kv(prob.q, prob.kv_start.cuda(), d(tokens),
                            d(prob.token_pos().numpy()[tokens]),
                            d(prob.token_req().numpy()[tokens]), o_ref, lse_ref,
                            softmax_scale=prob.scale, n_split=n_split, workspace=ws,
                            sink=prob.sink, topk_idx=prob.idx, **cpmla.kv_kwargs(prob))
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    # two calls in a row of the entry point that allocates nothing
    for call in range(2):
        o = torch.full((prob.T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((prob.T, H), float("nan"), dtype=torch.float32, device="cuda")
        args, keep = _args(prob, tokens, o, lse, n_split)
        rc = lib.mla_attn_split_kv_noalloc(*args)
        assert rc == cpmla.CPMLA_OK, lib.cpmla_last_error()
        torch.cuda.synchronize()
        assert cpmla.device_status() == 0, call
        _assert_close(o, lse, o_ref, lse_ref)
    # and both against the oracle on a few rows
    few = tokens[:3]
    ro, rl = pu.oracle_tokens(prob, few)
    pu.compare(o[:3], lse[:3], ro, rl)


def test_no_alloc_rejects_more_scratch_than_its_array():
    """Checked on the host before any device work: 64 heads x 64 parts x 64
    tokens need ~537 MB of scratch."""
    cbuild.build()
    lib = cpmla.lib()
    need = lib.mla_attn_split_kv_workspace_size(64, 64, 64)
    assert need > STATIC_BYTES
    rc = lib.mla_attn_split_kv_noalloc(None, 576 * 64, 64, 0, None, None, None, None, 16, None,
                                       None, None, None, 64, None, 0, 64, 0.07, None, 64, None,
                                       None, None)
    assert rc == cpmla.CPMLA_ERR_ARG
    msg = lib.cpmla_last_error().decode()
    assert "static array" in msg and str(need) in msg
    # an empty call is a no-op
    assert lib.mla_attn_split_kv_noalloc(None, 576 * 64, 64, 0, None, None, None, None, 16, None,
                                         None, None, None, 0, None, 0, 8, 0.07, None, 1, None,
                                         None, None) == cpmla.CPMLA_OK

"""Split-KV attention of decode rows (one query, long context or top-k list):
each row's keys cut into parts computed side by side, merged with the sink
once; against the fp64 oracle at the stated tolerance."""
import numpy as np
import pytest
import torch

from context_sparse_mla_gb300 import build as cbuild
from context_sparse_mla_gb300 import cpmla, synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cbuild.build()
    cpmla.lib()
    cpmla.device_status(clear=True)
    yield
    torch.cuda.synchronize()


def _decode_problem(ctx, H, topk, kv_format="bf16", seed=0, prefill=()):
    return synth.make_problem("varlen_p8_h64", prefill_lens=list(prefill), decode_ctx=list(ctx),
                              H=H, topk=topk, kv_format=kv_format, device="cuda", seed=seed)


def _run_split(prob, n_split, tokens=None, pos=None, req=None):
    part = cpmla.pcp_dualchunk_partition(prob.P, prob.cu_seqlens.numpy(),
                                         prob.q_start_pos.numpy(), prob.is_decode.numpy())
    if tokens is None:
        tokens = np.flatnonzero(np.repeat(prob.is_decode.numpy(),
                                          np.diff(prob.cu_seqlens.numpy())))
    tokens = np.asarray(tokens, np.int32)
    if pos is None:
        pos = prob.token_pos().numpy()[tokens]
        req = prob.token_req().numpy()[tokens]
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    o = torch.zeros((prob.T, prob.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((prob.T, prob.H), 7.0, dtype=torch.float32, device="cuda")
    ws = cpmla.split_kv_workspace(prob.H, len(tokens), n_split)
    cpmla.mla_attn_split_kv(prob.q, prob.kv_start.cuda(), d(tokens), d(pos), d(req), o, lse,
                            softmax_scale=prob.scale, n_split=n_split, workspace=ws,
                            sink=prob.sink, topk_idx=prob.idx, **cpmla.kv_kwargs(prob))
    torch.cuda.synchronize()
    return o, lse, tokens, part


@pytest.mark.parametrize("n_split", [1, 5, 16])
def test_split_kv_dense_decode_rows_up_to_131072_keys(n_split):
    """Dense decode rows over contexts of 4096 .. 131072 keys (1024 key tiles
    for the longest, cut into n_split parts)."""
    prob = _decode_problem([4096, 33333, 131072, 70001], H=8, topk=0, seed=31)
    o, lse, toks, _ = _run_split(prob, n_split)
    assert cpmla.device_status() == 0
    ro, rl = pu.oracle_tokens(prob, toks)
    ti = torch.as_tensor(toks, device="cuda")
    print(pu.compare(o[ti], lse[ti], ro, rl))


@pytest.mark.parametrize("n_split", [1, 8])
def test_split_kv_sparse_decode_rows_h64(n_split):
    """Top-2048 decode rows, 64 heads (the varlen workload's decode rows)."""
    prob = _decode_problem([4096, 50000, 131072, 9999, 77777], H=64, topk=2048, seed=32)
    o, lse, toks, _ = _run_split(prob, n_split)
    assert cpmla.device_status() == 0
    ro, rl = pu.oracle_tokens(prob, toks)
    ti = torch.as_tensor(toks, device="cuda")
    pu.compare(o[ti], lse[ti], ro, rl)


def test_split_kv_sparse_fp8_decode_rows():
    prob = _decode_problem([4096, 131072, 20000], H=16, topk=2048, kv_format="fp8", seed=33)
    o, lse, toks, _ = _run_split(prob, 4)
    assert cpmla.device_status() == 0
    ro, rl = pu.oracle_tokens(prob, toks)
    ti = torch.as_tensor(toks, device="cuda")
    pu.compare(o[ti], lse[ti], ro, rl)


def test_split_kv_writes_only_the_listed_tokens():
    prob = _decode_problem([5000, 6000, 7000], H=16, topk=512, seed=34)
    o, lse, toks, _ = _run_split(prob, 3, tokens=[2, 0])
    assert cpmla.device_status() == 0
    assert (o[1].float() == 0).all() and (lse[1] == 7.0).all()
    ro, rl = pu.oracle_tokens(prob, [2, 0])
    pu.compare(o[[2, 0]], lse[[2, 0]], ro, rl)


def test_split_kv_more_parts_than_keys_and_a_bad_token():
    """A 5-key context cut into 16 parts (most parts empty); a token outside
    [0, T) is skipped and recorded."""
    prob = _decode_problem([5, 3000], H=16, topk=0, seed=35)
    o, lse, toks, _ = _run_split(prob, 16)
    assert cpmla.device_status() == 0
    ro, rl = pu.oracle_tokens(prob, toks)
    pu.compare(o[torch.as_tensor(toks, device="cuda")], lse[torch.as_tensor(toks, device="cuda")],
               ro, rl)
    # the second listed token's id is outside [0, T) (its position and request
    # are valid): its parts are computed, its merged row is not written
    o2, lse2, _, _ = _run_split(prob, 2, tokens=[0, prob.T + 4],
                                pos=prob.token_pos().numpy()[[0, 1]],
                                req=prob.token_req().numpy()[[0, 1]])
    assert cpmla.device_status(clear=True) == cpmla.CPMLA_ERR_INDEX
    assert (lse2[1] == 7.0).all()
    pu.compare(o2[:1], lse2[:1], ro[:1], rl[:1])


@pytest.mark.parametrize("topk,kv_format", [(2048, "bf16"), (0, "bf16"), (2048, "fp8")])
def test_pcp_path_with_split_decode_rows(topk, kv_format):
    """The whole path on a varlen batch: prefill rows through the merged
    launch (the decode tokens left out of it), decode rows through split-KV
    with one part per shard."""
    prob = synth.make_problem("varlen_p8_h64", prefill_lens=[2500, 1100, 7],
                              decode_ctx=[4100, 9000, 131072], H=16, topk=topk,
                              kv_format=kv_format, device="cuda", seed=36)
    plan = cpmla.plan_for(prob, merged=True, split_decode=True)
    assert plan.dec is not None and plan.dec["tokens"].numel() == 3
    o, lse = plan(prob.q, softmax_scale=prob.scale, sink=prob.sink, idx=prob.idx,
                  **cpmla.kv_kwargs(prob))
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    toks = np.concatenate([pu.sample_tokens(prob, 200), np.arange(prob.T - 3, prob.T)])
    toks = np.unique(toks)
    ro, rl = pu.oracle_tokens(prob, toks)
    ti = torch.as_tensor(toks, device="cuda")
    pu.compare(o[ti], lse[ti], ro, rl)

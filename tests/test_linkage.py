"""The library's ratio-2 linkage (host, through the C ABI) against the oracle,
bit for bit, and the device row gather against the rows it copies."""
import numpy as np
import pytest
import torch

from context_sparse_mla_gb300 import build as cbuild
from context_sparse_mla_gb300 import cpmla, synth
from oracle import oracle as orc
from tests.test_linkage_oracle import _golden_cases, _random_batch

KEYS = ("first", "last", "pred", "pred_shard", "flags")


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return cpmla.lib()


def _same(got, want):
    for k in KEYS:
        assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_linkage_golden_cases(lib, case):
    _same(cpmla.pcp_ratio2_linkage(case["P"], case["cu"], case["qs"], case["dec"]),
          orc.ratio2_linkage(case["P"], case["cu"], case["qs"], case["dec"]))


@pytest.mark.parametrize("seed", range(60))
def test_linkage_bit_exact_against_oracle(lib, seed):
    P, cu, qs, dec = _random_batch(np.random.default_rng(1000 + seed))
    _same(cpmla.pcp_ratio2_linkage(P, cu, qs, dec), orc.ratio2_linkage(P, cu, qs, dec))


@pytest.mark.parametrize("name", ["dense_s8192_h16_p2", "sparse_s32k_h32_p4", "varlen_p8_h64"])
def test_linkage_full_size_workloads(lib, name):
    """The workloads' request structure (tensors are not needed): odd chunk
    starts appear wherever S is not a multiple of 2P."""
    spec = dict(synth.WORKLOADS[name])
    g = torch.Generator().manual_seed(0)
    if spec.get("varlen"):
        plens = torch.randint(spec["len_lo"], spec["len_hi"] + 1, (spec["n_prefill"],),
                              generator=g).tolist()
        dctx = torch.randint(spec["ctx_lo"], spec["ctx_hi"] + 1, (spec["n_decode"],),
                             generator=g).tolist()
    else:
        plens, dctx = [spec["S"]], []
    lens = plens + [1] * len(dctx)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    qs = np.array([0] * len(plens) + [c - 1 for c in dctx], np.int32)
    dec = np.array([0] * len(plens) + [1] * len(dctx), np.uint8)
    got = cpmla.pcp_ratio2_linkage(spec["P"], cu, qs, dec)
    _same(got, orc.ratio2_linkage(spec["P"], cu, qs, dec))
    assert len(got["first"]) == 2 * spec["P"] * len(plens)


def test_linkage_argument_checks(lib):
    with pytest.raises(cpmla.CpmlaError):
        cpmla.pcp_ratio2_linkage(0, [0, 4], [0], [0])
    with pytest.raises(cpmla.CpmlaError):
        cpmla.pcp_ratio2_linkage(2, [0, 4, 2], [0, 0], [0, 0])  # decreasing offsets
    with pytest.raises(cpmla.CpmlaError):
        cpmla.pcp_ratio2_linkage(2, [0, 4], [-1], [0])  # negative position
    f = lib.pcp_gather_rows_f32
    assert f(None, 8, 4, 8, 0, None, None, 8, None) == cpmla.CPMLA_OK  # empty
    assert f(None, 8, 4, 6, 2, None, None, 8, None) == cpmla.CPMLA_ERR_ARG  # D % 4
    assert f(None, 4, 4, 8, 2, None, None, 8, None) == cpmla.CPMLA_ERR_ARG  # stride < D
    assert f(None, 8, 4, 8, 2, None, None, 8, None) == cpmla.CPMLA_ERR_ARG  # NULL
    assert b"pcp_gather_rows_f32" in lib.cpmla_last_error()


@pytest.mark.gpu
def test_gather_rows_copies_each_chunks_predecessor_row():
    """Each chunk's predecessor row, copied out of the rows every shard shares
    on one GPU, bit for bit (fp32 rows of 516 values, a ragged width); chunks
    with no predecessor get zeros; a bad index is recorded and zeroed."""
    cbuild.build()
    P, cu, qs, dec = 4, np.array([0, 37, 50, 51, 150], np.int32), \
        np.array([0, 3, 80, 0], np.int32), np.array([0, 0, 1, 0], np.uint8)
    lk = cpmla.pcp_ratio2_linkage(P, cu, qs, dec)
    T, D = int(cu[-1]), 516
    src = torch.randn((T, D + 4), device="cuda")[:, :D]  # a row stride of D + 4
    idx = torch.from_numpy(lk["pred"]).cuda()
    assert (idx >= 0).any() and (idx < 0).any()
    cpmla.device_status(clear=True)
    out = torch.empty((idx.numel(), D), device="cuda")
    cpmla.lib().pcp_gather_rows_f32(
        cpmla._ptr(src), src.stride(0), T, D, idx.numel(), cpmla._ptr(idx), cpmla._ptr(out),
        out.stride(0), cpmla._stream(None))
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    want = torch.zeros_like(out)
    have = idx >= 0
    want[have] = src[idx[have].long()]
    assert torch.equal(out, want)
    # the all-gathered buffer of every chunk's last row, and a bad index
    last = torch.from_numpy(lk["last"]).cuda()
    last[0] = T + 3
    g = cpmla.pcp_gather_rows_f32(src.contiguous(), last)
    torch.cuda.synchronize()
    assert cpmla.device_status(clear=True) == cpmla.CPMLA_ERR_INDEX
    ok = last >= 0
    ok[0] = False
    assert torch.equal(g[ok], src[last[ok].long()]) and (g[~ok] == 0).all()

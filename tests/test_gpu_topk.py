"""GPU parity of the indexer's top-k selection (mla_topk_select through the C
ABI) with the oracle: bit-exact index lists on seeded logits ("[Feat][NVIDIA]
DeepSeek-V4.1: Prefill support CP with multistream forward prepare (4/N)":
topk_v2 after mqa_logits; the rule is the total order with ties to the
smaller column).  The cases cover rows at or below k, rows short enough to be
all candidates, sampled rows, ties that overflow the candidate buffer (the
fallback over the whole row), signed zeros and -inf, a wide k, and the full
32768-token causal workload the benchmark times."""
import numpy as np
import pytest
import torch

from context_sparse_mla_gb300 import build as cbuild
from context_sparse_mla_gb300 import cpmla, synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cbuild.build()
    cpmla.lib()
    cpmla.device_status(clear=True)
    yield
    torch.cuda.synchronize()


def _case(row_len, width, k, kind, seed):
    x = synth.indexer_logits(len(row_len), width, seed=seed, kind=kind, device="cuda")
    rl = torch.as_tensor(np.asarray(row_len, np.int32), device="cuda")
    got = cpmla.mla_topk_select(x, rl, k)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    want = orc.topk_select(x.cpu().numpy(), np.asarray(row_len), k)
    g = got.cpu().numpy()
    bad = np.nonzero((g != want).any(axis=1))[0]
    assert bad.size == 0, "rows %s differ (row_len %s)" % (bad[:5], np.asarray(row_len)[bad[:5]])


def test_causal_rows_normal():
    # rows 1..3000 with k = 256: at or below k, all-candidate (<= 2k + 2048)
    # and sampled rows, ragged lengths (not multiples of 4 or 32)
    _case(np.arange(1, 3001), 3000, 256, "normal", 1)


def test_random_lengths_every_path():
    rng = np.random.default_rng(2)
    lens = rng.integers(0, 20001, 400)
    lens[:4] = [0, 1, 64, 20000]
    _case(lens, 20000, 512, "normal", 2)


def test_row_to_row_scale_changes_take_the_sample():
    """A CTA's threshold for a row is extrapolated from its previous row and
    checked by the filter's count; rows whose scale and offset change at
    random (x 1000, +- 40) make that guess miss, so those rows take the
    sampled threshold and a second filter pass -- the lists stay exact."""
    n_rows, width, k = 3000, 12000, 512
    x = synth.indexer_logits(n_rows, width, seed=21, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(21)
    big = torch.rand((n_rows, 1), generator=g, device="cuda") < 0.5
    shift = (torch.rand((n_rows, 1), generator=g, device="cuda") - 0.5) * 80.0
    x = (torch.where(big, x * 1000.0, x) + shift).contiguous()
    rl = torch.as_tensor(np.linspace(width, k + 1, n_rows).astype(np.int32), device="cuda")
    got = cpmla.mla_topk_select(x, rl, k)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    want = orc.topk_select(x.cpu().numpy(), rl.cpu().numpy(), k)
    g_ = got.cpu().numpy()
    bad = np.nonzero((g_ != want).any(axis=1))[0]
    assert bad.size == 0, "rows %s differ" % bad[:5]


def test_ties_overflow_the_candidates():
    # seven distinct values and k = 16: the top value alone fills a seventh
    # of a row, beyond the 2k + 2048 candidates for rows over 14560, so the
    # selection of those rows runs over the whole row
    rng = np.random.default_rng(3)
    _case(rng.integers(100, 20001, 120), 20000, 16, "ties", 3)


def test_signed_zeros_inf_and_repeats():
    rng = np.random.default_rng(4)
    _case(rng.integers(1, 16001, 200), 16000, 1024, "mixed", 4)


def test_all_equal_rows():
    x = torch.full((6, 4096), 0.5, device="cuda")
    x[1] = -0.0
    x[2, ::2] = 0.0  # +0 above -0: the even columns first
    x[2, 1::2] = -0.0
    rl = torch.tensor([4096, 4096, 4096, 100, 5000 // 2, 4093], dtype=torch.int32, device="cuda")
    got = cpmla.mla_topk_select(x, rl, 64).cpu().numpy()
    want = orc.topk_select(x.cpu().numpy(), rl.cpu().numpy(), 64)
    assert np.array_equal(got, want)
    assert list(got[0][:3]) == [0, 1, 2] and list(got[2][:3]) == [0, 2, 4]


def test_wide_k():
    rng = np.random.default_rng(5)
    _case(rng.integers(6000, 24001, 48), 24000, 8192, "normal", 5)


def test_bad_row_len_is_recorded_and_skipped():
    x = synth.indexer_logits(3, 256, seed=6, device="cuda")
    rl = torch.tensor([200, 300, 100], dtype=torch.int32, device="cuda")  # 300 > max_row_len
    got = cpmla.mla_topk_select(x, rl, 16, max_row_len=256)
    torch.cuda.synchronize()
    assert cpmla.device_status(clear=True) == cpmla.CPMLA_ERR_INDEX
    assert (got[1] == -1).all()
    want = orc.topk_select(x.cpu().numpy(), [200, 0, 100], 16)
    assert np.array_equal(got.cpu().numpy(), want)


def test_full_size_causal_32k_sampled_rows():
    """The 32768-token request with k = 2048 (the sparse workload's index
    lists), in the launch the benchmark times: every row checked for shape
    and validity, 600 seeded rows (and the longest) against the oracle."""
    S, k = 32768, 2048
    x = synth.indexer_logits(S, S, seed=7, device="cuda")
    rl = torch.arange(1, S + 1, dtype=torch.int32, device="cuda")
    got = cpmla.mla_topk_select(x, rl, k)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    n = torch.clamp(rl, max=k)
    valid = got >= 0
    assert torch.equal(valid.sum(1).to(torch.int32), n)
    assert bool((got < rl[:, None]).all())
    sel = got[:, 1:][valid[:, 1:]]
    assert bool((got[:, 1:] > got[:, :-1])[valid[:, 1:]].all()) and sel.numel() > 0
    rows = np.random.default_rng(8).choice(S, 600, replace=False)
    rows = np.concatenate([rows, [S - 1, k - 1, k, k + 1]])
    ti = torch.as_tensor(rows, device="cuda")
    want = orc.topk_select(x[ti].cpu().numpy(), rl[ti].cpu().numpy(), k)
    assert np.array_equal(got[ti].cpu().numpy(), want)


def test_selected_lists_drive_the_sparse_attention():
    """The index producer feeding the sparse attention: lists selected from
    seeded logits (varlen requests with decode rows, request-local causal
    prefixes) are the oracle's, and the sparse path run on them matches the
    oracle's attention over the same lists."""
    from tests import parity_util as pu
    prob = synth.make_problem("varlen_p8_h64", prefill_lens=[2500, 700, 3], decode_ctx=[3000, 40],
                              H=16, P=4, topk=512, device="cuda", seed=9)
    pos = prob.token_pos()
    row_len = (pos + 1).to(torch.int32)
    width = (int(row_len.max()) + 3) // 4 * 4
    x = synth.indexer_logits(prob.T, width, seed=10, device="cuda")
    idx = cpmla.mla_topk_select(x, row_len.cuda(), prob.topk)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    want = orc.topk_select(x.cpu().numpy(), row_len.numpy(), prob.topk)
    assert np.array_equal(idx.cpu().numpy(), want)
    prob.idx = idx
    o, lse, _ = pu.run_path(prob)
    toks = np.arange(prob.T)
    ro, rl = pu.oracle_tokens(prob, toks)
    pu.compare(o, lse, ro, rl)


def test_maximum_row_length():
    # rows of up to 2^20 columns: a 128 KB column bitmap per CTA
    w = 1 << 20
    _case([w, w - 3, 5000, 0], w, 2048, "normal", 11)


def test_maximum_k_takes_the_whole_row_path():
    # k = 65536 exceeds the candidate buffer, so every row longer than k is
    # selected over the row in global memory
    _case([70000, 65536, 65537, 100], 70000, 65536, "normal", 12)

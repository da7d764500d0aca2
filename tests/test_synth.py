"""The seeded generator draws valid inputs: top-k lists sorted, unique, inside
the causal prefix, with min(t+1, k) entries and -1 padding; varlen structure as
described; deterministic under a seed."""
import numpy as np
import torch

from context_sparse_mla_gb300 import synth


def _check_idx(idx, pos, k):
    idx = idx.numpy()
    for t, row in zip(pos.tolist(), idx):
        v = row[row >= 0]
        assert len(v) == min(t + 1, k)
        assert np.all(row[len(v):] == -1)
        assert np.all(np.diff(v) > 0) and v[0] >= 0 and v[-1] <= t


def test_topk_lists_valid_all_three_regimes():
    g = torch.Generator().manual_seed(0)
    k = 16
    pos = torch.tensor([0, 3, 15, 16, 17, 40, 63, 64, 65, 500, 5000], dtype=torch.int32)
    idx = synth.sample_topk(pos, k, g, "cpu")
    _check_idx(idx, pos, k)


def test_topk_uniform_marginals():
    # each position of [0, t] is picked with probability k / (t + 1)
    g = torch.Generator().manual_seed(1)
    k, t, n = 8, 99, 4000
    for tt in (t, 9 * t):  # both drawing regimes
        idx = synth.sample_topk(torch.full((n,), tt, dtype=torch.int32), k, g, "cpu")
        counts = np.bincount(idx.numpy().ravel(), minlength=tt + 1)
        p = k / (tt + 1)
        expect = n * p
        sd = np.sqrt(n * p * (1 - p))
        assert np.abs(counts - expect).max() < 6 * sd


def test_problem_deterministic_and_shapes():
    a = synth.make_problem("varlen_p8_h64", prefill_lens=[40, 9], decode_ctx=[30, 70], H=2, topk=8)
    b = synth.make_problem("varlen_p8_h64", prefill_lens=[40, 9], decode_ctx=[30, 70], H=2, topk=8)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.idx, b.idx)
    assert a.T == 40 + 9 + 2 and a.kv.shape == (40 + 9 + 30 + 70, 576)
    assert a.kv_start.tolist() == [0, 40, 49, 79]
    assert a.q_start_pos.tolist() == [0, 0, 29, 69] and a.is_decode.tolist() == [0, 0, 1, 1]
    _check_idx(a.idx, a.token_pos(), 8)


def test_fp8_problem_fields():
    p = synth.make_problem("sparse_s128k_h16_p2_fp8", S=300, H=2, topk=32)
    assert p.kv is None and p.kv_fp8.dtype == torch.uint8 and p.kv_fp8.shape == (300, 512)
    assert p.kv_scale.shape == (300, 4) and float(p.kv_scale.min()) >= 0.5 and float(p.kv_scale.max()) <= 2.0
    assert p.kv_rope.dtype == torch.bfloat16 and p.kv_rope.shape == (300, 64)


def test_default_workload_shapes():
    p = synth.make_problem("dense_s256_h4_p2")
    assert p.q.shape == (256, 4, 576) and p.kv.shape == (256, 576) and p.P == 2 and p.topk == 0
    assert synth.attended_keys(p) == 256 * 257 // 2

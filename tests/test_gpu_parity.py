"""GPU parity: the CUDA path (partition -> partial attention -> merge with sink,
all through the C ABI) against the fp64 oracle, element by element, on seeded
inputs.  Small cases compare every token; the full-size workloads compare a
seeded sample of >= 4096 tokens (all heads, all 512 channels each) in the same
launch configuration the benchmark times."""
import numpy as np
import pytest
import torch

from context_sparse_mla_gb300 import build as cbuild
from context_sparse_mla_gb300 import cpmla, synth
from oracle import oracle as orc
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cbuild.build()
    cpmla.lib()
    cpmla.device_status(clear=True)
    yield
    torch.cuda.synchronize()


def _check_all(prob):
    o, lse, _ = pu.run_path(prob)
    toks = np.arange(prob.T)
    ro, rl = pu.oracle_tokens(prob, toks)
    return pu.compare(o, lse, ro, rl)


def _check_sample(prob, n, seed=0):
    o, lse, _ = pu.run_path(prob)
    toks = pu.sample_tokens(prob, n, seed)
    ro, rl = pu.oracle_tokens(prob, toks)
    ti = torch.as_tensor(toks, device=o.device)
    return pu.compare(o[ti], lse[ti], ro, rl)


# ----------------------------------------------------------------- dense
def test_dense_tiny_workload_every_token():
    prob = synth.make_problem("dense_s256_h4_p2", device="cuda")
    _check_all(prob)


def test_dense_ragged_multi_tile_every_token():
    prob = synth.make_problem("dense_s8192_h16_p2", S=1000, device="cuda", seed=3)
    _check_all(prob)


@pytest.mark.parametrize("H", [1, 5, 8, 24, 32, 40, 64, 128])
def test_dense_head_groupings(H):
    """Heads per work item: hc = H (at most 64) over 64 // hc tokens.  A
    multiple of 8 takes Q by TMA: 8 (eight tokens), 24 (48 of 64 rows, the
    rest zero padding), 40 (one token, 24 padding rows); others load Q
    through registers."""
    prob = synth.make_problem("dense_s8192_h16_p2", S=300, H=H, P=3, device="cuda", seed=H)
    _check_all(prob)


def test_dense_varlen_with_decode_rows():
    prob = synth.make_problem("varlen_p8_h64", prefill_lens=[700, 5, 260], decode_ctx=[900, 33],
                              H=8, P=3, topk=0, device="cuda", seed=5)
    _check_all(prob)


def test_dense_fewer_tokens_than_chunks():
    prob = synth.make_problem("dense_s256_h4_p2", S=5, P=4, device="cuda", seed=8)
    _check_all(prob)


# ----------------------------------------------------------------- sparse
def test_sparse_bf16_h32_p4():
    prob = synth.make_problem("sparse_s32k_h32_p4", S=3000, device="cuda", seed=1)
    _check_sample(prob, 300)


def test_sparse_fp8_h16_p2():
    prob = synth.make_problem("sparse_s128k_h16_p2_fp8", S=2600, device="cuda", seed=2)
    _check_sample(prob, 300)


def test_sparse_fp8_subnormal_codes_decode_exactly():
    """A latent of E4M3 zeros and subnormals only (exponent field 0, values
    m * 2^-9), scaled by 32 so they carry values up to ~0.44: a decode that
    flushed subnormals to zero would zero V and the latent part of every
    score."""
    prob = synth.make_problem("sparse_s128k_h16_p2_fp8", S=400, topk=128, device="cuda", seed=17)
    g = torch.Generator().manual_seed(17)
    shape = tuple(prob.kv_fp8.shape)
    codes = torch.randint(0, 8, shape, generator=g) | (torch.randint(0, 2, shape, generator=g) << 7)
    prob.kv_fp8 = codes.to(torch.uint8).to("cuda")
    prob.kv_scale = torch.full_like(prob.kv_scale, 32.0)
    _check_all(prob)


@pytest.mark.parametrize("name", ["sparse_s32k_h32_p4", "sparse_s128k_h16_p2_fp8"])
def test_sparse_max_heads(name):
    """H = 128, the largest head count: four (bf16) or eight (fp8) head groups
    per token, each CTA gathering the token's keys for its own group."""
    prob = synth.make_problem(name, S=600, H=128, topk=256, device="cuda", seed=18)
    _check_sample(prob, 96)


@pytest.mark.parametrize("H", [8, 64])
def test_sparse_wide_topk(H):
    """k = 8192: 64 key tiles per token, far past the 16 of the workloads."""
    prob = synth.make_problem("sparse_s32k_h32_p4", S=9000, H=H, topk=8192, device="cuda",
                              seed=19)
    _check_sample(prob, 48)


def test_sparse_varlen_h64_p8_decode():
    prob = synth.make_problem("varlen_p8_h64", prefill_lens=[2500, 1100], decode_ctx=[4100, 9000],
                              device="cuda", seed=4)
    _check_sample(prob, 200)


@pytest.mark.parametrize("H", [1, 16, 24, 40, 64])
def test_sparse_unsorted_lists_with_holes(H):
    """Top-k lists need not be sorted and may hold -1 anywhere."""
    prob = synth.make_problem("sparse_s32k_h32_p4", S=700, H=H, topk=200, device="cuda", seed=H)
    g = torch.Generator(device="cuda").manual_seed(11)
    idx = prob.idx.clone()
    perm = torch.argsort(torch.rand(idx.shape, generator=g, device="cuda"), dim=1)
    idx = torch.gather(idx, 1, perm)
    holes = torch.rand(idx.shape, generator=g, device="cuda") < 0.2
    holes[:, 0] = False
    idx[holes & (torch.arange(idx.shape[0], device="cuda")[:, None] > 0)] = -1
    prob.idx = idx.contiguous()
    _check_all(prob)


@pytest.mark.parametrize("H", [16, 24, 64])
def test_sparse_rows_with_empty_lists(H):
    """Rows whose top-k list holds no key (all -1) get O = 0 and LSE = -inf;
    their neighbours are unaffected."""
    prob = synth.make_problem("sparse_s32k_h32_p4", S=500, H=H, topk=160, device="cuda", seed=25)
    idx = prob.idx.clone()
    idx[7] = -1
    idx[250:260] = -1
    idx[499] = -1
    prob.idx = idx.contiguous()
    _check_all(prob)


@pytest.mark.parametrize("H", [16, 64])
def test_sparse_out_of_prefix_index_is_skipped_and_flagged(H):
    prob = synth.make_problem("sparse_s32k_h32_p4", S=400, H=H, topk=64, device="cuda", seed=6)
    bad_tok = 300
    idx = prob.idx.clone()
    idx[bad_tok, 0] = 350  # outside [0, 300]
    prob.idx = idx
    plan = cpmla.plan_for(prob)
    o, lse = plan(prob.q, softmax_scale=prob.scale, sink=prob.sink, idx=prob.idx,
                  **cpmla.kv_kwargs(prob))
    assert cpmla.device_status(clear=True) == cpmla.CPMLA_ERR_INDEX
    fixed = idx.clone()
    fixed[bad_tok, 0] = -1
    prob.idx = fixed
    ro, rl = pu.oracle_tokens(prob, [bad_tok])
    pu.compare(o[bad_tok:bad_tok + 1], lse[bad_tok:bad_tok + 1], ro, rl)


# ----------------------------------------------------------------- merge
def test_kv_split_partials_merge_to_full_attention():
    """General N-partial merge: every row's keys split into the 2P DualChunkSwap
    KV chunks, one partial per chunk (restricted by kv_lo/kv_hi), merged by the
    GPU merge with the sink once."""
    S, H, P = 700, 16, 2
    prob = synth.make_problem("dense_s8192_h16_p2", S=S, H=H, P=P, device="cuda", seed=9)
    dev = "cuda"
    base, rem = divmod(S, 2 * P)
    bounds, st = [], 0
    for c in range(2 * P):
        ln = base + (1 if c < rem else 0)
        bounds.append((st, st + ln - 1))
        st += ln
    C = len(bounds)
    rows = torch.arange(S, dtype=torch.int32, device=dev).repeat(C)
    pos = rows.clone()
    req = torch.zeros_like(rows)
    lo = torch.tensor([b[0] for b in bounds], dtype=torch.int32, device=dev).repeat_interleave(S)
    hi = torch.tensor([b[1] for b in bounds], dtype=torch.int32, device=dev).repeat_interleave(S)
    kv_start = prob.kv_start.to(dev)
    o_part = torch.empty((C * S, H, 512), dtype=torch.float32, device=dev)
    lse_part = torch.empty((C * S, H), dtype=torch.float32, device=dev)
    cpmla.mla_partial_attn_dense(prob.q, kv_start, rows, pos, req, o_part, lse_part,
                                 softmax_scale=prob.scale, kv=prob.kv, kv_lo=lo, kv_hi=hi)
    off = torch.arange(0, C * S + 1, C, dtype=torch.int32, device=dev)
    contrib = (torch.arange(S, dtype=torch.int32, device=dev)[:, None]
               + S * torch.arange(C, dtype=torch.int32, device=dev)[None, :]).reshape(-1)
    o = torch.empty((S, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((S, H), dtype=torch.float32, device=dev)
    cpmla.lse_merge_with_sink(o_part, lse_part, contrib.contiguous(), o, lse, contrib_off=off,
                              sink=prob.sink)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    # partials of rows whose chunk lies wholly after them are empty
    assert torch.isneginf(lse_part[S * (C - 1)]).all()
    ro, rl = pu.oracle_tokens(prob, np.arange(S))
    pu.compare(o, lse, ro, rl)


# ------------------------------------------------ merge folded into attention
@pytest.mark.parametrize("name,kw", [
    ("dense_s8192_h16_p2", dict(S=1000, seed=21)),
    ("dense_s8192_h16_p2", dict(S=700, H=24, seed=26)),
    ("sparse_s32k_h32_p4", dict(S=3000, seed=22)),
    ("sparse_s128k_h16_p2_fp8", dict(S=2600, seed=23)),
    ("varlen_p8_h64", dict(prefill_lens=[2500, 1100], decode_ctx=[4100, 9000], seed=24)),
])
def test_merged_epilogue_matches_oracle_and_two_launch_path(name, kw):
    """The single-partial merge folded into the attention epilogue: parity
    with the oracle, and the same bits as partial attention + merge kernel
    (both compute (O / l) * 1 / (1 + e^(sink - L)) in fp32 in that order)."""
    prob = synth.make_problem(name, device="cuda", **kw)
    o2, l2, _ = pu.run_path(prob)
    plan = cpmla.plan_for(prob, merged=True)
    o1, l1 = plan(prob.q, softmax_scale=prob.scale, sink=prob.sink, idx=prob.idx,
                  **cpmla.kv_kwargs(prob))
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    toks = pu.sample_tokens(prob, 256)
    ro, rl = pu.oracle_tokens(prob, toks)
    ti = torch.as_tensor(toks, device=o1.device)
    pu.compare(o1[ti], l1[ti], ro, rl)


def test_merged_epilogue_full_size_dense_sampled():
    prob = synth.make_problem("dense_s8192_h16_p2", device="cuda", seed=0)
    plan = cpmla.plan_for(prob, merged=True)
    o, lse = plan(prob.q, softmax_scale=prob.scale, sink=prob.sink, **cpmla.kv_kwargs(prob))
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    toks = pu.sample_tokens(prob, 4096)
    ro, rl = pu.oracle_tokens(prob, toks)
    ti = torch.as_tensor(toks, device=o.device)
    pu.compare(o[ti], lse[ti], ro, rl)


# ------------------------------------------------------------- cache insertion
def _insert_case(n, s_cache, seed, fmt):
    g = torch.Generator().manual_seed(seed)
    kv = (torch.randn((n, 576), generator=g) * torch.exp(torch.randn((n, 1), generator=g)))
    kv = kv.to(torch.bfloat16)
    kv[min(3, n - 1), 128:256] = 0  # an all-zero group
    slot = torch.randperm(s_cache, generator=g)[:n].to(torch.int64)
    slot[:: max(1, n // 7)] = -1  # skipped tokens
    bits = kv.view(torch.int16).numpy().view(np.uint16)
    want = orc.kv_insert(bits, slot.numpy(), fmt=fmt, s_cache=s_cache)
    if fmt == 0:
        cache = torch.zeros((s_cache, 576), dtype=torch.bfloat16, device="cuda")
        cpmla.mla_kv_cache_insert(kv.cuda(), slot.cuda(), cache=cache)
        got = dict(kv=cache.cpu().view(torch.int16).numpy().view(np.uint16))
    else:
        c8 = torch.zeros((s_cache, 512), dtype=torch.uint8, device="cuda")
        cs = torch.zeros((s_cache, 4), dtype=torch.float32, device="cuda")
        cr = torch.zeros((s_cache, 64), dtype=torch.bfloat16, device="cuda")
        cpmla.mla_kv_cache_insert(kv.cuda(), slot.cuda(), cache_fp8=c8, cache_scale=cs,
                                  cache_rope=cr)
        got = dict(kv_fp8=c8.cpu().numpy(), kv_scale=cs.cpu().numpy(),
                   kv_rope=cr.cpu().view(torch.int16).numpy().view(np.uint16))
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    for k in want:  # bytes and binary32 scales: bit-exact
        assert np.array_equal(got[k].view(np.uint8), want[k].view(np.uint8)), k


@pytest.mark.parametrize("fmt", [0, 1])
def test_kv_cache_insert_bit_exact(fmt):
    _insert_case(3001, 4000, 30 + fmt, fmt)


def test_kv_cache_insert_fp8_full_size():
    """The fp8 cache of the 131072-token sparse workload, every token inserted."""
    _insert_case(131072, 131072 + 5, 32, 1)


def _rounding_boundary_rows(n, seed):
    """bf16 KV rows whose fp8 quotients x / scale sit on E4M3 rounding
    midpoints but for the rounding of the scale itself: per 128-channel group
    the amax A = (32 + u) 2^a has six significant bits (so A / 448 = A / (7 .
    64) is inexact unless 7 divides 32 + u), and element x = +-3 A 2^(E - 10)
    gives x / (A / 448) = 21 . 2^(E - 4) = 2^(E) (1 + 5/16), the midpoint
    between two E4M3 values of that binade; the binary32 quotient lands one
    ulp to one side of it, so a division off by one ulp flips the code."""
    rng = np.random.default_rng(seed)
    x = np.zeros((n, 576), np.float32)
    for t in range(n):
        for g in range(4):
            u = int(rng.integers(0, 32))
            a = int(rng.integers(-24, 24))
            A = np.float32((32 + u) * 2.0 ** a)
            grp = np.float32(A) * rng.integers(-31, 32, 128).astype(np.float32) / np.float32(64)
            grp[0] = A
            for k in range(1, 40):
                E = -6 + (k % 15)
                grp[k] = np.float32((1 if rng.random() < 0.5 else -1) * 3.0 * float(A) * 2.0 ** (E - 10))
            x[t, 128 * g:128 * (g + 1)] = grp
        x[t, 512:] = rng.standard_normal(64)
    kv = torch.from_numpy(x).to(torch.bfloat16)  # the filler rounds; A and the +-3 A 2^(E-10) do not
    lat = kv[:, :512].float().view(n, 4, 128)
    want = torch.from_numpy(x[:, :512]).view(n, 4, 128)
    assert torch.equal(lat[:, :, :40], want[:, :, :40]), "boundary elements not bf16-exact"
    assert (lat.abs().amax(-1) == want[:, :, 0]).all(), "A is not the group's amax"
    return kv


def test_kv_cache_insert_fp8_rounding_boundaries():
    """The fp8 insertion's quotients next to E4M3 rounding midpoints: codes
    and scales bit-exact with the oracle's binary32 division."""
    n, s_cache = 2048, 2048
    kv = _rounding_boundary_rows(n, 41)
    slot = torch.arange(n, dtype=torch.int64)
    bits = kv.view(torch.int16).numpy().view(np.uint16)
    want = orc.kv_insert(bits, slot.numpy(), fmt=1, s_cache=s_cache)
    c8 = torch.zeros((s_cache, 512), dtype=torch.uint8, device="cuda")
    cs = torch.zeros((s_cache, 4), dtype=torch.float32, device="cuda")
    cr = torch.zeros((s_cache, 64), dtype=torch.bfloat16, device="cuda")
    cpmla.mla_kv_cache_insert(kv.cuda(), slot.cuda(), cache_fp8=c8, cache_scale=cs, cache_rope=cr)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    assert np.array_equal(cs.cpu().numpy().view(np.uint32), want["kv_scale"].view(np.uint32))
    assert np.array_equal(c8.cpu().numpy(), want["kv_fp8"])


def test_merge_kernel_against_oracle_merge():
    rng = np.random.default_rng(17)
    n_part, H, T = 300, 6, 120
    op = rng.standard_normal((n_part, H, 512)).astype(np.float32)
    lp = (rng.standard_normal((n_part, H)) * 3).astype(np.float32)
    lp[rng.random((n_part, H)) < 0.1] = -np.inf
    counts = rng.integers(0, 4, T)
    counts[:3] = [1, 2, 3]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    contrib = rng.integers(0, n_part, off[-1]).astype(np.int32)
    sink = rng.standard_normal(H).astype(np.float32)
    for s in (sink, None):
        ro, rl = orc.merge(op.astype(np.float64), lp.astype(np.float64), off, contrib, sink=s)
        d = lambda a: torch.from_numpy(a).cuda()
        o = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
        cpmla.lse_merge_with_sink(d(op), d(lp), d(contrib), o, lse, contrib_off=d(off),
                                  sink=None if s is None else d(s))
        torch.cuda.synchronize()
        og = o.float().cpu().numpy().astype(np.float64)
        # the stated bounds: |d| <= 1e-2 + 2^-8 |O_ref| (the bf16 output's own
        # rounding), mean |d| <= 1e-3, LSE |d| <= 1e-3
        d = np.abs(og - ro)
        assert (d - pu.O_REL * np.abs(ro)).max() <= pu.O_MAX, d.max()
        assert d.mean() <= pu.O_MEAN, d.mean()
        fin = np.isfinite(rl)
        lg = lse.cpu().numpy()
        assert np.array_equal(np.isfinite(lg), fin)
        assert np.abs(lg[fin] - rl[fin]).max() <= pu.LSE_MAX
        assert (og[counts == 0] == 0).all()


def test_merge_flags_a_bad_partial_row_even_when_it_is_the_only_one():
    """A token whose only contrib row lies outside [0, n_part) gets O = 0 and
    LSE = -inf, and the bad index is recorded in the status word."""
    n_part, H, T = 8, 2, 3
    op = torch.randn((n_part, H, 512), device="cuda")
    lp = torch.randn((n_part, H), device="cuda")
    off = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device="cuda")
    contrib = torch.tensor([2, n_part + 5, 4], dtype=torch.int32, device="cuda")
    o = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    cpmla.device_status(clear=True)
    cpmla.lse_merge_with_sink(op, lp, contrib, o, lse, contrib_off=off)
    assert cpmla.device_status(clear=True) == cpmla.CPMLA_ERR_INDEX
    assert (o[1].float() == 0).all() and torch.isneginf(lse[1]).all()
    assert torch.equal(lse[0], lp[2]) and torch.equal(lse[2], lp[4])


def test_repeat_runs_bitwise_identical():
    prob = synth.make_problem("dense_s8192_h16_p2", S=900, device="cuda", seed=12)
    o1, l1, _ = pu.run_path(prob)
    o2, l2, _ = pu.run_path(prob)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


@pytest.mark.parametrize("name,kw", [
    ("sparse_s128k_h16_p2_fp8", dict(S=6000, seed=5)),
    ("sparse_s32k_h32_p4", dict(S=3000, H=16, seed=31)),
    ("sparse_s32k_h32_p4", dict(S=3000, seed=22)),
    ("varlen_p8_h64", dict(prefill_lens=[2500, 1100], decode_ctx=[4100, 9000], seed=24)),
])
def test_sparse_repeat_runs_bitwise_identical(name, kw):
    """The sparse kernel's warps hand shared-memory slots to one another
    through mbarriers; a missing wait shows up as a run that differs from the
    others (a few whole tokens, not rounding).  Twelve merged-output runs of
    each kernel shape (fp8 16 heads, bf16 16 / 32 / 64 heads) must agree bit
    for bit."""
    prob = synth.make_problem(name, device="cuda", **kw)
    plan = cpmla.plan_for(prob, merged=True)
    kv = cpmla.kv_kwargs(prob)
    ref = None
    for _ in range(12):
        o, lse = plan(prob.q, softmax_scale=prob.scale, sink=prob.sink, idx=prob.idx, **kv)
        torch.cuda.synchronize()
        assert cpmla.device_status() == 0
        if ref is None:
            ref = (o.clone(), lse.clone())
        else:
            assert torch.equal(o.view(torch.int16), ref[0].view(torch.int16))
            assert torch.equal(lse, ref[1])


@pytest.mark.parametrize("merged", [False, True])
def test_dense_repeat_runs_bitwise_identical(merged):
    """The dense kernel's warps hand ring slots, S^T buffers, P^T and O^T to
    one another through mbarriers; a phase passed one use early shows up as a
    run that differs from the others (whole rows, not rounding).  Twelve runs
    of 750 work items (several waves of CTAs) must agree bit for bit, with the
    two-launch path and with the merged epilogue."""
    prob = synth.make_problem("dense_s8192_h16_p2", S=3000, device="cuda", seed=27)
    plan = cpmla.plan_for(prob, merged=merged)
    kv = cpmla.kv_kwargs(prob)
    ref = None
    for _ in range(12):
        o, lse = plan(prob.q, softmax_scale=prob.scale, sink=prob.sink, idx=prob.idx, **kv)
        torch.cuda.synchronize()
        assert cpmla.device_status() == 0
        if ref is None:
            ref = (o.clone(), lse.clone())
        else:
            assert torch.equal(o.view(torch.int16), ref[0].view(torch.int16))
            assert torch.equal(lse, ref[1])


# ----------------------------------------------------- full-size workloads
@pytest.mark.parametrize("name", ["dense_s8192_h16_p2", "sparse_s32k_h32_p4",
                                  "sparse_s128k_h16_p2_fp8", "varlen_p8_h64"])
def test_full_size_workload_sampled_4096_tokens(name):
    torch.cuda.empty_cache()
    prob = synth.make_problem(name, device="cuda", seed=0)
    stats = _check_sample(prob, 4096, seed=1)
    print(name, stats)
    del prob
    torch.cuda.empty_cache()


# ------------------------------------------------------ failure detection
def test_bounded_wait_times_out_and_context_survives():
    """A pipeline wait that is never satisfied gives up after its limit,
    records CPMLA_ERR_TIMEOUT in the status word and exits normally; the CUDA
    context keeps working (the small dense workload still matches)."""
    import time
    t0 = time.time()
    assert cpmla.selftest_wait_timeout(200) == cpmla.CPMLA_ERR_TIMEOUT
    assert time.time() - t0 < 30
    assert cpmla.device_status() == 0
    prob = synth.make_problem("dense_s256_h4_p2", device="cuda", seed=1)
    _check_all(prob)


# ------------------------------------------------------ more edge cases
def test_sparse_fp8_two_head_groups():
    prob = synth.make_problem("sparse_s128k_h16_p2_fp8", S=900, H=32, topk=256, device="cuda",
                              seed=13)
    _check_sample(prob, 200)


@pytest.mark.parametrize("H", [16, 48])
def test_sparse_topk_width_not_a_tile_multiple(H):
    prob = synth.make_problem("sparse_s32k_h32_p4", S=700, H=H, topk=300, device="cuda", seed=14)
    _check_all(prob)


@pytest.mark.parametrize("H", [16, 64])
def test_sparse_kv_split_partials_merge_to_full_attention(H):
    """KV-split on the sparse path: each row's top-k keys restricted to the
    2P chunks in turn, merged on the GPU with the sink once."""
    S, P, k = 600, 2, 64
    prob = synth.make_problem("sparse_s32k_h32_p4", S=S, H=H, P=P, topk=k, device="cuda", seed=15)
    dev = "cuda"
    base, rem = divmod(S, 2 * P)
    bounds, st = [], 0
    for c in range(2 * P):
        ln = base + (1 if c < rem else 0)
        bounds.append((st, st + ln - 1))
        st += ln
    C = len(bounds)
    rows = torch.arange(S, dtype=torch.int32, device=dev).repeat(C)
    req = torch.zeros_like(rows)
    lo = torch.tensor([b[0] for b in bounds], dtype=torch.int32, device=dev).repeat_interleave(S)
    hi = torch.tensor([b[1] for b in bounds], dtype=torch.int32, device=dev).repeat_interleave(S)
    o_part = torch.empty((C * S, H, 512), dtype=torch.float32, device=dev)
    lse_part = torch.empty((C * S, H), dtype=torch.float32, device=dev)
    cpmla.mla_partial_attn_sparse(prob.q, prob.kv_start.to(dev), rows, rows.clone(), req, prob.idx,
                                  o_part, lse_part, softmax_scale=prob.scale, kv=prob.kv,
                                  kv_lo=lo, kv_hi=hi)
    off = torch.arange(0, C * S + 1, C, dtype=torch.int32, device=dev)
    contrib = (torch.arange(S, dtype=torch.int32, device=dev)[:, None]
               + S * torch.arange(C, dtype=torch.int32, device=dev)[None, :]).reshape(-1)
    o = torch.empty((S, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((S, H), dtype=torch.float32, device=dev)
    cpmla.lse_merge_with_sink(o_part, lse_part, contrib.contiguous(), o, lse, contrib_off=off,
                              sink=prob.sink)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    ro, rl = pu.oracle_tokens(prob, np.arange(S))
    pu.compare(o, lse, ro, rl)


def test_empty_calls_are_no_ops():
    prob = synth.make_problem("dense_s256_h4_p2", device="cuda", seed=2)
    z = torch.zeros(0, dtype=torch.int32, device="cuda")
    o = torch.empty((0, 4, 512), dtype=torch.float32, device="cuda")
    l = torch.empty((0, 4), dtype=torch.float32, device="cuda")
    cpmla.mla_partial_attn_dense(prob.q, prob.kv_start.cuda(), z, z, z, o, l,
                                 softmax_scale=prob.scale, kv=prob.kv)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0

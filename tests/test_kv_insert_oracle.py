"""Pins of the oracle's KV-cache insertion ("[Core] Add MRV2 virtual-batch PCP
for MLA", Summary: sparse MLA cache insertion; the fp8_ds_mla cache dtype of
"[Feature][PCP] Add DeepSeek-V4.1-Flash support") and of its E4M3 encoder,
against the format's own values, an independent library conversion and the
properties the quantisation rule (per-128-channel amax / 448 scale, round to
nearest even) fixes."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc

FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_encode_round_trips_every_finite_code():
    vals = orc.e4m3_to_float64(np.array(FINITE, np.uint8)).astype(np.float32)
    assert list(orc.e4m3_encode(vals)) == FINITE


def test_encode_rounds_midpoints_to_even_codes():
    # between adjacent codes c < c+1 of one sign the midpoint has five
    # significant bits, so it is a binary32 value; it must go to the code with
    # the even last fraction bit (the even code, also across a binade)
    for base in (0x00, 0x80):
        for c in range(base, base + 0x7E):
            lo, hi = orc.e4m3_to_float64(np.array([c, c + 1], np.uint8))
            mid = np.float32((lo + hi) / 2)
            want = c if c % 2 == 0 else c + 1
            assert orc.e4m3_encode(np.array([mid]))[0] == want, hex(c)


def test_encode_saturates_and_keeps_nan_and_signed_zero():
    x = np.array([448.0, 463.9, 464.0, 480.0, 1e30, np.inf, -448.5, -np.inf, np.nan, 0.0, -0.0],
                 np.float32)
    assert list(orc.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F,
                                        0x00, 0x80]
    # below the smallest subnormal 2^-9: half of it ties to zero, more rounds up
    x = np.array([2.0 ** -10, 1.25 * 2.0 ** -10, 0.5 * 2.0 ** -10], np.float32)
    assert list(orc.e4m3_encode(x)) == [0x00, 0x01, 0x00]


def test_encode_matches_torch_float8_e4m3fn_inside_the_finite_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-3, 2, 20000),
                        rng.uniform(-447.9, 447.9, 5000)]).astype(np.float32)
    x = x[np.abs(x) < 448.0]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(x), want)


def _random_kv(n, seed):
    g = torch.Generator().manual_seed(seed)
    kv = torch.randn((n, 576), generator=g) * torch.exp(torch.randn((n, 1), generator=g))
    return kv.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_fp8_insert_properties():
    n, s_cache = 64, 100
    kv = _random_kv(n, 1)
    kv[3, 128:256] = 0  # an all-zero group
    slot = np.random.default_rng(2).permutation(s_cache)[:n].astype(np.int64)
    slot[5] = -1
    c = orc.kv_insert(kv, slot, fmt=1, s_cache=s_cache)
    x = orc.bf16_to_float64(kv).astype(np.float32)
    for t in range(n):
        s = slot[t]
        if s < 0:
            continue
        assert np.array_equal(c["kv_rope"][s], kv[t, 512:])
        for g in range(4):
            xg = x[t, 128 * g:128 * (g + 1)]
            codes = c["kv_fp8"][s, 128 * g:128 * (g + 1)]
            scale = c["kv_scale"][s, g]
            amax = np.float32(np.abs(xg).max())
            if amax == 0:
                assert scale == 1.0 and not codes.any()
                continue
            assert scale == amax / np.float32(448.0)
            # the largest magnitude lands on +-448
            assert (codes[np.abs(xg) == amax] & 0x7F == 0x7E).all()
            # dequantised within half a step: 2^-4 relative for normals,
            # 2^-10 * scale for subnormals
            back = orc.e4m3_to_float64(codes) * scale
            assert (np.abs(back - xg) <= 2.0 ** -4 * np.abs(xg) + 2.0 ** -10 * scale + 1e-12).all()
    untouched = np.setdiff1d(np.arange(s_cache), slot[slot >= 0])
    assert not c["kv_fp8"][untouched].any() and not c["kv_scale"][untouched].any()


def test_bf16_insert_is_a_copy_and_rejects_bad_slots():
    kv = _random_kv(10, 3)
    slot = np.array([9, 0, -1, 4, 5, 6, 7, 8, 1, 2], np.int64)
    c = orc.kv_insert(kv, slot, fmt=0, s_cache=10)
    for t in range(10):
        if slot[t] >= 0:
            assert np.array_equal(c["kv"][slot[t]], kv[t])
    assert not c["kv"][3].any()
    with pytest.raises(ValueError):
        orc.kv_insert(kv, np.array([0] * 9 + [10], np.int64), fmt=0, s_cache=10)

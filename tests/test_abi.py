"""The C-ABI library builds, loads without a GPU, exports every entry point its
header declares, partitions bit-exactly like the oracle, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from context_sparse_mla_gb300 import build as cbuild
from context_sparse_mla_gb300 import cpmla
from oracle import oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return cpmla.lib()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"pcp_dualchunk_partition", "mla_partial_attn_dense", "mla_partial_attn_sparse",
            "lse_merge_with_sink", "mla_attn_dense_merged", "mla_attn_sparse_merged",
            "mla_kv_cache_insert", "mla_topk_select"} <= set(names)
    h = ctypes.CDLL(cpmla.LIB_PATH)
    for n in names:
        assert hasattr(h, n), n
    assert lib.cpmla_version() >= 100


@pytest.mark.parametrize("seed", range(6))
def test_partition_bit_exact_against_oracle(lib, seed):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(1, 9))
    B = int(rng.integers(1, 7))
    dec = (rng.random(B) < 0.3).astype(np.uint8)
    lens = np.where(dec == 1, 1, rng.integers(0, 200, B))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    qs = np.where(dec == 1, rng.integers(1, 1000, B), 0).astype(np.int32)
    got = cpmla.pcp_dualchunk_partition(P, cu, qs, dec)
    want = orc.partition(P, cu, qs, dec)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


def test_partition_full_size_workloads_bit_exact(lib):
    from context_sparse_mla_gb300 import synth
    for name, P, cu, qs, dec in [
        ("dense_s8192", 2, [0, 8192], [0], [0]),
        ("sparse_s32k", 4, [0, 32768], [0], [0]),
        ("sparse_s128k", 2, [0, 131072], [0], [0]),
    ]:
        got = cpmla.pcp_dualchunk_partition(P, cu, qs, dec)
        want = orc.partition(P, cu, qs, dec)
        for k in want:
            assert np.array_equal(got[k], want[k]), (name, k)
    # the varlen workload's structure (lengths drawn by the generator, no tensors)
    g = torch.Generator().manual_seed(0)
    plens = torch.randint(1024, 65537, (8,), generator=g).tolist()
    dctx = torch.randint(4096, 131073, (32,), generator=g).tolist()
    cu = np.concatenate([[0], np.cumsum(plens + [1] * 32)]).astype(np.int32)
    qs = np.array([0] * 8 + [c - 1 for c in dctx], np.int32)
    dec = np.array([0] * 8 + [1] * 32, np.uint8)
    got = cpmla.pcp_dualchunk_partition(8, cu, qs, dec)
    want = orc.partition(8, cu, qs, dec)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


def test_partition_rejects_bad_arguments(lib):
    with pytest.raises(cpmla.CpmlaError) as e:
        cpmla.pcp_dualchunk_partition(0, [0, 4], [0], [0])
    assert e.value.code == cpmla.CPMLA_ERR_ARG
    with pytest.raises(cpmla.CpmlaError):
        cpmla.pcp_dualchunk_partition(2, [0, 5, 3], [0, 0], [0, 0])  # decreasing offsets
    with pytest.raises(cpmla.CpmlaError):
        cpmla.pcp_dualchunk_partition(2, [1, 5], [0], [0])  # offsets not starting at 0
    with pytest.raises(cpmla.CpmlaError):
        cpmla.pcp_dualchunk_partition(2, [0, 5], [-3], [0])  # negative position


def _raw_dense(lib, **over):
    a = dict(q=None, qs=576 * 4, H=4, fmt=0, kv=None, kv8=None, ksc=None, krope=None, s_kv=16,
             kv_start=None, rows=None, pos=None, req=None, n=1, lo=None, hi=None, scale=0.07,
             o=None, lse=None, stream=None)
    a.update(over)
    return lib.mla_partial_attn_dense(*a.values())


def test_attention_argument_checks_fail_before_the_device(lib):
    assert _raw_dense(lib, n=0) == cpmla.CPMLA_OK  # empty is a no-op
    assert _raw_dense(lib) == cpmla.CPMLA_ERR_ARG  # NULL pointers
    assert _raw_dense(lib, H=0) == cpmla.CPMLA_ERR_ARG
    assert _raw_dense(lib, H=96) == cpmla.CPMLA_ERR_ARG
    assert b"H=96" in lib.cpmla_last_error()
    assert _raw_dense(lib, qs=100) == cpmla.CPMLA_ERR_ARG
    assert _raw_dense(lib, scale=float("nan")) == cpmla.CPMLA_ERR_ARG
    assert _raw_dense(lib, fmt=1) == cpmla.CPMLA_ERR_UNSUPPORTED  # dense takes bf16 KV only
    assert _raw_dense(lib, fmt=7) == cpmla.CPMLA_ERR_ARG
    rc = lib.mla_partial_attn_sparse(None, 576, 1, 0, None, None, None, None, 16, None, None, None,
                                     None, 1, None, None, None, 0, 0.07, None, None, None)
    assert rc == cpmla.CPMLA_ERR_ARG  # k = 0
    # sparse over the fp8 cache takes 16 heads a CTA: H = 24 is refused, 48 passes this check
    rc = lib.mla_partial_attn_sparse(None, 576 * 24, 24, 1, None, None, None, None, 16, None, None,
                                     None, None, 1, None, None, None, 8, 0.07, None, None, None)
    assert rc == cpmla.CPMLA_ERR_UNSUPPORTED
    assert b"H=24" in lib.cpmla_last_error()
    rc = lib.mla_partial_attn_sparse(None, 576 * 48, 48, 1, None, None, None, None, 16, None, None,
                                     None, None, 1, None, None, None, 8, 0.07, None, None, None)
    assert rc == cpmla.CPMLA_ERR_ARG  # past the head check: NULL pointers


def test_merged_attention_argument_checks(lib):
    base = [None, 576 * 4, 4, 0, None, None, None, None, 16, None, None, None, None]
    # empty is a no-op; otherwise o_out, owner_row and lse_out are required
    assert lib.mla_attn_dense_merged(*base, 0, None, None, 0.07, None, 0, None, None, None,
                                     None) == cpmla.CPMLA_OK
    assert lib.mla_attn_dense_merged(*base, 1, None, None, 0.07, None, 4, None, None, None,
                                     None) == cpmla.CPMLA_ERR_ARG
    assert b"o_out" in lib.cpmla_last_error()
    assert lib.mla_attn_sparse_merged(*base, 1, None, None, None, 8, 0.07, None, -1, None, None,
                                      None, None) == cpmla.CPMLA_ERR_ARG


def test_kv_cache_insert_argument_checks(lib):
    f = lib.mla_kv_cache_insert
    assert f(None, 576, 0, None, 0, None, None, None, None, 16, None) == cpmla.CPMLA_OK
    assert f(None, 576, 4, None, 0, None, None, None, None, 16, None) == cpmla.CPMLA_ERR_ARG
    assert f(None, 576, 4, None, 5, None, None, None, None, 16, None) == cpmla.CPMLA_ERR_ARG
    assert f(None, 500, 4, None, 0, None, None, None, None, 16, None) == cpmla.CPMLA_ERR_ARG
    assert f(None, 576, 4, None, 0, None, None, None, None, 0, None) == cpmla.CPMLA_ERR_ARG
    assert f(None, 576, -1, None, 0, None, None, None, None, 16, None) == cpmla.CPMLA_ERR_ARG
    assert b"mla_kv_cache_insert" in lib.cpmla_last_error()


def test_topk_select_argument_checks(lib):
    f = lib.mla_topk_select
    assert f(None, 64, 0, None, 64, 8, None, None) == cpmla.CPMLA_OK
    assert f(None, 64, 4, None, 64, 0, None, None) == cpmla.CPMLA_ERR_ARG  # k = 0
    assert f(None, 64, 4, None, 64, 65537, None, None) == cpmla.CPMLA_ERR_ARG
    assert f(None, 62, 4, None, 60, 8, None, None) == cpmla.CPMLA_ERR_ARG  # stride % 4
    assert f(None, 64, 4, None, 65, 8, None, None) == cpmla.CPMLA_ERR_ARG  # stride < max_row_len
    assert f(None, 1 << 21, 4, None, (1 << 20) + 1, 8, None, None) == cpmla.CPMLA_ERR_ARG
    assert f(None, 64, -1, None, 64, 8, None, None) == cpmla.CPMLA_ERR_ARG
    assert f(None, 64, 4, None, 64, 8, None, None) == cpmla.CPMLA_ERR_ARG  # row_len NULL
    assert b"mla_topk_select" in lib.cpmla_last_error()


def test_merge_argument_checks(lib):
    assert lib.lse_merge_with_sink(None, None, 0, 4, None, None, 0, None, None, None, None) == 0
    assert lib.lse_merge_with_sink(None, None, 0, 0, None, None, 3, None, None, None, None) == -1
    assert lib.lse_merge_with_sink(None, None, 5, 4, None, None, 3, None, None, None, None) == -1
    msg = lib.cpmla_last_error().decode()
    assert "NULL" in msg


def test_selftest_limit_checked_before_the_device(lib):
    assert lib.cpmla_selftest_wait_timeout(0, None) == cpmla.CPMLA_ERR_ARG
    assert lib.cpmla_selftest_wait_timeout(5000, None) == cpmla.CPMLA_ERR_ARG


def test_split_kv_argument_checks(lib):
    size = lib.mla_attn_split_kv_workspace_size
    assert size(64, 32, 8) >= 32 * 8 * 64 * (512 * 4 + 4)
    assert size(64, 32, 8) < size(64, 32, 9) and size(0, 1, 1) == 0 and size(4, 1, 0) == 0
    f = lib.mla_attn_split_kv
    base = [None, 576 * 4, 4, 0, None, None, None, None, 16, None]
    # empty is a no-op; n_split outside 1..64; a missing or short workspace
    assert f(*base, None, None, None, 0, None, 0, 4, 0.07, None, 1, None, None, None, 0,
             None) == cpmla.CPMLA_OK
    assert f(*base, None, None, None, 1, None, 0, 0, 0.07, None, 1, None, None, None, 0,
             None) == cpmla.CPMLA_ERR_ARG
    assert f(*base, None, None, None, 1, None, 0, 65, 0.07, None, 1, None, None, None, 0,
             None) == cpmla.CPMLA_ERR_ARG
    buf = ctypes.create_string_buffer(1 << 12)
    addr = (ctypes.addressof(buf) + 255) & ~255
    assert f(*base, 8, 8, 8, 1, None, 0, 2, 0.07, None, 1, 8, 8, addr, 16,
             None) == cpmla.CPMLA_ERR_ARG
    assert b"workspace" in lib.cpmla_last_error()

"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on chosen global tokens, and compare with the stated
tolerances.

O: |d| <= 1e-2 + 2^-8 * |O_ref| per element and mean |d| <= 1e-3; LSE:
|d| <= 1e-3.  The absolute 1e-2 is the stated bound for unit-scale outputs;
the output is bf16, whose own rounding of a value of magnitude m reaches
m * 2^-8 (half a unit in the last place of an 8-bit significand), so each
element may also carry its own rounding on top of it.  Rows with very few
keys have O close to a single value row (up to ~4.5 for N(0,1) data, ~10 for
the fp8 cache's scaled values), which is where that term matters."""
import numpy as np
import torch

from context_sparse_mla_gb300 import cpmla
from oracle import oracle as orc

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3
O_REL = 2.0 ** -8  # bf16 output rounding of the element itself


def run_path(prob):
    plan = cpmla.plan_for(prob)
    o, lse = plan(prob.q, softmax_scale=prob.scale, sink=prob.sink, idx=prob.idx,
                  **cpmla.kv_kwargs(prob))
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    return o, lse, plan


def bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def kv_host(prob):
    if prob.kv is not None:
        return dict(kv_bf16=bits(prob.kv))
    return dict(kv_fp8=prob.kv_fp8.cpu().numpy(), kv_scale=prob.kv_scale.cpu().numpy(),
                kv_rope=bits(prob.kv_rope))


def oracle_tokens(prob, tokens, kvh=None):
    """fp64 plain-definition attention (sink applied, LSE without it) of the
    given global tokens."""
    tokens = np.asarray(tokens, np.int64)
    pos = prob.token_pos().numpy()[tokens]
    req = prob.token_req().numpy()[tokens]
    q = bits(prob.q[torch.as_tensor(tokens, device=prob.q.device)])
    idx = None
    if prob.idx is not None:
        idx = prob.idx[torch.as_tensor(tokens, device=prob.idx.device)].cpu().numpy()
    return orc.attention(q, pos, prob.kv_start.numpy()[req], topk=idx, scale=prob.scale,
                         sink=prob.sink.cpu().numpy(), **(kvh or kv_host(prob)))


def compare(o_gpu, lse_gpu, o_ref, lse_ref):
    og = o_gpu.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.float().cpu().numpy().astype(np.float64)
    d = np.abs(og - o_ref)
    dl = np.abs(lg - lse_ref)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin), "LSE finiteness differs"
    excess = d - O_REL * np.abs(o_ref)  # what is left after the element's own rounding
    stats = dict(o_max=float(d.max()), o_max_excess=float(excess.max()), o_mean=float(d.mean()),
                 o_max_unit=float(d[np.abs(o_ref) <= 1.0].max()) if (np.abs(o_ref) <= 1).any()
                 else 0.0,
                 lse_max=float(dl[fin].max()) if fin.any() else 0.0)
    assert stats["o_max_excess"] <= O_MAX, stats
    assert stats["o_mean"] <= O_MEAN, stats
    assert stats["lse_max"] <= LSE_MAX, stats
    return stats


def sample_tokens(prob, n, seed=0):
    """Seeded sample of n global tokens, always including the first and last
    token of every request and the DualChunkSwap chunk edges of each prefill."""
    T = prob.T
    must = set()
    for b in range(prob.B):
        a, e = int(prob.cu_seqlens[b]), int(prob.cu_seqlens[b + 1])
        if e == a:
            continue
        must.update([a, e - 1])
        S = e - a
        if not int(prob.is_decode[b]):
            base, rem = divmod(S, 2 * prob.P)
            st = 0
            for c in range(2 * prob.P):
                ln = base + (1 if c < rem else 0)
                if ln:
                    must.update([a + st, a + st + ln - 1])
                st += ln
    rng = np.random.default_rng(seed)
    rest = rng.choice(T, size=min(T, max(0, n - len(must))), replace=False)
    return np.array(sorted(must.union(rest.tolist())), np.int64)

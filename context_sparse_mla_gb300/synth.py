"""Seeded synthetic inputs shaped like the long-context prefill workloads of the
source pages (vLLM ``bench serve`` random prompts of exact lengths, 8K-1M
tokens; see "[Feature][PCP] Add DeepSeek-V4.1-Flash support", benchmark
tables, and "[DeepSeekV4][PCP] ...", TTFT tables).

This module only draws random numbers and lays them out.  It holds none of the
method's arithmetic (no partition, no attention, no merge), so both the CUDA
path and the CPU oracle can be fed from it.

Workloads (``WORKLOADS``):
  dense_s256_h4_p2      1 request, 256 tokens, 4 heads, P=2, dense causal
  dense_s8192_h16_p2    1 request, 8192 tokens, 16 heads, P=2, dense causal
  sparse_s32k_h32_p4    1 request, 32768 tokens, 32 heads, P=4, top-2048
  sparse_s128k_h16_p2_fp8  131072 tokens, 16 heads, P=2, top-2048, fp8 latent
  varlen_p8_h64         8 prefills of U[1024,65536] tokens + 32 decode rows
                        over contexts U[4096,131072], 64 heads, P=8, top-2048
  varlen_p8_h64_s16k, sparse_s12k_h32_p4   smaller cases of the same shapes
All values bf16 ~N(0,1); sink ~N(0,1) fp32 per head; softmax scale 1/sqrt(192).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

DQK, DV, DROPE, GROUP = 576, 512, 64, 128
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)


@dataclass
class Problem:
    name: str
    P: int
    H: int
    topk: int                      # 0 = dense causal
    kv_format: str                 # "bf16" or "fp8"
    cu_seqlens: torch.Tensor       # int32 [B+1], host
    q_start_pos: torch.Tensor      # int32 [B], host
    is_decode: torch.Tensor        # uint8 [B], host
    kv_start: torch.Tensor         # int64 [B], host: KV row of position 0
    q: torch.Tensor                # bf16 [T, H, 576]
    sink: torch.Tensor             # fp32 [H]
    kv: Optional[torch.Tensor] = None        # bf16 [S_kv, 576]
    kv_fp8: Optional[torch.Tensor] = None    # uint8 [S_kv, 512] (E4M3 codes)
    kv_scale: Optional[torch.Tensor] = None  # fp32 [S_kv, 4]
    kv_rope: Optional[torch.Tensor] = None   # bf16 [S_kv, 64]
    idx: Optional[torch.Tensor] = None       # int32 [T, topk], -1 padded
    scale: float = SOFTMAX_SCALE
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def B(self) -> int:
        return len(self.cu_seqlens) - 1

    def token_pos(self) -> torch.Tensor:
        """Position of every global token within its request (int32, host)."""
        out = torch.empty(self.T, dtype=torch.int32)
        for b in range(self.B):
            a, e = int(self.cu_seqlens[b]), int(self.cu_seqlens[b + 1])
            out[a:e] = torch.arange(e - a, dtype=torch.int32) + int(self.q_start_pos[b])
        return out

    def token_req(self) -> torch.Tensor:
        out = torch.empty(self.T, dtype=torch.int32)
        for b in range(self.B):
            out[int(self.cu_seqlens[b]):int(self.cu_seqlens[b + 1])] = b
        return out


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def sample_topk(pos: torch.Tensor, k: int, gen: torch.Generator, device,
                batch_rows: int = 4096) -> torch.Tensor:
    """Per query row at position t: sorted unique indices drawn uniformly from
    [0, t] (every position when t + 1 <= k), -1 padded to k.

    A uniformly random k-subset is drawn in one of two exact ways:
      * n = t + 1 <= 4k: random priorities for all n positions, keep the k
        smallest (a uniform random k-subset);
      * n > 4k: 3k iid uniform draws, duplicates dropped, then a uniform
        random k-subset of the distinct values (uniform by exchangeability);
        a row with fewer than k distinct draws is redrawn the first way.
    """
    pos = pos.to(device=device, dtype=torch.int64)
    T = pos.numel()
    out = torch.full((T, k), -1, dtype=torch.int32, device=device)
    if T == 0 or k == 0:
        return out
    n_all = pos + 1
    ar_k = torch.arange(k, device=device)
    # rows that take every position
    small = torch.nonzero(n_all <= k).flatten()
    for s in range(0, small.numel(), batch_rows):
        rows = small[s:s + batch_rows]
        n = n_all[rows]
        vals = ar_k.unsqueeze(0).expand(rows.numel(), k)
        out[rows] = torch.where(vals < n.unsqueeze(1), vals, torch.full_like(vals, -1)).to(torch.int32)

    def by_priority(rows):
        n = n_all[rows]
        nmax = int(n.max())
        pri = torch.rand((rows.numel(), nmax), generator=gen, device=device)
        cols = torch.arange(nmax, device=device).unsqueeze(0)
        pri = torch.where(cols < n.unsqueeze(1), pri, torch.full_like(pri, 2.0))
        sel = torch.topk(pri, k, dim=1, largest=False).indices
        return torch.sort(sel, dim=1).values.to(torch.int32)

    mid = torch.nonzero((n_all > k) & (n_all <= 4 * k)).flatten()
    for s in range(0, mid.numel(), batch_rows // 4 or 1):
        rows = mid[s:s + (batch_rows // 4 or 1)]
        out[rows] = by_priority(rows)
    big = torch.nonzero(n_all > 4 * k).flatten()
    m = 3 * k
    for s in range(0, big.numel(), batch_rows):
        rows = big[s:s + batch_rows]
        n = n_all[rows].unsqueeze(1)
        u = torch.rand((rows.numel(), m), generator=gen, device=device, dtype=torch.float64)
        draws = torch.clamp((u * n).floor().to(torch.int64), max=n - 1)
        draws = torch.sort(draws, dim=1).values
        dup = torch.zeros_like(draws, dtype=torch.bool)
        dup[:, 1:] = draws[:, 1:] == draws[:, :-1]
        pri = torch.rand((rows.numel(), m), generator=gen, device=device)
        pri = torch.where(dup, torch.full_like(pri, 2.0), pri)
        sel = torch.topk(pri, k, dim=1, largest=False).indices
        picked = torch.gather(draws, 1, sel)
        ok = torch.gather(dup, 1, sel).logical_not().all(dim=1)
        out[rows] = torch.sort(picked, dim=1).values.to(torch.int32)
        redo = rows[~ok]
        if redo.numel():
            out[redo] = by_priority(redo)
    return out


def quantize_e4m3(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even to OCP E4M3 and return the stored bytes (uint8)."""
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def make_problem(name: str, *, seed: int = 0, device="cpu", S: int | None = None,
                 H: int | None = None, P: int | None = None, topk: int | None = None,
                 kv_format: str | None = None, prefill_lens=None, decode_ctx=None) -> Problem:
    """Build a seeded problem.  ``name`` picks a workload from ``WORKLOADS``;
    keyword overrides give smaller parity cases of the same structure."""
    spec = dict(WORKLOADS[name])
    for k_, v_ in dict(S=S, H=H, P=P, topk=topk, kv_format=kv_format,
                       prefill_lens=prefill_lens, decode_ctx=decode_ctx).items():
        if v_ is not None:
            spec[k_] = v_
    gen_host = _gen(seed, "cpu")
    # request structure
    if spec.get("varlen"):
        if spec.get("prefill_lens") is not None:
            plens = [int(x) for x in spec["prefill_lens"]]
        else:
            plens = torch.randint(spec["len_lo"], spec["len_hi"] + 1, (spec["n_prefill"],),
                                  generator=gen_host).tolist()
        if spec.get("decode_ctx") is not None:
            dctx = [int(x) for x in spec["decode_ctx"]]
        else:
            dctx = torch.randint(spec["ctx_lo"], spec["ctx_hi"] + 1, (spec["n_decode"],),
                                 generator=gen_host).tolist()
    else:
        plens, dctx = [spec["S"]], []
    q_lens = plens + [1] * len(dctx)
    B = len(q_lens)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    q_start = torch.tensor([0] * len(plens) + [c - 1 for c in dctx], dtype=torch.int32)
    is_dec = torch.tensor([0] * len(plens) + [1] * len(dctx), dtype=torch.uint8)
    kv_lens = plens + dctx
    kv_start = torch.zeros(B, dtype=torch.int64)
    if B > 1:
        kv_start[1:] = torch.cumsum(torch.tensor(kv_lens[:-1], dtype=torch.int64), 0)
    S_kv = int(sum(kv_lens))
    T = int(cu[-1])
    Hn = spec["H"]
    gen = _gen(seed + 1, device)
    q = normal_bf16((T, Hn, DQK), gen, device)
    sink = torch.randn((Hn,), generator=gen_host, dtype=torch.float32).to(device)
    prob = Problem(name=name, P=spec["P"], H=Hn, topk=spec.get("topk", 0),
                   kv_format=spec.get("kv_format", "bf16"), cu_seqlens=cu, q_start_pos=q_start,
                   is_decode=is_dec, kv_start=kv_start, q=q, sink=sink,
                   meta=dict(prefill_lens=plens, decode_ctx=dctx, S_kv=S_kv, seed=seed))
    if prob.kv_format == "bf16":
        prob.kv = normal_bf16((S_kv, DQK), gen, device)
    else:
        lat = torch.randn((S_kv, DV), generator=gen, device=device, dtype=torch.float32)
        prob.kv_fp8 = quantize_e4m3(lat)
        prob.kv_scale = torch.rand((S_kv, DV // GROUP), generator=gen, device=device) * 1.5 + 0.5
        prob.kv_rope = normal_bf16((S_kv, DROPE), gen, device)
    if prob.topk:
        prob.idx = sample_topk(prob.token_pos(), prob.topk, gen, device)
    return prob


WORKLOADS = {
    "dense_s256_h4_p2": dict(S=256, H=4, P=2, topk=0, kv_format="bf16"),
    "dense_s8192_h16_p2": dict(S=8192, H=16, P=2, topk=0, kv_format="bf16"),
    "sparse_s32k_h32_p4": dict(S=32768, H=32, P=4, topk=2048, kv_format="bf16"),
    "sparse_s128k_h16_p2_fp8": dict(S=131072, H=16, P=2, topk=2048, kv_format="fp8"),
    "varlen_p8_h64": dict(varlen=True, n_prefill=8, len_lo=1024, len_hi=65536, n_decode=32,
                          ctx_lo=4096, ctx_hi=131072, H=64, P=8, topk=2048, kv_format="bf16"),
    # smaller cases of the same kernels, for profiler captures (inputs larger
    # than L2: 1.2 GB of Q, 168 MB of KV; 3.8 GB of Q, 38 MB of KV; 302 MB of
    # Q, 11 MB of fp8 KV)
    "varlen_p8_h64_s16k": dict(varlen=True, prefill_lens=[9000, 7000], decode_ctx=[40000, 90000],
                               H=64, P=8, topk=2048, kv_format="bf16"),
    "sparse_s12k_h32_p4": dict(S=12288, H=32, P=4, topk=2048, kv_format="bf16"),
    "sparse_s16k_h16_p2_fp8": dict(S=16384, H=16, P=2, topk=2048, kv_format="fp8"),
}


def attended_keys(prob: Problem) -> int:
    """Number of (query token, key) pairs the workload attends: the causal
    triangle for dense, the valid top-k entries for sparse.  Each decode row
    is counted once."""
    pos = prob.token_pos().to(torch.int64)
    if prob.topk == 0:
        return int((pos + 1).sum())
    return int(torch.clamp(pos + 1, max=prob.topk).sum())


# ------------------------------------------------------------ indexer logits
def indexer_logits(n_rows: int, width: int, *, seed: int = 0, kind: str = "normal",
                   device="cpu") -> torch.Tensor:
    """Seeded fp32 [n_rows, width] stand-in for an indexer's scores (trained
    indexer weights are not available):
      normal  N(0,1) per entry
      ties    integers in [-3, 3] (long runs of equal values)
      mixed   N(0,1) with 10% +0, 5% -0, 5% -inf and 10% copies of one value
    Drawn on ``device`` with a generator of that device."""
    gen = torch.Generator(device=device).manual_seed(seed)
    if kind == "ties":
        return torch.randint(-3, 4, (n_rows, width), generator=gen, device=device).float()
    x = torch.randn((n_rows, width), generator=gen, device=device)
    if kind == "mixed":
        u = torch.rand((n_rows, width), generator=gen, device=device)
        x[u < 0.10] = 0.0
        x[(u >= 0.10) & (u < 0.15)] = -0.0
        x[(u >= 0.15) & (u < 0.20)] = -math.inf
        x[(u >= 0.20) & (u < 0.30)] = 0.75
    elif kind != "normal":
        raise ValueError("unknown logits kind %r" % kind)
    return x

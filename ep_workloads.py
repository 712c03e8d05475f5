"""Seeded synthetic inputs for MoE dispatch / combine.

This module only draws random inputs; it holds none of the dispatch or
combine arithmetic.  Both the CPU oracle (through the tests) and the CUDA
path (through the tests, ``bench.py`` and the smoke run) take their inputs
from here, so both sides always see the same bytes.

Every array is drawn on the CPU from a ``torch.Generator`` with a fixed seed.
The five named workloads follow the routing regimes the DeepEP pages describe
(DeepEP README, "Performance" tables: 4096-token prefill batches with hidden
7168, top-4 groups and top-8 experts; 128-token-per-rank decode batches with
hidden 7168 and top-8).  There is no public dataset behind those numbers; the
recipes below stand in for real router outputs.

Routing recipes
---------------
uniform   top-k experts chosen uniformly without replacement per token.
group     DeepSeek-V3 group-limited routing: logits N(0,1) over the experts,
          group score = max logit in the group, keep the top groups, then the
          top-k logits among their experts; weights = sigmoid(logit) divided by
          their sum over the chosen experts.
zipf      top-k sampled without replacement from a Zipf(s) expert popularity
          p_e ~ (e+1)^-s (skewed load).
softmax   top-k of softmax(N(0,1) logits); the weights are the top-k
          probabilities, not renormalised.
An optional Bernoulli(p_drop) mask sets slots to -1 (empty slot).  Weights of
empty slots are 0; for "uniform" and "zipf" the weights are a softmax of
N(0,1) logits over the valid slots only.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_tokens: int            # T
    hidden: int                # H
    num_experts: int           # E
    num_ranks: int             # R (logical ranks; experts are split in contiguous blocks)
    num_topk: int              # K
    num_max_tokens_per_rank: int  # M; token t comes from logical rank t // M
    expert_alignment: int      # A
    routing: str               # uniform | group | zipf | softmax
    drop_prob: float = 0.0     # Bernoulli probability of an empty (-1) slot
    num_groups: int = 0        # group routing: number of expert groups
    topk_groups: int = 0       # group routing: groups kept per token
    zipf_s: float = 0.0        # zipf routing exponent
    use_fp8: bool = False
    col_major_sf: bool = False
    do_expand: bool = False
    do_zero_padding: bool = False
    do_cpu_sync: bool = True
    expert_bias_std: float = 0.0  # >0: per-expert BF16 bias [E, H] ~ N(0, std)
    fixed_capacity: bool = False  # fixed-capacity per-expert layout (M * R rows per expert)


WORKLOADS = {
    "tiny": Workload("tiny", 128, 256, 16, 4, 2, 32, 8, "uniform", drop_prob=0.05,
                     do_expand=True, do_zero_padding=True, do_cpu_sync=True),
    "decode": Workload("decode", 1024, 7168, 256, 8, 8, 128, 1, "uniform",
                       use_fp8=True, col_major_sf=False, do_expand=False,
                       do_cpu_sync=False),
    "prefill": Workload("prefill", 4096, 7168, 256, 8, 8, 512, 128, "group",
                        num_groups=8, topk_groups=4, use_fp8=True, col_major_sf=True,
                        do_expand=True, do_zero_padding=True, do_cpu_sync=True),
    "skewed": Workload("skewed", 16384, 4096, 64, 8, 6, 2048, 1, "zipf", drop_prob=0.02,
                       zipf_s=1.2, do_expand=False, do_cpu_sync=True, expert_bias_std=0.1),
    "decode_ll": Workload("decode_ll", 1024, 7168, 256, 8, 8, 128, 1, "uniform",
                          use_fp8=True, col_major_sf=True, do_expand=True, do_cpu_sync=False,
                          fixed_capacity=True),
    "large": Workload("large", 32768, 7168, 256, 32, 8, 1024, 128, "softmax",
                      use_fp8=True, col_major_sf=True, do_expand=True,
                      do_zero_padding=True, do_cpu_sync=False),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _masked_softmax(logits: torch.Tensor, valid: torch.Tensor) -> torch.Tensor:
    z = logits.masked_fill(~valid, float("-inf"))
    w = torch.softmax(z, dim=1)
    return torch.nan_to_num(w, nan=0.0).masked_fill(~valid, 0.0)


def make_routing(wl: Workload, seed: int, num_tokens: Optional[int] = None):
    """Return ``(topk_idx int64 [T,K], topk_weights float32 [T,K])``."""
    T = wl.num_tokens if num_tokens is None else num_tokens
    E, K = wl.num_experts, wl.num_topk
    g = _gen(seed)
    if wl.routing == "uniform":
        idx = torch.rand(T, E, generator=g).topk(K, dim=1).indices
        logits = torch.randn(T, K, generator=g)
        weights = None
    elif wl.routing == "group":
        logits_all = torch.randn(T, E, generator=g)
        G = wl.num_groups
        gscore = logits_all.view(T, G, E // G).amax(dim=2)
        keep = gscore.topk(wl.topk_groups, dim=1).indices
        gmask = torch.zeros(T, G, dtype=torch.bool).scatter_(1, keep, True)
        emask = gmask.repeat_interleave(E // G, dim=1)
        sel = logits_all.masked_fill(~emask, float("-inf")).topk(K, dim=1)
        idx = sel.indices
        s = torch.sigmoid(sel.values)
        weights = s / s.sum(dim=1, keepdim=True)
        logits = None
    elif wl.routing == "zipf":
        p = (torch.arange(E, dtype=torch.float64) + 1.0).pow(-wl.zipf_s)
        idx = torch.multinomial(p.to(torch.float32).expand(T, E).contiguous(), K,
                                replacement=False, generator=g)
        logits = torch.randn(T, K, generator=g)
        weights = None
    elif wl.routing == "softmax":
        probs = torch.softmax(torch.randn(T, E, generator=g), dim=1)
        sel = probs.topk(K, dim=1)
        idx, weights, logits = sel.indices, sel.values, None
    else:
        raise ValueError(f"unknown routing {wl.routing!r}")
    idx = idx.to(torch.int64)
    if wl.drop_prob > 0.0:
        drop = torch.rand(T, K, generator=g) < wl.drop_prob
        idx = idx.masked_fill(drop, -1)
    valid = idx >= 0
    if weights is None:
        weights = _masked_softmax(logits, valid)
    else:
        weights = weights.masked_fill(~valid, 0.0)
    return idx.contiguous(), weights.to(torch.float32).contiguous()


def make_x(wl: Workload, seed: int, num_tokens: Optional[int] = None,
           std: float = 1.0) -> torch.Tensor:
    """Token activations, BF16 N(0, std^2) [T, H]."""
    T = wl.num_tokens if num_tokens is None else num_tokens
    g = _gen(seed + 1_000_003)
    return (torch.randn(T, wl.hidden, generator=g) * std).to(torch.bfloat16)


def make_expert_bias(wl: Workload, seed: int) -> Optional[torch.Tensor]:
    if wl.expert_bias_std <= 0.0:
        return None
    g = _gen(seed + 2_000_003)
    return (torch.randn(wl.num_experts, wl.hidden, generator=g)
            * wl.expert_bias_std).to(torch.bfloat16)


def make_bf16_rows(rows: int, hidden: int, seed: int, std: float = 1.0) -> torch.Tensor:
    """Generic BF16 N(0, std^2) matrix, e.g. expert outputs or per-token bias."""
    g = _gen(seed + 3_000_017)
    return (torch.randn(rows, hidden, generator=g) * std).to(torch.bfloat16)


def make_inputs(name_or_wl, seed: int = 0, num_tokens: Optional[int] = None) -> dict:
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    idx, w = make_routing(wl, seed, num_tokens)
    return {
        "workload": wl,
        "topk_idx": idx,
        "topk_weights": w,
        "x": make_x(wl, seed, num_tokens),
        "expert_bias": make_expert_bias(wl, seed),
    }


def replace(wl: Workload, **kw) -> Workload:
    return dataclasses.replace(wl, **kw)


def hashed_bf16_rows(rows, hidden: int, seed: int, device="cpu") -> torch.Tensor:
    """Counter-based BF16 matrix: element (r, c) depends only on (seed, r, c).

    Rows can be produced one subset at a time and on any device with
    identical bits, so the CPU side can rebuild exactly the rows it needs of
    a large matrix that lives in device memory.  Integer arithmetic only
    (every product stays below 2^62, so nothing overflows int64).  Values
    are +-m * 2^k with k in [-3, 1], roughly unit scale.
    """
    r = torch.as_tensor(rows, dtype=torch.int64, device=device).reshape(-1, 1)
    c = torch.arange(hidden, dtype=torch.int64, device=device).reshape(1, -1)
    m31 = 0x7FFFFFFF
    h = (r * 40503 + c * 2654435 + seed * 97 + 12345) & m31
    for _ in range(3):
        h = ((h * 1103515245 + 12345) & m31) ^ (h >> 13)
    sign = (h & 1) << 15
    expo = 124 + ((h >> 1) % 5)                # biased exponent 124..128
    mant = (h >> 4) & 0x7F
    bits = sign | (expo << 7) | mant
    bits = torch.where(bits >= 0x8000, bits - 0x10000, bits).to(torch.int16)
    return bits.view(torch.bfloat16)

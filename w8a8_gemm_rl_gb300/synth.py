"""Seeded synthetic workloads shared by the tests, the smoke check and the bench.

This module only draws random numbers and rounds them to BF16; it holds none
of the quantization or GEMM arithmetic.  The shapes and value distributions
stand in for the workloads the FP8-RL pages train on (Qwen3-8B dense and
Qwen3-30B-A3B MoE rollouts), which are not available here:

* activations: N(0, 1) with 0.1% of the entries multiplied by 50 (outliers),
  drawn in FP32 and rounded to BF16 (round to nearest even);
* weights: N(0, 0.02);
* KV cache: x * g[h, d] with x ~ N(0, 1) and a per-channel gain
  g ~ LogNormal(0, 0.5) over the 8 x 128 (kv head, head dim) channels;
* MoE routing: softmax of N(0, 1) logits over the experts, top-8 per token
  (ties to the lower expert id), tokens listed expert by expert in ascending
  token order.

All tensors are returned as torch tensors on ``device``; BF16 data is
``torch.bfloat16``.
"""
from dataclasses import dataclass

import torch

# Qwen3-8B linear shapes (N, K) per layer; 36 layers.
QWEN3_8B_LAYERS = 36
QWEN3_8B_LINEARS = {
    "qkv": (6144, 4096),
    "o": (4096, 4096),
    "gate_up": (24576, 4096),
    "down": (4096, 12288),
}
# Qwen3-30B-A3B MoE layer.
MOE_TOKENS = 4096
MOE_HIDDEN = 2048
MOE_EXPERTS = 128
MOE_INTER = 768
MOE_TOPK = 8
# KV cache [batch, seq, kv heads, head dim].
KV_SHAPE = (32, 8192, 8, 128)


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def activations(m: int, k: int, seed: int, device="cpu", outlier_frac=0.001,
                outlier_mult=50.0) -> torch.Tensor:
    """BF16 [m, k]: N(0,1) in FP32, round(outlier_frac * numel) entries x50."""
    g = generator(seed, device)
    x = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
    n = m * k
    n_out = int(round(outlier_frac * n))
    if n_out:
        idx = torch.randperm(n, generator=g, device=device)[:n_out]
        x.view(-1)[idx] *= outlier_mult
    return x.to(torch.bfloat16)


def weights(n: int, k: int, seed: int, device="cpu", std=0.02) -> torch.Tensor:
    """BF16 [n, k] ~ N(0, std)."""
    g = generator(seed, device)
    w = torch.randn(n, k, generator=g, device=device, dtype=torch.float32) * std
    return w.to(torch.bfloat16)


def kv_cache(seed: int, shape=KV_SHAPE, device="cpu") -> torch.Tensor:
    """BF16 tensor x * g[h, d] with x ~ N(0,1) and g ~ LogNormal(0, 0.5)."""
    g = generator(seed, device)
    heads, dim = shape[-2], shape[-1]
    gain = torch.exp(torch.randn(heads, dim, generator=g, device=device) * 0.5)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    x *= gain
    return x.to(torch.bfloat16)


@dataclass
class Routing:
    row_idx: torch.Tensor        # int32 [tokens * topk]: source token of each routed row
    group_offsets: torch.Tensor  # int32 [experts + 1]
    counts: torch.Tensor         # int64 [experts]


def moe_routing(tokens: int, experts: int, topk: int, seed: int, device="cpu") -> Routing:
    """softmax(N(0,1) logits) -> top-k -> rows grouped by expert, tokens ascending."""
    g = generator(seed, device)
    logits = torch.randn(tokens, experts, generator=g, device=device, dtype=torch.float32)
    probs = torch.softmax(logits, dim=-1)
    # ties go to the lower expert id: sort by (-prob, expert) with a stable sort
    order = torch.sort(-probs, dim=-1, stable=True).indices[:, :topk]
    expert_of = order.reshape(-1)
    token_of = torch.arange(tokens, device=device).repeat_interleave(topk)
    # stable sort by expert keeps tokens ascending inside each expert
    perm = torch.sort(expert_of, stable=True).indices
    row_idx = token_of[perm].to(torch.int32)
    counts = torch.bincount(expert_of, minlength=experts)
    offsets = torch.zeros(experts + 1, dtype=torch.int64, device=device)
    offsets[1:] = torch.cumsum(counts, 0)
    return Routing(row_idx=row_idx.contiguous(), group_offsets=offsets.to(torch.int32),
                   counts=counts)


def random_groups(total_rows: int, groups: int, seed: int, device="cpu",
                  allow_empty=True) -> torch.Tensor:
    """int32 [groups + 1] offsets splitting total_rows into random ragged groups."""
    g = generator(seed, "cpu")
    if groups == 0:
        return torch.zeros(1, dtype=torch.int32, device=device)
    cuts = torch.randint(0, total_rows + 1, (groups - 1,), generator=g)
    if not allow_empty:
        raise ValueError("not used")
    cuts, _ = torch.sort(cuts)
    off = torch.cat([torch.zeros(1, dtype=torch.int64), cuts, torch.tensor([total_rows])])
    return off.to(torch.int32).to(device)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a BF16 tensor's bytes (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")

"""Seeded synthetic inputs shaped like the FP8-RL pages' workloads.

This module only draws random numbers and lays them out; it holds none of the
quantisation or GEMM arithmetic.  Both the CUDA path and the CPU oracle are fed
from it, so a parity test hands the same bytes to both sides.

Recipes (every tensor has its own stream id under one seed):

* Qwen3-8B-shaped decoder layer (the dense model of the FP8-RL page, section
  "Results"): seven bf16 linears ~ N(0, 0.02); 0.1 % of entries, picked by an
  independent uniform draw u < 0.001, are multiplied by 20 (outliers).
* Activations for the GEMM sweep: X[m, k] = N(0, 1) * f_k with one lognormal
  factor f_k = exp(N(0, 1)) per K channel (outlier channels).
* Qwen3-30B-A3B-shaped MoE layer: 128 experts, each with a fused gate-up
  [1536, 2048] and a down [2048, 768] bf16 matrix ~ N(0, 0.02); T tokens route
  to top-8 experts by the softmax of N(0, 1) router logits (ties go to the lower
  expert index).  The indices are fixed integers, replayed as the R3 post
  describes; the combine weights are the chosen experts' renormalised
  probabilities.  Grouping the token rows by expert is the dispatch step,
  not part of this module.

Small inputs are drawn with numpy on the host (``device='cpu'``); the
multi-gigabyte benchmark inputs are drawn with torch's generator directly on
the GPU.  The two generators give different numbers for the same seed: a test
always draws once and hands that one draw to both sides.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np
import torch

QWEN3_8B_LAYER = (
    # name, N (out features), K (in features)
    ("q_proj", 4096, 4096),
    ("k_proj", 1024, 4096),
    ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096),
    ("gate_proj", 12288, 4096),
    ("up_proj", 12288, 4096),
    ("down_proj", 4096, 12288),
)
QWEN3_8B_LAYERS = 36

# GEMM sweep: fused projections of the same layer as (N, K)
QWEN3_8B_GEMMS = (
    ("qkv", 6144, 4096),
    ("o_proj", 4096, 4096),
    ("gate_up", 24576, 4096),
    ("down", 4096, 12288),
)
GEMM_SWEEP_M = (16, 128, 1024, 8192)

# Qwen3-30B-A3B-shaped MoE layer
MOE_EXPERTS = 128
MOE_TOPK = 8
MOE_HIDDEN = 2048
MOE_INTER = 768
MOE_LAYERS = 48
MOE_TOKENS = 4096

WEIGHT_STD = 0.02
OUTLIER_RATE = 1e-3
OUTLIER_GAIN = 20.0


def stream_seed(seed: int, *stream) -> int:
    """A 63-bit seed for one named stream under a global seed."""
    h = hashlib.blake2b(repr((int(seed),) + tuple(stream)).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def _np_rng(seed: int, *stream) -> np.random.Generator:
    return np.random.default_rng(stream_seed(seed, *stream))


def _torch_gen(device, seed: int, *stream) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(stream_seed(seed, *stream))
    return g


def _is_cpu(device) -> bool:
    return torch.device(device).type == "cpu"


def normal_bf16(shape, std: float, seed: int, *stream, device="cpu") -> torch.Tensor:
    """bf16 tensor of N(0, std^2) draws (fp32 draw, one RNE rounding to bf16)."""
    if _is_cpu(device):
        a = _np_rng(seed, *stream).standard_normal(shape, dtype=np.float32) * np.float32(std)
        return torch.from_numpy(a).to(torch.bfloat16)
    g = _torch_gen(device, seed, *stream)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(torch.bfloat16)


def weight_bf16(n: int, k: int, seed: int, *stream, outliers: bool = True,
                device="cpu") -> torch.Tensor:
    """A weight matrix ~ N(0, 0.02) with optional 0.1 % x20 outliers."""
    if _is_cpu(device):
        rng = _np_rng(seed, *stream)
        a = rng.standard_normal((n, k), dtype=np.float32) * np.float32(WEIGHT_STD)
        if outliers:
            u = _np_rng(seed, *stream, "outlier").random((n, k), dtype=np.float32)
            a[u < OUTLIER_RATE] *= np.float32(OUTLIER_GAIN)
        return torch.from_numpy(a).to(torch.bfloat16)
    g = _torch_gen(device, seed, *stream)
    t = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
    t.mul_(WEIGHT_STD)
    if outliers:
        gu = _torch_gen(device, seed, *stream, "outlier")
        u = torch.rand((n, k), generator=gu, device=device, dtype=torch.float32)
        t.mul_(torch.where(u < OUTLIER_RATE, OUTLIER_GAIN, 1.0))
        del u
    return t.to(torch.bfloat16)


def activation_bf16(m: int, k: int, seed: int, *stream, device="cpu") -> torch.Tensor:
    """X[m, k] = N(0,1) * f_k with per-channel lognormal(0, 1) factors f_k."""
    if _is_cpu(device):
        z = _np_rng(seed, *stream).standard_normal((m, k), dtype=np.float32)
        f = np.exp(_np_rng(seed, *stream, "channel").standard_normal(k)).astype(np.float32)
        return torch.from_numpy(z * f[None, :]).to(torch.bfloat16)
    g = _torch_gen(device, seed, *stream)
    z = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
    gf = _torch_gen(device, seed, *stream, "channel")
    f = torch.randn((k,), generator=gf, device=device, dtype=torch.float32).exp_()
    z.mul_(f[None, :])
    return z.to(torch.bfloat16)


# --------------------------------------------------------------------------- tiny linear

def tiny_linear(seed: int = 0, device="cpu"):
    """W bf16 [256, 256] ~ N(0, 0.02) with the 128x128 block at (row-block 0,
    K-block 1) set to zero, and X bf16 [16, 256] ~ N(0, 1)."""
    w = normal_bf16((256, 256), WEIGHT_STD, seed, "tiny", "w", device=device)
    w[0:128, 128:256] = 0
    x = normal_bf16((16, 256), 1.0, seed, "tiny", "x", device=device)
    return w, x


# --------------------------------------------------------------------------- dense model

def qwen3_8b_layer(layer: int = 0, seed: int = 0, device="cpu", shapes=QWEN3_8B_LAYER):
    """The seven bf16 linears of one decoder layer, as a list of (name, tensor)."""
    return [(name, weight_bf16(n, k, seed, "qwen3-8b", layer, name, device=device))
            for name, n, k in shapes]


# --------------------------------------------------------------------------- MoE routing

@dataclass
class Routing:
    topk: np.ndarray   # int32 [T, k] expert indices (fixed, replayed)
    gate: np.ndarray   # fp32 [T, k] the router's weights of those experts (renormalised over the k)


def moe_routing(tokens: int = MOE_TOKENS, experts: int = MOE_EXPERTS, topk: int = MOE_TOPK,
                seed: int = 0, layer: int = 0) -> Routing:
    """Top-k experts per token from softmax(N(0,1) logits); lower index wins ties.

    The indices are drawn once and then treated as fixed integers (the
    dispatch never sees the logits).  The combine weights are the chosen
    experts' softmax probabilities renormalised to sum to 1, as the MoE layer
    of Qwen3-30B-A3B forms them."""
    logits = _np_rng(seed, "router", layer).standard_normal((tokens, experts))
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")  # stable: equal p keeps the lower index first
    idx = order[:, :topk].astype(np.int32)
    w = np.take_along_axis(p, order[:, :topk], axis=1)
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return Routing(topk=idx, gate=w)


def routing_with_counts(counts, seed: int = 0) -> np.ndarray:
    """Offsets for explicit per-expert row counts (edge cases: empty experts)."""
    counts = np.asarray(counts, dtype=np.int64)
    offsets = np.zeros(counts.size + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return offsets


def moe_expert_weights(n: int, k: int, experts: int, seed: int, layer: int, which: str,
                       device="cpu") -> torch.Tensor:
    """bf16 [experts, n, k] ~ N(0, 0.02) (no outliers)."""
    if _is_cpu(device):
        a = _np_rng(seed, "moe", layer, which).standard_normal((experts, n, k), dtype=np.float32)
        return torch.from_numpy(a * np.float32(WEIGHT_STD)).to(torch.bfloat16)
    g = _torch_gen(device, seed, "moe", layer, which)
    out = torch.empty((experts, n, k), device=device, dtype=torch.bfloat16)
    for e in range(experts):
        t = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
        out[e].copy_(t.mul_(WEIGHT_STD))
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (a host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------- rollout log-probabilities (TIS)

ROLLOUT_RESPONSES = 512
ROLLOUT_MAX_LEN = 16384


def rollout_logprobs(responses: int = ROLLOUT_RESPONSES, max_len: int = ROLLOUT_MAX_LEN, seed: int = 0,
                     device="cpu"):
    """Per-token log-probabilities of a padded rollout batch, flattened
    [responses * max_len]: (lp_train fp32, lp_rollout fp32, mask uint8).

    Response lengths ~ uniform{1..max_len}; mask = 1 on a response's tokens,
    0 on its padding.  lp_rollout = -Exp(mean 0.5) (mostly confident
    samples); lp_train = lp_rollout + N(0, 0.05), and for 1 % of tokens an
    extra N(0, 1) (tokens where the two precisions disagree), so that some
    ratios pass the truncation."""
    n = responses * max_len
    g = _torch_gen(device, seed, "rollout", "len")
    lens = torch.randint(1, max_len + 1, (responses,), generator=g, device=device)
    pos = torch.arange(max_len, device=device)
    mask = (pos[None, :] < lens[:, None]).reshape(n).to(torch.uint8)
    g = _torch_gen(device, seed, "rollout", "lp")
    lp_rollout = torch.empty(n, device=device, dtype=torch.float32).exponential_(2.0, generator=g).neg_()
    noise = torch.randn(n, generator=g, device=device, dtype=torch.float32).mul_(0.05)
    big = torch.rand(n, generator=g, device=device, dtype=torch.float32) < 0.01
    noise += torch.randn(n, generator=g, device=device, dtype=torch.float32) * big
    lp_train = lp_rollout + noise
    return lp_train, lp_rollout, mask

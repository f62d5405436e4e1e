"""Seeded synthetic inputs shared by the tests, the benchmark and smoke().

This module holds none of the method's arithmetic: it only draws seeded
normal samples (torch's CPU generator, fp32), scales them, plants outliers and
rounds to bf16 (round to nearest even).  The same bytes are handed to the CUDA
library and to the CPU oracle.

Recipe (shapes and distributions of the workloads):
  activations  ~ N(0, 1)                       seed = workload seed
  decode acts  ~ N(0, 1), exactly round(0.001 * M * K) positions (a seeded
                 permutation) multiplied by 50 before bf16 rounding
  weights      ~ N(0, 0.02)                    seed = workload seed + 100
  router logits ~ N(0, 1), fp32                seed = workload seed + 200
"""
import numpy as np
import torch


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_f32(shape, seed, std=1.0):
    x = torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def randn_bf16(shape, seed, std=1.0):
    """[shape] bf16 CPU tensor, N(0, std^2) rounded to bf16."""
    return randn_f32(shape, seed, std).to(torch.bfloat16)


def activations_with_outliers(m, k, seed, frac=0.001, factor=50.0):
    """Decode-shaped activations: N(0,1) with round(frac*m*k) entries x factor."""
    x = randn_f32((m, k), seed)
    n_out = int(round(frac * m * k))
    if n_out:
        idx = torch.randperm(m * k, generator=_gen(seed + 1))[:n_out]
        x.view(-1)[idx] *= factor
    return x.to(torch.bfloat16)


def weights_bf16(n, k, seed, std=0.02):
    return randn_bf16((n, k), seed, std)


def expert_weights_bf16(n_experts, n, k, seed, std=0.02):
    """[E, n, k] bf16, one seeded draw per expert (seed + e)."""
    out = torch.empty((n_experts, n, k), dtype=torch.bfloat16)
    for e in range(n_experts):
        out[e] = randn_bf16((n, k), seed * 1000 + e, std)
    return out


def router_logits(t, e, seed):
    return randn_f32((t, e), seed)


def u16(t):
    """bf16 tensor -> numpy uint16 bit patterns (what the oracle consumes)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)

"""Seeded synthetic workloads for the verify step (shared by tests and bench).

Only input generation lives here: random logits with the shapes and value
distributions of the five workloads, and draft tokens drawn from the draft
distribution (the draft model's own sampling step, which comes before the
verify step).  Nothing in this module computes any part of the verify step.

Recipes (the readings are listed in the design notes):
  sample_b1      B=1,   gamma=4, V=32000,  fp32: z_t ~ N(0, 2^2), z_d = z_t + N(0, 0.5^2), T=1
  greedy_b64     B=64,  gamma=5, V=32000,  bf16: z_t ~ N(0, 3^2), z_d = z_t + N(0, 1), x = argmax z_d
  sample_b64     B=64,  gamma=4, V=128256, bf16: z_t ~ N(0, 2^2) + bias, bias of the token at
                 rank k (ranks = a seeded permutation of the vocabulary) = -1.1 ln k (Zipf 1.1);
                 z_d = z_t + N(0, sigma^2), sigma in {0.25, 1, 4}, T = 0.8
  sample_b256    B=256, gamma=8, V=152064, bf16: z_t ~ N(0, 2^2); per batch row T_b ~ U[0.5, 1.5],
                 sigma_b ~ U[0.1, 3]; each draft row independently w.p. 0.1 gets -inf on
                 floor(0.01 V) distinct random tokens
  lmhead_b32     B=32,  gamma=4, V=128256: h_t [160, 4096], h_d [128, 2048] ~ N(0, 1) bf16,
                 W_t [4096, V], W_d [2048, V] ~ N(0, 0.02^2) bf16, T = 1
Draft tokens are drawn from q = softmax(z_d / T) with torch.multinomial.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

GEN_DEVICE_DEFAULT = "cuda"


@dataclass
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    dtype: torch.dtype
    temperature: float
    zt: torch.Tensor
    zd: torch.Tensor | None
    xt: torch.Tensor
    row_temperature: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)

    @property
    def logit_bytes(self) -> int:
        n = self.zt.numel() + (self.zd.numel() if self.zd is not None else 0)
        return n * self.zt.element_size()


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def draw_from_logits(zd: torch.Tensor, temperature, gen: torch.Generator) -> torch.Tensor:
    """Draft tokens x ~ softmax(z_d / T) (the draft model's sampling), int32 [B, gamma]."""
    B, g, V = zd.shape
    out = torch.empty((B, g), dtype=torch.int32, device=zd.device)
    T = temperature if torch.is_tensor(temperature) else torch.full((B,), float(temperature),
                                                                     device=zd.device)
    for b0 in range(0, B, 16):  # bounded temporary memory
        b1 = min(B, b0 + 16)
        probs = torch.softmax(zd[b0:b1].float() / T[b0:b1, None, None].float(), dim=-1)
        out[b0:b1] = torch.multinomial(probs.reshape(-1, V), 1, generator=gen).reshape(
            b1 - b0, g).to(torch.int32)
    return out


def sample_b1(seed: int = 1001, device=GEN_DEVICE_DEFAULT, B: int = 1, gamma: int = 4,
              V: int = 32000) -> Workload:
    g = _gen(seed, device)
    zt = torch.randn((B, gamma + 1, V), generator=g, device=device) * 2.0
    zd = zt[:, :gamma] + torch.randn((B, gamma, V), generator=g, device=device) * 0.5
    zt, zd = zt.float().contiguous(), zd.float().contiguous()
    xt = draw_from_logits(zd, 1.0, g)
    return Workload("sample_b1", B, gamma, V, torch.float32, 1.0, zt, zd, xt)


def greedy_b64(seed: int = 1002, device=GEN_DEVICE_DEFAULT, B: int = 64, gamma: int = 5,
               V: int = 32000) -> Workload:
    g = _gen(seed, device)
    zt = (torch.randn((B, gamma + 1, V), generator=g, device=device) * 3.0).to(torch.bfloat16)
    zd = (zt[:, :gamma].float() + torch.randn((B, gamma, V), generator=g, device=device)).to(
        torch.bfloat16)
    xt = zd.float().argmax(dim=-1).to(torch.int32)  # first maximal index
    return Workload("greedy_b64", B, gamma, V, torch.bfloat16, 0.0, zt.contiguous(), None,
                    xt.contiguous(), extra={"zd": zd})


def zipf_bias(V: int, gen: torch.Generator, device, s: float = 1.1) -> torch.Tensor:
    ranks = torch.randperm(V, generator=gen, device=device) + 1  # rank of each token, 1..V
    return -s * torch.log(ranks.float())


def sample_b64(sigma: float = 1.0, seed: int = 1003, device=GEN_DEVICE_DEFAULT, B: int = 64,
               gamma: int = 4, V: int = 128256, temperature: float = 0.8) -> Workload:
    g = _gen(seed * 1000 + int(round(sigma * 100)), device)
    bias = zipf_bias(V, g, device)
    zt = torch.randn((B, gamma + 1, V), generator=g, device=device) * 2.0 + bias
    zd = zt[:, :gamma] + torch.randn((B, gamma, V), generator=g, device=device) * sigma
    zt, zd = zt.to(torch.bfloat16).contiguous(), zd.to(torch.bfloat16).contiguous()
    xt = draw_from_logits(zd, temperature, g)
    return Workload(f"sample_b64_s{sigma:g}", B, gamma, V, torch.bfloat16, temperature, zt, zd,
                    xt, extra={"sigma": sigma})


def sample_b256(seed: int = 1004, device=GEN_DEVICE_DEFAULT, B: int = 256, gamma: int = 8,
                V: int = 152064, mask_prob: float = 0.1, mask_frac: float = 0.01) -> Workload:
    g = _gen(seed, device)
    T = torch.rand((B,), generator=g, device=device) * 1.0 + 0.5
    sig = torch.rand((B,), generator=g, device=device) * 2.9 + 0.1
    zt = (torch.randn((B, gamma + 1, V), generator=g, device=device) * 2.0).to(torch.bfloat16)
    zd = torch.empty((B, gamma, V), dtype=torch.bfloat16, device=device)
    nmask = int(math.floor(mask_frac * V))
    masked = torch.rand((B, gamma), generator=g, device=device) < mask_prob
    for b in range(B):
        zd[b] = (zt[b, :gamma].float() + torch.randn((gamma, V), generator=g, device=device)
                 * sig[b]).to(torch.bfloat16)
    idx = masked.nonzero().tolist()
    for b, i in idx:
        toks = torch.randperm(V, generator=g, device=device)[:nmask]
        zd[b, i, toks] = float("-inf")
    xt = draw_from_logits(zd, T, g)
    return Workload("sample_b256", B, gamma, V, torch.bfloat16, 1.0, zt.contiguous(),
                    zd.contiguous(), xt, row_temperature=T.float().contiguous(),
                    extra={"sigma": sig, "masked_rows": masked})


def lmhead_b32(seed: int = 1005, device=GEN_DEVICE_DEFAULT, B: int = 32, gamma: int = 4,
               V: int = 128256, Ht: int = 4096, Hd: int = 2048) -> Workload:
    g = _gen(seed, device)
    h_t = torch.randn((B * (gamma + 1), Ht), generator=g, device=device).to(torch.bfloat16)
    h_d = torch.randn((B * gamma, Hd), generator=g, device=device).to(torch.bfloat16)
    W_t = (torch.randn((Ht, V), generator=g, device=device) * 0.02).to(torch.bfloat16)
    W_d = (torch.randn((Hd, V), generator=g, device=device) * 0.02).to(torch.bfloat16)
    # draft tokens from the draft model's own head (its sampling step)
    zd = (h_d.float() @ W_d.float()).reshape(B, gamma, V)
    xt = draw_from_logits(zd, 1.0, g)
    del zd
    return Workload("lmhead_b32", B, gamma, V, torch.bfloat16, 1.0, h_t, None, xt,
                    extra={"h_t": h_t, "W_t": W_t, "h_d": h_d, "W_d": W_d})


def three_token(n: int, seed: int = 1006, device=GEN_DEVICE_DEFAULT) -> Workload:
    """The three-token example (p = (0.6, 0.3, 0.1), q = (0.2, 0.5, 0.3)) as fp32 logits,
    one batch row per draw."""
    g = _gen(seed, device)
    p = torch.tensor([0.6, 0.3, 0.1], device=device)
    q = torch.tensor([0.2, 0.5, 0.3], device=device)
    zt = torch.log(p).float().expand(n, 2, 3).contiguous()
    zd = torch.log(q).float().expand(n, 1, 3).contiguous()
    xt = torch.multinomial(q.expand(n, 3), 1, replacement=True, generator=g).to(torch.int32)
    return Workload("three_token", n, 1, 3, torch.float32, 1.0, zt, zd, xt.contiguous())


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (the oracle's bf16 input format)."""
    import numpy as np
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_oracle(t: torch.Tensor):
    """Device logits -> numpy array the oracle reads (float32 or bf16 bits)."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.float().cpu().numpy()

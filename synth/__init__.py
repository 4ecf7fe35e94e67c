"""Seeded synthetic inputs for the selective log-prob / GRPO loss path.

This module serves both the CUDA library's callers (tests, bench) and the
oracle's callers. It holds none of the path's arithmetic: it only draws
tensors with the shapes and value distributions of the workloads below.

Workloads (flattened tokens N = prompts x G completions x T tokens):

=================  =======  ====  ====  ======  ============================
name               prompts   G     T      D      V        padding
=================  =======  ====  ====  ======  ============================
tiny                  1       4     64    256     4096    none
qwen2.5-1.5b          2       4   1024   1536   151936    lengths ~ U[256, 1024]
llama-3.1-8b          1       4   4096   4096   128256    none
qwen3-8b-long         1       8  16384   4096   151936    lengths ~ U[1024, 16384]
gpt-oss-20b-long      1       2  65536   2880   201088    none
=================  =======  ====  ====  ======  ============================

Value recipe (all workloads): hidden ~ N(0, 1) and lm_head W ~ N(0, 0.02^2),
both rounded to bf16 (round-to-nearest-even); token ids uniform in [0, V)
(also on padding, where they are never read); one Bernoulli(0.5) reward per
completion; advantage = (r - mean_group) / (std_group + 1e-4) with the
Bessel-corrected standard deviation; old and reference log-probs are a base
log-prob (supplied by the caller) plus independent N(0, 0.05^2) noise;
eps = 0.2 both sides, beta = 0.001; padding is trailing, masked with 0.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

WORKLOADS = {
    "tiny": dict(prompts=1, G=4, T=64, D=256, V=4096, lengths=None),
    "qwen2.5-1.5b": dict(prompts=2, G=4, T=1024, D=1536, V=151936,
                         lengths=(256, 1024)),
    "llama-3.1-8b": dict(prompts=1, G=4, T=4096, D=4096, V=128256,
                         lengths=None),
    "qwen3-8b-long": dict(prompts=1, G=8, T=16384, D=4096, V=151936,
                          lengths=(1024, 16384)),
    "gpt-oss-20b-long": dict(prompts=1, G=2, T=65536, D=2880, V=201088,
                             lengths=None),
}

EPS = 0.2
BETA = 0.001
LOGP_NOISE_STD = 0.05
HIDDEN_STD = 1.0
WEIGHT_STD = 0.02

# Stream ids: every tensor has its own generator, so changing one tensor's
# shape leaves the others unchanged.
_S_HIDDEN, _S_WEIGHT, _S_IDS, _S_LEN, _S_REWARD, _S_OLD, _S_REF = range(7)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1009 + stream * 7919 + 17)
    return g


@dataclass
class Problem:
    """One batch of synthetic inputs. Tensors live on ``device``."""

    name: str
    n_tokens: int
    seq_len: int
    hidden_size: int
    vocab: int
    group: int
    hidden: torch.Tensor      # [N, D] bf16
    weight: torch.Tensor      # [V, D] bf16
    ids: torch.Tensor         # [N] int32
    mask: torch.Tensor        # [N] uint8
    lengths: torch.Tensor     # [B] int64 valid tokens per completion
    rewards: torch.Tensor     # [B] float64
    adv: torch.Tensor         # [B] float32
    old_noise: torch.Tensor   # [N] float32
    ref_noise: torch.Tensor   # [N] float32
    eps_low: float = EPS
    eps_high: float = EPS
    beta: float = BETA

    @property
    def n_seqs(self) -> int:
        return self.n_tokens // self.seq_len

    @property
    def n_valid(self) -> int:
        return int(self.lengths.sum().item())

    def old_ref(self, base_logp: torch.Tensor):
        """old/ref log-probs = base log-prob + independent N(0, 0.05^2)."""
        base = base_logp.to(self.old_noise.device, torch.float32)
        return base + self.old_noise, base + self.ref_noise


def group_advantages(rewards: torch.Tensor, group: int) -> torch.Tensor:
    """(r - mean_g) / (std_g + 1e-4) per group of G completions, in float64."""
    r = rewards.to(torch.float64).reshape(-1, group)
    mean = r.mean(dim=1, keepdim=True)
    std = r.std(dim=1, keepdim=True, unbiased=True) if group > 1 else torch.zeros_like(mean)
    return ((r - mean) / (std + 1e-4)).reshape(-1)


def make_problem(name: str = "tiny", seed: int = 0, device="cpu", *,
                 prompts=None, G=None, T=None, D=None, V=None, lengths="cfg",
                 weight_std: float = WEIGHT_STD,
                 hidden_std: float = HIDDEN_STD) -> Problem:
    """Draw one workload (optionally with any shape field overridden)."""
    cfg = dict(WORKLOADS[name])
    for k, v in (("prompts", prompts), ("G", G), ("T", T), ("D", D), ("V", V)):
        if v is not None:
            cfg[k] = v
    if lengths != "cfg":
        cfg["lengths"] = lengths
    B = cfg["prompts"] * cfg["G"]
    Tn, Dn, Vn = cfg["T"], cfg["D"], cfg["V"]
    N = B * Tn
    dev = torch.device(device)

    hidden = (torch.randn(N, Dn, generator=_gen(seed, _S_HIDDEN, dev), device=dev)
              * hidden_std).to(torch.bfloat16)
    weight = (torch.randn(Vn, Dn, generator=_gen(seed, _S_WEIGHT, dev), device=dev)
              * weight_std).to(torch.bfloat16)
    ids = torch.randint(0, Vn, (N,), generator=_gen(seed, _S_IDS, dev), device=dev,
                        dtype=torch.int64).to(torch.int32)
    if cfg["lengths"] is None:
        lens = torch.full((B,), Tn, dtype=torch.int64)
    else:
        lo, hi = cfg["lengths"]
        lens = torch.randint(lo, hi + 1, (B,), generator=_gen(seed, _S_LEN, "cpu"),
                             dtype=torch.int64)
    pos = torch.arange(Tn, dtype=torch.int64)
    mask = (pos[None, :] < lens[:, None]).reshape(-1).to(torch.uint8).to(dev)
    rewards = torch.bernoulli(torch.full((B,), 0.5, dtype=torch.float64),
                              generator=_gen(seed, _S_REWARD, "cpu"))
    adv = group_advantages(rewards, cfg["G"]).to(torch.float32).to(dev)
    old_noise = torch.randn(N, generator=_gen(seed, _S_OLD, dev), device=dev) * LOGP_NOISE_STD
    ref_noise = torch.randn(N, generator=_gen(seed, _S_REF, dev), device=dev) * LOGP_NOISE_STD
    return Problem(name=name, n_tokens=N, seq_len=Tn, hidden_size=Dn, vocab=Vn,
                   group=cfg["G"], hidden=hidden, weight=weight, ids=ids, mask=mask,
                   lengths=lens, rewards=rewards, adv=adv, old_noise=old_noise,
                   ref_noise=ref_noise)

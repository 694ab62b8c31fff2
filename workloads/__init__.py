"""Seeded synthetic inputs for the fused MoE layer.

Shared by the tests, the smoke check and the benchmark for both the CUDA
path and the oracle.  This module holds only random draws and their recipe:
none of the layer's arithmetic (no routing, no quantisation, no GEMM).

Recipe (the pages measure serving on real models; these synthetic tensors
stand in for them -- no dataset or trained weight is used):
  * one ``torch.Generator`` seeded per workload, on the device the tensors are
    made on; draw order: logits, x, router bias (Standard) or x_b, counts,
    padding garbage (Batched); then w1, w2 -- so the activations of a seed do
    not depend on whether its weights are drawn;
  * hidden states x ~ N(0, 1) rounded to bf16; router logits ~ N(0, 1) fp32;
  * w1 (E, 2N, K) ~ N(0, 1/K), w2 (E, K, N) ~ N(0, 1/N), drawn in bf16;
  * skewed routing (DeepSeek-V3-shaped prefill): a per-expert bias
    b_e = -s * ln(rank_e), rank a seeded permutation of 1..E and s = 1.1 --
    the log of a Zipf(s) probability up to a constant, added to the logits;
  * batched masked format: counts[e] ~ U{0..T} with two experts forced to 0
    and one to T (positions drawn), valid rows N(0, 1), padded rows
    N(0, 10^2) garbage that must not reach the output.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

SOFTMAX, SIGMOID = 0, 1
BF16, FP8, FP8_CHANNEL, FP8_TENSOR = 0, 1, 2, 3


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    M: int                 # tokens (Standard) -- or T, max tokens per expert (Batched)
    K: int                 # hidden size
    N: int                 # intermediate size (w1 has 2N rows per expert)
    E: int                 # experts
    topk: int
    dtype: int = BF16      # BF16, FP8 (e4m3, 1x128 activation / 128x128 weight scales) or
                           # FP8_CHANNEL (e4m3, one scale per token / per weight row) or
                           # FP8_TENSOR (e4m3, one scale per activation tensor / per weight row)
    score_fn: int = SOFTMAX
    n_groups: int = 1
    topk_groups: int = 1
    zipf_bias: bool = False
    renorm: bool = True
    batched: bool = False  # BatchedExperts (E, T, K) masked by counts
    seed: int = 0

    @property
    def P(self) -> int:
        return self.M * self.topk

    @property
    def requant_h(self) -> bool:
        return self.dtype != BF16


# The workloads the layer is specified on.
TINY = MoEConfig("tiny_bf16_M64_K256_N128_E8_top2", M=64, K=256, N=128, E=8,
                 topk=2, seed=0)
MIXTRAL_PREFILL = MoEConfig("mixtral8x7b_prefill_bf16_M4096_K4096_N14336_E8_top2",
                            M=4096, K=4096, N=14336, E=8, topk=2, seed=2)
DSV3_PREFILL_FP8 = MoEConfig("dsv3_prefill_fp8_M8192_K7168_N2048_E256_top8",
                             M=8192, K=7168, N=2048, E=256, topk=8, dtype=FP8,
                             score_fn=SIGMOID, n_groups=8, topk_groups=4,
                             zipf_bias=True, seed=3)
DSV3_DECODE = MoEConfig("dsv3_decode_bf16_M64_K7168_N2048_E256_top8",
                        M=64, K=7168, N=2048, E=256, topk=8, score_fn=SIGMOID,
                        n_groups=8, topk_groups=4, seed=4)
BATCHED_MASKED = MoEConfig("batched_masked_bf16_E32_T1024_K7168_N2048",
                           M=1024, K=7168, N=2048, E=32, topk=1, batched=True,
                           seed=5000)
# the same shapes with e4m3 activations and block-scaled weights
BATCHED_MASKED_FP8 = MoEConfig("batched_masked_fp8_E32_T1024_K7168_N2048",
                               M=1024, K=7168, N=2048, E=32, topk=1, batched=True,
                               dtype=FP8, seed=6000)

# Smaller cases of the same kinds, for parity tests that the oracle finishes in
# seconds while still spanning several tiles and a ragged tail.
SMALL_BF16 = MoEConfig("small_bf16_M300_K512_N384_E8_top2", M=300, K=512, N=384,
                       E=8, topk=2, seed=11)
SMALL_SIGMOID = MoEConfig("small_sigmoid_bf16_M200_K384_N256_E64_top6",
                          M=200, K=384, N=256, E=64, topk=6, score_fn=SIGMOID,
                          n_groups=8, topk_groups=4, zipf_bias=True, seed=12)
SMALL_FP8 = MoEConfig("small_fp8_M256_K512_N256_E16_top4", M=256, K=512, N=256,
                      E=16, topk=4, dtype=FP8, score_fn=SIGMOID, n_groups=4,
                      topk_groups=2, zipf_bias=True, seed=13)
SMALL_BATCHED = MoEConfig("small_batched_bf16_E6_T200_K256_N256", M=200, K=256,
                          N=256, E=6, topk=1, batched=True, seed=14)

# Small cases whose experts average 128 rows or more (M*topk >= 128*E, or
# T >= 128 for the batched format): the bf16 GEMMs run on CTA pairs with
# 256-row tiles, here with ragged last tiles in M and, for K = 640, a down
# n-tile of 128 columns.  SMALL_BATCHED_SHORT (T < 128) stays on the 1-SM
# kernel.
SMALL_PAIR = MoEConfig("small_pair_bf16_M300_K384_N256_E2_top1", M=300, K=384,
                       N=256, E=2, topk=1, seed=15)
SMALL_PAIR_TOP2 = MoEConfig("small_pair_bf16_M520_K640_N384_E4_top2", M=520, K=640,
                            N=384, E=4, topk=2, seed=16)
# e4m3 with a down n-tile of 128 columns (K = 640) and 150 rows per expert
SMALL_FP8_K640 = MoEConfig("small_fp8_M300_K640_N256_E4_top2", M=300, K=640, N=256,
                           E=4, topk=2, dtype=FP8, seed=18)
# e4m3 with every expert at 1..64 rows (the operand-swapped narrow tile) and
# K = 640 (the last down tile's second half lies past K)
SMALL_FP8_NARROW = MoEConfig("small_fp8_narrow_M48_K640_N256_E8_top2", M=48, K=640, N=256,
                             E=8, topk=2, dtype=FP8, seed=29)
SMALL_BATCHED_SHORT = MoEConfig("small_batched_bf16_E5_T100_K384_N256", M=100, K=384,
                                N=256, E=5, topk=1, batched=True, seed=17)
# the BatchedExperts format with e4m3 activations (1 x 128 group scales) and
# block-scaled weights: several m-tiles per expert, and T < 128 with K = 640
# (the last down tile's second half lies past K)
SMALL_BATCHED_FP8 = MoEConfig("small_batched_fp8_E6_T300_K256_N256", M=300, K=256,
                              N=256, E=6, topk=1, batched=True, dtype=FP8, seed=41)
SMALL_BATCHED_FP8_K640 = MoEConfig("small_batched_fp8_E5_T100_K640_N256", M=100, K=640,
                                   N=256, E=5, topk=1, batched=True, dtype=FP8, seed=42)

# e4m3 with per-token / per-channel scales: a small sigmoid-routed case with
# 64 rows per expert, one with 150 rows per expert and K = 640, and the
# DeepSeek-V3-shaped prefill in this format.
SMALL_FP8CH = MoEConfig("small_fp8ch_M256_K512_N256_E16_top4", M=256, K=512, N=256,
                        E=16, topk=4, dtype=FP8_CHANNEL, score_fn=SIGMOID, n_groups=4,
                        topk_groups=2, zipf_bias=True, seed=19)
SMALL_FP8CH_PAIR = MoEConfig("small_fp8ch_M300_K640_N384_E4_top2", M=300, K=640, N=384,
                             E=4, topk=2, dtype=FP8_CHANNEL, seed=20)
DSV3_PREFILL_FP8CH = MoEConfig("dsv3_prefill_fp8ch_M8192_K7168_N2048_E256_top8",
                               M=8192, K=7168, N=2048, E=256, topk=8, dtype=FP8_CHANNEL,
                               score_fn=SIGMOID, n_groups=8, topk_groups=4, zipf_bias=True,
                               seed=3)

# e4m3 with one scale per activation tensor: cases small enough for the
# oracle's two passes over every token, and the DeepSeek-V3-shaped prefill
# in this format (timed; its parity is covered by the smaller cases, since a
# per-tensor scale couples every token)
SMALL_FP8T = MoEConfig("small_fp8t_M256_K512_N256_E8_top2", M=256, K=512, N=256, E=8,
                       topk=2, dtype=FP8_TENSOR, seed=27)
MID_FP8T = MoEConfig("mid_fp8t_M384_K768_N384_E16_top4", M=384, K=768, N=384, E=16,
                     topk=4, dtype=FP8_TENSOR, score_fn=SIGMOID, n_groups=4, topk_groups=2,
                     zipf_bias=True, seed=28)
DSV3_PREFILL_FP8T = MoEConfig("dsv3_prefill_fp8t_M8192_K7168_N2048_E256_top8",
                              M=8192, K=7168, N=2048, E=256, topk=8, dtype=FP8_TENSOR,
                              score_fn=SIGMOID, n_groups=8, topk_groups=4, zipf_bias=True,
                              seed=3)

ALL = [TINY, MIXTRAL_PREFILL, DSV3_PREFILL_FP8, DSV3_DECODE, BATCHED_MASKED]

# Small cases of the same kernels for profiler captures: operands larger than
# the 129 MB L2, a few hundred MB to ~1 GB on the device.
PROFILE_BF16 = MoEConfig("profile_bf16_M2048_K4096_N14336_E2_top1", M=2048, K=4096,
                         N=14336, E=2, topk=1, seed=21)
PROFILE_FP8 = MoEConfig("profile_fp8_M2048_K7168_N2048_E16_top2", M=2048, K=7168,
                        N=2048, E=16, topk=2, dtype=FP8, score_fn=SIGMOID,
                        n_groups=4, topk_groups=2, seed=22)
PROFILE_FP8CH = MoEConfig("profile_fp8ch_M2048_K7168_N2048_E16_top2", M=2048, K=7168,
                          N=2048, E=16, topk=2, dtype=FP8_CHANNEL, score_fn=SIGMOID,
                          n_groups=4, topk_groups=2, seed=22)
PROFILE_BATCHED = MoEConfig("profile_batched_bf16_E8_T512_K7168_N2048", M=512, K=7168,
                            N=2048, E=8, topk=1, batched=True, seed=24)
PROFILE_DECODE = MoEConfig("profile_decode_bf16_M16_K7168_N2048_E32_top4", M=16,
                           K=7168, N=2048, E=32, topk=4, score_fn=SIGMOID,
                           n_groups=4, topk_groups=2, seed=23)

BY_NAME = {c.name: c for c in ALL + [SMALL_BF16, SMALL_SIGMOID, SMALL_FP8,
                                     SMALL_BATCHED, SMALL_PAIR, SMALL_PAIR_TOP2, SMALL_FP8_K640,
                                     SMALL_FP8CH, SMALL_FP8CH_PAIR, DSV3_PREFILL_FP8CH,
                                     PROFILE_FP8CH, SMALL_FP8T, MID_FP8T, DSV3_PREFILL_FP8T,
                                     SMALL_BATCHED_SHORT, PROFILE_BF16, PROFILE_FP8, PROFILE_DECODE,
                                     PROFILE_BATCHED, SMALL_FP8_NARROW, SMALL_BATCHED_FP8,
                                     SMALL_BATCHED_FP8_K640, BATCHED_MASKED_FP8]}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, std=1.0, dtype=torch.float32):
    t = torch.randn(shape, generator=g, device=device, dtype=dtype)
    if std != 1.0:
        t.mul_(std)
    return t


def _weights(cfg: MoEConfig, g, device) -> dict:
    return {"w1": _randn((cfg.E, 2 * cfg.N, cfg.K), g, device,
                         std=1.0 / math.sqrt(cfg.K), dtype=torch.bfloat16),
            "w2": _randn((cfg.E, cfg.K, cfg.N), g, device,
                         std=1.0 / math.sqrt(cfg.N), dtype=torch.bfloat16)}


def _standard_acts(cfg: MoEConfig, g, device) -> dict:
    out = {"logits": _randn((cfg.M, cfg.E), g, device)}
    out["x"] = _randn((cfg.M, cfg.K), g, device).to(torch.bfloat16)
    out["bias"] = None
    if cfg.zipf_bias:
        rank = torch.randperm(cfg.E, generator=g, device=device).to(torch.float32) + 1.0
        out["bias"] = (-1.1 * torch.log(rank)).to(torch.float32)
    return out


def _batched_acts(cfg: MoEConfig, g, device) -> dict:
    E, T = cfg.E, cfg.M
    xb = _randn((E, T, cfg.K), g, device)
    counts = torch.randint(0, T + 1, (E,), generator=g, device=device,
                           dtype=torch.int64)
    pos = torch.randperm(E, generator=g, device=device)
    if E >= 3:
        counts[pos[0]] = 0
        counts[pos[1]] = 0
        counts[pos[2]] = T
    counts = counts.to(torch.int32)
    rows = torch.arange(T, device=device).view(1, T, 1)
    pad = rows >= counts.view(E, 1, 1).to(rows.dtype)
    garbage = _randn((E, T, cfg.K), g, device, std=10.0)
    return {"x_b": torch.where(pad, garbage, xb).to(torch.bfloat16), "counts": counts}


def make_standard(cfg: MoEConfig, device="cpu", seed: Optional[int] = None,
                  with_weights: bool = True) -> dict:
    """Inputs of the Standard format: logits (M, E) fp32, x (M, K) bf16,
    bias (E) fp32 or None, w1 (E, 2N, K) bf16, w2 (E, K, N) bf16."""
    g = _gen(cfg.seed if seed is None else seed, device)
    out = _standard_acts(cfg, g, device)
    if with_weights:
        out.update(_weights(cfg, g, device))
    return out


def make_batched(cfg: MoEConfig, device="cpu", seed: Optional[int] = None,
                 with_weights: bool = True) -> dict:
    """Inputs of the BatchedExperts format: x_b (E, T, K) bf16 whose rows
    r >= counts[e] are N(0, 10^2) garbage, counts (E) int32, w1, w2."""
    assert cfg.batched
    g = _gen(cfg.seed if seed is None else seed, device)
    out = _batched_acts(cfg, g, device)
    if with_weights:
        out.update(_weights(cfg, g, device))
    return out


def make_weights(cfg: MoEConfig, device="cpu", seed: Optional[int] = None) -> dict:
    """Only the expert weights: the same draws make_inputs gives for this
    seed (the activations are drawn first and dropped)."""
    g = _gen(cfg.seed if seed is None else seed, device)
    if cfg.batched:
        _batched_acts(cfg, g, device)
    else:
        _standard_acts(cfg, g, device)
    return _weights(cfg, g, device)


def make_inputs(cfg: MoEConfig, device="cpu", seed: Optional[int] = None,
                with_weights: bool = True) -> dict:
    if cfg.batched:
        return make_batched(cfg, device, seed, with_weights)
    return make_standard(cfg, device, seed, with_weights)


@dataclasses.dataclass(frozen=True)
class EpConfig:
    """Expert-parallel worst-tokens layout: G shards of up to M tokens each
    (a device count of valid ones per shard), E routed experts split evenly
    over the shards (E / G each), top-k routing; worst_tokens rows of static
    receive capacity per expert (G * M: every token of every shard)."""
    name: str
    G: int
    M: int
    K: int
    N: int
    E: int
    topk: int
    score_fn: int = SOFTMAX
    n_groups: int = 1
    topk_groups: int = 1
    seed: int = 0

    @property
    def worst_tokens(self) -> int:
        return self.G * self.M


EP2 = EpConfig("ep_worst_tokens_G2_M96_K512_N256_E32_top4", G=2, M=96, K=512, N=256, E=32,
               topk=4, seed=71)
EP4 = EpConfig("ep_worst_tokens_G4_M64_K384_N256_E64_top6", G=4, M=64, K=384, N=256, E=64,
               topk=6, score_fn=SIGMOID, n_groups=8, topk_groups=4, seed=72)
# DeepSeek-V3-shaped experts split over eight shards (an EP8 layer's shards
# emulated in one GPU's memory), 256 tokens per shard
EP8_DSV3 = EpConfig("ep_worst_tokens_G8_M256_K7168_N2048_E256_top8", G=8, M=256, K=7168,
                    N=2048, E=256, topk=8, score_fn=SIGMOID, n_groups=8, topk_groups=4, seed=73)


def make_ep_inputs(cfg: EpConfig, device="cpu", seed: Optional[int] = None,
                   with_weights: bool = True) -> dict:
    """x (G, M, K) bf16 and logits (G, M, E) fp32 with N(0, 1) valid rows and
    N(0, 10^2) garbage in the padded rows of each shard, num_tokens (G) int32
    ~ U{M/2..M} with one shard at M; then w1 (E, 2N, K), w2 (E, K, N) as for
    the Standard workloads."""
    g = _gen(cfg.seed if seed is None else seed, device)
    G, M = cfg.G, cfg.M
    n = torch.randint(M // 2, M + 1, (G,), generator=g, device=device, dtype=torch.int64)
    n[int(torch.randint(0, G, (1,), generator=g, device=device).item())] = M
    rows = torch.arange(M, device=device).view(1, M, 1)
    pad = rows >= n.view(G, 1, 1)
    x = torch.where(pad, _randn((G, M, cfg.K), g, device, std=10.0),
                    _randn((G, M, cfg.K), g, device))
    logits = torch.where(pad, _randn((G, M, cfg.E), g, device, std=10.0),
                         _randn((G, M, cfg.E), g, device))
    out = {"x": x.to(torch.bfloat16), "logits": logits.contiguous(),
           "num_tokens": n.to(torch.int32)}
    if with_weights:
        out["w1"] = _randn((cfg.E, 2 * cfg.N, cfg.K), g, device, std=1.0 / math.sqrt(cfg.K),
                           dtype=torch.bfloat16)
        out["w2"] = _randn((cfg.E, cfg.K, cfg.N), g, device, std=1.0 / math.sqrt(cfg.N),
                           dtype=torch.bfloat16)
    return out


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bits (on the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def flops(cfg: MoEConfig, rows: int) -> float:
    """Algorithmic FLOPs of the two expert GEMMs for `rows` routed rows:
    4*K*N for the gate/up GEMM plus 2*K*N for the down GEMM per row."""
    return 6.0 * cfg.K * cfg.N * rows

"""Shared helpers of the GPU parity tests: run the CUDA path through the C-ABI
binding, build the oracle's view of the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc
import workloads as WL

TOL = {WL.BF16: 2e-2, WL.FP8: 5e-2, WL.FP8_CHANNEL: 5e-2, WL.FP8_TENSOR: 5e-2}  # max|d| <= tol * max|ref|


def gbmoe():
    import mixture_experts_layer_count_gb300 as g
    g.load()
    return g


def assert_close_rel(got, ref, tol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    assert err <= tol * scale, f"{what}: max|d|={err:.4e} > {tol}*max|ref|={tol * scale:.4e}"
    return err / scale if scale > 0 else 0.0


class GpuWeights:
    """The expert weights as the CUDA path takes them: bf16 tensors, or e4m3
    codes + 128 x 128 block scales (FP8) or one scale per row (FP8_CHANNEL,
    FP8_TENSOR) made by the library's own quantiser."""

    def __init__(self, cfg, w1, w2):
        g = gbmoe()
        self.dtype = cfg.dtype
        if cfg.dtype == WL.BF16:
            self.w1, self.w2, self.w1s, self.w2s = w1, w2, None, None
        elif cfg.dtype in (WL.FP8_CHANNEL, WL.FP8_TENSOR):  # per-row weight scales
            E, N, K = cfg.E, cfg.N, cfg.K
            self.w1 = torch.empty((E, 2 * N, K), dtype=torch.uint8, device=w1.device)
            self.w2 = torch.empty((E, K, N), dtype=torch.uint8, device=w1.device)
            self.w1s = torch.empty((E, 2 * N), dtype=torch.float32, device=w1.device)
            self.w2s = torch.empty((E, K), dtype=torch.float32, device=w1.device)
            g.moe_quant_fp8_group(w1.view(E * 2 * N, K), self.w1.view(E * 2 * N, K),
                                  self.w1s.view(E * 2 * N, 1), group=K)
            g.moe_quant_fp8_group(w2.view(E * K, N), self.w2.view(E * K, N),
                                  self.w2s.view(E * K, 1), group=N)
        else:
            E, N, K = cfg.E, cfg.N, cfg.K
            self.w1 = torch.empty((E, 2 * N, K), dtype=torch.uint8, device=w1.device)
            self.w2 = torch.empty((E, K, N), dtype=torch.uint8, device=w1.device)
            self.w1s = torch.empty((E, 2 * N // 128, K // 128), dtype=torch.float32, device=w1.device)
            self.w2s = torch.empty((E, K // 128, N // 128), dtype=torch.float32, device=w1.device)
            g.moe_quant_fp8_block(w1, self.w1, self.w1s)
            g.moe_quant_fp8_block(w2, self.w2, self.w2s)


def oracle_weights(cfg, w1, w2, experts=None):
    """The oracle's weights for the listed experts (all when None), made from
    the bf16 tensors by the oracle's own quantiser for FP8."""
    experts = range(cfg.E) if experts is None else sorted(set(int(e) for e in experts))
    blocks = {}
    for e in experts:
        b1 = WL.bf16_bits(w1[e])
        b2 = WL.bf16_bits(w2[e])
        if cfg.dtype == WL.BF16:
            blocks[e] = (b1, b2)
        elif cfg.dtype in (WL.FP8_CHANNEL, WL.FP8_TENSOR):  # one scale per weight row
            q1, s1 = orc.quant_fp8_group(b1, group=cfg.K)
            q2, s2 = orc.quant_fp8_group(b2, group=cfg.N)
            blocks[e] = (q1, q2, s1[:, 0], s2[:, 0])
        else:
            q1, s1 = orc.quant_fp8_block(b1)
            q2, s2 = orc.quant_fp8_block(b2)
            blocks[e] = (q1, q2, s1, s2)
    return orc.Weights(cfg.dtype, experts=blocks, E=cfg.E, N=cfg.N, K=cfg.K)


def run_forward(cfg, d, gw, stream=None):
    """The whole Standard layer on the GPU; returns out, ids, weights, err."""
    g = gbmoe()
    dev = d["x"].device
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    out = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    ids = torch.empty((M, k), dtype=torch.int32, device=dev)
    wts = torch.empty((M, k), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype, device=dev)
    g.moe_forward(d["x"], d["logits"], d["bias"], N, E, k, cfg.score_fn,
                  cfg.n_groups, cfg.topk_groups, cfg.renorm, cfg.dtype, gw.w1,
                  gw.w1s, gw.w2, gw.w2s, out, ws, topk_ids=ids, topk_weights=wts,
                  err_word=err, stream=stream)
    return out, ids, wts, err


def oracle_forward(cfg, d, W, tokens=None, nthreads=0):
    return orc.moe_forward(WL.bf16_bits(d["x"]), d["logits"].cpu().numpy(),
                           None if d["bias"] is None else d["bias"].cpu().numpy(),
                           cfg.topk, cfg.score_fn, W, cfg.n_groups, cfg.topk_groups,
                           cfg.renorm, cfg.requant_h, tokens=tokens,
                           nthreads=nthreads)


def check_ids(gpu_ids, ref_ids, margin, what=""):
    """Router ids are compared bit for bit.  A token may differ only when the
    oracle reports a group-key margin below 1e-6 (a last-bit difference
    between two exp implementations could flip it); such tokens are counted
    and must stay rare."""
    diff = np.flatnonzero((gpu_ids != ref_ids).any(1))
    near = [t for t in diff if margin[t] < 1e-6]
    assert len(diff) == len(near), f"{what}: ids differ on tokens {diff[:10]}"
    assert len(near) <= max(1, len(ref_ids) // 1000), f"{what}: {len(near)} near-ties"
    return diff

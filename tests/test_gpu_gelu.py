"""activation "gelu" (gelu_and_mul) through the C ABI against the oracle:
the one-call layer in bf16 and FP8, the gate/up GEMM entry point, and the
batched masked format."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as WL
from gpu_common import TOL, GpuWeights, assert_close_rel, gbmoe, oracle_weights

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


@pytest.mark.parametrize("cfg", [WL.SMALL_BF16, WL.SMALL_FP8, WL.SMALL_PAIR_TOP2,
                                 WL.SMALL_FP8_K640, WL.SMALL_FP8CH_PAIR],
                         ids=lambda c: c.name)
def test_forward_gelu(cfg):
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    out = torch.empty((cfg.M, cfg.K), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_FORWARD, cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk, cfg.dtype)
    g.moe_forward(d["x"], d["logits"], d["bias"], cfg.N, cfg.E, cfg.topk, cfg.score_fn,
                  cfg.n_groups, cfg.topk_groups, cfg.renorm, cfg.dtype, gw.w1, gw.w1s, gw.w2,
                  gw.w2s, out, ws, err_word=err, activation=g.ACT_GELU)
    torch.cuda.synchronize()
    assert err.item() == 0
    W = oracle_weights(cfg, d["w1"], d["w2"])
    W.act = orc.GELU
    ref, _, _ = orc.moe_forward(WL.bf16_bits(d["x"]), d["logits"].cpu().numpy(),
                                None if d["bias"] is None else d["bias"].cpu().numpy(),
                                cfg.topk, cfg.score_fn, W, cfg.n_groups, cfg.topk_groups,
                                cfg.renorm, cfg.requant_h)
    assert_close_rel(out.float().cpu().numpy(), ref, TOL[cfg.dtype], cfg.name)


def test_gate_up_gelu_entry_point():
    g = gbmoe()
    cfg = WL.TINY
    d = WL.make_inputs(cfg, DEV)
    rid, rw, _ = orc.route(d["logits"].cpu().numpy(), None, cfg.topk, orc.SOFTMAX)
    ids = torch.from_numpy(rid).to(DEV)
    P = cfg.P
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)
    srt = torch.empty(P, dtype=torch.int32, device=DEV)
    inv = torch.empty(P, dtype=torch.int32, device=DEV)
    g.moe_align_permute(ids, cfg.E, None, offsets, srt, inv,
                        g.workspace(g.WS_ALIGN, cfg.M, cfg.E, 0, 0, cfg.topk, 0))
    A = torch.empty((P, cfg.K), dtype=torch.bfloat16, device=DEV)
    g.moe_permute_rows(d["x"], None, srt, offsets, cfg.topk, cfg.E, g.BF16, A)
    H = torch.empty((P, cfg.N), dtype=torch.bfloat16, device=DEV)
    g.moe_grouped_gemm_gate_up_gelu(A, None, offsets, cfg.M, cfg.topk, cfg.E, cfg.N, cfg.K,
                                    d["w1"], None, g.BF16, H, None)
    torch.cuda.synchronize()
    W = orc.Weights(orc.BF16, WL.bf16_bits(d["w1"]), WL.bf16_bits(d["w2"]), act=orc.GELU)
    s = srt.cpu().numpy()
    href = np.stack([orc.expert_row(WL.bf16_bits(d["x"]), p // cfg.topk, rid.ravel()[p], W)[0]
                     for p in s])
    assert_close_rel(H.float().cpu().numpy(), href, TOL[WL.BF16], "H (gelu)")


@pytest.mark.parametrize("cfg", [WL.SMALL_BATCHED, WL.SMALL_BATCHED_FP8],
                         ids=lambda c: c.name)
def test_batched_gelu(cfg):
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV)
    yb = torch.full((cfg.E, cfg.M, cfg.K), 5.0, dtype=torch.bfloat16, device=DEV)
    ws = g.workspace(g.WS_BATCHED, cfg.M, cfg.E, cfg.N, cfg.K, 1, cfg.dtype)
    if cfg.dtype == WL.FP8:
        gw = GpuWeights(cfg, d["w1"], d["w2"])
        E, T, K = cfg.E, cfg.M, cfg.K
        q = torch.empty((E, T, K), dtype=torch.uint8, device=DEV)
        sc = torch.empty((E * T, K // 128), dtype=torch.float32, device=DEV)
        g.moe_quant_fp8_group(d["x_b"].reshape(E * T, K), q.view(E * T, K), sc)
        g.moe_batched_masked_experts(q, d["counts"], cfg.N, gw.w1, gw.w2, yb, ws, dtype=WL.FP8,
                                     x_b_scales=sc, w1_scales=gw.w1s, w2_scales=gw.w2s,
                                     activation=g.ACT_GELU)
    else:
        g.moe_batched_masked_experts(d["x_b"], d["counts"], cfg.N, d["w1"], d["w2"], yb, ws,
                                     activation=g.ACT_GELU)
    torch.cuda.synchronize()
    W = oracle_weights(cfg, d["w1"], d["w2"])
    W.act = orc.GELU
    ref, n = orc.batched_experts(WL.bf16_bits(d["x_b"]), d["counts"].cpu().numpy(), W,
                                 requant_h=cfg.dtype == WL.FP8)
    mask = ~np.isnan(ref[..., 0])
    assert_close_rel(yb.float().cpu().numpy()[mask], ref[mask], TOL[cfg.dtype], f"{cfg.name} gelu")

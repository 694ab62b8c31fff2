"""The layer at the edges of its argument ranges, against the oracle: the
largest expert count (512) with grouped sigmoid routing, the largest top-k
(32), every expert picked by every token (topk = E), a single expert, the
largest K and N of the block-scaled e4m3 GEMMs (16384: 128 scale blocks,
the whole per-tile scale table), a single token in every dtype, and empty
inputs (no token, or no valid row) in every dtype."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as WL
from gpu_common import TOL, GpuWeights, assert_close_rel, check_ids, gbmoe, oracle_forward, \
    oracle_weights, run_forward

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


CASES = [
    # 512 experts in 8 groups of 64, top-4 groups, top-8 (the route kernel's
    # widest rows, the GEMMs' full tile table)
    WL.MoEConfig("edge_E512_top8_grouped", M=96, K=256, N=128, E=512, topk=8,
                 score_fn=WL.SIGMOID, n_groups=8, topk_groups=4, zipf_bias=True, seed=51),
    # the largest top-k: 32 of 64 experts (the top-8 reduce in four batches)
    WL.MoEConfig("edge_E64_top32", M=40, K=256, N=128, E=64, topk=32, seed=52),
    # every token on every expert, weights renormalised over all of them
    WL.MoEConfig("edge_topk_eq_E", M=100, K=384, N=256, E=4, topk=4, seed=53),
    # one expert: the dense gated MLP
    WL.MoEConfig("edge_E1_bf16", M=70, K=256, N=256, E=1, topk=1, seed=54),
    WL.MoEConfig("edge_E1_fp8", M=70, K=256, N=256, E=1, topk=1, dtype=WL.FP8, seed=55),
    # block-scaled e4m3 at the largest K (gate/up: 128 K blocks) and N (down)
    WL.MoEConfig("edge_fp8_K16384", M=40, K=16384, N=256, E=4, topk=2, dtype=WL.FP8, seed=56),
    WL.MoEConfig("edge_fp8_N16384", M=24, K=256, N=16384, E=2, topk=1, dtype=WL.FP8, seed=57),
    # a single token (a decode step of batch one) in every dtype
    WL.MoEConfig("edge_M1_bf16", M=1, K=512, N=256, E=8, topk=2, seed=58),
    WL.MoEConfig("edge_M1_fp8_grouped", M=1, K=512, N=256, E=64, topk=8, dtype=WL.FP8,
                 score_fn=WL.SIGMOID, n_groups=8, topk_groups=4, zipf_bias=True, seed=59),
    WL.MoEConfig("edge_M1_fp8ch", M=1, K=512, N=256, E=16, topk=4, dtype=WL.FP8_CHANNEL,
                 seed=60),
    WL.MoEConfig("edge_M1_fp8t", M=1, K=512, N=256, E=16, topk=4, dtype=WL.FP8_TENSOR, seed=61),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_edge_shapes_match_the_oracle(cfg):
    d = WL.make_inputs(cfg, DEV)
    out, ids, wts, err = run_forward(cfg, d, GpuWeights(cfg, d["w1"], d["w2"]))
    torch.cuda.synchronize()
    assert err.item() == 0
    W = oracle_weights(cfg, d["w1"], d["w2"])
    ref, ref_ids, ref_w = oracle_forward(cfg, d, W)
    logits = d["logits"].cpu().numpy()
    bias = None if d["bias"] is None else d["bias"].cpu().numpy()
    _, _, margin = orc.route(logits, bias, cfg.topk, cfg.score_fn, cfg.n_groups,
                             cfg.topk_groups, cfg.renorm)
    gi = ids.cpu().numpy()
    diff = check_ids(gi, ref_ids, margin, cfg.name, cfg, logits, bias)
    same = np.setdiff1d(np.arange(cfg.M), diff)
    if cfg.topk == cfg.E:
        assert np.all(np.sort(gi, axis=1) == np.arange(cfg.E))
    np.testing.assert_allclose(wts.cpu().numpy()[same], ref_w[same], rtol=0, atol=2e-6)
    assert_close_rel(out.float().cpu().numpy()[same], ref[same], TOL[cfg.dtype], cfg.name)


def test_fp8_block_k_and_n_above_the_limit_are_rejected():
    """K or N beyond 16384 with block-scaled e4m3 is refused before any
    launch (INVALID_ARG), and the output is left alone."""
    g = gbmoe()
    for K, N in ((16512, 128), (128, 16512)):
        assert g.moe_workspace_size(g.WS_FORWARD, 4, 2, N, K, 1, g.FP8_E4M3) == 0
    cfg = WL.MoEConfig("edge_reject", M=4, K=16512, N=128, E=2, topk=1, seed=58)
    x = torch.zeros((4, cfg.K), dtype=torch.bfloat16, device=DEV)
    logits = torch.zeros((4, 2), dtype=torch.float32, device=DEV)
    w1 = torch.zeros((2, 256, cfg.K), dtype=torch.uint8, device=DEV)
    w2 = torch.zeros((2, cfg.K, 128), dtype=torch.uint8, device=DEV)
    s1 = torch.ones((2, 2, cfg.K // 128), dtype=torch.float32, device=DEV)
    s2 = torch.ones((2, cfg.K // 128, 1), dtype=torch.float32, device=DEV)
    out = torch.full((4, cfg.K), 3.0, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(1 << 26, dtype=torch.uint8, device=DEV)
    with pytest.raises(RuntimeError) as ei:
        g.moe_forward(x, logits, None, 128, 2, 1, WL.SOFTMAX, 1, 1, True, g.FP8_E4M3,
                      w1, s1, w2, s2, out, ws)
    assert ei.value.status == 1  # GBMOE_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


@pytest.mark.parametrize("chunked", [False, True], ids=["one_call", "chunked"])
@pytest.mark.parametrize("dtype,static", [(WL.FP8, False), (WL.FP8_CHANNEL, False),
                                          (WL.FP8_TENSOR, False), (WL.FP8_TENSOR, True)],
                         ids=["fp8_block", "fp8_channel", "fp8_tensor", "fp8_tensor_static"])
def test_empty_input_is_a_no_op_in_every_dtype(dtype, static, chunked):
    """M = 0 in every e4m3 mode (the bf16 case is in the parity tests):
    GBMOE_OK, no error bit, and nothing written."""
    cfg = WL.MoEConfig("edge_M0", M=0, K=256, N=256, E=8, topk=2, dtype=dtype, seed=62)
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    g = gbmoe()
    out = torch.full((1, cfg.K), 3.0, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_FORWARD, 0, cfg.E, cfg.N, cfg.K, cfg.topk, dtype, device=DEV)
    kw = {}
    if static:
        kw = dict(a1_scale=torch.full((1,), 0.01, device=DEV),
                  a2_scale=torch.full((1,), 0.01, device=DEV))
    args = (d["x"], d["logits"], None, cfg.N, cfg.E, cfg.topk, cfg.score_fn, 1, 1, True,
            dtype, gw.w1, gw.w1s, gw.w2, gw.w2s, out, ws)
    if chunked:
        g.moe_forward_chunked(*args, 64, err_word=err, **kw)
    else:
        g.moe_forward(*args, err_word=err, **kw)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.all(out == 3.0)


@pytest.mark.parametrize("dtype", [WL.BF16, WL.FP8], ids=["bf16", "fp8_block"])
def test_batched_with_every_count_zero_writes_nothing(dtype):
    """Every expert's device count is 0: no row is computed, no row of the
    output is written, no error bit is set."""
    E, T, K, N = 4, 96, 256, 256
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(63)
    xb = torch.randn((E, T, K), generator=gen, device=DEV).to(torch.bfloat16)
    w1 = (torch.randn((E, 2 * N, K), generator=gen, device=DEV) / 16).to(torch.bfloat16)
    w2 = (torch.randn((E, K, N), generator=gen, device=DEV) / 16).to(torch.bfloat16)
    counts = torch.zeros(E, dtype=torch.int32, device=DEV)
    yb = torch.empty((E, T, K), dtype=torch.bfloat16, device=DEV)
    yb.view(torch.int16).fill_(0x7E7E)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_BATCHED, T, E, N, K, 1, dtype, device=DEV)
    if dtype == WL.BF16:
        g.moe_batched_masked_experts(xb, counts, N, w1, w2, yb, ws, err_word=err)
    else:
        cfg = WL.MoEConfig("edge_batched_zero", M=T, K=K, N=N, E=E, topk=1, dtype=WL.FP8)
        gw = GpuWeights(cfg, w1, w2)
        q = torch.empty((E, T, K), dtype=torch.uint8, device=DEV)
        sc = torch.empty((E * T, K // 128), dtype=torch.float32, device=DEV)
        g.moe_quant_fp8_group(xb.reshape(E * T, K), q.view(E * T, K), sc)
        g.moe_batched_masked_experts(q, counts, N, gw.w1, gw.w2, yb, ws, dtype=WL.FP8,
                                     x_b_scales=sc, w1_scales=gw.w1s, w2_scales=gw.w2s,
                                     err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.all(yb.view(torch.int16) == 0x7E7E)

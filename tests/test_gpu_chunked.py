"""In-graph chunking: the layer run in chunks of tokens with a workspace
sized for one chunk equals the unchunked layer bit for bit (the
"chunked == unchunked" property of _maybe_chunk_fused_experts), and the
chunk loop is capturable because no count ever goes to the host."""
import pytest
import torch

import workloads as WL
from gpu_common import TOL, GpuWeights, assert_close_rel, gbmoe, oracle_forward, oracle_weights

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


@pytest.mark.parametrize("cfg,chunk", [(WL.SMALL_SIGMOID, 64), (WL.SMALL_FP8, 100),
                                       (WL.SMALL_BF16, 300), (WL.SMALL_FP8CH, 96),
                                       (WL.SMALL_PAIR_TOP2, 200),
                                       # the e4m3 prefill in the 2048-token chunks the bench times
                                       (WL.DSV3_PREFILL_FP8, 2048)],
                         ids=lambda v: str(getattr(v, "name", v)))
def test_chunked_equals_unchunked(cfg, chunk):
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    args = (d["logits"], d["bias"], N, E, k, cfg.score_fn, cfg.n_groups, cfg.topk_groups,
            cfg.renorm, cfg.dtype, gw.w1, gw.w1s, gw.w2, gw.w2s)
    ref = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    g.moe_forward(d["x"], *args, ref, g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype))
    out = torch.empty_like(ref)
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_FORWARD, min(M, chunk), E, N, K, k, cfg.dtype)
    g.moe_forward_chunked(d["x"], *args, out, ws, chunk, topk_ids=ids)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # captured: the chunk loop replays with new tokens
    x = d["x"].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.moe_forward_chunked(x, *args, out, ws, chunk)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.moe_forward_chunked(x, *args, out, ws, chunk)
    x2 = WL.make_inputs(cfg, DEV, seed=cfg.seed + 9, with_weights=False)["x"]
    x.copy_(x2)
    graph.replay()
    g.moe_forward(x2, *args, ref, g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_chunked_fp8_tensor_dynamic_scales_are_taken_per_chunk():
    """Per-tensor e4m3 with dynamic scales: each chunk quantises with its own
    tensor maxima, as if the chunk were the whole input.  Chunk by chunk
    (two full chunks and a ragged one), the chunked layer equals the one-call
    layer run on that chunk alone, bit for bit, and the oracle's layer on
    that chunk alone."""
    cfg, chunk = WL.SMALL_FP8T, 96
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    args = (cfg.score_fn, cfg.n_groups, cfg.topk_groups, cfg.renorm, cfg.dtype,
            gw.w1, gw.w1s, gw.w2, gw.w2s)
    out = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    g.moe_forward_chunked(d["x"], d["logits"], d["bias"], N, E, k, *args, out,
                          g.workspace(g.WS_FORWARD, chunk, E, N, K, k, cfg.dtype), chunk,
                          err_word=err)
    W = oracle_weights(cfg, d["w1"], d["w2"])
    whole = torch.empty_like(out)
    g.moe_forward(d["x"], d["logits"], d["bias"], N, E, k, *args, whole,
                  g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype))
    torch.cuda.synchronize()
    assert err.item() == 0
    assert not torch.equal(out.view(torch.int16), whole.view(torch.int16))  # scales differ
    for c0 in range(0, M, chunk):
        c1 = min(M, c0 + chunk)
        xc, lc = d["x"][c0:c1].contiguous(), d["logits"][c0:c1].contiguous()
        one = torch.empty((c1 - c0, K), dtype=torch.bfloat16, device=DEV)
        g.moe_forward(xc, lc, d["bias"], N, E, k, *args, one,
                      g.workspace(g.WS_FORWARD, c1 - c0, E, N, K, k, cfg.dtype))
        torch.cuda.synchronize()
        assert torch.equal(out[c0:c1].view(torch.int16), one.view(torch.int16)), (c0, c1)
        ref, _, _ = oracle_forward(cfg, {"x": xc, "logits": lc, "bias": d["bias"]}, W)
        assert_close_rel(out[c0:c1].float().cpu().numpy(), ref, TOL[cfg.dtype],
                         f"chunk [{c0}, {c1})")

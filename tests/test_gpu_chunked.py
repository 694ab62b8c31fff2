"""In-graph chunking: the layer run in chunks of tokens with a workspace
sized for one chunk equals the unchunked layer bit for bit (the
"chunked == unchunked" property of _maybe_chunk_fused_experts), and the
chunk loop is capturable because no count ever goes to the host."""
import pytest
import torch

import workloads as WL
from gpu_common import GpuWeights, gbmoe

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


@pytest.mark.parametrize("cfg,chunk", [(WL.SMALL_SIGMOID, 64), (WL.SMALL_FP8, 100),
                                       (WL.SMALL_BF16, 300), (WL.SMALL_FP8CH, 96),
                                       (WL.SMALL_PAIR_TOP2, 200)],
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

"""Expert-parallel dispatch / combine in the worst-tokens mode, G = 2 and 4
shards in this GPU's memory: route -> dispatch -> per-shard masked grouped
GEMMs reading the device counts -> combine, captured once in a CUDA graph and
replayed with fresh data, routing and valid-token counts per replay (50 for
G = 2, 20 for G = 4).  Every replay equals the eager run bit for bit; the
per-expert counts and every pair's receive row equal the oracle's stable
counting sort of the valid pairs (bit-exact); the outputs of the valid tokens
match the oracle's layer over all experts within the bf16 tolerance; rows of
padded tokens are never written."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as WL
from gpu_common import TOL, assert_close_rel, check_ids, gbmoe, oracle_weights

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = 0x7E7E


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


class EpLayer:
    """Static buffers of the sharded layer and its launch sequence (bf16, or
    e4m3: tokens quantised per 128-group before the dispatch, block-scaled
    weights)."""

    def __init__(self, cfg, w1, w2, dtype=WL.BF16):
        g = gbmoe()
        self.cfg, self.g, self.dtype = cfg, g, dtype
        G, M, K, N, E, k = cfg.G, cfg.M, cfg.K, cfg.N, cfg.E, cfg.topk
        W = cfg.worst_tokens
        i32 = torch.int32
        self.x = torch.empty((G, M, K), dtype=torch.bfloat16, device=DEV)
        self.logits = torch.empty((G, M, E), dtype=torch.float32, device=DEV)
        self.num_tokens = torch.empty(G, dtype=i32, device=DEV)
        self.ids = torch.empty((G, M, k), dtype=i32, device=DEV)
        self.wts = torch.empty((G, M, k), dtype=torch.float32, device=DEV)
        fp8 = dtype == WL.FP8
        self.recv_x = torch.empty((E, W, K), dtype=torch.uint8 if fp8 else torch.bfloat16,
                                  device=DEV)
        if fp8:
            self.xq = torch.empty((G, M, K), dtype=torch.uint8, device=DEV)
            self.xs = torch.empty((G * M, K // 128), dtype=torch.float32, device=DEV)
            self.recv_s = torch.empty((E * W, K // 128), dtype=torch.float32, device=DEV)
            q1 = torch.empty((E, 2 * N, K), dtype=torch.uint8, device=DEV)
            q2 = torch.empty((E, K, N), dtype=torch.uint8, device=DEV)
            s1 = torch.empty((E, 2 * N // 128, K // 128), dtype=torch.float32, device=DEV)
            s2 = torch.empty((E, K // 128, N // 128), dtype=torch.float32, device=DEV)
            g.moe_quant_fp8_block(w1, q1, s1)
            g.moe_quant_fp8_block(w2, q2, s2)
            w1, w2 = q1, q2
        self.recv_y = torch.empty((E, W, K), dtype=torch.bfloat16, device=DEV)
        self.recv_counts = torch.empty(E, dtype=i32, device=DEV)
        self.recv_pos = torch.empty((G, M, k), dtype=i32, device=DEV)
        self.out = torch.empty((G, M, K), dtype=torch.bfloat16, device=DEV)
        self.err = torch.zeros(1, dtype=i32, device=DEV)
        self.ws = g.workspace(g.WS_EP_DISPATCH, M, E, G, K, k, 0)
        El = E // G
        self.El = El
        self.w1 = [w1[s * El:(s + 1) * El] for s in range(G)]
        self.w2 = [w2[s * El:(s + 1) * El] for s in range(G)]
        self.kw = [{} for _ in range(G)]
        if fp8:
            for s_ in range(G):
                self.kw[s_] = dict(dtype=WL.FP8, x_b_scales=self.recv_s[s_ * El * W:(s_ + 1) * El * W],
                                   w1_scales=s1[s_ * El:(s_ + 1) * El],
                                   w2_scales=s2[s_ * El:(s_ + 1) * El])
        self.bws = [g.workspace(g.WS_BATCHED, W, El, N, K, 1, dtype) for _ in range(G)]

    def step(self):
        c, g = self.cfg, self.g
        G, M, E, k = c.G, c.M, c.E, c.topk
        g.moe_topk_route(self.logits.view(G * M, E), None, k, c.score_fn, c.n_groups,
                         c.topk_groups, True, self.ids.view(G * M, k), self.wts.view(G * M, k))
        if self.dtype == WL.FP8:
            g.moe_quant_fp8_group(self.x.view(G * M, c.K), self.xq.view(G * M, c.K), self.xs)
            g.moe_ep_dispatch(self.xq, self.num_tokens, self.ids, E, c.worst_tokens, self.recv_x,
                              self.recv_counts, self.recv_pos, self.ws, self.err, dtype=WL.FP8,
                              x_scales=self.xs, recv_scales=self.recv_s)
        else:
            g.moe_ep_dispatch(self.x, self.num_tokens, self.ids, E, c.worst_tokens, self.recv_x,
                              self.recv_counts, self.recv_pos, self.ws, self.err)
        for s in range(G):  # each shard's masked grouped GEMMs on its own receive block
            sl = slice(s * self.El, (s + 1) * self.El)
            g.moe_batched_masked_experts(self.recv_x[sl], self.recv_counts[sl], c.N, self.w1[s],
                                         self.w2[s], self.recv_y[sl], self.bws[s],
                                         err_word=self.err, **self.kw[s])
        g.moe_ep_combine(self.recv_y, self.ids, self.recv_pos, self.wts, self.num_tokens,
                         self.out)

    def load(self, d):
        self.x.copy_(d["x"])
        self.logits.copy_(d["logits"])
        self.num_tokens.copy_(d["num_tokens"])
        self.out.view(torch.int16).fill_(SENTINEL)


def _oracle_check(cfg, layer, d, W, dtype=WL.BF16):
    n = d["num_tokens"].cpu().numpy()
    G, M, E, k = cfg.G, cfg.M, cfg.E, cfg.topk
    xv = torch.cat([d["x"][r, :n[r]] for r in range(G)])
    lv = torch.cat([d["logits"][r, :n[r]] for r in range(G)]).cpu().numpy()
    rid, rw, _ = orc.route(lv, None, k, cfg.score_fn, cfg.n_groups, cfg.topk_groups, True)
    # per-expert counts and the receive row of every valid pair
    rc, bad = orc.count(rid, E)
    ro, rs, ri = orc.align(rid, E)
    assert bad == 0
    assert np.array_equal(layer.recv_counts.cpu().numpy(), rc)
    pos_ref = ri - ro[rid.ravel()]
    gpos = layer.recv_pos.cpu().numpy()
    gids = layer.ids.cpu().numpy()
    got_pos = np.concatenate([gpos[r, :n[r]].ravel() for r in range(G)])
    got_ids = np.concatenate([gids[r, :n[r]] for r in range(G)])
    assert np.array_equal(got_ids, rid)
    assert np.array_equal(got_pos, pos_ref)
    for r in range(G):  # pairs of padded tokens are not dispatched
        assert np.all(gpos[r, n[r]:] == -1)
    # values: the layer over all experts, token by token
    ref, rid2, _ = orc.moe_forward(WL.bf16_bits(xv), lv, None, k, cfg.score_fn, W,
                                   cfg.n_groups, cfg.topk_groups, True,
                                   requant_h=dtype == WL.FP8)
    got = torch.cat([layer.out[r, :n[r]] for r in range(G)]).float().cpu().numpy()
    assert_close_rel(got, ref, TOL[dtype], cfg.name)
    bits = layer.out.view(torch.int16).cpu().numpy()
    for r in range(G):
        assert np.all(bits[r, n[r]:] == np.int16(SENTINEL)), f"shard {r}: padded rows written"


@pytest.mark.parametrize("cfg,replays", [(WL.EP2, 50), (WL.EP4, 20)], ids=["G2", "G4"])
def test_ep_worst_tokens_graph_replays(cfg, replays):
    d0 = WL.make_ep_inputs(cfg, DEV)
    layer = EpLayer(cfg, d0["w1"], d0["w2"])
    W = oracle_weights(WL.MoEConfig("ep_all", M=1, K=cfg.K, N=cfg.N, E=cfg.E, topk=cfg.topk),
                       d0["w1"], d0["w2"])
    layer.load(d0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.step()  # warm up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.step()
    eager = EpLayer(cfg, d0["w1"], d0["w2"])
    for r in range(replays):
        dr = WL.make_ep_inputs(cfg, DEV, seed=cfg.seed * 1000 + r + 1, with_weights=False)
        layer.load(dr)
        graph.replay()
        eager.load(dr)
        eager.step()
        torch.cuda.synchronize()
        assert layer.err.item() == 0 and eager.err.item() == 0, f"replay {r}"
        for name in ("out", "recv_counts", "recv_pos", "ids"):
            a, b = getattr(layer, name), getattr(eager, name)
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), f"replay {r}: {name} differs from the eager run"
        if r % 5 == 0:
            _oracle_check(cfg, layer, dr, W)


@pytest.mark.parametrize("cfg,replays", [(WL.EP2, 20), (WL.EP4, 10)], ids=["G2", "G4"])
def test_ep_worst_tokens_fp8_graph_replays(cfg, replays):
    """The same sharded layer with the tokens quantised to e4m3 (1 x 128
    group scales) before the dispatch, the scales carried with the rows, and
    block-scaled e4m3 experts on each shard: 20 (G = 2) or 10 (G = 4)
    replays, each equal to the eager run bit for bit (receive rows and scales
    included), every fifth against the oracle's e4m3 layer (h requantised)."""
    d0 = WL.make_ep_inputs(cfg, DEV)
    layer = EpLayer(cfg, d0["w1"], d0["w2"], WL.FP8)
    W = oracle_weights(WL.MoEConfig("ep_all_fp8", M=1, K=cfg.K, N=cfg.N, E=cfg.E, topk=cfg.topk,
                                    dtype=WL.FP8), d0["w1"], d0["w2"])
    layer.load(d0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.step()
    eager = EpLayer(cfg, d0["w1"], d0["w2"], WL.FP8)
    for r in range(replays):
        dr = WL.make_ep_inputs(cfg, DEV, seed=cfg.seed * 1000 + 500 + r, with_weights=False)
        layer.load(dr)
        graph.replay()
        eager.load(dr)
        eager.step()
        torch.cuda.synchronize()
        assert layer.err.item() == 0 and eager.err.item() == 0, f"replay {r}"
        for name in ("out", "recv_counts", "recv_pos", "ids"):
            a, b = getattr(layer, name), getattr(eager, name)
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), f"replay {r}: {name} differs from the eager run"
        # the received rows (codes and scales) below each count agree too
        cnt = layer.recv_counts.cpu().numpy()
        for e in range(cfg.E):
            c = int(cnt[e])
            assert torch.equal(layer.recv_x[e, :c], eager.recv_x[e, :c]), f"replay {r} expert {e}"
            row0 = e * cfg.worst_tokens
            assert torch.equal(layer.recv_s[row0:row0 + c], eager.recv_s[row0:row0 + c])
        if r % 5 == 0:
            # every dispatched pair's receive row holds its token's codes and
            # scales, byte for byte
            pos, ids = layer.recv_pos, layer.ids
            sh, tk, _ = torch.nonzero(pos >= 0, as_tuple=True)
            pe, pp = ids[pos >= 0].long(), pos[pos >= 0].long()
            assert torch.equal(layer.recv_x[pe, pp], layer.xq[sh, tk])
            assert torch.equal(layer.recv_s[pe * cfg.worst_tokens + pp], layer.xs[sh * cfg.M + tk])
            _oracle_check(cfg, layer, dr, W, WL.FP8)


def test_ep_dispatch_flags_overflow_of_the_static_shape():
    """A receive capacity below the real per-expert count: the count is
    clamped, the extra pairs are dropped (pos -1) and the error bit is set;
    nothing is written past the static shape."""
    g = gbmoe()
    cfg = WL.EP2
    d = WL.make_ep_inputs(cfg, DEV, with_weights=False)
    G, M, E, k, K = cfg.G, cfg.M, cfg.E, cfg.topk, cfg.K
    ids = torch.zeros((G, M, k), dtype=torch.int32, device=DEV)
    ids[..., 1] = 1
    ids[..., 2] = 2
    ids[..., 3] = 3   # every token on experts 0..3: counts = sum(num_tokens)
    worst = 16
    flat = torch.empty(E * worst * K + 4096, dtype=torch.bfloat16, device=DEV)
    flat.view(torch.int16).fill_(SENTINEL)
    recv_x = flat[:E * worst * K].view(E, worst, K)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    pos = torch.empty((G, M, k), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_EP_DISPATCH, M, E, G, K, k, 0)
    g.moe_ep_dispatch(d["x"], d["num_tokens"], ids, E, worst, recv_x, counts, pos, ws, err)
    torch.cuda.synchronize()
    assert err.item() & g.ERR_COUNT_RANGE
    assert torch.all(counts[:4] == worst) and torch.all(counts[4:] == 0)
    assert int((pos >= 0).sum()) == 4 * worst
    assert int(pos.max()) == worst - 1
    # the first `worst` valid tokens (in shard, token order) fill each block
    n = d["num_tokens"].cpu().numpy()
    xv = torch.cat([d["x"][r, :n[r]] for r in range(G)])
    for e in range(4):
        assert torch.equal(recv_x[e].view(torch.int16), xv[:worst].view(torch.int16))
    assert torch.all(recv_x[4:].view(torch.int16) == SENTINEL)      # experts with no rows
    assert torch.all(flat[E * worst * K:].view(torch.int16) == SENTINEL)  # past the shape


def test_ep_worst_tokens_fp8_full_size():
    """The sharded e4m3 layer at the size the bench times: 8 shards of up to
    256 tokens, K = 7168, N = 2048, 256 experts, grouped sigmoid top-8.
    Captured and replayed once, the replay equals the eager run bit for bit.
    Against the oracle: the router ids of every valid token (near-ties
    validated); the per-expert counts and every valid pair's receive position,
    bit-exact against the oracle's stable counting sort of those ids; the
    tokens' 1 x 128 codes and scales, bit-exact, which every receive row
    holds byte for byte; the outputs of 16 sampled valid tokens against the
    oracle's e4m3 layer (h requantised).  Padded tokens' pairs are not
    dispatched and their output rows are not written."""
    cfg = WL.EP8_DSV3
    G, M, K, N, E, k = cfg.G, cfg.M, cfg.K, cfg.N, cfg.E, cfg.topk
    Wt = cfg.worst_tokens
    d = WL.make_ep_inputs(cfg, DEV)
    layer = EpLayer(cfg, d["w1"], d["w2"], WL.FP8)
    layer.load(d)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.step()
    layer.load(d)
    graph.replay()
    eager = EpLayer(cfg, d["w1"], d["w2"], WL.FP8)
    eager.load(d)
    eager.step()
    torch.cuda.synchronize()
    assert layer.err.item() == 0 and eager.err.item() == 0
    for name in ("out", "recv_counts", "recv_pos", "ids"):
        a, b = getattr(layer, name), getattr(eager, name)
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), f"{name} differs from the eager run"
    del eager
    n = d["num_tokens"].cpu().numpy()
    xv = torch.cat([d["x"][r, :n[r]] for r in range(G)])
    lv = torch.cat([d["logits"][r, :n[r]] for r in range(G)]).cpu().numpy()
    rid, _, margin = orc.route(lv, None, k, cfg.score_fn, cfg.n_groups, cfg.topk_groups, True)
    gids = layer.ids.cpu().numpy()
    got_ids = np.concatenate([gids[r, :n[r]] for r in range(G)])
    diff = check_ids(got_ids, rid, margin, cfg.name, cfg, lv, None)
    # the dispatch of the GPU's (validated) routing
    rc, bad = orc.count(got_ids, E)
    ro, _, ri = orc.align(got_ids, E)
    assert bad == 0
    assert np.array_equal(layer.recv_counts.cpu().numpy(), rc)
    gpos = layer.recv_pos.cpu().numpy()
    got_pos = np.concatenate([gpos[r, :n[r]].ravel() for r in range(G)])
    assert np.array_equal(got_pos, ri - ro[got_ids.ravel()])
    for r in range(G):
        assert np.all(gpos[r, n[r]:] == -1)
    q_ref, s_ref = orc.quant_fp8_group(WL.bf16_bits(xv))
    xq = torch.cat([layer.xq[r, :n[r]] for r in range(G)]).cpu().numpy()
    xs = torch.cat([layer.xs[r * M:r * M + n[r]] for r in range(G)]).cpu().numpy()
    assert np.array_equal(xq, q_ref)
    assert np.array_equal(xs.view(np.uint32), s_ref.view(np.uint32))
    pos, ids = layer.recv_pos, layer.ids
    sh, tk, _ = torch.nonzero(pos >= 0, as_tuple=True)
    pe, pp = ids[pos >= 0].long(), pos[pos >= 0].long()
    assert torch.equal(layer.recv_x[pe, pp], layer.xq[sh, tk])
    assert torch.equal(layer.recv_s[pe * Wt + pp], layer.xs[sh * M + tk])
    # values of sampled valid tokens
    rng = np.random.default_rng(6)
    tokens = np.setdiff1d(np.sort(rng.choice(len(xv), 16, replace=False)), diff)
    W = oracle_weights(WL.MoEConfig("ep8_fp8", M=1, K=K, N=N, E=E, topk=k, dtype=WL.FP8),
                       d["w1"], d["w2"], np.unique(rid[tokens]))
    ref, rid_s, _ = orc.moe_forward(WL.bf16_bits(xv), lv, None, k, cfg.score_fn, W,
                                    cfg.n_groups, cfg.topk_groups, True, requant_h=True,
                                    tokens=tokens)
    assert np.array_equal(rid_s, rid[tokens])
    got = torch.cat([layer.out[r, :n[r]] for r in range(G)])[torch.from_numpy(tokens).to(DEV)]
    assert_close_rel(got.float().cpu().numpy(), ref, TOL[WL.FP8], cfg.name)
    bits = layer.out.view(torch.int16).cpu().numpy()
    for r in range(G):
        assert np.all(bits[r, n[r]:] == np.int16(SENTINEL)), f"shard {r}: padded rows written"

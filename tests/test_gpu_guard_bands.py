"""Guard bands around every buffer the library writes.  Each output buffer
and each workspace of every entry point sits between two 4 KiB bands of
sentinel bytes, and the bands must be unchanged after the call.  An
out-of-bounds write anywhere in the kernels (a tile tail, a scatter index, a
workspace carve, a vector store past a row) changes a sentinel byte.  The
shapes are small and ragged, with tails in every tile dimension, and cover
every dtype, both activation formats, the one-call layers and the
expert-parallel dispatch / combine.  This is the stand-in for a device
memory checker, which is not available here."""
import numpy as np
import pytest
import torch

import workloads as WL
from gpu_common import Guarded, GpuWeights, gbmoe, run_forward, run_stages

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


STANDARD = [WL.TINY, WL.SMALL_BF16, WL.SMALL_SIGMOID, WL.SMALL_PAIR, WL.SMALL_PAIR_TOP2,
            WL.SMALL_FP8, WL.SMALL_FP8_K640, WL.SMALL_FP8_NARROW, WL.SMALL_FP8CH,
            WL.SMALL_FP8CH_PAIR, WL.SMALL_FP8T]


@pytest.mark.parametrize("cfg", STANDARD, ids=lambda c: c.name)
def test_separate_calls_write_only_their_buffers(cfg):
    """route, align, quantise (x and H), gather, both grouped GEMMs and the
    reduce, every buffer guarded; per-tensor e4m3 with dynamic and with
    static scales."""
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    g = gbmoe()
    guard = Guarded()
    ids, wts = guard((cfg.M, cfg.topk), torch.int32), guard((cfg.M, cfg.topk), torch.float32)
    g.moe_topk_route(d["logits"], d["bias"], cfg.topk, cfg.score_fn, cfg.n_groups,
                     cfg.topk_groups, cfg.renorm, ids, wts)
    g.moe_count_expert_tokens(ids, cfg.E, guard((cfg.E,), torch.int32))
    st = run_stages(cfg, d, gw, ids, wts, alloc=guard)
    guard.check(cfg.name)
    assert st["err"].item() == 0
    if cfg.dtype == WL.FP8_TENSOR:
        guard2 = Guarded()
        one = torch.full((1,), 0.02, dtype=torch.float32, device=DEV)
        st = run_stages(cfg, d, gw, ids, wts, a1_scale=one, a2_scale=one, alloc=guard2)
        guard2.check(cfg.name + " static scales")
        assert st["err"].item() == 0


@pytest.mark.parametrize("cfg", STANDARD, ids=lambda c: c.name)
def test_one_call_layers_write_only_their_buffers(cfg):
    """moe_forward, moe_forward_chunked (a ragged last chunk) and
    moe_forward_shared (the shared expert in the layer's dtype family), with
    outputs and workspaces guarded."""
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    g = gbmoe()
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    guard = Guarded()
    _, _, _, err = run_forward(cfg, d, gw, alloc=guard)
    guard.check(cfg.name + " one call")
    assert err.item() == 0

    chunk = max(1, (M + 2) // 3)
    guard = Guarded()
    args = (d["logits"], d["bias"], N, E, k, cfg.score_fn, cfg.n_groups, cfg.topk_groups,
            cfg.renorm, cfg.dtype, gw.w1, gw.w1s, gw.w2, gw.w2s)
    out = guard((M, K), torch.bfloat16)
    ids, wts = guard((M, k), torch.int32), guard((M, k), torch.float32)
    ws = guard.ws(g.WS_FORWARD, chunk, E, N, K, k, cfg.dtype)
    g.moe_forward_chunked(d["x"], *args, out, ws, chunk, topk_ids=ids, topk_weights=wts)
    guard.check(cfg.name + " chunked")

    Ns = 256
    sdt = {WL.BF16: WL.BF16, WL.FP8: WL.FP8}.get(cfg.dtype, WL.FP8_CHANNEL)
    gen = torch.Generator(device=DEV).manual_seed(7)
    w1s = (torch.randn((2 * Ns, K), generator=gen, device=DEV) / K ** 0.5).to(torch.bfloat16)
    w2s = (torch.randn((K, Ns), generator=gen, device=DEV) / Ns ** 0.5).to(torch.bfloat16)
    sh = WL.MoEConfig("shared", M=M, K=K, N=Ns, E=1, topk=1, dtype=sdt)
    sw = GpuWeights(sh, w1s.unsqueeze(0), w2s.unsqueeze(0))
    s1 = None if sdt == WL.BF16 else sw.w1s[0]
    s2 = None if sdt == WL.BF16 else sw.w2s[0]
    guard = Guarded()
    out = guard((M, K), torch.bfloat16)
    out_sh = guard((M, K), torch.bfloat16)
    aux = torch.cuda.Stream()
    g.moe_forward_shared(d["x"], *args, out, guard.ws(g.WS_FORWARD, M, E, N, K, k, cfg.dtype),
                         Ns, sw.w1[0], sw.w2[0], out_sh,
                         guard.ws(g.WS_SHARED, M, 1, Ns, K, 1, sdt), aux_stream=aux,
                         ev_input_ready=torch.cuda.Event(), ev_output_ready=torch.cuda.Event(),
                         shared_dtype=sdt, w1s_scales=s1, w2s_scales=s2)
    guard.check(cfg.name + " with a shared expert")


@pytest.mark.parametrize("cfg", [WL.SMALL_BATCHED, WL.SMALL_BATCHED_SHORT, WL.SMALL_BATCHED_FP8,
                                 WL.SMALL_BATCHED_FP8_K640], ids=lambda c: c.name)
def test_batched_writes_only_its_buffers(cfg):
    _batched_guarded(cfg)


def _batched_guarded(cfg):
    d = WL.make_inputs(cfg, DEV)
    g = gbmoe()
    E, T, K = cfg.E, cfg.M, cfg.K
    guard = Guarded()
    yb = guard((E, T, K), torch.bfloat16)
    ws = guard.ws(g.WS_BATCHED, T, E, cfg.N, K, 1, cfg.dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if cfg.dtype == WL.BF16:
        g.moe_batched_masked_experts(d["x_b"], d["counts"], cfg.N, d["w1"], d["w2"], yb, ws,
                                     err_word=err)
    else:
        gw = GpuWeights(cfg, d["w1"], d["w2"])
        q = guard((E, T, K), torch.uint8)
        sc = guard((E * T, K // 128), torch.float32)
        g.moe_quant_fp8_group(d["x_b"].reshape(E * T, K), q.view(E * T, K), sc)
        g.moe_batched_masked_experts(q, d["counts"], cfg.N, gw.w1, gw.w2, yb, ws, dtype=WL.FP8,
                                     x_b_scales=sc, w1_scales=gw.w1s, w2_scales=gw.w2s,
                                     err_word=err)
    guard.check(cfg.name)
    assert err.item() == 0


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
def test_ep_dispatch_and_combine_write_only_their_buffers(fp8):
    cfg = WL.EP4
    g = gbmoe()
    d = WL.make_ep_inputs(cfg, DEV)
    G, M, K, E, k, W = cfg.G, cfg.M, cfg.K, cfg.E, cfg.topk, cfg.worst_tokens
    guard = Guarded()
    ids, wts = guard((G, M, k), torch.int32), guard((G, M, k), torch.float32)
    g.moe_topk_route(d["logits"].view(G * M, E), None, k, cfg.score_fn, cfg.n_groups,
                     cfg.topk_groups, True, ids.view(G * M, k), wts.view(G * M, k))
    recv_counts, recv_pos = guard((E,), torch.int32), guard((G, M, k), torch.int32)
    ws = guard.ws(g.WS_EP_DISPATCH, M, E, G, K, k, 0)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if fp8:
        xq, xs = guard((G, M, K), torch.uint8), guard((G * M, K // 128), torch.float32)
        g.moe_quant_fp8_group(d["x"].view(G * M, K), xq.view(G * M, K), xs)
        recv_x, recv_s = guard((E, W, K), torch.uint8), guard((E * W, K // 128), torch.float32)
        g.moe_ep_dispatch(xq, d["num_tokens"], ids, E, W, recv_x, recv_counts, recv_pos, ws, err,
                          dtype=WL.FP8, x_scales=xs, recv_scales=recv_s)
    else:
        recv_x = guard((E, W, K), torch.bfloat16)
        g.moe_ep_dispatch(d["x"], d["num_tokens"], ids, E, W, recv_x, recv_counts, recv_pos, ws,
                          err)
    recv_y = guard((E, W, K), torch.bfloat16)
    recv_y.view(torch.int16).fill_(0)
    out = guard((G, M, K), torch.bfloat16)
    g.moe_ep_combine(recv_y, ids, recv_pos, wts, d["num_tokens"], out)
    guard.check("EP dispatch / combine")
    assert err.item() == 0


def test_quantisers_write_only_their_buffers():
    """The weight-block quantiser (ragged in neither dimension by contract,
    but over several experts), the per-tensor quantisers with a device row
    count, and the three quantise-and-permute calls."""
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(11)
    guard = Guarded()
    w = torch.randn((3, 384, 640), generator=gen, device=DEV).to(torch.bfloat16)
    g.moe_quant_fp8_block(w, guard((3, 384, 640), torch.uint8), guard((3, 3, 5), torch.float32))
    M, K, k = 77, 640, 3
    x = torch.randn((M, K), generator=gen, device=DEV).to(torch.bfloat16)
    n_rows = torch.tensor([50], dtype=torch.int32, device=DEV)
    g.moe_quant_fp8_tensor(x, guard((M, K), torch.uint8), guard((M,), torch.float32),
                           guard((1,), torch.int32), n_rows=n_rows)
    g.moe_quant_fp8_tensor_static(x, torch.full((1,), 0.01, device=DEV),
                                  guard((M, K), torch.uint8), guard((M,), torch.float32))
    inv = torch.randperm(M * k, generator=gen, device=DEV).to(torch.int32)
    inv[::7] = -1  # pairs not computed here are not written
    ld = (M * k + 3) // 4 * 4
    g.moe_quant_fp8_group_permute(x, inv, k, guard((M * k, K), torch.uint8),
                                  guard((K // 128, ld), torch.float32))
    g.moe_quant_fp8_row_permute(x, inv, k, guard((M * k, K), torch.uint8),
                                guard((M * k,), torch.float32))
    g.moe_quant_fp8_tensor_permute(x, inv, k, guard((M * k, K), torch.uint8),
                                   guard((M * k,), torch.float32),
                                   amax_ws=guard((1,), torch.int32))
    guard.check("quantisers")


@pytest.mark.parametrize("cfg", [WL.MIXTRAL_PREFILL, WL.DSV3_DECODE, WL.DSV3_PREFILL_FP8,
                                 WL.DSV3_PREFILL_FP8CH, WL.DSV3_PREFILL_FP8T],
                         ids=lambda c: c.name)
def test_full_size_layers_write_only_their_buffers(cfg):
    """The one-call layer at the bench's sizes (many tile waves, the CTA-pair
    and block-scaled kernels' full schedules): outputs and the workspace
    guarded."""
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    guard = Guarded()
    _, _, _, err = run_forward(cfg, d, gw, alloc=guard)
    guard.check(cfg.name)
    assert err.item() == 0


@pytest.mark.parametrize("cfg", [WL.BATCHED_MASKED, WL.BATCHED_MASKED_FP8], ids=lambda c: c.name)
def test_full_size_batched_writes_only_its_buffers(cfg):
    """The batched masked layer at the bench's sizes (32 experts x 1024
    rows, K = 7168), bf16 and e4m3."""
    _batched_guarded(cfg)

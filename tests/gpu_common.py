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
    blocks = oracle_blocks(cfg, w1, w2, experts)
    return orc.Weights(cfg.dtype, experts=blocks, E=cfg.E, N=cfg.N, K=cfg.K)


def oracle_blocks(cfg, w1, w2, experts=None):
    """{expert: (w1e, w2e[, w1se, w2se])} in the oracle's weight format."""
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
    return blocks


GUARD = 4096  # bytes on each side; a multiple of 256 keeps the inner buffer's alignment
GUARD_BYTE = 0xA5


class Guarded:
    """An allocator (shape, dtype) -> tensor whose buffers each sit between two
    bands of GUARD sentinel bytes; check() asserts that no band changed."""

    def __init__(self, device="cuda"):
        self.device = device
        self.bufs = []

    def __call__(self, shape, dtype):
        shape = tuple(int(v) for v in shape)
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((GUARD + n + GUARD,), GUARD_BYTE, dtype=torch.uint8,
                         device=self.device)
        self.bufs.append((raw, n, f"{dtype} {shape}"))
        return raw[GUARD:GUARD + n].view(dtype).view(shape)

    def ws(self, which, *args):
        n = gbmoe().moe_workspace_size(which, *args)
        assert n > 0
        return self((n,), torch.uint8)

    def check(self, what):
        if torch.device(self.device).type == "cuda":
            torch.cuda.synchronize()
        assert self.bufs
        for raw, n, name in self.bufs:
            head, tail = raw[:GUARD], raw[GUARD + n:]
            bad_h = int((head != GUARD_BYTE).sum())
            bad_t = int((tail != GUARD_BYTE).sum())
            assert bad_h == 0 and bad_t == 0, \
                f"{what}: {name}: {bad_h} bytes before and {bad_t} after the buffer overwritten"


def _torch_alloc(dev):
    return lambda shape, dtype: torch.empty(shape, dtype=dtype, device=dev)


def run_forward(cfg, d, gw, stream=None, a1_scale=None, a2_scale=None, alloc=None):
    """The whole Standard layer on the GPU (per-tensor e4m3: static activation
    scales a1_scale / a2_scale, device fp32 scalars, when given); returns
    out, ids, weights, err.  alloc(shape, dtype) makes the output buffers and
    the workspace (default: torch.empty on x's device)."""
    g = gbmoe()
    dev = d["x"].device
    alloc = alloc or _torch_alloc(dev)
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    out = alloc((M, K), torch.bfloat16)
    ids = alloc((M, k), torch.int32)
    wts = alloc((M, k), torch.float32)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = alloc((g.moe_workspace_size(g.WS_FORWARD, M, E, N, K, k, cfg.dtype),), torch.uint8)
    g.moe_forward(d["x"], d["logits"], d["bias"], N, E, k, cfg.score_fn,
                  cfg.n_groups, cfg.topk_groups, cfg.renorm, cfg.dtype, gw.w1,
                  gw.w1s, gw.w2, gw.w2s, out, ws, topk_ids=ids, topk_weights=wts,
                  err_word=err, stream=stream, a1_scale=a1_scale, a2_scale=a2_scale)
    return out, ids, wts, err


def oracle_forward(cfg, d, W, tokens=None, nthreads=0, static_scales=None):
    return orc.moe_forward(WL.bf16_bits(d["x"]), d["logits"].cpu().numpy(),
                           None if d["bias"] is None else d["bias"].cpu().numpy(),
                           cfg.topk, cfg.score_fn, W, cfg.n_groups, cfg.topk_groups,
                           cfg.renorm, cfg.requant_h, tokens=tokens,
                           nthreads=nthreads, static_scales=static_scales)


def _grouped_choice_is_valid(v, ids_row, topk, n_groups, topk_groups, tol):
    """Whether ids_row is one correct result of the sigmoid group-limited
    top-k on the fp32 values v = l + b of one token when group keys closer
    than `tol` count as tied: there must be a set S of topk_groups groups that
    holds every group whose fp64 key is above the topk_groups-th largest key
    by more than tol, only groups within tol of that key besides, every group
    ids_row uses, and whose experts' top-k by v (ties: lower id, descending
    order) is ids_row.  The fp64 key of a group is the sum of the sigmoids of
    its two largest v (ties: lower id)."""
    import itertools
    E = v.size
    gs = E // n_groups
    key = np.empty(n_groups)
    for gi in range(n_groups):
        vg = v[gi * gs:(gi + 1) * gs].astype(np.float64)
        order = np.lexsort((np.arange(gs), -vg))[:min(2, gs)]
        key[gi] = np.sum(1.0 / (1.0 + np.exp(-vg[order])))
    kth = np.sort(key)[::-1][topk_groups - 1]
    sure = [gi for gi in range(n_groups) if key[gi] > kth + tol]
    border = [gi for gi in range(n_groups) if abs(key[gi] - kth) <= tol]
    used = set(int(e) // gs for e in ids_row)
    if not used <= set(sure) | set(border):
        return False
    need = topk_groups - len(sure)
    if need < 0 or need > len(border):
        return False
    for extra in itertools.combinations(border, need):
        groups = set(sure) | set(extra)
        if not used <= groups:
            continue
        cand = np.array([e for e in range(E) if e // gs in groups])
        order = np.lexsort((cand, -v[cand].astype(np.float64)))
        if np.array_equal(cand[order[:topk]], np.asarray(ids_row)):
            return True
    return False


def check_ids(gpu_ids, ref_ids, margin, what="", cfg=None, logits=None, bias=None):
    """Router ids are compared bit for bit.  A token may differ only when the
    oracle reports a group-key margin below 1e-6 (a last-bit difference
    between two exp implementations could flip a group choice); there
    several results are correct, so the GPU's ids must be one of them (given
    cfg and the host logits / bias: the valid-choice check above), and such
    tokens must stay rare.  Returns the tokens that differ."""
    diff = np.flatnonzero((gpu_ids != ref_ids).any(1))
    near = [t for t in diff if margin[t] < 1e-6]
    assert len(diff) == len(near), f"{what}: ids differ on tokens {diff[:10]}"
    assert len(near) <= max(1, len(ref_ids) // 1000), f"{what}: {len(near)} near-ties"
    if len(near):
        assert cfg is not None and logits is not None, \
            f"{what}: near-tie tokens {near[:10]} need the routing inputs to be validated"
        for t in near:
            v = logits[t].astype(np.float32) + (np.zeros_like(logits[t], np.float32)
                                                if bias is None else bias.astype(np.float32))
            assert _grouped_choice_is_valid(v, gpu_ids[t], cfg.topk, cfg.n_groups,
                                            cfg.topk_groups, 1e-6), \
                f"{what}: token {t}: GPU ids {gpu_ids[t]} are not a valid near-tie choice"
    return diff


def run_stages(cfg, d, gw, ids, wts, a1_scale=None, a2_scale=None, keep_hidden=False,
               alloc=None):
    """The Standard layer as its separate calls, on the given routing (ids
    (M, topk) int32 and weights (M, topk) fp32 on the device): align, [FP8
    quantise], gather, gate/up GEMM, [quantise H], down GEMM into the
    (M, topk, K) slots, and the ordered reduce (per-tensor e4m3: static
    scales a1_scale / a2_scale when given).  Returns the device tensors
    counts, offsets, sorted, inv, y_slot, out, err and amax (the per-tensor
    maxima of x and H as float bits, dynamic per-tensor e4m3 only); with
    keep_hidden (per-token and per-tensor e4m3) also xq / xs (x's codes and
    row scales), Hb (the bf16 hidden rows) and H / Hs (their codes and row
    scales).  alloc(shape, dtype) makes every buffer the calls write
    (default: torch.empty on x's device)."""
    g = gbmoe()
    dev = d["x"].device
    alloc = alloc or _torch_alloc(dev)
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    P = M * k
    i32, f32 = torch.int32, torch.float32
    counts = alloc((E,), i32).fill_(-7)
    offsets = alloc((E + 1,), i32)
    srt = alloc((P,), i32).fill_(-5)
    inv = alloc((P,), i32)
    err = torch.zeros(1, dtype=i32, device=dev)
    g.moe_align_permute(ids, E, counts, offsets, srt, inv,
                        alloc((g.moe_workspace_size(g.WS_ALIGN, M, E, 0, 0, k, 0),), torch.uint8),
                        err)
    fp8 = cfg.dtype != WL.BF16
    tensor = cfg.dtype == WL.FP8_TENSOR
    ch = cfg.dtype == WL.FP8_CHANNEL or tensor   # one scale per row of A and of H
    amax = alloc((2,), i32)
    ld = (P + 3) // 4 * 4  # group-major FP8 row scales
    if fp8:
        sk = 1 if ch else K // 128
        xq = alloc((M, K), torch.uint8)
        xs = alloc((M, sk), f32)
        if tensor and a1_scale is not None:
            g.moe_quant_fp8_tensor_static(d["x"], a1_scale, xq, xs.view(-1))
        elif tensor:
            g.moe_quant_fp8_tensor(d["x"], xq, xs.view(-1), amax[0:1])
        else:
            g.moe_quant_fp8_group(d["x"], xq, xs, group=K if ch else 128)
        A = alloc((P, K), torch.uint8)
        As = alloc((sk, ld), f32)
        g.moe_permute_rows(xq, xs, srt, offsets, k, E, cfg.dtype, A, As)
    else:
        A = alloc((P, K), torch.bfloat16)
        As = None
        g.moe_permute_rows(d["x"], None, srt, offsets, k, E, cfg.dtype, A, None)
    if ch:
        Hb = alloc((P, N), torch.bfloat16)
        g.moe_grouped_gemm_gate_up_silu(A, As, offsets, M, k, E, N, K, gw.w1, gw.w1s,
                                        cfg.dtype, Hb, None, err)
        H = alloc((P, N), torch.uint8)
        Hs = alloc((P, 1), f32)
        if tensor and a2_scale is not None:  # rows of pairs computed here: offsets[E]
            g.moe_quant_fp8_tensor_static(Hb, a2_scale, H, Hs.view(-1), n_rows=offsets[E:])
        elif tensor:
            g.moe_quant_fp8_tensor(Hb, H, Hs.view(-1), amax[1:2], n_rows=offsets[E:])
        else:
            g.moe_quant_fp8_group(Hb, H, Hs, group=N)
        if not keep_hidden:
            del Hb
    elif fp8:
        H = alloc((P, N), torch.uint8)
        Hs = alloc((N // 128, ld), f32)
        g.moe_grouped_gemm_gate_up_silu(A, As, offsets, M, k, E, N, K, gw.w1, gw.w1s,
                                        cfg.dtype, H, Hs, err)
    else:
        H = alloc((P, N), torch.bfloat16)
        Hs = None
        g.moe_grouped_gemm_gate_up_silu(A, None, offsets, M, k, E, N, K, gw.w1, None,
                                        cfg.dtype, H, None, err)
    del A, As
    y = alloc((M, k, K), torch.bfloat16)
    g.moe_grouped_gemm_down(H, Hs, srt, offsets, wts, M, k, E, N, K, gw.w2, gw.w2s,
                            cfg.dtype, y, err)
    out = alloc((M, K), torch.bfloat16)
    g.moe_unpermute_weighted_reduce(y, inv, M, k, K, out)
    res = {"counts": counts, "offsets": offsets, "sorted": srt, "inv": inv,
           "y_slot": y, "out": out, "err": err, "amax": amax}
    if keep_hidden and ch:
        res.update(xq=xq, xs=xs, Hb=Hb, H=H, Hs=Hs)
    return res


def oracle_pair_rows(cfg, d, w1, w2, rid, pairs):
    """The oracle's unweighted expert output y = expert_e(x_t) (fp64, (n, K))
    for the listed pairs p = t*topk + j with e = rid[t, j]: the rows of each
    expert are laid out as one BatchedExperts block (built from the oracle's
    own routing) and computed by the oracle's batched form on all host
    cores."""
    pairs = np.asarray(pairs, np.int64)
    t_of, j_of = pairs // cfg.topk, pairs % cfg.topk
    e_of = rid[t_of, j_of]
    experts = sorted(set(int(e) for e in e_of))
    local = {e: i for i, e in enumerate(experts)}
    slot = np.zeros(pairs.size, np.int64)
    per = {e: 0 for e in experts}
    for n, e in enumerate(e_of):
        slot[n] = per[int(e)]
        per[int(e)] += 1
    T = max(per.values())
    xbits = WL.bf16_bits(d["x"])
    xb = np.zeros((len(experts), T, cfg.K), np.uint16)
    for n in range(pairs.size):
        xb[local[int(e_of[n])], slot[n]] = xbits[t_of[n]]
    counts = np.array([per[e] for e in experts], np.int32)
    blocks = {local[e]: blk for e, blk in oracle_blocks(cfg, w1, w2, experts).items()}
    Wl = orc.Weights(cfg.dtype, experts=blocks, E=len(experts), N=cfg.N, K=cfg.K)
    yb, n_rows = orc.batched_experts(xb, counts, Wl, requant_h=cfg.requant_h)
    assert n_rows == pairs.size
    return np.stack([yb[local[int(e_of[n])], slot[n]] for n in range(pairs.size)])

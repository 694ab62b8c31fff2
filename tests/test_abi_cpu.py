"""Host-side checks of the C-ABI library that need no GPU: it builds, loads,
exports every function include/gbmoe.h declares, and sizes workspaces."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"^\s*[\w\s\*]*?\b(\w+)\s*\(", txt, flags=re.M))
    return {n for n in names if n.startswith(("moe_", "gbmoe_"))}


def test_header_is_plain_c():
    """include/gbmoe.h is a C header: it compiles warning-free as C (and C++)."""
    import shutil
    import subprocess
    hdr = os.path.join(ROOT, "include", "gbmoe.h")
    for cc, lang in (("gcc", "c"), ("g++", "c++")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not found")
        r = subprocess.run([cc, "-fsyntax-only", "-Wall", "-Wextra", "-Werror", "-x", lang, hdr],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_c_caller_builds(tmp_path):
    """A C program that uses the library through include/gbmoe.h alone
    compiles warning-free and links against libgbmoe.so and the CUDA runtime."""
    import c_example
    try:
        exe = c_example.build(str(tmp_path))
    except FileNotFoundError as e:
        pytest.skip(str(e))
    assert os.access(exe, os.X_OK)


def test_library_exports_every_declared_symbol():
    import mixture_experts_layer_count_gb300 as g
    lib = g.load()
    declared = _declared()
    assert len(declared) >= 14, declared
    for name in declared:
        assert hasattr(lib, name), name


def test_binding_covers_every_entry_point():
    import mixture_experts_layer_count_gb300 as g
    for name in _declared():
        if name.startswith("moe_"):
            assert callable(getattr(g, name, None)), name


def test_workspace_sizes():
    import mixture_experts_layer_count_gb300 as g
    # Standard layer: ids, weights, counts, offsets, sorted, inv, chunk
    # histograms, gathered rows, H and the weighted slots, each 256-aligned
    M, E, N, K, k = 64, 8, 128, 256, 2
    n = g.moe_workspace_size(g.WS_FORWARD, M, E, N, K, k, g.BF16)
    P = M * k
    expect = sum(-(-b // 256) * 256 for b in (
        P * 4, P * 4, E * 4, (E + 1) * 4, P * 4, P * 4, 1 * E * 4,
        P * K * 2, P * N * 2, P * K * 2))  # A, H, y_slot
    assert n == expect
    assert g.moe_workspace_size(g.WS_FORWARD, M, E, 100, K, k, g.BF16) == 0  # N % 128
    # batched: H (E*T, N) in the operand type; for e4m3 also H's and x_b's
    # group-major scales with E*T rounded up to 4 rows
    T, E, N, K = 15, 4, 256, 384
    R, ld = E * T, (E * T + 3) // 4 * 4
    assert g.moe_workspace_size(g.WS_BATCHED, T, E, N, K, 1, g.BF16) == -(-R * N * 2 // 256) * 256
    assert g.moe_workspace_size(g.WS_BATCHED, T, E, N, K, 1, g.FP8_E4M3) == sum(
        -(-b // 256) * 256 for b in (R * N, ld * (N // 128) * 4, ld * (K // 128) * 4))
    assert g.moe_workspace_size(g.WS_BATCHED, T, E, N, K, 1, g.FP8_E4M3_CHANNEL) == 0
    # block-scaled e4m3 GEMMs take K and N up to 16384 (128 scale blocks)
    assert g.moe_workspace_size(g.WS_FORWARD, 4, 2, 128, 16384, 1, g.FP8_E4M3) > 0
    assert g.moe_workspace_size(g.WS_FORWARD, 4, 2, 128, 16512, 1, g.FP8_E4M3) == 0
    assert g.moe_workspace_size(g.WS_FORWARD, 4, 2, 16512, 128, 1, g.FP8_E4M3) == 0
    assert g.moe_workspace_size(g.WS_FORWARD, 4, 2, 16512, 128, 1, g.BF16) > 0
    assert g.moe_workspace_size(g.WS_ALIGN, 8192, 256, 0, 0, 8, 0) == 32 * 256 * 4
    # shared experts (M rows, Ns = N): H; e4m3 also H's group-major scales,
    # the codes of x, x's scales row-major and group-major
    M, Ns, K = 100, 256, 384
    ld = (M + 3) // 4 * 4
    assert g.moe_workspace_size(g.WS_SHARED, M, 1, Ns, K, 1, g.BF16) == -(-M * Ns * 2 // 256) * 256
    assert g.moe_workspace_size(g.WS_SHARED, M, 1, Ns, K, 1, g.FP8_E4M3) == sum(
        -(-b // 256) * 256 for b in (M * Ns, ld * (Ns // 128) * 4, M * K, M * (K // 128) * 4,
                                     ld * (K // 128) * 4))
    # per-channel e4m3: H, H's scale per row, H in bf16, the codes of x, x's scale per row
    assert g.moe_workspace_size(g.WS_SHARED, M, 1, Ns, K, 1, g.FP8_E4M3_CHANNEL) == sum(
        -(-b // 256) * 256 for b in (M * Ns, M * 4, M * Ns * 2, M * K, M * 4))
    assert g.moe_workspace_size(g.WS_SHARED, M, 1, Ns, K, 1, g.FP8_E4M3_TENSOR) == 0
    # EP dispatch (M tokens per shard, E routed experts, N = G shards): the
    # pairs' ids, the map, counts, offsets, sorted, inv, chunk histograms
    G, M, E, k = 4, 100, 64, 6
    P = G * M * k
    expect = sum(-(-b // 256) * 256 for b in (P * 4, (E + 1) * 4, E * 4, (E + 1) * 4, P * 4,
                                               P * 4, -(-P // 2048) * E * 4))
    assert g.moe_workspace_size(g.WS_EP_DISPATCH, M, E, G, 256, k, 0) == expect
    assert g.moe_workspace_size(g.WS_EP_DISPATCH, M, E, 5, 256, k, 0) == 0  # E % G


def test_status_strings():
    import mixture_experts_layer_count_gb300 as g
    lib = g.load()
    assert lib.gbmoe_status_string(0) == b"ok"
    assert lib.gbmoe_status_string(1) == b"invalid argument"


# ---------------------------------------------------------------------------
# Argument checks: every call below is invalid and must be refused on the
# host, before any device query or launch.  The pointers are stand-ins that
# are never dereferenced.  Skipped where a CUDA device is visible, so that a
# mistake in the checks could never turn into a launch on garbage pointers.

P16 = 1 << 20          # a 16-byte aligned stand-in pointer
P_ODD = (1 << 20) + 4  # misaligned for TMA / vector access


@pytest.fixture
def lib():
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-side argument checks run where no device is visible")
    import mixture_experts_layer_count_gb300 as g
    return g.load()


INVALID, UNSUPPORTED = 1, 2


def test_route_rejects_bad_arguments(lib):
    f = lib.moe_topk_route
    #        logits bias  M   E  topk fn ng tg rn ids  w   err stream
    assert f(P16, None, 8, 8, 9, 0, 1, 1, 1, P16, P16, None, None) == INVALID   # topk > E
    assert f(P16, None, 8, 64, 33, 0, 1, 1, 1, P16, P16, None, None) == INVALID  # topk > 32
    assert f(P16, None, 8, 513, 2, 0, 1, 1, 1, P16, P16, None, None) == INVALID  # E > 512
    assert f(P16, P16, 8, 8, 2, 0, 1, 1, 1, P16, P16, None, None) == INVALID     # bias with softmax
    assert f(P16, None, 8, 10, 2, 1, 4, 2, 1, P16, P16, None, None) == INVALID   # E % groups
    assert f(P16, None, 8, 16, 5, 1, 4, 1, 1, P16, P16, None, None) == INVALID   # topk > kept experts
    assert f(P16, None, 8, 8, 2, 7, 1, 1, 1, P16, P16, None, None) == INVALID    # score function
    assert f(None, None, 8, 8, 2, 0, 1, 1, 1, P16, P16, None, None) == INVALID   # null logits


def test_count_align_reject_bad_arguments(lib):
    c = lib.moe_count_expert_tokens
    #        ids  M  k  Eg map  E  counts err  s
    assert c(P16, 8, 2, 8, None, 8, None, None, None) == INVALID
    assert c(P16, -1, 2, 8, None, 8, P16, None, None) == INVALID
    assert c(None, 8, 2, 8, None, 8, P16, None, None) == INVALID
    assert c(P16, 8, 2, 16, None, 8, P16, None, None) == INVALID  # no map: Eg must equal E
    assert c(P16, 8, 2, 0, P16, 8, P16, None, None) == INVALID    # no routed experts
    a = lib.moe_align_permute
    #        ids  M  k  Eg map   E  cnt  off  srt  inv  ws   wsb  err  s
    assert a(P16, 8, 2, 8, None, 8, None, P16, P16, P16, P16, 0, None, None) == INVALID  # ws too small
    assert a(P16, 8, 2, 600, None, 600, None, P16, P16, P16, P16, 1 << 20, None, None) == INVALID
    assert a(P16, 8, 2, 12, None, 8, None, P16, P16, P16, P16, 1 << 20, None, None) == INVALID
    # the no-workspace variant refuses sizes beyond its fixed array
    assert lib.moe_align_permute_no_ws(P16, 65536, 8, 512, None, P16, P16, P16, None, None) == INVALID


def test_quant_rejects_bad_arguments(lib):
    q = lib.moe_quant_fp8_group
    assert q(P16, None, 4, 256, 64, P16, P16, None) == INVALID     # group
    assert q(P16, None, 4, 200, 128, P16, P16, None) == INVALID    # K % 128
    assert q(P_ODD, None, 4, 256, 128, P16, P16, None) == INVALID  # alignment
    assert lib.moe_quant_fp8_block(P16, 100, 256, 128, P16, P16, None) == INVALID  # R % 128
    assert lib.moe_quant_fp8_block(P16, 128, 256, 128, None, P16, None) == INVALID


def test_gemm_calls_reject_bad_arguments(lib):
    g = lib.moe_grouped_gemm_gate_up_silu
    #        A   As    off  M  k  E  N    K    w1   w1s  dt H    Hs   err  s
    assert g(P16, None, P16, 8, 2, 8, 100, 256, P16, None, 0, P16, None, None, None) == INVALID
    assert g(P16, None, P16, 8, 2, 8, 128, 256, P16, None, 5, P16, None, None, None) == UNSUPPORTED
    assert g(P_ODD, None, P16, 8, 2, 8, 128, 256, P16, None, 0, P16, None, None, None) == INVALID
    assert g(P16, None, P16, 8, 2, 8, 128, 256, P16, None, 1, P16, None, None, None) == INVALID  # fp8 w/o scales
    assert g(P16, None, P16, 8, 2, 8, 128, 256, None, None, 0, P16, None, None, None) == INVALID
    d = lib.moe_grouped_gemm_down
    assert d(P16, None, P16, P16, P16, 8, 2, 8, 128, 256, P16, None, 1, P16, None, None) == INVALID
    assert d(P16, None, None, P16, None, 8, 2, 8, 128, 256, P16, None, 0, P16, None, None) == INVALID  # no sorted ids
    pr = lib.moe_permute_rows
    #         x   xs    rw    srt  off  M  k  E  K    dt A    As   s
    assert pr(P16, None, None, P16, P16, 8, 2, 8, 256, 9, P16, None, None) == UNSUPPORTED
    assert pr(P16, None, None, P16, P16, 8, 2, 8, 200, 0, P16, None, None) == INVALID
    assert pr(None, None, None, P16, P16, 8, 2, 8, 256, 0, P16, None, None) == INVALID
    # FP8 rows take the router weight in the quantiser, not in the gather
    assert pr(P16, P16, P16, P16, P16, 8, 1, 8, 256, 1, P16, P16, None) == INVALID
    assert lib.moe_unpermute_weighted_reduce(P16, None, 8, 2, 12, P16, None) == INVALID
    ed = lib.moe_ep_dispatch
    #         x    xs    ntok ids  G  M   K    E   k  worst dt rx   rs    rc   rp   ws   wsb      err   s
    assert ed(P16, None, P16, P16, 3, 16, 256, 32, 4, 48, 0, P16, None, P16, P16, P16, 1 << 20, None, None) == INVALID  # E % G
    assert ed(P16, None, P16, P16, 2, 16, 250, 32, 4, 32, 0, P16, None, P16, P16, P16, 1 << 20, None, None) == INVALID  # K % 8
    assert ed(P16, None, P16, P16, 2, 16, 256, 32, 4, 32, 0, P16, None, P16, P16, P16, 16, None, None) == INVALID       # ws too small
    assert ed(P16, None, None, P16, 2, 16, 256, 32, 4, 32, 0, P16, None, P16, P16, P16, 1 << 20, None, None) == INVALID  # no counts
    assert ed(P_ODD, None, P16, P16, 2, 16, 256, 32, 4, 32, 0, P16, None, P16, P16, P16, 1 << 20, None, None) == INVALID
    assert ed(P16, None, P16, P16, 2, 16, 256, 32, 33, 32, 0, P16, None, P16, P16, P16, 1 << 20, None, None) == INVALID  # topk
    assert ed(P16, None, P16, P16, 2, 16, 256, 32, 4, 32, 2, P16, None, P16, P16, P16, 1 << 20, None, None) == UNSUPPORTED
    # e4m3: both scale arrays, K a multiple of 128
    assert ed(P16, None, P16, P16, 2, 16, 256, 32, 4, 32, 1, P16, P16, P16, P16, P16, 1 << 20, None, None) == INVALID
    assert ed(P16, P16, P16, P16, 2, 16, 256, 32, 4, 32, 1, P16, None, P16, P16, P16, 1 << 20, None, None) == INVALID
    assert ed(P16, P16, P16, P16, 2, 16, 192, 32, 4, 32, 1, P16, P16, P16, P16, P16, 1 << 20, None, None) == INVALID
    ec = lib.moe_ep_combine
    #         ry   ids  pos  w    ntok G  M   K    E   k  worst out  s
    assert ec(P16, P16, P16, P16, P16, 2, 16, 256, 32, 4, 0, P16, None) == INVALID    # worst < 1
    assert ec(P16, P16, P16, None, P16, 2, 16, 256, 32, 4, 32, P16, None) == INVALID  # no weights
    assert ec(P16, P16, P16, P16, P16, 2, 16, 256, 32, 4, 32, P_ODD, None) == INVALID
    assert lib.moe_unpermute_weighted_reduce(P16, None, 8, 33, 256, P16, None) == INVALID
    qp = lib.moe_quant_fp8_group_permute
    #         x    rw    M   K    inv  k  A    As   s
    assert qp(P16, None, 16, 200, P16, 4, P16, P16, None) == INVALID   # K % 128
    assert qp(P16, P16, 16, 256, P16, 2, P16, P16, None) == INVALID    # row weights need top-1
    assert qp(P16, None, 16, 256, None, 4, P16, P16, None) == INVALID  # no inverse map
    assert qp(P_ODD, None, 16, 256, P16, 4, P16, P16, None) == INVALID
    assert qp(P16, None, 16, 256, P16, 4, P16, P16 + 2, None) == INVALID
    rp = lib.moe_quant_fp8_row_permute
    #         x    rw    M   K    inv  k  A    As   s
    assert rp(P16, None, 16, 200, P16, 4, P16, P16, None) == INVALID   # K % 128
    assert rp(P16, P16, 16, 256, P16, 2, P16, P16, None) == INVALID    # row weights need top-1
    assert rp(P16, None, 16, 256, P16, 33, P16, P16, None) == INVALID  # topk > 32
    assert rp(P16, None, 16, 256, None, 4, P16, P16, None) == INVALID  # no inverse map
    assert rp(P_ODD, None, 16, 256, P16, 4, P16, P16, None) == INVALID
    tp = lib.moe_quant_fp8_tensor_permute
    #         x    rw    M   K    inv  k  scale q    As   amax  s
    assert tp(P16, None, 16, 256, P16, 4, None, P16, P16, None, None) == INVALID      # no scale, no amax
    assert tp(P16, None, 16, 256, P16, 4, P16 + 2, P16, P16, None, None) == INVALID   # misaligned scale
    assert tp(P16, P16, 16, 256, P16, 2, P16, P16, P16, None, None) == INVALID        # row weights need top-1
    assert tp(P16, None, 16, 200, P16, 4, P16, P16, P16, None, None) == INVALID       # K % 128
    b = lib.moe_batched_masked_experts
    #        xb  xbs   cnt E  T   N    K    w1   w1s  w2   w2s  dt ac yb   ws   wsb  err  s
    assert b(P16, None, P16, 4, 16, 128, 256, P16, None, P16, None, 2, 0, P16, P16, 1 << 30, None, None) == UNSUPPORTED
    # e4m3 with block scales: all three scale arrays are required, x_b's 4-byte aligned
    assert b(P16, None, P16, 4, 16, 128, 256, P16, P16, P16, P16, 1, 0, P16, P16, 1 << 30, None, None) == INVALID
    assert b(P16, P16, P16, 4, 16, 128, 256, P16, None, P16, P16, 1, 0, P16, P16, 1 << 30, None, None) == INVALID
    assert b(P16, P16, P16, 4, 16, 128, 256, P16, P16, P16, None, 1, 0, P16, P16, 1 << 30, None, None) == INVALID
    assert b(P16, P16 + 2, P16, 4, 16, 128, 256, P16, P16, P16, P16, 1, 0, P16, P16, 1 << 30, None, None) == INVALID
    assert b(P16, P16, P16, 4, 16, 128, 256, P16, P16, P16, P16, 1, 0, P16, P16, 1000, None, None) == INVALID
    assert b(P16, None, P16, 4, 16, 128, 256, P16, None, P16, None, 0, 0, P16, P16, 16, None, None) == INVALID
    assert b(P16, None, None, 4, 16, 128, 256, P16, None, P16, None, 0, 0, P16, P16, 1 << 30, None, None) == INVALID
    assert b(P16, None, P16, 4, 16, 128, 256, P16, None, P16, None, 0, 5, P16, P16, 1 << 30, None, None) == INVALID


def test_forward_rejects_bad_arguments(lib):
    f = lib.moe_forward
    #       x    lg   bias  M   K    N    Eg map   E  k  fn ng tg rn woi act dt
    args = [P16, P16, None, 64, 256, 128, 8, None, 8, 2, 0, 1, 1, 1, 0, 0, 0,
            P16, None, P16, None, None, None, P16, None, None, P16, 1 << 30, None, None]
    #       w1   w1s   w2   w2s   a1s   a2s   out  ids   wts   ws   wsb      err   s
    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a27=1024) == INVALID          # workspace too small
    assert call(a2=P16) == INVALID            # bias with a softmax router
    assert call(a23=P_ODD) == INVALID         # misaligned output
    assert call(a16=1) == INVALID             # FP8 weights without their scales
    assert call(a14=1) == INVALID             # weight on input needs topk 1
    assert call(a6=16) == INVALID             # 16 routed experts, 8 local, no map
    assert call(a15=7) == INVALID             # activation
    assert call(a16=9) == UNSUPPORTED         # dtype
    # static activation scales: per-tensor e4m3 only, 4-byte aligned
    assert call(a21=P16) == INVALID                                  # with bf16
    assert call(a16=1, a18=P16, a20=P16, a22=P16) == INVALID        # with 1 x 128 groups
    assert call(a16=3, a18=P16, a20=P16, a21=P16 + 2) == INVALID    # misaligned a1_scale
    c = lib.moe_forward_chunked
    #         x    lg   bias  M   K    N    Eg map   E  k  fn ng tg rn woi act dt
    assert c(P16, P16, None, 64, 256, 128, 8, None, 8, 2, 0, 1, 1, 1, 0, 0, 0,
             P16, None, P16, None, P16, None, P16, None, None, 32, P16, 1 << 30, None,
             None) == INVALID                                       # a1_scale with bf16
    #        w1   w1s   w2   w2s   a1s  a2s   out  ids   wts   cs  ws   wsb      err
    q = lib.moe_quant_fp8_tensor_static
    #        x    rw    M  K    n    scale q    rs   s
    assert q(P16, None, 4, 256, None, None, P16, P16, None) == INVALID      # no scale
    assert q(P16, None, 4, 256, None, P16 + 2, P16, P16, None) == INVALID   # misaligned
    assert q(P16, None, 4, 200, None, P16, P16, P16, None) == INVALID       # K % 128


def test_shared_experts_reject_bad_arguments(lib):
    f = lib.moe_shared_expert_forward
    #       x    M   K    Ns   w1s  w1ss  w2s  w2ss  dt act out  ws   wsb      err   s
    args = [P16, 64, 256, 128, P16, None, P16, None, 0, 0, P16, P16, 1 << 30, None, None]

    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a8=3) == UNSUPPORTED                  # per-tensor e4m3
    assert call(a8=2) == INVALID                      # per-channel e4m3 without scales
    assert call(a8=2, a5=P16, a7=P16 + 4) == INVALID  # per-channel scales not 16-byte aligned
    assert call(a8=1) == INVALID                      # e4m3 weights without scales
    assert call(a8=1, a5=P16) == INVALID              # ... without w2s's scales
    assert call(a8=1, a5=P16 + 2, a7=P16) == INVALID  # scales not 4-byte aligned
    assert call(a3=100) == INVALID                    # Ns % 128
    assert call(a2=16512, a8=1, a5=P16, a7=P16) == INVALID  # block-scaled K above 16384
    assert call(a12=256) == INVALID                   # workspace too small
    assert call(a9=3) == INVALID                      # activation
    assert call(a4=P_ODD) == INVALID                  # misaligned weights
    fs = lib.moe_forward_shared
    #       x    lg   bias  M   K    N    Eg map   E  k  fn ng tg rn woi act dt
    fargs = [P16, P16, None, 64, 256, 128, 8, None, 8, 2, 0, 1, 1, 1, 0, 0, 0,
             P16, None, P16, None, None, None, P16, P16, 1 << 30, 128, P16, None, P16, None, 0,
             P16, P16, 1 << 30, None, None, None, None, None]
    #        w1   w1s   w2   w2s   a1s   a2s   out  ws   wsb     Ns   w1sh  ss   w2sh  ss  sdt
    #        outsh wssh wsshb    err   s     aux   ev    ev

    def fcall(**kw):
        a = list(fargs)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return fs(*a)
    assert fcall(a31=3) == UNSUPPORTED          # shared experts in per-tensor e4m3
    assert fcall(a31=1) == INVALID              # e4m3 shared experts without scales
    assert fcall(a34=64) == INVALID             # shared workspace too small
    assert fcall(a37=P16) == INVALID            # aux stream without its events
    assert fcall(a16=9) == UNSUPPORTED          # routed dtype
    assert fcall(a22=P16) == INVALID            # a2_scale with bf16


def test_selftest_rejects_bad_arguments(lib):
    s = lib.gbmoe_selftest_bounded_wait
    assert s(None, 1000, None) == INVALID          # no error word
    assert s(P16, 0, None) == INVALID              # limit below 1 us
    assert s(P16, 1000001, None) == INVALID        # limit above 1 s

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
    assert g.moe_workspace_size(g.WS_BATCHED, 16, 4, 128, 256, 1, g.FP8_E4M3) == 0
    assert g.moe_workspace_size(g.WS_ALIGN, 8192, 256, 0, 0, 8, 0) == 32 * 256 * 4


def test_status_strings():
    import mixture_experts_layer_count_gb300 as g
    lib = g.load()
    assert lib.gbmoe_status_string(0) == b"ok"
    assert lib.gbmoe_status_string(1) == b"invalid argument"

"""CPU oracle for the fused MoE hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never links, loads or calls it, and this package imports nothing
from the CUDA library: the two share only the seeded input generators in
``workloads``.

The arithmetic lives in ``moe_oracle.c`` (plain C loops, fp64 sums, fp32
routing and quantisation decisions); this module compiles it with gcc and
marshals numpy arrays into it.  See the header of ``moe_oracle.c`` for the
passages of the pages it follows and the readings it takes where they are
silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# FP8: 1x128 / 128x128 scales; FP8_CHANNEL: per token / per weight row;
# FP8_TENSOR: one scale per activation tensor / per weight row
BF16, FP8, FP8_CHANNEL, FP8_TENSOR = 0, 1, 2, 3
SOFTMAX, SIGMOID = 0, 1
SILU, GELU = 0, 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so (gcc, OpenMP, no FP contraction,
    so that fp32 decisions are the same on x86-64 and aarch64)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.orc_e4m3_value.restype = ctypes.c_double
            lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_route.restype = None
            lib.orc_route.argtypes = [P, P, I, I, I, I, I, I, I, P, P, P]
            lib.orc_count.restype = I
            lib.orc_count.argtypes = [P, I, I, P]
            lib.orc_count_mapped.restype = I
            lib.orc_count_mapped.argtypes = [P, I, I, P, I, P]
            lib.orc_align.restype = None
            lib.orc_align.argtypes = [P, I, I, P, P, P]
            lib.orc_align_mapped.restype = None
            lib.orc_align_mapped.argtypes = [P, I, I, P, I, P, P, P]
            lib.orc_quant_fp8_group_w.restype = None
            lib.orc_quant_fp8_group_w.argtypes = [P, P, I, I, I, P, P]
            lib.orc_moe_forward_ep.restype = None
            lib.orc_moe_forward_ep.argtypes = [P, P, P, I, I, I, I, I, I, I, I, I,
                                               I, I, P, I, I, P, P, P, P, P, I,
                                               P, P, P, I, I, P]
            lib.orc_permute_rows.restype = None
            lib.orc_permute_rows.argtypes = [P, P, I, I, I, P]
            lib.orc_unpermute_reduce.restype = None
            lib.orc_unpermute_reduce.argtypes = [P, P, P, I, I, I, P]
            lib.orc_quant_fp8_group.restype = None
            lib.orc_quant_fp8_group.argtypes = [P, I, I, I, P, P]
            lib.orc_quant_fp8_block.restype = None
            lib.orc_quant_fp8_block.argtypes = [P, I, I, I, P, P]
            lib.orc_quant_fp8_tensor.restype = None
            lib.orc_quant_fp8_tensor.argtypes = [P, P, I, I, P, P]
            lib.orc_quant_fp8_tensor_static.restype = None
            lib.orc_quant_fp8_tensor_static.argtypes = [P, P, I, I, ctypes.c_float, P]
            lib.orc_expert_row.restype = None
            lib.orc_expert_row.argtypes = [I, P, I, I, I, I, I, P, P, P, P, I,
                                           P, P, I]
            lib.orc_moe_forward.restype = None
            lib.orc_moe_forward.argtypes = [P, P, P, I, I, I, I, I, I, I, I, I,
                                            I, I, P, P, P, P, P, I, P, P, P, I]
            lib.orc_batched_experts.restype = I
            lib.orc_batched_experts.argtypes = [P, P, I, I, I, I, I, I, P, P,
                                                P, P, P, I, P, I, I]
            lib.orc_max_threads.restype = I
            lib.orc_max_threads.argtypes = []
            _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    if isinstance(a, ctypes.Array):
        return ctypes.cast(a, ctypes.c_void_p)
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """C-contiguous numpy array of the given dtype (a view when possible)."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        if dtype in (np.uint16, np.uint8) and a.dtype.itemsize == np.dtype(dtype).itemsize:
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def max_threads() -> int:
    return int(_load().orc_max_threads())


def e4m3_value(code: int) -> float:
    return float(_load().orc_e4m3_value(int(code)))


def e4m3_encode(x) -> np.ndarray:
    lib = _load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_e4m3_encode(float(v)) for v in x], dtype=np.uint8)


def route(logits, bias, topk, score_fn, n_groups=1, topk_groups=1,
          renorm=True):
    """[Router]: returns ids (M, topk) int32, weights (M, topk) fp64 and the
    per-token decision margin (fp64; +inf for softmax)."""
    lib = _load()
    logits = _c(logits, np.float32)
    M, E = logits.shape
    bias = _c(bias, np.float32)
    ids = np.empty((M, topk), np.int32)
    w = np.empty((M, topk), np.float64)
    margin = np.empty((M,), np.float64)
    lib.orc_route(_p(logits), _p(bias), M, E, topk, score_fn, n_groups,
                  topk_groups, int(renorm), _p(ids), _p(w), _p(margin))
    return ids, w, margin


def count(ids, E, expert_map=None, E_local=None):
    """Per-(local-)expert counts; returns (counts, number of invalid ids).
    With expert_map (E global ids -> local id or -1), counts has E_local
    entries and pairs of experts that are not local are left out."""
    lib = _load()
    ids = _c(ids, np.int32).ravel()
    El = E if E_local is None else E_local
    counts = np.empty((El,), np.int32)
    m = _c(expert_map, np.int32)
    bad = lib.orc_count_mapped(_p(ids), ids.size, E, _p(m), El, _p(counts))
    return counts, int(bad)


def align(ids, E, expert_map=None, E_local=None):
    """Returns offsets (E_local+1), sorted pair ids (offsets[-1]), inv (P)."""
    lib = _load()
    ids = _c(ids, np.int32).ravel()
    P = ids.size
    El = E if E_local is None else E_local
    offsets = np.empty((El + 1,), np.int32)
    sorted_ids = np.full((P,), -1, np.int32)
    inv = np.empty((P,), np.int32)
    m = _c(expert_map, np.int32)
    lib.orc_align_mapped(_p(ids), P, E, _p(m), El, _p(offsets), _p(sorted_ids), _p(inv))
    return offsets, sorted_ids[: offsets[El]].copy(), inv


def permute_rows(x, sorted_ids, topk):
    lib = _load()
    x = _c(x, np.float64)
    sorted_ids = _c(sorted_ids, np.int32)
    n, K = sorted_ids.size, x.shape[1]
    out = np.empty((n, K), np.float64)
    lib.orc_permute_rows(_p(x), _p(sorted_ids), n, topk, K, _p(out))
    return out


def unpermute_reduce(yperm, inv, w):
    lib = _load()
    yperm = _c(yperm, np.float64)
    w = _c(w, np.float64)
    M, topk = w.shape
    inv = _c(inv, np.int32)
    K = yperm.shape[1]
    out = np.empty((M, K), np.float64)
    lib.orc_unpermute_reduce(_p(yperm), _p(inv), _p(w), M, topk, K, _p(out))
    return out


def quant_fp8_group(x_bf16_bits, group=128, row_weights=None):
    """x (M, K) as uint16 bf16 bits -> q (M, K) uint8 codes, scales (M, K/group).
    row_weights (M) fp32 or None: rows multiplied (in fp32) before quantising."""
    lib = _load()
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, K // group), np.float32)
    rw = _c(row_weights, np.float32)
    lib.orc_quant_fp8_group_w(_p(x), _p(rw), M, K, group, _p(q), _p(s))
    return q, s


def quant_fp8_tensor(x_bf16_bits, row_weights=None, scale=None):
    """x (M, K) bf16 bits -> q (M, K) codes and the one scale of the tensor
    (rows multiplied by row_weights in fp32 first when given).  With `scale`
    (a static activation scale, Q8) the codes use it instead of the
    tensor's maximum (saturating at +-448) and it is returned."""
    lib = _load()
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    rw = _c(row_weights, np.float32)
    if scale is not None:
        lib.orc_quant_fp8_tensor_static(_p(x), _p(rw), M, K, float(np.float32(scale)), _p(q))
        return q, np.float32(scale)
    s = np.empty((1,), np.float32)
    lib.orc_quant_fp8_tensor(_p(x), _p(rw), M, K, _p(q), _p(s))
    return q, s[0]


def quant_fp8_block(w_bf16_bits, block=128):
    """w (R, C) bf16 bits -> q (R, C) codes, scales (R/block, C/block)."""
    lib = _load()
    w = _c(w_bf16_bits, np.uint16)
    R, C = w.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty((R // block, C // block), np.float32)
    lib.orc_quant_fp8_block(_p(w), R, C, block, _p(q), _p(s))
    return q, s


class Weights:
    """Expert weights as the oracle reads them: bf16 bits (dtype BF16), or
    e4m3 codes plus 128 x 128 block scales (dtype FP8), or e4m3 codes plus
    one scale per row (dtypes FP8_CHANNEL and FP8_TENSOR), one block per
    expert.

    Either pass full arrays w1 (E, 2N, K), w2 (E, K, N) [+ w1s (E, 2N/128,
    K/128), w2s (E, K/128, N/128) for FP8; w1s (E, 2N), w2s (E, K) for
    FP8_CHANNEL and FP8_TENSOR], or ``experts={e: (w1e, w2e[, w1se, w2se])}`` with
    ``E, N, K`` for a subset of the experts (the rest are absent; routing a
    computed token to one of them is a caller error)."""

    def __init__(self, dtype, w1=None, w2=None, w1s=None, w2s=None,
                 experts=None, E=None, N=None, K=None, act=SILU):
        self.dtype = dtype
        self.act = act  # the experts' gated activation: SILU or GELU
        bits = np.uint16 if dtype == BF16 else np.uint8
        if experts is None:
            w1 = _c(w1, bits)
            w2 = _c(w2, bits)
            self.E, twoN, self.K = w1.shape
            self.N = twoN // 2
            assert w2.shape == (self.E, self.K, self.N)
            experts = {}
            for e in range(self.E):
                blk = (w1[e], w2[e])
                if dtype != BF16:
                    blk = blk + (_c(w1s, np.float32)[e], _c(w2s, np.float32)[e])
                experts[e] = blk
        else:
            self.E, self.N, self.K = E, N, K
        self.present = sorted(experts)
        self._keep = []
        arrs = [(ctypes.c_void_p * self.E)() for _ in range(4)]
        for e, blk in experts.items():
            blk = list(blk)
            blk[0] = _c(blk[0], bits)
            blk[1] = _c(blk[1], bits)
            assert blk[0].shape == (2 * self.N, self.K), blk[0].shape
            assert blk[1].shape == (self.K, self.N), blk[1].shape
            if dtype != BF16:
                blk[2] = _c(blk[2], np.float32)
                blk[3] = _c(blk[3], np.float32)
            self._keep.append(blk)
            for i, a in enumerate(blk):
                arrs[i][e] = a.ctypes.data
        self.w1, self.w2, self.w1s, self.w2s = arrs
        if dtype == BF16:
            self.w1s = self.w2s = None


def expert_row(x_bf16_bits, t, e, W: Weights, requant_h=False):
    """h (N) and y (K) of expert e on row t of x, fp64."""
    lib = _load()
    x = _c(x_bf16_bits, np.uint16)
    h = np.empty((W.N,), np.float64)
    y = np.empty((W.K,), np.float64)
    lib.orc_expert_row(W.dtype, _p(x), int(t), int(e), W.E, W.N, W.K,
                       _p(W.w1), _p(W.w1s), _p(W.w2), _p(W.w2s),
                       int(requant_h), _p(h), _p(y), int(W.act))
    return h, y


def moe_forward(x_bf16_bits, logits, bias, topk, score_fn, W: Weights,
                n_groups=1, topk_groups=1, renorm=True, requant_h=False,
                tokens=None, nthreads=0, expert_map=None,
                weight_on_input=False, static_scales=None):
    """The layer in the Standard format for the listed tokens (all when None).
    logits (M, E) cover the E routed (global) experts; W holds W.E local
    experts, reached through expert_map (E) when given (-1: not local, the
    pair adds nothing).  weight_on_input: the router weight scales the
    expert's input instead of its output.  static_scales (FP8_TENSOR only):
    (scale of x, scale of H) given instead of the tensors' maxima (Q8).
    Returns out (n, K) fp64, ids (n, topk) int32 (global), weights (n, topk)."""
    lib = _load()
    x = _c(x_bf16_bits, np.uint16)
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    M, K = x.shape
    E = logits.shape[1]
    assert K == W.K
    assert (expert_map is None and E == W.E) or expert_map is not None
    emap = _c(expert_map, np.int32)
    tok = None if tokens is None else _c(np.asarray(tokens), np.int32)
    n = M if tok is None else tok.size
    out = np.empty((n, K), np.float64)
    ids = np.empty((n, topk), np.int32)
    w = np.empty((n, topk), np.float64)
    assert static_scales is None or W.dtype == FP8_TENSOR
    ss = None if static_scales is None else np.asarray(static_scales, np.float32).reshape(2)
    lib.orc_moe_forward_ep(_p(x), _p(logits), _p(bias), M, K, W.N, E, topk,
                           score_fn, n_groups, topk_groups, int(renorm), W.dtype,
                           int(requant_h), _p(emap), W.E, int(weight_on_input),
                           _p(W.w1), _p(W.w1s), _p(W.w2), _p(W.w2s), _p(tok), n,
                           _p(ids), _p(w), _p(out), int(nthreads), int(W.act), _p(ss))
    return out, ids, w


def batched_experts(xb_bf16_bits, counts, W: Weights, rows=None,
                    requant_h=False, nthreads=0, out=None):
    """BatchedExperts format: y_b[e, r] = expert_e(x_b[e, r]) for
    r < min(counts[e], T).  Returns y_b (E, T, K) fp64 holding NaN at the rows
    not computed, and the number of rows computed."""
    lib = _load()
    xb = _c(xb_bf16_bits, np.uint16)
    E, T, K = xb.shape
    counts = _c(counts, np.int32)
    if out is None:
        out = np.full((E, T, K), np.nan, np.float64)
    r = None if rows is None else _c(np.asarray(rows).reshape(-1, 2), np.int32)
    n = lib.orc_batched_experts(_p(xb), _p(counts), E, T, W.N, K, W.dtype,
                                int(requant_h), _p(W.w1), _p(W.w1s), _p(W.w2),
                                _p(W.w2s), _p(r), 0 if r is None else r.shape[0],
                                _p(out), int(nthreads), int(W.act))
    return out, int(n)

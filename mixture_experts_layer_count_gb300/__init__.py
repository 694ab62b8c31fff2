"""Python binding of libgbmoe.so, the GB300 (sm_103a) fused MoE layer.

Argument marshalling only: every function here has the name of a C entry
point of ``include/gbmoe.h``, takes torch tensors (device memory) and plain
ints, passes their pointers and the current CUDA stream through ctypes, and
raises ``GbmoeError`` when the call returns a non-OK status.  All arithmetic
runs in the library's CUDA kernels; there is no fallback path: if the
library cannot be built or loaded, importing this package fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

BF16, FP8_E4M3, FP8_E4M3_CHANNEL, FP8_E4M3_TENSOR = 0, 1, 2, 3  # dtype codes of include/gbmoe.h
SOFTMAX, SIGMOID = 0, 1
ACT_SILU, ACT_GELU = 0, 1
WS_ALIGN, WS_BATCHED, WS_FORWARD, WS_SHARED, WS_EP_DISPATCH = 0, 2, 3, 4, 6
ERR_BAD_EXPERT_ID, ERR_COUNT_RANGE, ERR_TIMEOUT = 0x1, 0x2, 0x4

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported dtype or device",
           3: "CUDA launch error"}

_lock = threading.Lock()
_lib = None


class GbmoeError(RuntimeError):
    def __init__(self, name, status, cuda_error=0):
        msg = f"{name}: {_STATUS.get(status, status)}"
        if status == 3:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)
        self.status = status


# C signatures: (name, restype, argtypes)
_P, _I, _Z, _L = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int64
_SIGS = {
    "gbmoe_status_string": (ctypes.c_char_p, [_I]),
    "gbmoe_last_cuda_error": (_I, []),
    "moe_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_topk_route": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_count_expert_tokens": (_I, [_P, _I, _I, _I, _P, _I, _P, _P, _P]),
    "moe_align_permute": (_I, [_P, _I, _I, _I, _P, _I, _P, _P, _P, _P, _P, _Z, _P, _P]),
    "moe_forward_chunked": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _I, _I, _I, _I, _I, _I,
                                 _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _Z, _P,
                                 _P]),
    "moe_shared_expert_forward": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P, _Z,
                                       _P, _P]),
    "moe_forward_shared": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _I, _I, _I, _I, _I, _I,
                                _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _I, _P, _P, _P,
                                _P, _I, _P, _P, _Z, _P, _P, _P, _P, _P]),
    "moe_align_permute_no_ws": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "gbmoe_selftest_bounded_wait": (_I, [_P, _I, _P]),
    "moe_quant_fp8_group": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_quant_fp8_tensor": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _P]),
    "moe_quant_fp8_tensor_static": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _P]),
    "moe_quant_fp8_row_permute": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _P]),
    "moe_quant_fp8_tensor_permute": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _P]),
    "moe_quant_fp8_block": (_I, [_P, _L, _I, _I, _P, _P, _P]),
    "moe_permute_rows": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_grouped_gemm_gate_up_silu": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P,
                                           _I, _P, _P, _P, _P]),
    "moe_grouped_gemm_gate_up_gelu": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P,
                                           _I, _P, _P, _P, _P]),
    "moe_grouped_gemm_down": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P,
                                   _I, _P, _P, _P]),
    "moe_unpermute_weighted_reduce": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_quant_fp8_group_permute": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _P]),
    "moe_ep_dispatch": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                             _Z, _P, _P]),
    "moe_ep_combine": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "moe_batched_masked_experts": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                        _I, _I, _P, _P, _Z, _P, _P]),
    "moe_forward": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _I, _I, _I, _I, _I, _I,
                         _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P, _P]),
}


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libgbmoe.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if not _build.up_to_date():
                _build.build()
            lib = ctypes.CDLL(_build.LIB)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, st):
    if st != 0:
        raise GbmoeError(name, st, load().gbmoe_last_cuda_error())


def moe_workspace_size(which, M_or_T, E, N, K, topk, dtype) -> int:
    return int(load().moe_workspace_size(which, M_or_T, E, N, K, topk, dtype))


def moe_topk_route(logits, bias, topk, score_fn, n_groups, topk_groups,
                   renormalize, topk_ids, topk_weights, err_word=None,
                   stream=None):
    M, E = logits.shape
    _check("moe_topk_route", load().moe_topk_route(
        _ptr(logits), _ptr(bias), M, E, topk, score_fn, n_groups, topk_groups,
        int(renormalize), _ptr(topk_ids), _ptr(topk_weights), _ptr(err_word),
        _stream(stream)))


def moe_count_expert_tokens(topk_ids, E, counts, err_word=None, stream=None,
                            expert_map=None, E_global=None):
    """counts (E) of the local experts; with expert_map (E_global) the ids are
    global and mapped (-1: not local)."""
    M, topk = topk_ids.shape
    Eg = E if E_global is None else E_global
    _check("moe_count_expert_tokens", load().moe_count_expert_tokens(
        _ptr(topk_ids), M, topk, Eg, _ptr(expert_map), E, _ptr(counts),
        _ptr(err_word), _stream(stream)))


def moe_align_permute(topk_ids, E, counts, offsets, sorted_pair_ids, inv, ws,
                      err_word=None, stream=None, expert_map=None, E_global=None):
    M, topk = topk_ids.shape
    Eg = E if E_global is None else E_global
    _check("moe_align_permute", load().moe_align_permute(
        _ptr(topk_ids), M, topk, Eg, _ptr(expert_map), E, _ptr(counts),
        _ptr(offsets), _ptr(sorted_pair_ids), _ptr(inv), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _ptr(err_word),
        _stream(stream)))


def moe_align_permute_no_ws(topk_ids, E, counts, offsets, sorted_pair_ids, inv,
                            err_word=None, stream=None):
    """moe_align_permute for callers that have no scratch buffer to give:
    the histograms live in a fixed 256 KiB array owned by the library (see
    include/gbmoe.h for the size limit and the rule against overlapping
    calls)."""
    M, topk = topk_ids.shape
    _check("moe_align_permute_no_ws", load().moe_align_permute_no_ws(
        _ptr(topk_ids), M, topk, E, _ptr(counts), _ptr(offsets),
        _ptr(sorted_pair_ids), _ptr(inv), _ptr(err_word), _stream(stream)))


def gbmoe_selftest_bounded_wait(err_word, limit_us, stream=None):
    """Runs the GEMM kernels' bounded pipeline wait on a barrier nothing
    completes: GBMOE_ERR_TIMEOUT lands in err_word after about limit_us."""
    _check("gbmoe_selftest_bounded_wait", load().gbmoe_selftest_bounded_wait(
        _ptr(err_word), int(limit_us), _stream(stream)))


def moe_quant_fp8_group(x, q, scales, group=128, stream=None, row_weights=None):
    M, K = x.shape
    _check("moe_quant_fp8_group", load().moe_quant_fp8_group(
        _ptr(x), _ptr(row_weights), M, K, group, _ptr(q), _ptr(scales),
        _stream(stream)))


def moe_quant_fp8_group_permute(x, inv, topk, A, A_scales, row_weights=None, stream=None):
    """x (M, K) bf16, inv (M*topk) int32 -> A (M*topk, K) e4m3 codes in
    permuted order, A_scales group-major (K/128, ld) fp32."""
    M, K = x.shape
    _check("moe_quant_fp8_group_permute", load().moe_quant_fp8_group_permute(
        _ptr(x), _ptr(row_weights), M, K, _ptr(inv), topk, _ptr(A), _ptr(A_scales),
        _stream(stream)))


def moe_quant_fp8_tensor(x, q, row_scales, amax_ws, n_rows=None, stream=None,
                         row_weights=None):
    """One scale for the whole tensor (rows < *n_rows when n_rows, a device
    int32, is given); row_scales (M) receives it for every such row;
    amax_ws: a 4-byte device buffer."""
    M, K = x.shape
    _check("moe_quant_fp8_tensor", load().moe_quant_fp8_tensor(
        _ptr(x), _ptr(row_weights), M, K, _ptr(n_rows), _ptr(q), _ptr(row_scales),
        _ptr(amax_ws), _stream(stream)))


def moe_quant_fp8_row_permute(x, inv, topk, A, A_scales, row_weights=None, stream=None):
    """One scale per token, quantised and written to the permuted rows in one
    pass: A[inv[p]] gets its token's codes and A_scales[inv[p]] its scale."""
    M, K = x.shape
    _check("moe_quant_fp8_row_permute", load().moe_quant_fp8_row_permute(
        _ptr(x), _ptr(row_weights), M, K, _ptr(inv), topk, _ptr(A), _ptr(A_scales),
        _stream(stream)))


def moe_quant_fp8_tensor_permute(x, inv, topk, A, A_scales, scale=None, amax_ws=None,
                                 row_weights=None, stream=None):
    """One scale for all of x -- the static `scale` (a device fp32), else its
    maximum / 448 (amax_ws: a 4-byte device buffer) -- quantised and written
    to the permuted rows in one pass (A[inv[p]], A_scales[inv[p]])."""
    M, K = x.shape
    _check("moe_quant_fp8_tensor_permute", load().moe_quant_fp8_tensor_permute(
        _ptr(x), _ptr(row_weights), M, K, _ptr(inv), topk, _ptr(scale), _ptr(A),
        _ptr(A_scales), _ptr(amax_ws), _stream(stream)))


def moe_quant_fp8_tensor_static(x, scale, q, row_scales, n_rows=None, stream=None,
                                row_weights=None):
    """The per-tensor quantiser with a static scale (a device fp32 scalar):
    q = e4m3(x / scale) saturating, row_scales (M) = scale for every row
    (rows < *n_rows when n_rows is given)."""
    M, K = x.shape
    _check("moe_quant_fp8_tensor_static", load().moe_quant_fp8_tensor_static(
        _ptr(x), _ptr(row_weights), M, K, _ptr(n_rows), _ptr(scale), _ptr(q), _ptr(row_scales),
        _stream(stream)))


def moe_quant_fp8_block(w, q, scales, block=128, stream=None):
    R = w.numel() // w.shape[-1]
    C = w.shape[-1]
    _check("moe_quant_fp8_block", load().moe_quant_fp8_block(
        _ptr(w), R, C, block, _ptr(q), _ptr(scales), _stream(stream)))


def moe_permute_rows(x, x_scales, sorted_pair_ids, offsets, topk, E, dtype, A,
                     A_scales=None, stream=None, row_weights=None):
    M, K = x.shape
    _check("moe_permute_rows", load().moe_permute_rows(
        _ptr(x), _ptr(x_scales), _ptr(row_weights), _ptr(sorted_pair_ids),
        _ptr(offsets), M, topk, E, K, dtype, _ptr(A), _ptr(A_scales),
        _stream(stream)))


def moe_grouped_gemm_gate_up_silu(A, A_scales, offsets, M, topk, E, N, K, w1,
                                  w1_scales, dtype, H, H_scales, err_word=None,
                                  stream=None):
    _check("moe_grouped_gemm_gate_up_silu", load().moe_grouped_gemm_gate_up_silu(
        _ptr(A), _ptr(A_scales), _ptr(offsets), M, topk, E, N, K, _ptr(w1),
        _ptr(w1_scales), dtype, _ptr(H), _ptr(H_scales), _ptr(err_word),
        _stream(stream)))


def moe_grouped_gemm_gate_up_gelu(A, A_scales, offsets, M, topk, E, N, K, w1,
                                  w1_scales, dtype, H, H_scales, err_word=None,
                                  stream=None):
    _check("moe_grouped_gemm_gate_up_gelu", load().moe_grouped_gemm_gate_up_gelu(
        _ptr(A), _ptr(A_scales), _ptr(offsets), M, topk, E, N, K, _ptr(w1),
        _ptr(w1_scales), dtype, _ptr(H), _ptr(H_scales), _ptr(err_word),
        _stream(stream)))


def moe_grouped_gemm_down(H, H_scales, sorted_pair_ids, offsets, topk_weights,
                          M, topk, E, N, K, w2, w2_scales, dtype, y_slot,
                          err_word=None, stream=None):
    _check("moe_grouped_gemm_down", load().moe_grouped_gemm_down(
        _ptr(H), _ptr(H_scales), _ptr(sorted_pair_ids), _ptr(offsets),
        _ptr(topk_weights), M, topk, E, N, K, _ptr(w2), _ptr(w2_scales), dtype,
        _ptr(y_slot), _ptr(err_word), _stream(stream)))


def moe_ep_dispatch(x, num_tokens, topk_ids, E, worst_tokens, recv_x, recv_counts, recv_pos,
                    ws, err_word=None, stream=None, dtype=BF16, x_scales=None,
                    recv_scales=None):
    """x (G, M, K) bf16, or e4m3 codes with x_scales (G*M, K/128); num_tokens
    (G) int32, topk_ids (G, M, topk) int32; recv_x (E, worst_tokens, K)
    [+ recv_scales (E*worst_tokens, K/128)], recv_counts (E), recv_pos
    (G, M, topk)."""
    G, M, K = x.shape
    topk = topk_ids.shape[-1]
    _check("moe_ep_dispatch", load().moe_ep_dispatch(
        _ptr(x), _ptr(x_scales), _ptr(num_tokens), _ptr(topk_ids), G, M, K, E, topk,
        worst_tokens, dtype, _ptr(recv_x), _ptr(recv_scales), _ptr(recv_counts),
        _ptr(recv_pos), _ptr(ws), ws.numel() * ws.element_size(), _ptr(err_word),
        _stream(stream)))


def moe_ep_combine(recv_y, topk_ids, recv_pos, topk_weights, num_tokens, out, stream=None):
    """recv_y (E, worst_tokens, K); topk_ids / recv_pos / topk_weights
    (G, M, topk); num_tokens (G); out (G, M, K)."""
    E, worst, K = recv_y.shape
    G, M, topk = topk_ids.shape
    _check("moe_ep_combine", load().moe_ep_combine(
        _ptr(recv_y), _ptr(topk_ids), _ptr(recv_pos), _ptr(topk_weights), _ptr(num_tokens),
        G, M, K, E, topk, worst, _ptr(out), _stream(stream)))


def moe_unpermute_weighted_reduce(y_slot, inv, M, topk, K, out, stream=None):
    _check("moe_unpermute_weighted_reduce", load().moe_unpermute_weighted_reduce(
        _ptr(y_slot), _ptr(inv), M, topk, K, _ptr(out), _stream(stream)))


def moe_batched_masked_experts(x_b, expert_num_tokens, N, w1, w2, y_b, ws,
                               dtype=BF16, x_b_scales=None, w1_scales=None,
                               w2_scales=None, err_word=None, stream=None,
                               activation=ACT_SILU):
    E, T, K = x_b.shape
    _check("moe_batched_masked_experts", load().moe_batched_masked_experts(
        _ptr(x_b), _ptr(x_b_scales), _ptr(expert_num_tokens), E, T, N, K,
        _ptr(w1), _ptr(w1_scales), _ptr(w2), _ptr(w2_scales), dtype,
        int(activation), _ptr(y_b),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(err_word),
        _stream(stream)))


def moe_forward(x, logits, bias, N, E, topk, score_fn, n_groups, topk_groups,
                renormalize, dtype, w1, w1_scales, w2, w2_scales, out, ws,
                topk_ids=None, topk_weights=None, err_word=None, stream=None,
                expert_map=None, apply_router_weight_on_input=False,
                activation=ACT_SILU, a1_scale=None, a2_scale=None):
    """The whole Standard layer.  E is the number of local experts (w1.shape[0]);
    the router picks among logits.shape[1] experts, mapped to local ones by
    expert_map when given.  a1_scale / a2_scale: static activation scales
    (device fp32 scalars) for FP8_E4M3_TENSOR, None for the dynamic ones."""
    M, K = x.shape
    E_global = logits.shape[1]
    _check("moe_forward", load().moe_forward(
        _ptr(x), _ptr(logits), _ptr(bias), M, K, N, E_global, _ptr(expert_map), E,
        topk, score_fn, n_groups, topk_groups, int(renormalize),
        int(apply_router_weight_on_input), int(activation), dtype, _ptr(w1),
        _ptr(w1_scales),
        _ptr(w2), _ptr(w2_scales), _ptr(a1_scale), _ptr(a2_scale), _ptr(out), _ptr(topk_ids),
        _ptr(topk_weights),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(err_word),
        _stream(stream)))


def moe_forward_chunked(x, logits, bias, N, E, topk, score_fn, n_groups, topk_groups,
                        renormalize, dtype, w1, w1_scales, w2, w2_scales, out, ws,
                        chunk_size, topk_ids=None, topk_weights=None, err_word=None,
                        stream=None, expert_map=None, apply_router_weight_on_input=False,
                        activation=ACT_SILU, a1_scale=None, a2_scale=None):
    """moe_forward in chunks of chunk_size tokens (ws sized for one chunk)."""
    M, K = x.shape
    E_global = logits.shape[1]
    _check("moe_forward_chunked", load().moe_forward_chunked(
        _ptr(x), _ptr(logits), _ptr(bias), M, K, N, E_global, _ptr(expert_map), E,
        topk, score_fn, n_groups, topk_groups, int(renormalize),
        int(apply_router_weight_on_input), int(activation), dtype, _ptr(w1),
        _ptr(w1_scales), _ptr(w2), _ptr(w2_scales), _ptr(a1_scale), _ptr(a2_scale), _ptr(out),
        _ptr(topk_ids), _ptr(topk_weights), int(chunk_size), _ptr(ws), ws.numel() * ws.element_size(),
        _ptr(err_word), _stream(stream)))


def moe_shared_expert_forward(x, Ns, w1s, w2s, out_shared, ws, dtype=BF16,
                              activation=ACT_SILU, err_word=None, stream=None,
                              w1s_scales=None, w2s_scales=None):
    """The shared experts (dense gated MLP) on every token of x; bf16, or e4m3
    weights with their 128 x 128 block scales (dtype FP8_E4M3)."""
    M, K = x.shape
    _check("moe_shared_expert_forward", load().moe_shared_expert_forward(
        _ptr(x), M, K, Ns, _ptr(w1s), _ptr(w1s_scales), _ptr(w2s), _ptr(w2s_scales), dtype,
        int(activation), _ptr(out_shared), _ptr(ws), ws.numel() * ws.element_size(),
        _ptr(err_word), _stream(stream)))


def _event(ev):
    """Raw cudaEvent_t of a torch.cuda.Event (recorded once if torch has not
    created it yet)."""
    if ev is None:
        return None
    if ev.cuda_event == 0:
        ev.record()
    return ev.cuda_event


def moe_forward_shared(x, logits, bias, N, E, topk, score_fn, n_groups,
                       topk_groups, renormalize, dtype, w1, w1_scales, w2,
                       w2_scales, out, ws, Ns, w1s, w2s, out_shared, ws_shared,
                       aux_stream=None, ev_input_ready=None, ev_output_ready=None,
                       err_word=None, stream=None, expert_map=None,
                       apply_router_weight_on_input=False, activation=ACT_SILU,
                       shared_dtype=BF16, w1s_scales=None, w2s_scales=None, a1_scale=None,
                       a2_scale=None):
    """moe_forward with the shared experts overlapped on aux_stream (a
    torch.cuda.Stream) through two torch.cuda.Event objects; the shared
    experts in shared_dtype (BF16, or FP8_E4M3 with block scales)."""
    M, K = x.shape
    E_global = logits.shape[1]
    _check("moe_forward_shared", load().moe_forward_shared(
        _ptr(x), _ptr(logits), _ptr(bias), M, K, N, E_global, _ptr(expert_map), E,
        topk, score_fn, n_groups, topk_groups, int(renormalize),
        int(apply_router_weight_on_input), int(activation), dtype, _ptr(w1),
        _ptr(w1_scales), _ptr(w2), _ptr(w2_scales), _ptr(a1_scale), _ptr(a2_scale), _ptr(out),
        _ptr(ws),
        ws.numel() * ws.element_size(), Ns, _ptr(w1s), _ptr(w1s_scales), _ptr(w2s),
        _ptr(w2s_scales), int(shared_dtype), _ptr(out_shared),
        _ptr(ws_shared), ws_shared.numel() * ws_shared.element_size(), _ptr(err_word),
        _stream(stream), None if aux_stream is None else aux_stream.cuda_stream,
        _event(ev_input_ready), _event(ev_output_ready)))


def workspace(which, M_or_T, E, N, K, topk, dtype, device="cuda"):
    """A device byte buffer of the size moe_workspace_size asks for."""
    n = moe_workspace_size(which, M_or_T, E, N, K, topk, dtype)
    if n == 0:
        raise GbmoeError("moe_workspace_size", 1)
    return torch.empty(n, dtype=torch.uint8, device=device)

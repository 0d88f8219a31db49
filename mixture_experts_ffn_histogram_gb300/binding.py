"""ctypes binding of libmoe.so: one Python function per C entry point, with the
same name, that only marshals arguments (torch tensors -> device pointers,
dims -> ``moe_dims``, stream -> ``cudaStream_t``) and raises on a non-OK
status.  Every step of the block runs in the library's CUDA kernels; there is
no other implementation behind these functions, and they fail loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_DEVICE = 4
MOE_ERR_TIMEOUT = 5

SCORE_SOFTMAX_TOPK = 0
SCORE_SIGMOID_NORM = 1
SCORE_GIVEN = 2

ENTRY_POINTS = (
    "moe_workspace_bytes", "moe_status_string", "moe_abi_version", "moe_route_histogram",
    "moe_permute", "moe_permute_bwd", "moe_grouped_gemm_fc1_swiglu",
    "moe_grouped_gemm_fc1_swiglu_bwd", "moe_grouped_gemm_fc2", "moe_grouped_gemm_fc2_bwd",
    "moe_combine", "moe_combine_bwd", "moe_selftest_bounded_wait", "moe_route_histogram_noalloc",
    "moe_mx_bytes", "moe_mx_quantize_wi", "moe_mx_quantize_wo", "moe_mx_permute_quantize",
    "moe_mx_grouped_gemm_fc1_swiglu", "moe_mx_grouped_gemm_fc2",
    "moe_grouped_gemm_fc1_swiglu_experts", "moe_grouped_gemm_fc1_bwd_experts",
    "moe_fused_forward", "moe_mx_combine_bwd", "moe_mx_quantize_rows", "moe_mx_quantize_tokens", "moe_mx_grouped_gemm_fc2_bwd",
    "moe_mx_grouped_gemm_fc1_bwd",
)

# moe_mx_buffer
(MX_XQ, MX_XSC, MX_WIQ, MX_WISC, MX_WOQ, MX_WOSC, MX_HQ, MX_HSC, MX_DYQ, MX_DYSC, MX_DZQ,
 MX_DZSC, MX_WIQ_BWD, MX_WISC_BWD, MX_WOQ_BWD, MX_WOSC_BWD, MX_XT, MX_XTSC, MX_HT, MX_HTSC,
 MX_DYT, MX_DYTSC, MX_DZT, MX_DZTSC) = range(24)

# int32 capacity of the fixed scratch behind moe_route_histogram_noalloc
NOALLOC_ROUTE_SCRATCH_INTS = 262144


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("D", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("F", ctypes.c_int32)]

    def __repr__(self):
        return f"MoeDims(T={self.T}, D={self.D}, E={self.E}, K={self.K}, F={self.F})"


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str | None = None):
        super().__init__(f"{fn}: {detail or status_string(status)} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def dims(T, D, E, K, F) -> MoeDims:
    return MoeDims(T, D, E, K, F)


def library_path() -> str:
    return LIB


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB):
            raise RuntimeError(
                f"libmoe.so not found at {LIB}; build it first "
                "(mixture_experts_ffn_histogram_gb300._build.build())")
        L = ctypes.CDLL(LIB)
        P, I, D_ = ctypes.c_void_p, ctypes.c_int, MoeDims
        sig = {
            "moe_workspace_bytes": ([D_], ctypes.c_size_t),
            "moe_status_string": ([I], ctypes.c_char_p),
            "moe_abi_version": ([], I),
            "moe_route_histogram": ([P, P, I, P, P, P, P, P, P, P, P, D_, P], I),
            "moe_permute": ([P, P, P, D_, P], I),
            "moe_permute_bwd": ([P, P, P, D_, P], I),
            "moe_grouped_gemm_fc1_swiglu": ([P, P, P, P, P, P, P, D_, P], I),
            "moe_grouped_gemm_fc1_swiglu_bwd": ([P, P, P, P, P, P, P, P, P, D_, P], I),
            "moe_grouped_gemm_fc2": ([P, P, P, P, P, P, D_, P], I),
            "moe_grouped_gemm_fc2_bwd": ([P, P, P, P, P, P, P, P, P, D_, P], I),
            "moe_combine": ([P, P, P, P, D_, P], I),
            "moe_fused_forward": ([P, P, P, P, P, P, P, P, P, P, P, D_, P], I),
            "moe_combine_bwd": ([P, P, P, P, P, P, D_, P], I),
            "moe_selftest_bounded_wait": ([P, ctypes.c_uint64, P], I),
            "moe_route_histogram_noalloc": ([P, P, I, P, P, P, P, P, P, P, D_, P], I),
            "moe_mx_bytes": ([D_, I], ctypes.c_size_t),
            "moe_grouped_gemm_fc1_swiglu_experts": ([P, P, P, I, I, P, P, P, P, D_, P], I),
            "moe_grouped_gemm_fc1_bwd_experts": ([P, P, P, P, I, I, P, P, P, P, D_, P], I),
            "moe_mx_quantize_wi": ([P, P, P, P, P, D_, P], I),
            "moe_mx_quantize_wo": ([P, P, P, P, P, D_, P], I),
            "moe_mx_permute_quantize": ([P, P, P, P, P, D_, P], I),
            "moe_mx_grouped_gemm_fc1_swiglu": ([P, P, P, P, P, P, P, P, P, P, D_, P], I),
            "moe_mx_grouped_gemm_fc2": ([P, P, P, P, P, P, P, D_, P], I),
            "moe_mx_combine_bwd": ([P] * 9 + [D_, P], I),
            "moe_mx_quantize_rows": ([P, I, P, P, P, D_, P], I),
            "moe_mx_quantize_tokens": ([P, P, I, P, P, P, D_, P], I),
            "moe_mx_grouped_gemm_fc2_bwd": ([P] * 13 + [D_, P], I),
            "moe_mx_grouped_gemm_fc1_bwd": ([P] * 12 + [D_, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ok(name, st):
    if st != MOE_OK:
        raise MoeError(name, st)


def moe_workspace_bytes(d: MoeDims) -> int:
    return int(lib().moe_workspace_bytes(d))


def moe_abi_version() -> int:
    return int(lib().moe_abi_version())


def moe_route_histogram(logits, bias, mode, ids, w, group_sizes, group_offsets, pos, row_src,
                        dev_status, ws, d: MoeDims, stream=None):
    _ok("moe_route_histogram", lib().moe_route_histogram(
        _p(logits), _p(bias), int(mode), _p(ids), _p(w), _p(group_sizes), _p(group_offsets),
        _p(pos), _p(row_src), _p(dev_status), _p(ws), d, _s(stream)))


def moe_route_histogram_noalloc(logits, bias, mode, ids, w, group_sizes, group_offsets, pos,
                                row_src, dev_status, d: MoeDims, stream=None):
    """moe_route_histogram with no workspace: for callers that cannot allocate
    device memory.  Its scratch is a fixed 1 MiB array inside the library,
    shared by every call (calls that overlap on the GPU race on it)."""
    st = lib().moe_route_histogram_noalloc(
        _p(logits), _p(bias), int(mode), _p(ids), _p(w), _p(group_sizes), _p(group_offsets),
        _p(pos), _p(row_src), _p(dev_status), d, _s(stream))
    if st == MOE_ERR_UNSUPPORTED:
        need = 2 * ((d.T + 255) // 256) * d.E
        if need > NOALLOC_ROUTE_SCRATCH_INTS:
            raise MoeError("moe_route_histogram_noalloc", st,
                           f"needs {need} int32 of fixed scratch (2*ceil(T/256)*E) but the "
                           f"library holds {NOALLOC_ROUTE_SCRATCH_INTS}")
    _ok("moe_route_histogram_noalloc", st)


def moe_permute(x, pos, xs, d: MoeDims, stream=None):
    _ok("moe_permute", lib().moe_permute(_p(x), _p(pos), _p(xs), d, _s(stream)))


def moe_permute_bwd(dxs, pos, dx, d: MoeDims, stream=None):
    _ok("moe_permute_bwd", lib().moe_permute_bwd(_p(dxs), _p(pos), _p(dx), d, _s(stream)))


def moe_grouped_gemm_fc1_swiglu(xs, wi, group_offsets, h, z, dev_status, ws, d: MoeDims,
                                stream=None):
    _ok("moe_grouped_gemm_fc1_swiglu", lib().moe_grouped_gemm_fc1_swiglu(
        _p(xs), _p(wi), _p(group_offsets), _p(h), _p(z), _p(dev_status), _p(ws), d, _s(stream)))


def moe_grouped_gemm_fc1_swiglu_bwd(grad, z, xs, wi, group_offsets, dxs, dwi, dev_status, ws,
                                    d: MoeDims, stream=None):
    _ok("moe_grouped_gemm_fc1_swiglu_bwd", lib().moe_grouped_gemm_fc1_swiglu_bwd(
        _p(grad), _p(z), _p(xs), _p(wi), _p(group_offsets), _p(dxs), _p(dwi), _p(dev_status),
        _p(ws), d, _s(stream)))


def moe_grouped_gemm_fc2(h, wo, group_offsets, ys, dev_status, ws, d: MoeDims, stream=None):
    _ok("moe_grouped_gemm_fc2", lib().moe_grouped_gemm_fc2(
        _p(h), _p(wo), _p(group_offsets), _p(ys), _p(dev_status), _p(ws), d, _s(stream)))


def moe_grouped_gemm_fc2_bwd(dys, h, wo, z, group_offsets, dh_or_dz, dwo, dev_status, ws,
                             d: MoeDims, stream=None):
    _ok("moe_grouped_gemm_fc2_bwd", lib().moe_grouped_gemm_fc2_bwd(
        _p(dys), _p(h), _p(wo), _p(z), _p(group_offsets), _p(dh_or_dz), _p(dwo),
        _p(dev_status), _p(ws), d, _s(stream)))


def moe_combine(ys, w, pos, out, d: MoeDims, stream=None):
    _ok("moe_combine", lib().moe_combine(_p(ys), _p(w), _p(pos), _p(out), d, _s(stream)))


def moe_fused_forward(x, w, row_src, group_offsets, wi, wo, h, acc, out, dev_status, ws,
                      d: MoeDims, stream=None):
    _ok("moe_fused_forward", lib().moe_fused_forward(
        _p(x), _p(w), _p(row_src), _p(group_offsets), _p(wi), _p(wo), _p(h), _p(acc), _p(out),
        _p(dev_status), _p(ws), d, _s(stream)))


def moe_combine_bwd(dout, ys, w, pos, dys, dw, d: MoeDims, stream=None):
    _ok("moe_combine_bwd", lib().moe_combine_bwd(
        _p(dout), _p(ys), _p(w), _p(pos), _p(dys), _p(dw), d, _s(stream)))


def moe_selftest_bounded_wait(dev_status, limit_ns: int, stream=None):
    _ok("moe_selftest_bounded_wait",
        lib().moe_selftest_bounded_wait(_p(dev_status), int(limit_ns), _s(stream)))


def moe_grouped_gemm_fc1_swiglu_experts(xs, wi_part, group_offsets, e_begin, e_end, h, z,
                                        dev_status, ws, d: MoeDims, stream=None):
    _ok("moe_grouped_gemm_fc1_swiglu_experts", lib().moe_grouped_gemm_fc1_swiglu_experts(
        _p(xs), _p(wi_part), _p(group_offsets), int(e_begin), int(e_end), _p(h), _p(z),
        _p(dev_status), _p(ws), d, _s(stream)))


def moe_grouped_gemm_fc1_bwd_experts(dz, xs, wi_part, group_offsets, e_begin, e_end, dxs,
                                     dwi_part, dev_status, ws, d: MoeDims, stream=None):
    _ok("moe_grouped_gemm_fc1_bwd_experts", lib().moe_grouped_gemm_fc1_bwd_experts(
        _p(dz), _p(xs), _p(wi_part), _p(group_offsets), int(e_begin), int(e_end), _p(dxs),
        _p(dwi_part), _p(dev_status), _p(ws), d, _s(stream)))


# ------------------------------------------------------------------ MXFP8
def moe_mx_bytes(d: MoeDims, which: int) -> int:
    return int(lib().moe_mx_bytes(d, int(which)))


def moe_mx_quantize_wi(wi, wq, wsc, d: MoeDims, stream=None, wq_bwd=None, wsc_bwd=None):
    _ok("moe_mx_quantize_wi", lib().moe_mx_quantize_wi(_p(wi), _p(wq), _p(wsc), _p(wq_bwd),
                                                       _p(wsc_bwd), d, _s(stream)))


def moe_mx_quantize_wo(wo, wq, wsc, d: MoeDims, stream=None, wq_bwd=None, wsc_bwd=None):
    _ok("moe_mx_quantize_wo", lib().moe_mx_quantize_wo(_p(wo), _p(wq), _p(wsc), _p(wq_bwd),
                                                       _p(wsc_bwd), d, _s(stream)))


def moe_mx_permute_quantize(x, pos, group_offsets, xq, xsc, d: MoeDims, stream=None):
    _ok("moe_mx_permute_quantize", lib().moe_mx_permute_quantize(
        _p(x), _p(pos), _p(group_offsets), _p(xq), _p(xsc), d, _s(stream)))


def moe_mx_grouped_gemm_fc1_swiglu(xq, xsc, wq, wsc, group_offsets, hq, hsc, h, dev_status,
                                   d: MoeDims, stream=None, z=None):
    _ok("moe_mx_grouped_gemm_fc1_swiglu", lib().moe_mx_grouped_gemm_fc1_swiglu(
        _p(xq), _p(xsc), _p(wq), _p(wsc), _p(group_offsets), _p(hq), _p(hsc), _p(h), _p(z),
        _p(dev_status), d, _s(stream)))


def moe_mx_grouped_gemm_fc2(hq, hsc, wq, wsc, group_offsets, ys, dev_status, d: MoeDims,
                            stream=None):
    _ok("moe_mx_grouped_gemm_fc2", lib().moe_mx_grouped_gemm_fc2(
        _p(hq), _p(hsc), _p(wq), _p(wsc), _p(group_offsets), _p(ys), _p(dev_status), d,
        _s(stream)))


def moe_mx_combine_bwd(dout, ys, w, pos, group_offsets, dys, dyq, dysc, dw, d: MoeDims,
                       stream=None):
    _ok("moe_mx_combine_bwd", lib().moe_mx_combine_bwd(
        _p(dout), _p(ys), _p(w), _p(pos), _p(group_offsets), _p(dys), _p(dyq), _p(dysc), _p(dw),
        d, _s(stream)))


def moe_mx_quantize_rows(src, C, group_offsets, q, sc, d: MoeDims, stream=None):
    _ok("moe_mx_quantize_rows", lib().moe_mx_quantize_rows(
        _p(src), int(C), _p(group_offsets), _p(q), _p(sc), d, _s(stream)))


def moe_mx_quantize_tokens(src, row_src, C, group_offsets, qt, sct, d: MoeDims, stream=None):
    _ok("moe_mx_quantize_tokens", lib().moe_mx_quantize_tokens(
        _p(src), _p(row_src), int(C), _p(group_offsets), _p(qt), _p(sct), d, _s(stream)))


def moe_mx_grouped_gemm_fc2_bwd(dyq, dysc, woq, wosc, z, ht, htsc, dyt, dytsc, group_offsets,
                                dz, dwo, dev_status, d: MoeDims, stream=None):
    _ok("moe_mx_grouped_gemm_fc2_bwd", lib().moe_mx_grouped_gemm_fc2_bwd(
        _p(dyq), _p(dysc), _p(woq), _p(wosc), _p(z), _p(ht), _p(htsc), _p(dyt), _p(dytsc),
        _p(group_offsets), _p(dz), _p(dwo), _p(dev_status), d, _s(stream)))


def moe_mx_grouped_gemm_fc1_bwd(dzq, dzsc, wiq, wisc, xt, xtsc, dzt, dztsc, group_offsets, dxs,
                                dwi, dev_status, d: MoeDims, stream=None):
    _ok("moe_mx_grouped_gemm_fc1_bwd", lib().moe_mx_grouped_gemm_fc1_bwd(
        _p(dzq), _p(dzsc), _p(wiq), _p(wisc), _p(xt), _p(xtsc), _p(dzt), _p(dztsc),
        _p(group_offsets), _p(dxs), _p(dwi), _p(dev_status), d, _s(stream)))

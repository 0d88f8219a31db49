"""CPU oracle for the sparse MoE expert block -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA path (the package
``mixture_experts_ffn_histogram_gb300``) never imports it, and the two share
no code: the oracle is ``oracle.c`` compiled with gcc (``-O3 -fopenmp
-ffp-contract=off``), wrapped here with ctypes over numpy arrays.

bf16 tensors cross this boundary as numpy ``uint16`` arrays of raw bit
patterns; see ``oracle.h`` for the definitions each function writes out.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

SOFTMAX_TOPK, SIGMOID_NORM, GIVEN = 0, 1, 2


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``oracle.c`` into a shared library with gcc; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(src),
                                              os.path.getmtime(os.path.join(_HERE, "oracle.h")))):
        return out
    base = ["gcc", "-std=c11", "-O3", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-I", _HERE, src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)   # no OpenMP runtime: 1 thread
    os.replace(out + ".tmp", out)
    return out


def load_library(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    sig = {
        "oracle_f32_to_bf16": ([ctypes.c_float], ctypes.c_uint16),
        "oracle_bf16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
        "oracle_route": ([P, P, I, I, I, I, P, P], I),
        "oracle_histogram": ([P, I, I, I, P, P, P, P], I),
        "oracle_permute": ([P, P, I, I, I, P], I),
        "oracle_fc1_swiglu": ([P, P, P, I, I, I, P, P], I),
        "oracle_fc2": ([P, P, P, I, I, I, P], I),
        "oracle_combine": ([P, P, P, I, I, I, P], I),
        "oracle_combine_bwd": ([P, P, P, P, I, I, I, P, P], I),
        "oracle_fc2_bwd": ([P, P, P, P, P, I, I, I, P, P], I),
        "oracle_swiglu_bwd": ([P, P, I, I, P], I),
        "oracle_fc1_bwd": ([P, P, P, P, I, I, I, P, P], I),
        "oracle_permute_bwd": ([P, P, I, I, I, P], I),
        "oracle_num_threads": ([], I),
        "oracle_e4m3_to_f64": ([ctypes.c_uint8], ctypes.c_double),
        "oracle_f64_to_e4m3": ([ctypes.c_double], ctypes.c_uint8),
        "oracle_mx_quantize": ([P, I, I, P, P], I),
        "oracle_mx_fc1_swiglu": ([P, P, P, P, P, I, I, I, P, P], I),
        "oracle_mx_fc2": ([P, P, P, P, P, I, I, I, P], I),
        "oracle_f32_to_bf16_array": ([P, ctypes.c_long, P], I),
        "oracle_mx_quantize_tokens": ([P, P, I, I, P, P, P], I),
        "oracle_mx_wgrad": ([P, P, P, P, P, P, I, I, I, P], I),
        "oracle_mx_fc2_dgrad_swiglu": ([P, P, P, P, P, P, I, I, I, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily route every wrapper through another build of the oracle
    (used by the test that plants mistakes in copies of ``oracle.c``)."""
    global _lib
    other = load_library(path)
    with _lock:
        old = _lib
        _lib = other
    try:
        yield
    finally:
        with _lock:
            _lib = old


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, name):
    if rc < 0:
        raise ValueError(f"{name}: bad arguments (rc={rc})")
    return rc


# ----------------------------------------------------------------- wrappers
def f32_to_bf16(a) -> np.ndarray:
    """RNE rounding of an fp32 array to bf16 bit patterns (elementwise)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    _check(lib().oracle_f32_to_bf16_array(_p(a), a.size, _p(out)), "f32_to_bf16")
    return out


def bf16_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def route(logits, bias, mode, T, E, K):
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    _check(lib().oracle_route(_p(logits), _p(bias), mode, T, E, K, _p(ids), _p(w)), "route")
    return ids, w


def histogram(ids, E):
    ids = _c(ids, np.int32)
    T, K = ids.shape
    gs = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    pos = np.empty((T, K), np.int32)
    row_src = np.empty(T * K, np.int32)
    bad = _check(lib().oracle_histogram(_p(ids), T, K, E, _p(gs), _p(off), _p(pos), _p(row_src)),
                 "histogram")
    return gs, off, pos, row_src, bad


def permute(x, pos):
    x = _c(x, np.uint16)
    pos = _c(pos, np.int32)
    T, D = x.shape
    K = pos.shape[1]
    xs = np.zeros((T * K, D), np.uint16)
    _check(lib().oracle_permute(_p(x), _p(pos), T, K, D, _p(xs)), "permute")
    return xs


def fc1_swiglu(xs, wi, offs, want_z=True):
    xs = _c(xs, np.uint16)
    wi = _c(wi, np.uint16)
    offs = _c(offs, np.int32)
    E, D, N = wi.shape
    F = N // 2
    R = int(offs[E])
    h = np.zeros((R, F), np.uint16)
    z = np.zeros((R, N), np.uint16) if want_z else None
    _check(lib().oracle_fc1_swiglu(_p(xs), _p(wi), _p(offs), E, D, F, _p(h), _p(z)), "fc1")
    return h, z


def fc2(h, wo, offs):
    h = _c(h, np.uint16)
    wo = _c(wo, np.uint16)
    offs = _c(offs, np.int32)
    E, F, D = wo.shape
    R = int(offs[E])
    ys = np.zeros((R, D), np.uint16)
    _check(lib().oracle_fc2(_p(h), _p(wo), _p(offs), E, F, D, _p(ys)), "fc2")
    return ys


def combine(ys, w, pos, T, D):
    ys = _c(ys, np.uint16)
    w = _c(w, np.float32)
    pos = _c(pos, np.int32)
    K = pos.shape[1]
    out = np.zeros((T, D), np.uint16)
    _check(lib().oracle_combine(_p(ys), _p(w), _p(pos), T, K, D, _p(out)), "combine")
    return out


def combine_bwd(dout, ys, w, pos):
    dout = _c(dout, np.uint16)
    ys = _c(ys, np.uint16)
    w = _c(w, np.float32)
    pos = _c(pos, np.int32)
    T, D = dout.shape
    K = pos.shape[1]
    dys = np.zeros((ys.shape[0], D), np.uint16)
    dw = np.zeros((T, K), np.float32)
    _check(lib().oracle_combine_bwd(_p(dout), _p(ys), _p(w), _p(pos), T, K, D, _p(dys), _p(dw)),
           "combine_bwd")
    return dys, dw


def fc2_bwd(dys, h, wo, z, offs, want_dlhs=True, want_drhs=True):
    dys = _c(dys, np.uint16)
    h = _c(h, np.uint16)
    wo = _c(wo, np.uint16)
    z = _c(z, np.uint16)
    offs = _c(offs, np.int32)
    E, F, D = wo.shape
    R = int(offs[E])
    g = np.zeros((R, 2 * F if z is not None else F), np.uint16) if want_dlhs else None
    dwo = np.zeros((E, F, D), np.uint16) if want_drhs else None
    _check(lib().oracle_fc2_bwd(_p(dys), _p(h), _p(wo), _p(z), _p(offs), E, F, D, _p(g), _p(dwo)),
           "fc2_bwd")
    return g, dwo


def swiglu_bwd(dh, z):
    dh = _c(dh, np.uint16)
    z = _c(z, np.uint16)
    R, F = dh.shape
    dz = np.zeros((R, 2 * F), np.uint16)
    _check(lib().oracle_swiglu_bwd(_p(dh), _p(z), R, F, _p(dz)), "swiglu_bwd")
    return dz


def fc1_bwd(dz, xs, wi, offs, want_dlhs=True, want_drhs=True):
    dz = _c(dz, np.uint16)
    xs = _c(xs, np.uint16)
    wi = _c(wi, np.uint16)
    offs = _c(offs, np.int32)
    E, D, N = wi.shape
    F = N // 2
    R = int(offs[E])
    dxs = np.zeros((R, D), np.uint16) if want_dlhs else None
    dwi = np.zeros((E, D, N), np.uint16) if want_drhs else None
    _check(lib().oracle_fc1_bwd(_p(dz), _p(xs), _p(wi), _p(offs), E, D, F, _p(dxs), _p(dwi)),
           "fc1_bwd")
    return dxs, dwi


def permute_bwd(dxs, pos, T, D):
    dxs = _c(dxs, np.uint16)
    pos = _c(pos, np.int32)
    K = pos.shape[1]
    dx = np.zeros((T, D), np.uint16)
    _check(lib().oracle_permute_bwd(_p(dxs), _p(pos), T, K, D, _p(dx)), "permute_bwd")
    return dx


def num_threads() -> int:
    return int(lib().oracle_num_threads())


# ------------------------------------------------------------------- MXFP8
def e4m3_to_f64(codes) -> np.ndarray:
    """Value of every E4M3 code in ``codes`` (elementwise)."""
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.oracle_e4m3_to_f64(int(v)) for v in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def f64_to_e4m3(values) -> np.ndarray:
    """E4M3 code of every value (nearest, ties to even, saturating)."""
    L = lib()
    v = np.asarray(values, dtype=np.float64)
    return np.array([L.oracle_f64_to_e4m3(float(x)) for x in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


def mx_quantize(x):
    """MXFP8 block quantization of fp32 rows ``x [rows, K]`` along K:
    returns (codes uint8 [rows, K], scales uint8 [rows, K/32])."""
    x = _c(x, np.float32)
    rows, K = x.shape
    q = np.zeros((rows, K), np.uint8)
    sc = np.zeros((rows, K // 32), np.uint8)
    _check(lib().oracle_mx_quantize(_p(x), rows, K, _p(q), _p(sc)), "mx_quantize")
    return q, sc


def mx_dequantize(q, sc) -> np.ndarray:
    """float64 values of MX codes ``q [rows, K]`` with scales ``sc [rows, K/32]``."""
    vals = e4m3_lut()[np.asarray(q, dtype=np.uint8)]
    return vals * np.exp2(np.repeat(np.asarray(sc, np.int64) - 127, 32, axis=-1))


_LUT = None


def e4m3_lut() -> np.ndarray:
    """The oracle's value of each of the 256 E4M3 codes."""
    global _LUT
    if _LUT is None:
        _LUT = e4m3_to_f64(np.arange(256, dtype=np.uint8))
    return _LUT


def mx_fc1_swiglu(xq, xsc, wq, wsc, offs, want_z=False):
    """FC1 + SwiGLU on MX operands (``wq [E, 2F, D]``, wi transposed);
    returns h fp32 [R, F], or (h, z) with z bf16 bits [R, 2F] when
    ``want_z``."""
    xq, xsc = _c(xq, np.uint8), _c(xsc, np.uint8)
    wq, wsc = _c(wq, np.uint8), _c(wsc, np.uint8)
    offs = _c(offs, np.int32)
    E, N, D = wq.shape
    F = N // 2
    R = int(offs[E])
    h = np.zeros((R, F), np.float32)
    z = np.zeros((R, N), np.uint16) if want_z else None
    _check(lib().oracle_mx_fc1_swiglu(_p(xq), _p(xsc), _p(wq), _p(wsc), _p(offs), E, D, F, _p(h),
                                      _p(z)), "mx_fc1")
    return (h, z) if want_z else h


def mx_fc2(hq, hsc, wq, wsc, offs):
    """FC2 on MX operands (``wq [E, D, F]``, wo transposed); returns ys bf16 bits."""
    hq, hsc = _c(hq, np.uint8), _c(hsc, np.uint8)
    wq, wsc = _c(wq, np.uint8), _c(wsc, np.uint8)
    offs = _c(offs, np.int32)
    E, D, F = wq.shape
    R = int(offs[E])
    ys = np.zeros((R, D), np.uint16)
    _check(lib().oracle_mx_fc2(_p(hq), _p(hsc), _p(wq), _p(wsc), _p(offs), E, F, D, _p(ys)),
           "mx_fc2")
    return ys


def mx_weights(wi, wo):
    """MX operands of the expert weights, quantized along each GEMM's
    contraction axis: wi [E, D, 2F] -> (wq [E, 2F, D], wsc [E, 2F, D/32]);
    wo [E, F, D] -> (oq [E, D, F], osc [E, D, F/32])."""
    wi = np.asarray(wi, np.uint16)
    wo = np.asarray(wo, np.uint16)
    E, D, N = wi.shape
    F = wo.shape[1]
    wit = np.ascontiguousarray(bf16_to_f32(wi).transpose(0, 2, 1)).reshape(E * N, D)
    wot = np.ascontiguousarray(bf16_to_f32(wo).transpose(0, 2, 1)).reshape(E * D, F)
    wq, wsc = mx_quantize(wit)
    oq, osc = mx_quantize(wot)
    return (wq.reshape(E, N, D), wsc.reshape(E, N, D // 32),
            oq.reshape(E, D, F), osc.reshape(E, D, F // 32))


def mx_weights_bwd(wi, wo):
    """MX operands of the expert weights for the dgrads, quantized along
    their last axis (the dgrads' contraction axis), in their own layout:
    wi [E, D, 2F] -> (q [E, D, 2F], sc [E, D, 2F/32]); wo [E, F, D] ->
    (q [E, F, D], sc [E, F, D/32])."""
    wi = np.asarray(wi, np.uint16)
    wo = np.asarray(wo, np.uint16)
    E, D, N = wi.shape
    F = wo.shape[1]
    iq, isc = mx_quantize(bf16_to_f32(wi).reshape(E * D, N))
    oq, osc = mx_quantize(bf16_to_f32(wo).reshape(E * F, D))
    return (iq.reshape(E, D, N), isc.reshape(E, D, N // 32),
            oq.reshape(E, F, D), osc.reshape(E, F, D // 32))


def mx_quantize_tokens(x, offs):
    """MX quantization of ``x`` fp32 [R, C] along the tokens of each group
    (blocks of 32 rows from the group's first row): returns (q [R, C],
    sc [NB, C], boff [E+1])."""
    x = _c(x, np.float32)
    offs = _c(offs, np.int32)
    R, C = x.shape
    E = len(offs) - 1
    sizes = np.diff(offs.astype(np.int64))
    NB = int(((sizes + 31) // 32).sum())
    q = np.zeros((R, C), np.uint8)
    sc = np.zeros((NB, C), np.uint8)
    boff = np.zeros(E + 1, np.int32)
    _check(lib().oracle_mx_quantize_tokens(_p(x), _p(offs), E, C, _p(q), _p(sc), _p(boff)),
           "mx_quantize_tokens")
    return q, sc, boff


def mx_dequantize_tokens(q, sc, offs, boff) -> np.ndarray:
    """float64 values of token-quantized codes ``q [R, C]``."""
    offs = np.asarray(offs, np.int64)
    R = int(offs[-1])
    blk = np.zeros(R, np.int64)
    for e in range(len(offs) - 1):
        r = np.arange(offs[e], offs[e + 1])
        blk[r] = boff[e] + (r - offs[e]) // 32
    return e4m3_lut()[np.asarray(q, np.uint8)] * np.exp2(np.asarray(sc, np.int64)[blk] - 127)


def mx_wgrad(a, b, offs):
    """Weight gradient out[e] = A_e^T B_e on token-quantized operands
    ``a = (aq, asc, boff)`` [R, Ca] and ``b`` [R, Cb] (from
    :func:`mx_quantize_tokens` with the same offsets); returns bf16 bits
    [E, Ca, Cb]."""
    aq, asc, boff = _c(a[0], np.uint8), _c(a[1], np.uint8), _c(a[2], np.int32)
    bq, bsc = _c(b[0], np.uint8), _c(b[1], np.uint8)
    offs = _c(offs, np.int32)
    E = len(offs) - 1
    Ca, Cb = aq.shape[1], bq.shape[1]
    out = np.zeros((E, Ca, Cb), np.uint16)
    _check(lib().oracle_mx_wgrad(_p(aq), _p(asc), _p(bq), _p(bsc), _p(offs), _p(boff), E, Ca, Cb,
                                 _p(out)), "mx_wgrad")
    return out


def mx_fc2_dgrad_swiglu(dq, dsc, wq, wsc, z, offs):
    """FC2 dgrad (``wq [E, F, D]``: wo quantized along D) followed by the
    SwiGLU backward at ``z`` bf16 [R, 2F]; returns dz bf16 bits [R, 2F]."""
    dq, dsc = _c(dq, np.uint8), _c(dsc, np.uint8)
    wq, wsc = _c(wq, np.uint8), _c(wsc, np.uint8)
    z, offs = _c(z, np.uint16), _c(offs, np.int32)
    E, F, D = wq.shape
    R = int(offs[E])
    dz = np.zeros((R, 2 * F), np.uint16)
    _check(lib().oracle_mx_fc2_dgrad_swiglu(_p(dq), _p(dsc), _p(wq), _p(wsc), _p(z), _p(offs), E,
                                            D, F, _p(dz)), "mx_fc2_dgrad_swiglu")
    return dz


def mx_block_forward(inp: dict) -> dict:
    """The MXFP8 forward in order: route, histogram, permute + quantize of
    the sorted rows, FC1 + SwiGLU on MX operands, quantize h, FC2 on MX
    operands, combine.  ``inp`` as for :func:`block_forward`."""
    wl = inp["workload"]
    T, D, E, K = wl.T, wl.D, wl.E, wl.K
    if wl.score_mode == GIVEN:
        ids, w = inp["ids"], inp["w"]
    else:
        ids, w = route(inp["logits"], inp["bias"], wl.score_mode, T, E, K)
    gs, off, pos, row_src, bad = histogram(ids, E)
    xs = permute(inp["x"], pos)
    xq, xsc = mx_quantize(bf16_to_f32(xs))
    wq, wsc, oq, osc = mx_weights(inp["wi"], inp["wo"])
    h, z = mx_fc1_swiglu(xq, xsc, wq, wsc, off, want_z=True)
    hq, hsc = mx_quantize(h)
    ys = mx_fc2(hq, hsc, oq, osc, off)
    out = combine(ys, w, pos, T, D)
    return dict(ids=ids, w=w, group_sizes=gs, group_offsets=off, pos=pos, row_src=row_src,
                xs=xs, xq=xq, xsc=xsc, wq=wq, wsc=wsc, oq=oq, osc=osc, h=h, z=z, hq=hq,
                hsc=hsc, ys=ys, out=out)


def mx_block_backward(inp: dict, fwd: dict, wgrad: str = "mx") -> dict:
    """The MXFP8 backward in order, after :func:`mx_block_forward`: combine
    backward (bf16, as in the bf16 block); dys quantized along D and wo along
    D for the FC2 dgrad, whose output passes through the SwiGLU backward;
    dz quantized along 2F and wi along 2F for the FC1 dgrad; permute
    backward; then xs, h (both as the bf16 copies the block keeps), dys and
    dz quantized along the tokens of each group for the two wgrads.

    ``wgrad="bf16"``: the two weight gradients instead take the same bf16
    operands unquantized, dwo = h^T dys and dwi = xs^T dz per expert, as
    :func:`fc2_bwd` and :func:`fc1_bwd` define them (the forward and the
    dgrads unchanged)."""
    if wgrad not in ("mx", "bf16"):
        raise ValueError(f"wgrad must be 'mx' or 'bf16', got {wgrad!r}")
    wl = inp["workload"]
    T, D = wl.T, wl.D
    off = fwd["group_offsets"]
    dys, dw = combine_bwd(inp["dy"], fwd["ys"], fwd["w"], fwd["pos"])
    dq, dsc = mx_quantize(bf16_to_f32(dys))
    iq, isc, oq, osc = mx_weights_bwd(inp["wi"], inp["wo"])
    dz = mx_fc2_dgrad_swiglu(dq, dsc, oq, osc, fwd["z"], off)
    dzq, dzsc = mx_quantize(bf16_to_f32(dz))
    dxs = mx_fc2(dzq, dzsc, iq, isc, off)
    dx = permute_bwd(dxs, fwd["pos"], T, D)
    hb = f32_to_bf16(fwd["h"])
    if wgrad == "bf16":
        _, dwo = fc2_bwd(dys, hb, inp["wo"], None, off, want_dlhs=False)
        _, dwi = fc1_bwd(dz, fwd["xs"], inp["wi"], off, want_dlhs=False)
        return dict(dys=dys, dw=dw, dq=dq, dsc=dsc, wiq_b=iq, wisc_b=isc, woq_b=oq, wosc_b=osc,
                    dz=dz, dzq=dzq, dzsc=dzsc, dxs=dxs, dx=dx, hb=hb, dwo=dwo, dwi=dwi)
    xt = mx_quantize_tokens(bf16_to_f32(fwd["xs"]), off)
    ht = mx_quantize_tokens(bf16_to_f32(hb), off)
    dyt = mx_quantize_tokens(bf16_to_f32(dys), off)
    dzt = mx_quantize_tokens(bf16_to_f32(dz), off)
    dwo = mx_wgrad(ht, dyt, off)
    dwi = mx_wgrad(xt, dzt, off)
    return dict(dys=dys, dw=dw, dq=dq, dsc=dsc, wiq_b=iq, wisc_b=isc, woq_b=oq, wosc_b=osc,
                dz=dz, dzq=dzq, dzsc=dzsc, dxs=dxs, dx=dx, hb=hb, xt=xt, ht=ht, dyt=dyt,
                dzt=dzt, dwo=dwo, dwi=dwi)


# ------------------------------------------------------- whole-block drivers
def block_forward(inp: dict, want_z: bool = True) -> dict:
    """Run the forward steps in order on numpy copies of ``inp`` (a dict from
    ``mixture_experts_ffn_histogram_gb300.inputs.make_inputs`` converted by
    :func:`to_numpy`).  Returns every intermediate."""
    wl = inp["workload"]
    T, D, E, K, F = wl.T, wl.D, wl.E, wl.K, wl.F
    if wl.score_mode == GIVEN:
        ids, w = inp["ids"], inp["w"]
    else:
        ids, w = route(inp["logits"], inp["bias"], wl.score_mode, T, E, K)
    gs, off, pos, row_src, bad = histogram(ids, E)
    xs = permute(inp["x"], pos)
    h, z = fc1_swiglu(xs, inp["wi"], off, want_z=want_z)
    ys = fc2(h, inp["wo"], off)
    out = combine(ys, w, pos, T, D)
    return dict(ids=ids, w=w, group_sizes=gs, group_offsets=off, pos=pos, row_src=row_src,
                bad=bad, xs=xs, h=h, z=z, ys=ys, out=out)


def block_backward(inp: dict, fwd: dict) -> dict:
    """The backward steps in order (fused SwiGLU backward inside FC2's)."""
    wl = inp["workload"]
    T, D = wl.T, wl.D
    dys, dw = combine_bwd(inp["dy"], fwd["ys"], fwd["w"], fwd["pos"])
    dz, dwo = fc2_bwd(dys, fwd["h"], inp["wo"], fwd["z"], fwd["group_offsets"])
    dxs, dwi = fc1_bwd(dz, fwd["xs"], inp["wi"], fwd["group_offsets"])
    dx = permute_bwd(dxs, fwd["pos"], T, D)
    return dict(dys=dys, dw=dw, dz=dz, dwo=dwo, dxs=dxs, dwi=dwi, dx=dx)


def to_numpy(inp: dict) -> dict:
    """Convert the torch tensors of an input dict to numpy (bf16 -> uint16 bits)."""
    import torch
    out = {}
    for k, v in inp.items():
        if isinstance(v, torch.Tensor):
            v = v.detach().contiguous().cpu()
            if v.dtype == torch.bfloat16:
                v = v.view(torch.int16).numpy().view(np.uint16)
            else:
                v = v.numpy()
        out[k] = v
    return out

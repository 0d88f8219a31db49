"""GPU parity of the MXFP8 forward (grouped quantize, block-scaled FC1 +
SwiGLU and FC2) against the CPU oracle.

Bars:
- every quantization the library performs from bf16 inputs is bit-exact:
  the weights' codes and scales, and the permuted tokens' codes and scales;
- FC1's bf16 h and FC2's ys are within |gpu - ref| <= 8e-3 |ref| + 1e-3 rms(ref).
  The products of MX elements are exact and the tensor cores sum them in fp32,
  so the error is the bf16 rounding of the output (<= 2^-8 relative) plus fp32
  summation error (~1e-6 relative);
- FC1's MX codes of h are decided from the kernel's fp32 h.  The oracle
  decides from its float64 h, so the two may differ where h lies within the
  fp32 accumulation bound of a decision boundary (a near-tie of a small
  element in a block of larger ones is the usual case).  The test therefore
  checks validity against that bound (mx_h_bound: D * 2^-24 * sum |x w| for
  gate and up, carried through SwiGLU).  A block's scale may differ only
  where its amax lies within the bound of a power of two, and every code
  must be the nearest E4M3 value, at the scale taken, of a value within the
  bound of the oracle's h;
- the block end to end (route -> quantize -> FC1 -> FC2 -> combine) is within
  2e-2 |ref| + 2e-2 rms(ref) of the oracle's MX forward.
Sizes span several 128-row tiles per group, ragged k-blocks (contraction
lengths that are odd multiples of 64), weight tiles whose second half lies
past the output columns, empty groups and the largest E.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.inputs import custom, make_inputs
from tests import mx_layout as L
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu

CASES = {
    # D = 320, F = 192: both contractions end half-way through a k-block;
    # 2F = 384 leaves FC1's second tile half empty, D = 320 FC2's
    "ragged": custom("mx_ragged", T=300, D=320, E=8, K=2, F=192),
    # ~1000 rows per group: eight 128-row tiles each, one ragged
    "long_groups": custom("mx_long", T=2048, D=256, E=4, K=2, F=128, bias_std=0.5),
    "zipf_given": custom("mx_zipf", T=640, D=384, E=24, K=4, F=320, score_mode=2, zipf_s=1.2),
    # the largest E: hundreds of empty groups, F = 64 (one k-step pair)
    "e_max": custom("mx_emax", T=300, D=128, E=1024, K=8, F=64, bias_std=0.5),
}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.fixture(params=sorted(CASES), scope="module")
def case(request):
    wl = CASES[request.param]
    inp = oracle.to_numpy(make_inputs(wl, "cpu"))
    ref = oracle.mx_block_forward(inp)
    return wl, inp, ref


def _dims(wl):
    return B.dims(wl.T, wl.D, wl.E, wl.K, wl.F)


def _u8(n):
    return torch.empty(int(n), dtype=torch.uint8, device="cuda")


def _sc(n):
    """A scale buffer prefilled with 0xFF (the E8M0 NaN): a GEMM that read a
    scale byte no quantize kernel wrote (tail k-steps, padding rows of partial
    tiles, weight rows past N) would turn its outputs into NaN."""
    return torch.full((int(n),), 0xFF, dtype=torch.uint8, device="cuda")


def _rms(a):
    return float(np.sqrt(np.mean(np.square(a.astype(np.float64))))) if a.size else 0.0


def _close(name, got_bits, want_bits, rtol, arel):
    want = oracle.bf16_to_f32(want_bits)
    assert_close(name, got_bits, want_bits, rtol=rtol, atol=arel * _rms(want))


def test_quantize_weights_exact(case):
    wl, inp, ref = case
    d = _dims(wl)
    E, D, F = wl.E, wl.D, wl.F
    wiq, wisc = _u8(B.moe_mx_bytes(d, B.MX_WIQ)), _sc(B.moe_mx_bytes(d, B.MX_WISC))
    woq, wosc = _u8(B.moe_mx_bytes(d, B.MX_WOQ)), _sc(B.moe_mx_bytes(d, B.MX_WOSC))
    assert wisc.numel() == L.weight_scale_bytes(E, 2 * F, D)
    assert wosc.numel() == L.weight_scale_bytes(E, D, F)
    B.moe_mx_quantize_wi(to_dev(inp["wi"]), wiq, wisc, d)
    B.moe_mx_quantize_wo(to_dev(inp["wo"]), woq, wosc, d)
    torch.cuda.synchronize()
    q, sc = L.unpack_weight(to_host(wiq).reshape(E, 2 * F, D), to_host(wisc), True)
    assert_exact("wi codes", q, ref["wq"])
    assert_exact("wi scales", sc, ref["wsc"])
    q, sc = L.unpack_weight(to_host(woq).reshape(E, D, F), to_host(wosc), False)
    assert_exact("wo codes", q, ref["oq"])
    assert_exact("wo scales", sc, ref["osc"])


def test_permute_quantize_exact(case):
    wl, inp, ref = case
    d = _dims(wl)
    R = wl.T * wl.K
    used = int(ref["group_offsets"][-1])
    xq, xsc = _u8(B.moe_mx_bytes(d, B.MX_XQ)), _sc(B.moe_mx_bytes(d, B.MX_XSC))
    B.moe_mx_permute_quantize(to_dev(inp["x"]), to_dev(ref["pos"]), to_dev(ref["group_offsets"]),
                              xq, xsc, d)
    torch.cuda.synchronize()
    got = to_host(xq).reshape(R, wl.D)[:used]
    assert_exact("xq codes", got, ref["xq"][:used])
    sc = L.unpack_act_scales(to_host(xsc), ref["group_offsets"], wl.D)
    assert_exact("xq scales", sc, ref["xsc"][:used])


def mx_h_bound(xq, xsc, wq, wsc, offs):
    """Bound on |h_kernel - h_oracle| per element: the kernel sums the exact
    products of FC1 in fp32, so its gate and up sums g, u each lie within
    D * 2^-24 * sum_d |x_d w_d| of the exact ones (the worst-case bound of a
    length-D fp32 sum); that moves h = silu(g) u by at most
    |silu'(g) u| dg + |silu(g)| du, plus the fp32 rounding of SwiGLU's own
    operations (4 * 2^-24 |h|)."""
    offs = np.asarray(offs, np.int64)
    E, N, D = wq.shape
    F = N // 2
    x = oracle.mx_dequantize(xq, xsc)
    w = oracle.mx_dequantize(wq.reshape(E * N, D), wsc.reshape(E * N, D // 32)).reshape(E, N, D)
    R = int(offs[-1])
    a = np.zeros((R, N))
    s = np.zeros((R, N))
    for e in range(E):   # one matmul per group
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r1 > r0:
            a[r0:r1] = x[r0:r1] @ w[e].T
            s[r0:r1] = np.abs(x[r0:r1]) @ np.abs(w[e]).T
    g, u = a[:, :F], a[:, F:]
    gamma = D * 2.0 ** -24
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    h = g * sig * u
    return np.abs(dsilu * u) * gamma * s[:, :F] + np.abs(g * sig) * gamma * s[:, F:] + \
        4 * 2.0 ** -24 * np.abs(h)


def _check_mx_codes(name, q, sc, h, offs, hb):
    """The codes of h written by the kernel are a valid quantization of h
    (see the module docstring): each is the nearest E4M3 value, at the
    block's scale, of some value within hb (mx_h_bound) of the oracle's h."""
    used = int(offs[-1])
    q, sc, h = q[:used], sc[:used].astype(np.int64), h[:used].astype(np.float64)
    hb = hb[:used]
    R, F = h.shape
    blocks = h.reshape(R, F // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    _, ex = np.frexp(amax)
    s_ref = np.where(amax == 0, -127, np.maximum(ex - 1 - 8, -127))
    s = sc - 127
    diff = s != s_ref
    # the block's amax may sit on either side of a power of two within hb
    p2 = np.exp2(np.round(np.log2(np.where(amax > 0, amax, 1.0))))
    near_pow2 = np.abs(amax - p2) <= hb.reshape(R, F // 32, 32).max(axis=2) + 1e-7 * amax
    assert not (diff & ~near_pow2).any(), \
        f"{name}: {int((diff & ~near_pow2).sum())} block scales are not floor(log2 amax) - 8"
    scale = np.exp2(np.repeat(s, 32, axis=1).astype(np.float64))
    v = np.abs(h) / scale
    deq = oracle.mx_dequantize(q, sc.astype(np.uint8))
    slack = hb / scale  # the bound in units of the scaled value
    sat = v - slack > 448
    assert np.all(deq[sat] == np.sign(h[sat]) * 448 * scale[sat]), f"{name}: saturation"
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    half_step = 0.5 * np.exp2(e - 3) * scale
    err = np.abs(deq - h)
    near_sat = (v + slack > 448) & ~sat   # within the bound of the saturation edge
    ok = sat | (err <= half_step * (1 + 1e-6) + hb) | (near_sat & (np.abs(deq) == 448 * scale))
    if not ok.all():
        r, c = np.argwhere(~ok)[0]
        b = c // 32
        raise AssertionError(
            f"{name}: {int((~ok).sum())} codes are not the nearest E4M3 value; first at row {r} "
            f"col {c}: h {h[r, c]!r} deq {deq[r, c]!r} code {int(q[r, c]):#04x} scale 2^{int(s[r, b])} "
            f"(oracle 2^{int(s_ref[r, b])}, block amax {amax[r, b]!r}) v {v[r, c]!r}; block h "
            f"{h[r, 32 * b:32 * b + 32].tolist()} codes {q[r, 32 * b:32 * b + 32].tolist()}")
    same = np.mean(q == oracle.mx_quantize(h.astype(np.float32))[0])
    assert same > 0.999, f"{name}: only {same:.4f} of the codes match the oracle's"


def test_fc1_swiglu(case):
    wl, inp, ref = case
    d = _dims(wl)
    R, D, F, E = wl.T * wl.K, wl.D, wl.F, wl.E
    offs = ref["group_offsets"]
    used = int(offs[-1])
    # the oracle's own operands, packed into the library's layouts
    xq = np.zeros((R, D), np.uint8)
    xq[:used] = ref["xq"]
    xsc = L.pack_act_scales(ref["xsc"], offs, B.moe_mx_bytes(d, B.MX_XSC))
    wq, wsc = L.pack_weight(ref["wq"], ref["wsc"], True)
    h = torch.zeros((R, F), dtype=torch.bfloat16, device="cuda")
    hq, hsc = _u8(B.moe_mx_bytes(d, B.MX_HQ)), _sc(B.moe_mx_bytes(d, B.MX_HSC))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_mx_grouped_gemm_fc1_swiglu(to_dev(xq), to_dev(xsc), to_dev(wq), to_dev(wsc),
                                     to_dev(offs), hq, hsc, h, st, d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = oracle.f32_to_bf16(ref["h"]) if used else np.zeros((0, F), np.uint16)
    _close("h", to_host(h)[:used], want, 8e-3, 1e-3)
    q = to_host(hq).reshape(R, F)
    sc = L.unpack_act_scales(to_host(hsc), offs, F)
    hb = mx_h_bound(ref["xq"], ref["xsc"], ref["wq"], ref["wsc"], offs)
    _check_mx_codes("hq", q, sc, ref["h"], offs, hb)


def test_fc2(case):
    wl, inp, ref = case
    d = _dims(wl)
    R, D, F = wl.T * wl.K, wl.D, wl.F
    offs = ref["group_offsets"]
    used = int(offs[-1])
    hq = np.zeros((R, F), np.uint8)
    hq[:used] = ref["hq"]
    hsc = L.pack_act_scales(ref["hsc"], offs, B.moe_mx_bytes(d, B.MX_HSC))
    wq, wsc = L.pack_weight(ref["oq"], ref["osc"], False)
    ys = torch.zeros((R, D), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_mx_grouped_gemm_fc2(to_dev(hq), to_dev(hsc), to_dev(wq), to_dev(wsc), to_dev(offs), ys,
                              st, d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _close("ys", to_host(ys)[:used], ref["ys"], 8e-3, 1e-3)


def mx_forward_gpu(wl, inp, stream=None):
    """The MX forward through the C ABI only: route + histogram, weight and
    token quantization, FC1 (MX h only), FC2, combine."""
    d = _dims(wl)
    T, K, E, D, F = wl.T, wl.K, wl.E, wl.D, wl.F
    R = T * K
    dev = {k: to_dev(v) for k, v in inp.items() if isinstance(v, np.ndarray)}
    ids = dev["ids"] if wl.score_mode == 2 else torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = dev["w"] if wl.score_mode == 2 else torch.empty((T, K), dtype=torch.float32, device="cuda")
    gs = torch.empty(E, dtype=torch.int32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty((T, K), dtype=torch.int32, device="cuda")
    row_src = torch.empty(R, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = _u8(max(B.moe_workspace_bytes(d), 16))
    B.moe_route_histogram(dev.get("logits"), dev.get("bias"), wl.score_mode, ids, w, gs, offs, pos,
                          row_src, st, ws, d)
    wiq, wisc = _u8(B.moe_mx_bytes(d, B.MX_WIQ)), _sc(B.moe_mx_bytes(d, B.MX_WISC))
    woq, wosc = _u8(B.moe_mx_bytes(d, B.MX_WOQ)), _sc(B.moe_mx_bytes(d, B.MX_WOSC))
    B.moe_mx_quantize_wi(dev["wi"], wiq, wisc, d)
    B.moe_mx_quantize_wo(dev["wo"], woq, wosc, d)
    xq, xsc = _u8(B.moe_mx_bytes(d, B.MX_XQ)), _sc(B.moe_mx_bytes(d, B.MX_XSC))
    B.moe_mx_permute_quantize(dev["x"], pos, offs, xq, xsc, d)
    hq, hsc = _u8(B.moe_mx_bytes(d, B.MX_HQ)), _sc(B.moe_mx_bytes(d, B.MX_HSC))
    B.moe_mx_grouped_gemm_fc1_swiglu(xq, xsc, wiq, wisc, offs, hq, hsc, None, st, d)
    ys = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")
    B.moe_mx_grouped_gemm_fc2(hq, hsc, woq, wosc, offs, ys, st, d)
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    B.moe_combine(ys, w, pos, out, d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return to_host(out)


def test_forward_end_to_end(case):
    wl, inp, ref = case
    out = mx_forward_gpu(wl, inp)
    _close("out", out, ref["out"], 2e-2, 2e-2)


def _edge(kind):
    """Small MX edge cases: one token with one slot; a single expert; every
    token routed to one expert of four (given routing)."""
    if kind == "one_row":
        wl = custom("mx_one_row", T=1, D=128, E=4, K=1, F=64)
        return wl, oracle.to_numpy(make_inputs(wl, "cpu"))
    if kind == "e1":
        wl = custom("mx_e1", T=200, D=192, E=1, K=1, F=128)
        return wl, oracle.to_numpy(make_inputs(wl, "cpu"))
    wl = custom("mx_all_to_one", T=300, D=128, E=4, K=1, F=64, score_mode=2)
    inp = oracle.to_numpy(make_inputs(wl, "cpu"))
    inp["ids"] = np.full((300, 1), 2, np.int32)
    inp["w"] = np.ones((300, 1), np.float32)
    return wl, inp


@pytest.mark.parametrize("kind", ["one_row", "e1", "all_to_one"])
def test_edge_cases(kind):
    wl, inp = _edge(kind)
    ref = oracle.mx_block_forward(inp)
    out = mx_forward_gpu(wl, inp)
    _close("out", out, ref["out"], 2e-2, 2e-2)


def test_t0_and_argument_errors():
    d0 = B.dims(0, 128, 4, 2, 64)
    z = _u8(16)
    B.moe_mx_permute_quantize(None, None, None, None, None, d0)
    B.moe_mx_grouped_gemm_fc2(None, None, None, None, None, None, None, d0)
    d = B.dims(8, 128, 4, 2, 64)
    with pytest.raises(B.MoeError) as ei:   # hq without hsc
        B.moe_mx_grouped_gemm_fc1_swiglu(z, z, z, z, z, z, None, None, None, d)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoeError) as ei:   # no output at all
        B.moe_mx_grouped_gemm_fc1_swiglu(z, z, z, z, z, None, None, None, None, d)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoeError) as ei:   # D not a multiple of 64
        B.moe_mx_quantize_wi(z, z, z, B.dims(8, 96, 4, 2, 64))
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
    assert B.moe_mx_bytes(B.dims(8, 96, 4, 2, 64), B.MX_XQ) == 0

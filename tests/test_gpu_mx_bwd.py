"""GPU parity of the MXFP8 backward against the CPU oracle.

The MX block in training (TransformerEngine "[DRAFT][JAX] Optimize MoE
block", Changes item 1): every backward GEMM on MX operands with blocks along
its own contraction axis -- the dgrads take the gradient rows and the weights
quantized along their last axis, the wgrads take both operands quantized
along the tokens of each group (32-row blocks from the group's first row).

Bars:
- every quantization from bf16 inputs is bit-exact (codes and scales): the
  weights along their last axis, dys and dz along their rows, and xs (read
  straight from x through row_src), h, dys and dz along tokens, whose
  padding columns must hold zero codes and the 32-token steps of padding
  only the scale of a zero block (byte 0);
- each GEMM on the oracle's own operands, packed into the library's
  layouts: |gpu - ref| <= 8e-3 |ref| + 1e-3 rms(ref).  Products of MX
  elements are exact and the tensor cores sum them in fp32, so the error is
  the bf16 rounding of the output (<= 2^-8 relative) plus the fp32 sums;
  the FC2 dgrad's SwiGLU backward adds a few fp32 roundings of its own;
- the block end to end (forward and backward through MoEBlockMX) within
  2e-2 |ref| + 2e-2 rms(ref) of the oracle's MX forward and backward: there
  the kernel's fp32 h and z are rounded and quantized where the oracle's
  float64 ones are, so a code may differ by one step where a value lies at
  a rounding boundary.
Output buffers are filled with NaN first, so an element no kernel writes
fails.  Cases: groups that span several 128-row tiles with ragged ends,
contraction and output lengths that are odd multiples of 64, given Zipf
routing with empty experts, E = 1024 with mostly empty experts, one token,
and T = 0.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.block import MoEBlockMX
from mixture_experts_ffn_histogram_gb300.inputs import custom, make_inputs
from tests import mx_layout as L
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu

CASES = {
    # D = 320, F = 192: contractions end half-way through a k-block; dwo's
    # rows (F = 192) end half-way through a 128-row tile
    "ragged": custom("mxb_ragged", T=300, D=320, E=8, K=2, F=192),
    # ~1000 rows per group: eight token tiles per group in the wgrads
    "long_groups": custom("mxb_long", T=2048, D=256, E=4, K=2, F=128, bias_std=0.5),
    "zipf_given": custom("mxb_zipf", T=640, D=384, E=24, K=4, F=320, score_mode=2, zipf_s=1.2),
    "e_max": custom("mxb_emax", T=300, D=128, E=1024, K=8, F=64, bias_std=0.5),
    "one_token": custom("mxb_one", T=1, D=128, E=4, K=1, F=64),
}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.fixture(params=sorted(CASES), scope="module")
def case(request):
    wl = CASES[request.param]
    inp = oracle.to_numpy(make_inputs(wl, "cpu", with_grad=True))
    ref = oracle.mx_block_forward(inp)
    refb = oracle.mx_block_backward(inp, ref)
    return wl, inp, ref, refb


def _dims(wl):
    return B.dims(wl.T, wl.D, wl.E, wl.K, wl.F)


def _u8(n):
    return torch.empty(int(n), dtype=torch.uint8, device="cuda")


def _sc(n):
    """Scale buffer prefilled with 0xFF (the E8M0 NaN), so that a scale no
    kernel wrote turns the GEMM's outputs into NaN."""
    return torch.full((int(n),), 0xFF, dtype=torch.uint8, device="cuda")


def _nan_bf16(shape):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")


def _rms(a):
    return float(np.sqrt(np.mean(np.square(a.astype(np.float64))))) if a.size else 0.0


def _close(name, got_bits, want_bits, rtol, arel):
    want = oracle.bf16_to_f32(want_bits)
    assert_close(name, got_bits, want_bits, rtol=rtol, atol=arel * _rms(want))


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ----------------------------------------------------------- quantization
def test_quantize_weights_bwd_exact(case):
    wl, inp, ref, refb = case
    d = _dims(wl)
    E, D, F = wl.E, wl.D, wl.F
    iq, isc = _u8(B.moe_mx_bytes(d, B.MX_WIQ_BWD)), _sc(B.moe_mx_bytes(d, B.MX_WISC_BWD))
    oq, osc = _u8(B.moe_mx_bytes(d, B.MX_WOQ_BWD)), _sc(B.moe_mx_bytes(d, B.MX_WOSC_BWD))
    assert isc.numel() == L.weight_scale_bytes(E, D, 2 * F)
    assert osc.numel() == L.weight_scale_bytes(E, F, D)
    # the dgrad copies alone, then both copies from one read: the same bytes
    B.moe_mx_quantize_wi(to_dev(inp["wi"]), None, None, d, wq_bwd=iq, wsc_bwd=isc)
    B.moe_mx_quantize_wo(to_dev(inp["wo"]), None, None, d, wq_bwd=oq, wsc_bwd=osc)
    torch.cuda.synchronize()
    fq, fsc = _u8(B.moe_mx_bytes(d, B.MX_WIQ)), _sc(B.moe_mx_bytes(d, B.MX_WISC))
    iq2, isc2 = _u8(iq.numel()), _sc(isc.numel())
    B.moe_mx_quantize_wi(to_dev(inp["wi"]), fq, fsc, d, wq_bwd=iq2, wsc_bwd=isc2)
    torch.cuda.synchronize()
    assert torch.equal(iq, iq2) and torch.equal(isc, isc2)
    q, sc = L.unpack_weight(to_host(fq).reshape(E, 2 * F, D), to_host(fsc), True)
    assert_exact("wi codes (along D, with the dgrad copy)", q, ref["wq"])
    assert_exact("wi scales (along D, with the dgrad copy)", sc, ref["wsc"])
    q, sc = L.unpack_weight(to_host(iq).reshape(E, D, 2 * F), to_host(isc), False)
    assert_exact("wi codes (along 2F)", q, refb["wiq_b"])
    assert_exact("wi scales (along 2F)", sc, refb["wisc_b"])
    q, sc = L.unpack_weight(to_host(oq).reshape(E, F, D), to_host(osc), False)
    assert_exact("wo codes (along D)", q, refb["woq_b"])
    assert_exact("wo scales (along D)", sc, refb["wosc_b"])


def test_quantize_rows_exact(case):
    wl, inp, ref, refb = case
    d = _dims(wl)
    R, D, F = wl.T * wl.K, wl.D, wl.F
    offs = ref["group_offsets"]
    used = int(offs[-1])
    for name, src, C, wq, wsc, which in (("dys", refb["dys"], D, refb["dq"], refb["dsc"], B.MX_DYQ),
                                         ("dz", refb["dz"], 2 * F, refb["dzq"], refb["dzsc"],
                                          B.MX_DZQ)):
        q, sc = _u8(B.moe_mx_bytes(d, which)), _sc(B.moe_mx_bytes(d, which + 1))
        B.moe_mx_quantize_rows(to_dev(src), C, to_dev(offs), q, sc, d)
        torch.cuda.synchronize()
        assert_exact(f"{name} row codes", to_host(q).reshape(R, C)[:used], wq[:used])
        assert_exact(f"{name} row scales", L.unpack_act_scales(to_host(sc), offs, C), wsc[:used])


def test_combine_bwd_quantize_exact(case):
    """moe_mx_combine_bwd on the oracle's ys: dys bit-exact (as
    moe_combine_bwd), its MX codes and scales along D bit-exact, dw within
    the tolerance."""
    wl, inp, ref, refb = case
    d = _dims(wl)
    R, D = wl.T * wl.K, wl.D
    offs = ref["group_offsets"]
    used = int(offs[-1])
    ys = np.zeros((R, D), np.uint16)
    ys[:used] = ref["ys"]
    dys = _nan_bf16((R, D))
    dw = torch.full((wl.T, wl.K), float("nan"), dtype=torch.float32, device="cuda")
    q, sc = _u8(B.moe_mx_bytes(d, B.MX_DYQ)), _sc(B.moe_mx_bytes(d, B.MX_DYSC))
    B.moe_mx_combine_bwd(to_dev(inp["dy"]), to_dev(ys), to_dev(ref["w"]), to_dev(ref["pos"]),
                         to_dev(offs), dys, q, sc, dw, d)
    torch.cuda.synchronize()
    assert_exact("dys", to_host(dys)[:used], refb["dys"])
    assert_exact("dys codes along D", to_host(q).reshape(R, D)[:used], refb["dq"][:used])
    assert_exact("dys scales along D", L.unpack_act_scales(to_host(sc), offs, D), refb["dsc"][:used])
    assert_close("dw", to_host(dw), refb["dw"], bf16=False, atol=2e-2 * _rms(refb["dw"]))


def test_quantize_tokens_exact(case):
    wl, inp, ref, refb = case
    d = _dims(wl)
    R, D, F = wl.T * wl.K, wl.D, wl.F
    offs = ref["group_offsets"]
    x, row_src = to_dev(inp["x"]), to_dev(ref["row_src"])
    cases = (("xs (gathered from x)", x, row_src, D, refb["xt"], B.MX_XT),
             ("h", to_dev(refb["hb"]), None, F, refb["ht"], B.MX_HT),
             ("dys", to_dev(refb["dys"]), None, D, refb["dyt"], B.MX_DYT),
             ("dz", to_dev(refb["dz"]), None, 2 * F, refb["dzt"], B.MX_DZT))
    for name, src, rs, C, want, which in cases:
        qt = torch.full((int(B.moe_mx_bytes(d, which)),), 0xAB, dtype=torch.uint8, device="cuda")
        sct = _sc(B.moe_mx_bytes(d, which + 1))
        assert qt.numel() == C * L.token_cols(R, wl.E)
        assert sct.numel() == L.token_scale_bytes(R, wl.E, C)
        B.moe_mx_quantize_tokens(src, rs, C, to_dev(offs), qt, sct, d)
        torch.cuda.synchronize()
        q, sc, pad, pad_sc = L.unpack_tokens(to_host(qt).reshape(C, -1), to_host(sct), offs)
        assert_exact(f"{name} token codes", q, want[0])
        assert_exact(f"{name} token scales", sc, want[1])
        assert not pad.any(), f"{name}: padding token columns must hold zero codes"
        assert not pad_sc.any(), f"{name}: steps of padding only must have scale byte 0"


# ------------------------------------------------ GEMMs on oracle operands
def _pack_rows(q, sc, offs, R, nbytes):
    full = np.zeros((R, q.shape[1]), np.uint8)
    full[: q.shape[0]] = q
    return to_dev(full), to_dev(L.pack_act_scales(sc, offs, nbytes))


def test_fc2_dgrad_swiglu(case):
    wl, inp, ref, refb = case
    d = _dims(wl)
    R, F = wl.T * wl.K, wl.F
    offs = ref["group_offsets"]
    used = int(offs[-1])
    dq, dsc = _pack_rows(refb["dq"], refb["dsc"], offs, R, B.moe_mx_bytes(d, B.MX_DYSC))
    wq, wsc = L.pack_weight(refb["woq_b"], refb["wosc_b"], False)
    z = np.zeros((R, 2 * F), np.uint16)
    z[:used] = ref["z"]
    dz = _nan_bf16((R, 2 * F))
    st = _status()
    B.moe_mx_grouped_gemm_fc2_bwd(dq, dsc, to_dev(wq), to_dev(wsc), to_dev(z), None, None, None,
                                  None, to_dev(offs), dz, None, st, d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _close("dz", to_host(dz)[:used], refb["dz"], 8e-3, 1e-3)


def test_fc1_dgrad(case):
    wl, inp, ref, refb = case
    d = _dims(wl)
    R, D = wl.T * wl.K, wl.D
    offs = ref["group_offsets"]
    used = int(offs[-1])
    zq, zsc = _pack_rows(refb["dzq"], refb["dzsc"], offs, R, B.moe_mx_bytes(d, B.MX_DZSC))
    wq, wsc = L.pack_weight(refb["wiq_b"], refb["wisc_b"], False)
    dxs = _nan_bf16((R, D))
    st = _status()
    B.moe_mx_grouped_gemm_fc1_bwd(zq, zsc, to_dev(wq), to_dev(wsc), None, None, None, None,
                                  to_dev(offs), dxs, None, st, d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _close("dxs", to_host(dxs)[:used], refb["dxs"], 8e-3, 1e-3)


def test_wgrads(case):
    wl, inp, ref, refb = case
    d = _dims(wl)
    R, E, D, F = wl.T * wl.K, wl.E, wl.D, wl.F
    offs = ref["group_offsets"]

    def pack(t):
        codes, buf = L.pack_tokens(t[0], t[1], offs, R, E)
        return to_dev(codes), to_dev(buf)

    ht, htsc = pack(refb["ht"])
    dyt, dytsc = pack(refb["dyt"])
    xt, xtsc = pack(refb["xt"])
    dzt, dztsc = pack(refb["dzt"])
    dwo, dwi = _nan_bf16((E, F, D)), _nan_bf16((E, D, 2 * F))
    st = _status()
    B.moe_mx_grouped_gemm_fc2_bwd(None, None, None, None, None, ht, htsc, dyt, dytsc,
                                  to_dev(offs), None, dwo, st, d)
    B.moe_mx_grouped_gemm_fc1_bwd(None, None, None, None, xt, xtsc, dzt, dztsc, to_dev(offs),
                                  None, dwi, st, d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _close("dwo", to_host(dwo), refb["dwo"], 8e-3, 1e-3)
    _close("dwi", to_host(dwi), refb["dwi"], 8e-3, 1e-3)
    empty = np.flatnonzero(np.diff(offs) == 0)
    if empty.size:
        assert not to_host(dwo)[empty].any() and not to_host(dwi)[empty].any()


# ------------------------------------------------------------ end to end
def _mx_train_step(wl, inp, wgrad="mx"):
    """Forward and backward through MoEBlockMX (the C ABI only)."""
    blk = MoEBlockMX(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=True, wgrad=wgrad)
    for t in (blk.dx, blk.dwi, blk.dwo, blk.dz, blk.dys, blk.out):
        t.fill_(float("nan"))
    blk.dw.fill_(float("nan"))
    g = {k: to_dev(v) for k, v in inp.items() if isinstance(v, np.ndarray)}
    blk.set_weights(g["wi"], g["wo"])
    blk.forward(g["x"], logits=g.get("logits"), bias=g.get("bias"), ids=g.get("ids"),
                w=g.get("w"))
    blk.backward(g["dy"])
    torch.cuda.synchronize()
    assert int(blk.status.item()) == 0
    return blk


def test_train_step_end_to_end(case):
    wl, inp, ref, refb = case
    blk = _mx_train_step(wl, inp)
    used = int(ref["group_offsets"][-1])
    assert_exact("group offsets", to_host(blk.group_offsets), ref["group_offsets"])
    _close("out", to_host(blk.out), ref["out"], 2e-2, 2e-2)
    _close("dys", to_host(blk.dys)[:used], refb["dys"], 2e-2, 2e-2)
    assert_close("dw", to_host(blk.dw), refb["dw"], bf16=False,
                 atol=2e-2 * _rms(refb["dw"].astype(np.float64)))
    _close("dz", to_host(blk.dz)[:used], refb["dz"], 2e-2, 2e-2)
    _close("dx", to_host(blk.dx), refb["dx"], 2e-2, 2e-2)
    _close("dwo", to_host(blk.dwo), refb["dwo"], 2e-2, 2e-2)
    _close("dwi", to_host(blk.dwi), refb["dwi"], 2e-2, 2e-2)


def test_train_step_bf16_wgrad(case):
    """The MX block with bf16 weight gradients (wgrad="bf16"): the forward
    and the dgrads are the same launches on the same inputs, so out, dys,
    dz and dx equal the all-MX step's bit for bit; dwo = h^T dys and dwi =
    xs^T dz on the bf16 grouped GEMM, against the oracle's bf16 products of
    its own MX-path operands (end-to-end bar)."""
    wl, inp, ref, refb = case
    refw = oracle.mx_block_backward(inp, ref, wgrad="bf16")
    mx = _mx_train_step(wl, inp)
    blk = _mx_train_step(wl, inp, wgrad="bf16")
    used = int(ref["group_offsets"][-1])
    for name in ("out", "dx", "dw"):
        assert_exact(name, to_host(getattr(blk, name)), to_host(getattr(mx, name)))
    for name in ("dys", "dz"):
        assert_exact(name, to_host(getattr(blk, name))[:used], to_host(getattr(mx, name))[:used])
    assert_exact("xs", to_host(blk.xs)[:used], ref["xs"])
    _close("dwo", to_host(blk.dwo), refw["dwo"], 2e-2, 2e-2)
    _close("dwi", to_host(blk.dwi), refw["dwi"], 2e-2, 2e-2)
    empty = np.flatnonzero(np.diff(ref["group_offsets"]) == 0)
    if empty.size:
        assert not to_host(blk.dwo)[empty].any() and not to_host(blk.dwi)[empty].any()


def test_all_tokens_to_one_expert():
    """Given routing of every token to expert 2 of 4: three experts get zero
    weight gradients, one gets a single group of 300 rows."""
    wl = custom("mxb_all_to_one", T=300, D=128, E=4, K=1, F=64, score_mode=2)
    inp = oracle.to_numpy(make_inputs(wl, "cpu", with_grad=True))
    inp["ids"] = np.full((300, 1), 2, np.int32)
    inp["w"] = np.ones((300, 1), np.float32)
    ref = oracle.mx_block_forward(inp)
    refb = oracle.mx_block_backward(inp, ref)
    blk = _mx_train_step(wl, inp)
    _close("dx", to_host(blk.dx), refb["dx"], 2e-2, 2e-2)
    dwi, dwo = to_host(blk.dwi), to_host(blk.dwo)
    _close("dwi", dwi, refb["dwi"], 2e-2, 2e-2)
    _close("dwo", dwo, refb["dwo"], 2e-2, 2e-2)
    assert not dwi[[0, 1, 3]].any() and not dwo[[0, 1, 3]].any()


def test_t0_and_argument_errors():
    d0 = B.dims(0, 128, 4, 2, 64)
    dwo = _nan_bf16((4, 64, 128))
    dwi = _nan_bf16((4, 128, 128))
    # no tokens: the weight gradients are zeros, nothing else is touched
    B.moe_mx_grouped_gemm_fc2_bwd(None, None, None, None, None, None, None, None, None, None,
                                  None, dwo, None, d0)
    B.moe_mx_grouped_gemm_fc1_bwd(None, None, None, None, None, None, None, None, None, None,
                                  dwi, None, d0)
    B.moe_mx_quantize_rows(None, 128, None, None, None, d0)
    B.moe_mx_quantize_tokens(None, None, 128, None, None, None, d0)
    torch.cuda.synchronize()
    assert not to_host(dwo).any() and not to_host(dwi).any()
    d = B.dims(8, 128, 4, 2, 64)
    z = _u8(16)
    with pytest.raises(B.MoeError) as ei:   # neither output
        B.moe_mx_grouped_gemm_fc2_bwd(z, z, z, z, z, z, z, z, z, z, None, None, None, d)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoeError) as ei:   # C is none of D, F, 2F
        B.moe_mx_quantize_tokens(z, None, 192, z, z, z, d)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoeError) as ei:   # rows: C must be D or 2F
        B.moe_mx_quantize_rows(z, 64, z, z, z, d)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoeError) as ei:   # neither copy of the weight
        B.moe_mx_quantize_wi(z, None, None, d)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoeError) as ei:   # codes without scales
        B.moe_mx_quantize_wo(z, z, None, d)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(RuntimeError):
        MoEBlockMX(8, 128, 4, 2, 64).backward(None)

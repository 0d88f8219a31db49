"""GPU parity of FC1 over expert ranges (the split-expert wi layout: wi held
as separate expert-range buffers, FC1 as chained grouped GEMM calls into one
output buffer).

For a split of [0, E) into ranges whose weights are separate tensors, the
chained calls must reproduce the whole-wi call bit for bit: h, z, dxs and
each range's slice of dwi.  Each output row or weight tile is computed by the
same kernel with the same reduction order either way; MOE_GEMM_PAIR pins the
tile path, so that both calls run the same one.  The results are also checked
against the oracle (2e-2 rel + 2e-2 abs).  Rows outside a call's range must
stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.inputs import custom, make_inputs
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu

CASES = {
    # uneven split, ragged N and K tails, 2-3 tiles per group
    "ragged": (custom("split_ragged", T=300, D=320, E=8, K=2, F=192, train=True), [0, 3, 8]),
    # skewed given routing with empty experts, split in three
    "zipf": (custom("split_zipf", T=640, D=256, E=24, K=4, F=256, score_mode=2, zipf_s=1.2,
                    train=True), [0, 5, 6, 24]),
}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.fixture(params=sorted(CASES), scope="module")
def case(request):
    wl, cuts = CASES[request.param]
    inp = oracle.to_numpy(make_inputs(wl, "cpu", with_grad=True))
    fwd = oracle.block_forward(inp)
    dys, _ = oracle.combine_bwd(inp["dy"], fwd["ys"], fwd["w"], fwd["pos"])
    dz, _ = oracle.fc2_bwd(dys, fwd["h"], inp["wo"], fwd["z"], fwd["group_offsets"],
                           want_drhs=False)
    dxs, dwi = oracle.fc1_bwd(dz, fwd["xs"], inp["wi"], fwd["group_offsets"])
    return wl, cuts, inp, fwd, dz, dxs, dwi


@pytest.mark.parametrize("pair", ["0", "1"], ids=["cta1", "cta2"])
def test_fc1_split_matches_whole(case, pair, monkeypatch):
    monkeypatch.setenv("MOE_GEMM_PAIR", pair)
    wl, cuts, inp, fwd, dz_ref, dxs_ref, dwi_ref = case
    d = B.dims(wl.T, wl.D, wl.E, wl.K, wl.F)
    R, D, F = wl.T * wl.K, wl.D, wl.F
    xs, wi, offs, dz = to_dev(fwd["xs"]), to_dev(inp["wi"]), to_dev(fwd["group_offsets"]), to_dev(dz_ref)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(B.moe_workspace_bytes(d), 256), dtype=torch.uint8, device="cuda")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    # the whole wi in one call
    h_w, z_w = torch.zeros((R, F), **bf), torch.zeros((R, 2 * F), **bf)
    B.moe_grouped_gemm_fc1_swiglu(xs, wi, offs, h_w, z_w, st, ws, d)
    dxs_w, dwi_w = torch.zeros((R, D), **bf), torch.zeros((wl.E, D, 2 * F), **bf)
    B.moe_grouped_gemm_fc1_swiglu_bwd(dz, None, xs, wi, offs, dxs_w, dwi_w, st, ws, d)
    # the same from separate expert-range buffers, chained into one h / z / dxs
    sentinel = -7.0
    h_s, z_s = torch.full((R, F), sentinel, **bf), torch.full((R, 2 * F), sentinel, **bf)
    dxs_s = torch.full((R, D), sentinel, **bf)
    parts = []
    used = int(fwd["group_offsets"][-1])
    for e0, e1 in zip(cuts[:-1], cuts[1:]):
        wi_part = wi[e0:e1].clone()          # a buffer of its own
        dwi_part = torch.full((e1 - e0, D, 2 * F), sentinel, **bf)
        B.moe_grouped_gemm_fc1_swiglu_experts(xs, wi_part, offs, e0, e1, h_s, z_s, st, ws, d)
        B.moe_grouped_gemm_fc1_bwd_experts(dz, xs, wi_part, offs, e0, e1, dxs_s, dwi_part, st, ws, d)
        parts.append(dwi_part)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for name, a, b in (("h", h_s, h_w), ("z", z_s, z_w), ("dxs", dxs_s, dxs_w)):
        assert_exact(name, to_host(a)[:used], to_host(b)[:used])
        if used < R:   # rows past the last group are never written
            assert torch.all(a[used:] == sentinel)
    assert_exact("dwi", to_host(torch.cat(parts)), to_host(dwi_w))
    # and against the oracle
    assert_close("h", to_host(h_s)[:used], fwd["h"])
    assert_close("dxs", to_host(dxs_s)[:used], dxs_ref)
    assert_close("dwi", to_host(torch.cat(parts)), dwi_ref)


def test_range_arguments():
    d = B.dims(8, 128, 4, 2, 64)
    z = torch.zeros(64, dtype=torch.uint8, device="cuda")
    for e0, e1 in ((-1, 2), (2, 2), (3, 2), (0, 5)):
        with pytest.raises(B.MoeError) as ei:
            B.moe_grouped_gemm_fc1_swiglu_experts(z, z, z, e0, e1, z, None, None, None, d)
        assert ei.value.status == B.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("pair", ["0", "1"], ids=["cta1", "cta2"])
def test_block_with_split_wi(case, pair, monkeypatch):
    """MoEBlock given wi as a list of expert-range tensors: the forward and
    backward equal those with the whole wi bit for bit; dwi_parts are the
    whole dwi's slices.  (A range call picks its tile path from all R rows
    over its own experts, so the path is pinned for the comparison.)"""
    monkeypatch.setenv("MOE_GEMM_PAIR", pair)
    from mixture_experts_ffn_histogram_gb300.block import MoEBlock
    wl, cuts, inp, *_ = case
    g = {k: to_dev(v) for k, v in inp.items() if isinstance(v, np.ndarray)}
    kw = dict(logits=g.get("logits"), bias=g.get("bias"), ids=g.get("ids"), w=g.get("w"))
    whole = MoEBlock(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=True)
    whole.forward(g["x"], g["wi"], g["wo"], **kw)
    whole.backward(g["dy"], g["wi"], g["wo"])
    split = MoEBlock(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=True)
    parts = [g["wi"][e0:e1].clone() for e0, e1 in zip(cuts[:-1], cuts[1:])]
    split.forward(g["x"], parts, g["wo"], **kw)
    split.backward(g["dy"], parts, g["wo"])
    torch.cuda.synchronize()
    assert int(split.status.item()) == 0
    for name in ("out", "dx", "dwo", "dw"):
        assert_exact(name, to_host(getattr(split, name)), to_host(getattr(whole, name)))
    assert_exact("dwi", to_host(torch.cat(split.dwi_parts)), to_host(whole.dwi))

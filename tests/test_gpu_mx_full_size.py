"""GPU parity of the MXFP8 forward at full size, in the configuration
bench.py times (MoEBlockMX on the whole workload).

Every check recomputes its expected values with the oracle from the original
inputs (sliced into sub-problems), never from GPU outputs:
  * the quantized weights of the largest, the smallest and a random expert,
    codes and scales, bit-exact;
  * the permuted-and-quantized rows of sampled sorted-order rows (edge rows
    of those experts included), codes and scales, bit-exact;
  * FC1's MX h on those rows: a valid MX quantization of the oracle's h
    (the check of tests/test_gpu_mx.py);
  * ys on those rows and out on sampled tokens: within 2e-2 |ref| +
    2e-2 rms(ref) of the oracle's MX forward of the sub-problem.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.block import MoEBlockMX
from mixture_experts_ffn_histogram_gb300.inputs import WORKLOADS, make_inputs
from tests import mx_layout as L
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_host
from tests.test_gpu_mx import _check_mx_codes, _rms, mx_h_bound

pytestmark = pytest.mark.gpu

FULL = ["token_sweep_T8192", "long_seq_train"]


@pytest.fixture(scope="module", params=FULL)
def run(request):
    need_gpu()
    wl = WORKLOADS[request.param]
    inp = make_inputs(wl, torch.device("cuda"), with_grad=False)
    blk = MoEBlockMX(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode)
    blk.set_weights(inp["wi"], inp["wo"])
    blk.forward(inp["x"], logits=inp["logits"], bias=inp["bias"], ids=inp["ids"], w=inp["w"])
    torch.cuda.synchronize()
    assert int(blk.status.item()) == 0
    if wl.score_mode == B.SCORE_GIVEN:
        ids_ref, w_ref = to_host(inp["ids"]), to_host(inp["w"])
    else:
        ids_ref, w_ref = oracle.route(to_host(inp["logits"]),
                                      None if inp["bias"] is None else to_host(inp["bias"]),
                                      wl.score_mode, wl.T, wl.E, wl.K)
    gs, off, pos, row_src, bad = oracle.histogram(ids_ref, wl.E)
    assert bad == 0
    assert_exact("group_offsets", to_host(blk.group_offsets), off)
    rng = np.random.Generator(np.random.PCG64(21))
    sizes = np.diff(off)
    experts = sorted({int(np.argmax(sizes)), int(np.argmin(np.where(sizes > 0, sizes, 1 << 30))),
                      int(rng.integers(0, wl.E))})
    yield dict(wl=wl, inp=inp, blk=blk, w=w_ref, off=off, pos=pos, row_src=row_src,
               experts=experts, rng=rng)
    del blk, inp
    torch.cuda.empty_cache()


def _quantized_expert(inp, e, F):
    """The oracle's MX operands of expert e: (wq [2F,D], wsc, oq [D,F], osc)."""
    wi_e = oracle.bf16_to_f32(to_host(inp["wi"][e]))      # [D, 2F]
    wo_e = oracle.bf16_to_f32(to_host(inp["wo"][e]))      # [F, D]
    wq, wsc = oracle.mx_quantize(np.ascontiguousarray(wi_e.T))
    oq, osc = oracle.mx_quantize(np.ascontiguousarray(wo_e.T))
    return wq, wsc, oq, osc


def test_quantized_weights_of_sampled_experts(run):
    wl, blk = run["wl"], run["blk"]
    E, D, F = wl.E, wl.D, wl.F
    wiq = to_host(blk.wiq)[:E * 2 * F * D].reshape(E, 2 * F, D)
    woq = to_host(blk.woq)[:E * D * F].reshape(E, D, F)
    wisc, wosc = to_host(blk.wisc), to_host(blk.wosc)
    for e in run["experts"]:
        wq, wsc, oq, osc = _quantized_expert(run["inp"], e, F)
        q, sc = L.unpack_weight_expert(wiq[e], wisc, e, 2 * F, D, True)
        assert_exact(f"wi codes e={e}", q, wq)
        assert_exact(f"wi scales e={e}", sc, wsc)
        q, sc = L.unpack_weight_expert(woq[e], wosc, e, D, F, False)
        assert_exact(f"wo codes e={e}", q, oq)
        assert_exact(f"wo scales e={e}", sc, osc)


def _sampled_rows(run):
    off, rng, R = run["off"], run["rng"], run["wl"].R
    rows = set(int(r) for r in rng.integers(0, R, 12))
    for e in run["experts"]:
        if off[e + 1] > off[e]:
            rows |= {int(off[e]), int(off[e]) + 127, int(off[e + 1] - 1)}
    return np.array(sorted(r for r in rows if r < off[-1]))


def test_forward_on_sampled_rows_and_tokens(run):
    wl, inp, blk = run["wl"], run["inp"], run["blk"]
    D, F, K = wl.D, wl.F, wl.K
    off = run["off"]
    # sampled rows, plus every row of a few sampled tokens (for out)
    tok = np.sort(run["rng"].choice(wl.T, size=4, replace=False))
    rows = np.union1d(_sampled_rows(run), run["pos"][tok].ravel())
    experts = np.searchsorted(off, rows, side="right") - 1
    uniq = np.unique(experts)
    sub_e = np.searchsorted(uniq, experts)
    order = np.lexsort((rows, sub_e))
    rows, sub_e = rows[order], sub_e[order]
    sub_off = np.concatenate([[0], np.cumsum(np.bincount(sub_e, minlength=len(uniq)))]).astype(np.int32)
    tokens = run["row_src"][rows] // K
    x = oracle.bf16_to_f32(to_host(inp["x"][torch.from_numpy(tokens).long().cuda()]))
    xq, xsc = oracle.mx_quantize(x)
    ops = [_quantized_expert(inp, int(e), F) for e in uniq]
    wq = np.stack([o[0] for o in ops]); wsc = np.stack([o[1] for o in ops])
    oq = np.stack([o[2] for o in ops]); osc = np.stack([o[3] for o in ops])
    h = oracle.mx_fc1_swiglu(xq, xsc, wq, wsc, sub_off)
    hq, hsc = oracle.mx_quantize(h)
    ys = oracle.mx_fc2(hq, hsc, oq, osc, sub_off)
    ri = torch.from_numpy(rows).long().cuda()
    # the permute + quantize, bit-exact
    assert_exact("xq rows", to_host(blk.xq.view(wl.R, D)[ri]), xq)
    xsc_buf = to_host(blk.xsc)
    assert_exact("xq scales", xsc_buf[L.act_scale_index_rows(off, rows, D)], xsc)
    # FC1's MX h: a valid quantization of the oracle's h
    hq_gpu = to_host(blk.hq.view(wl.R, F)[ri])
    hsc_gpu = to_host(blk.hsc)[L.act_scale_index_rows(off, rows, F)]
    hb = mx_h_bound(xq, xsc, wq, wsc, sub_off)
    _check_mx_codes("hq", hq_gpu, hsc_gpu, h, np.array([0, len(rows)]), hb)
    # ys and out
    want = oracle.bf16_to_f32(ys)
    assert_close("ys", to_host(blk.ys[ri]), ys, rtol=2e-2, atol=2e-2 * _rms(want))
    where = {int(r): i for i, r in enumerate(rows)}
    pos_sub = np.array([[where[int(r)] for r in run["pos"][t]] for t in tok], np.int32)
    out_ref = oracle.combine(ys, run["w"][tok], pos_sub, len(tok), D)
    want = oracle.bf16_to_f32(out_ref)
    ti = torch.from_numpy(tok).long().cuda()
    assert_close("out", to_host(blk.out[ti]), out_ref, rtol=2e-2, atol=2e-2 * _rms(want))

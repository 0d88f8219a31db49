"""GPU parity of the MXFP8 training step at full size, in the configuration
bench.py times (MoEBlockMX with train=True on long_seq_train: the weights
quantized with their dgrad copies, the MX forward, the MX backward).

Every output buffer is filled with NaN first and must come back finite.
Expected values are recomputed by the oracle from the original inputs,
sliced into sub-problems, never from GPU outputs:
  * sampled tokens (all their slots; with the tokens of the first, 128th
    and last rows of the largest, the smallest and a random expert): the
    MX forward and backward of the sub-problem they form -- dys, dw, dz,
    dxs, dx -- within 2e-2 |ref| + 2e-2 rms(ref);
  * the weight gradients of those experts on their whole groups: a few full
    rows f of dwo and full columns n of dwi.  Both token-axis quantizations
    and the MX FC1 are per column, so the oracle needs only FC1's columns
    f and F + f, wo's row f of the dgrad copy and xs, dys of the group.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.block import MoEBlockMX
from mixture_experts_ffn_histogram_gb300.inputs import WORKLOADS, make_inputs
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_host

pytestmark = pytest.mark.gpu


def _rms(a):
    a = np.asarray(a, np.float64)
    return float(np.sqrt(np.mean(np.square(a)))) if a.size else 0.0


def _close_bits(name, got_bits, want_bits):
    want = oracle.bf16_to_f32(want_bits)
    assert_close(name, got_bits, want_bits, rtol=2e-2, atol=2e-2 * _rms(want))


def _dev_rows(t, idx):
    return to_host(t[torch.from_numpy(np.asarray(idx)).long().cuda()])


@pytest.fixture(scope="module")
def run():
    need_gpu()
    wl = WORKLOADS["long_seq_train"]
    inp = make_inputs(wl, torch.device("cuda"), with_grad=True)
    blk = MoEBlockMX(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=True)
    for t in (blk.out, blk.ys, blk.h, blk.z, blk.dys, blk.dz, blk.dxs, blk.dx, blk.dwi, blk.dwo):
        t.fill_(float("nan"))
    blk.dw.fill_(float("nan"))
    blk.set_weights(inp["wi"], inp["wo"])
    blk.forward(inp["x"], logits=inp["logits"], bias=inp["bias"])
    blk.backward(inp["dy"])
    torch.cuda.synchronize()
    assert int(blk.status.item()) == 0
    ids_ref, w_ref = oracle.route(to_host(inp["logits"]), to_host(inp["bias"]), wl.score_mode,
                                  wl.T, wl.E, wl.K)
    gs, off, pos, row_src, bad = oracle.histogram(ids_ref, wl.E)
    assert bad == 0
    assert_exact("group_offsets", to_host(blk.group_offsets), off)
    rng = np.random.Generator(np.random.PCG64(23))
    sizes = np.diff(off)
    experts = sorted({int(np.argmax(sizes)), int(np.argmin(np.where(sizes > 0, sizes, 1 << 30))),
                      int(rng.integers(0, wl.E))})
    yield dict(wl=wl, inp=inp, blk=blk, w=w_ref, off=off, pos=pos, row_src=row_src,
               experts=experts, rng=rng)
    del blk, inp
    torch.cuda.empty_cache()


def test_every_output_written(run):
    blk, wl = run["blk"], run["wl"]
    R = int(run["off"][-1])
    for name, t in (("out", blk.out), ("dx", blk.dx), ("dw", blk.dw), ("dwi", blk.dwi),
                    ("dwo", blk.dwo), ("dys", blk.dys[:R]), ("dz", blk.dz[:R]),
                    ("dxs", blk.dxs[:R]), ("h", blk.h[:R]), ("z", blk.z[:R])):
        assert bool(torch.isfinite(t).all()), f"{name}: elements left unwritten (NaN) or not finite"


def _sub_problem(run, tok):
    """The sampled tokens as a block of their own: given routing over the
    experts they use (renumbered in order), those experts' weights."""
    from types import SimpleNamespace
    wl, inp = run["wl"], run["inp"]
    ids_ref = oracle.route(to_host(inp["logits"][torch.from_numpy(tok).long().cuda()]),
                           to_host(inp["bias"]), wl.score_mode, len(tok), wl.E, wl.K)[0]
    uniq = np.unique(ids_ref)
    ui = torch.from_numpy(uniq).long().cuda()
    ti = torch.from_numpy(tok).long().cuda()
    sub = SimpleNamespace(T=len(tok), D=wl.D, E=len(uniq), K=wl.K, F=wl.F, score_mode=oracle.GIVEN)
    return dict(workload=sub, x=to_host(inp["x"][ti]), wi=to_host(inp["wi"][ui]),
                wo=to_host(inp["wo"][ui]), dy=to_host(inp["dy"][ti]),
                ids=np.searchsorted(uniq, ids_ref).astype(np.int32), w=run["w"][tok],
                logits=None, bias=None), uniq


def test_forward_and_backward_on_sampled_tokens(run):
    wl, blk, off, pos, row_src = run["wl"], run["blk"], run["off"], run["pos"], run["row_src"]
    K = wl.K
    tok = set(int(t) for t in run["rng"].choice(wl.T, size=4, replace=False))
    for e in run["experts"]:
        for r in (off[e], off[e] + 127, off[e + 1] - 1):
            if off[e] <= r < off[e + 1]:
                tok.add(int(row_src[r]) // K)
    tok = np.array(sorted(tok))
    inp_sub, _ = _sub_problem(run, tok)
    f = oracle.mx_block_forward(inp_sub)
    g = oracle.mx_block_backward(inp_sub, f)
    # sub row -> the full block's row of the same (token, slot)
    rs = f["row_src"]
    grow = pos[tok[rs // K], rs % K]
    _close_bits("out (sampled tokens)", _dev_rows(blk.out, tok), f["out"])
    _close_bits("dys", _dev_rows(blk.dys, grow), g["dys"])
    _close_bits("dz", _dev_rows(blk.dz, grow), g["dz"])
    _close_bits("dxs", _dev_rows(blk.dxs, grow), g["dxs"])
    _close_bits("dx (sampled tokens)", _dev_rows(blk.dx, tok), g["dx"])
    assert_close("dw (sampled tokens)", _dev_rows(blk.dw, tok), g["dw"], bf16=False,
                 atol=2e-2 * _rms(g["dw"]))


def test_weight_gradients_of_sampled_experts(run):
    """dwo[e][f, :] and dwi[e][:, n] for a few f (n = f and F + f) of the
    largest, the smallest and a random expert, on the expert's whole group."""
    wl, inp, blk, off, row_src = run["wl"], run["inp"], run["blk"], run["off"], run["row_src"]
    D, F, K = wl.D, wl.F, wl.K
    dy_all = inp["dy"]
    for e in run["experts"]:
        n = int(off[e + 1] - off[e])
        if n == 0:
            continue
        j = row_src[off[e]:off[e + 1]]
        t, k = j // K, j % K
        ti = torch.from_numpy(t).long().cuda()
        sel = np.array(sorted({0, F - 1, int(run["rng"].integers(0, F))}))
        m = len(sel)
        g1 = [0, n]
        # xs and dys of the group's rows (dys = bf16(w * dy), the combine
        # backward with one slot per row)
        xs = to_host(inp["x"][ti])
        dys, _ = oracle.combine_bwd(to_host(dy_all[ti]), np.zeros((n, D), np.uint16),
                                    run["w"][t, k][:, None], np.arange(n, dtype=np.int32)[:, None])
        # FC1 columns f and F + f only: wi's MX codes are per output column
        wi_e = oracle.bf16_to_f32(to_host(inp["wi"][e]))          # [D, 2F]
        cols = np.concatenate([sel, F + sel])
        wq, wsc = oracle.mx_quantize(np.ascontiguousarray(wi_e[:, cols].T))
        xq, xsc = oracle.mx_quantize(oracle.bf16_to_f32(xs))
        h, z = oracle.mx_fc1_swiglu(xq, xsc, wq.reshape(1, 2 * m, D), wsc.reshape(1, 2 * m, -1),
                                    np.array(g1, np.int32), want_z=True)
        # dwo rows f: h (bf16) and dys along the group's tokens
        ht = oracle.mx_quantize_tokens(oracle.bf16_to_f32(oracle.f32_to_bf16(h)), g1)
        dyt = oracle.mx_quantize_tokens(oracle.bf16_to_f32(dys), g1)
        want = oracle.mx_wgrad(ht, dyt, g1)[0]                     # [m, D]
        got = to_host(blk.dwo[e][torch.from_numpy(sel).long().cuda()])
        _close_bits(f"dwo[{e}] rows {sel.tolist()}", got, want)
        # dwi columns f, F + f: dz of those columns from wo's rows f (dgrad
        # copy, blocks along D) and z, then xs and dz along tokens
        wo_e = oracle.bf16_to_f32(to_host(inp["wo"][e]))          # [F, D]
        oq, osc = oracle.mx_quantize(np.ascontiguousarray(wo_e[sel]))
        dq, dsc = oracle.mx_quantize(oracle.bf16_to_f32(dys))
        dz = oracle.mx_fc2_dgrad_swiglu(dq, dsc, oq.reshape(1, m, D), osc.reshape(1, m, -1), z,
                                        np.array(g1, np.int32))      # [n, 2m]
        xt = oracle.mx_quantize_tokens(oracle.bf16_to_f32(xs), g1)
        dzt = oracle.mx_quantize_tokens(oracle.bf16_to_f32(dz), g1)
        want = oracle.mx_wgrad(xt, dzt, g1)[0]                     # [D, 2m]
        got = to_host(blk.dwi[e][:, torch.from_numpy(cols).long().cuda()])
        _close_bits(f"dwi[{e}] columns {cols.tolist()}", got, want)


@pytest.fixture(scope="module")
def run_bw():
    """The same step with the weight gradients on the bf16 GEMM
    (MoEBlockMX(wgrad="bf16"), as bench.py's mxfp8_train_bf16_wgrad)."""
    need_gpu()
    wl = WORKLOADS["long_seq_train"]
    inp = make_inputs(wl, torch.device("cuda"), with_grad=True)
    blk = MoEBlockMX(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=True, wgrad="bf16")
    for t in (blk.out, blk.h, blk.z, blk.dys, blk.dz, blk.dxs, blk.dx, blk.dwi, blk.dwo, blk.xs):
        t.fill_(float("nan"))
    blk.set_weights(inp["wi"], inp["wo"])
    blk.forward(inp["x"], logits=inp["logits"], bias=inp["bias"])
    blk.backward(inp["dy"])
    torch.cuda.synchronize()
    assert int(blk.status.item()) == 0
    ids_ref, w_ref = oracle.route(to_host(inp["logits"]), to_host(inp["bias"]), wl.score_mode,
                                  wl.T, wl.E, wl.K)
    gs, off, pos, row_src, bad = oracle.histogram(ids_ref, wl.E)
    rng = np.random.Generator(np.random.PCG64(29))
    sizes = np.diff(off)
    experts = sorted({int(np.argmax(sizes)), int(np.argmin(np.where(sizes > 0, sizes, 1 << 30))),
                      int(rng.integers(0, wl.E))})
    yield dict(wl=wl, inp=inp, blk=blk, w=w_ref, off=off, row_src=row_src, experts=experts,
               rng=rng)
    del blk, inp
    torch.cuda.empty_cache()


def test_bf16_weight_gradients_of_sampled_experts(run_bw):
    """With bf16 weight gradients: every output written; dwo[e][f, :] =
    h_f^T dys and dwi[e][:, n] = xs^T dz_n for a few f (n = f, F + f) of the
    largest, the smallest and a random expert on their whole groups, with
    h, dys and dz of those columns recomputed by the oracle's MX forward and
    dgrad, the products by its bf16 fc2_bwd / fc1_bwd."""
    wl, inp, blk, off, row_src = (run_bw[k] for k in ("wl", "inp", "blk", "off", "row_src"))
    D, F, K = wl.D, wl.F, wl.K
    R = int(off[-1])
    for name, t in (("dwi", blk.dwi), ("dwo", blk.dwo), ("dx", blk.dx), ("xs", blk.xs[:R])):
        assert bool(torch.isfinite(t).all()), f"{name}: elements left unwritten (NaN) or not finite"
    for e in run_bw["experts"]:
        n = int(off[e + 1] - off[e])
        if n == 0:
            continue
        j = row_src[off[e]:off[e + 1]]
        t, k = j // K, j % K
        ti = torch.from_numpy(t).long().cuda()
        sel = np.array(sorted({0, F - 1, int(run_bw["rng"].integers(0, F))}))
        m = len(sel)
        g1 = np.array([0, n], np.int32)
        xs = to_host(inp["x"][ti])
        dys, _ = oracle.combine_bwd(to_host(inp["dy"][ti]), np.zeros((n, D), np.uint16),
                                    run_bw["w"][t, k][:, None],
                                    np.arange(n, dtype=np.int32)[:, None])
        wi_e = oracle.bf16_to_f32(to_host(inp["wi"][e]))          # [D, 2F]
        cols = np.concatenate([sel, F + sel])
        wq, wsc = oracle.mx_quantize(np.ascontiguousarray(wi_e[:, cols].T))
        xq, xsc = oracle.mx_quantize(oracle.bf16_to_f32(xs))
        h, z = oracle.mx_fc1_swiglu(xq, xsc, wq.reshape(1, 2 * m, D), wsc.reshape(1, 2 * m, -1),
                                    g1, want_z=True)
        hb = oracle.f32_to_bf16(h)                                 # [n, m]
        wo_sub = to_host(inp["wo"][e][torch.from_numpy(sel).long().cuda()])[None]  # [1, m, D]
        _, want = oracle.fc2_bwd(dys, hb, wo_sub, None, g1, want_dlhs=False)
        got = to_host(blk.dwo[e][torch.from_numpy(sel).long().cuda()])
        _close_bits(f"dwo[{e}] rows {sel.tolist()} (bf16)", got, want[0])
        wo_e = oracle.bf16_to_f32(to_host(inp["wo"][e]))          # [F, D]
        oq, osc = oracle.mx_quantize(np.ascontiguousarray(wo_e[sel]))
        dq, dsc = oracle.mx_quantize(oracle.bf16_to_f32(dys))
        dz = oracle.mx_fc2_dgrad_swiglu(dq, dsc, oq.reshape(1, m, D), osc.reshape(1, m, -1), z,
                                        g1)                         # [n, 2m]
        wi_sub = np.ascontiguousarray(to_host(inp["wi"][e])[:, cols])[None]        # [1, D, 2m]
        _, want = oracle.fc1_bwd(dz, xs, wi_sub, g1, want_dlhs=False)
        got = to_host(blk.dwi[e][:, torch.from_numpy(cols).long().cuda()])
        _close_bits(f"dwi[{e}] columns {cols.tolist()} (bf16)", got, want[0])

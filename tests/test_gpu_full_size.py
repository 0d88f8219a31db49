"""GPU parity at the workloads' full sizes, in the configuration bench.py times.

The block runs whole on the GPU (MoEBlock, the default GEMM path choice).
Checks:
  * routing ids, group sizes/offsets, pos and row_src against the oracle,
    whole and bit-exact; routing weights within tolerance;
  * the permutation by its definition at full size (xs == x[row_src // K],
    exact);
  * FC1 (h, z), FC2 (ys), combine (out) and every backward (dys, dw, dz,
    dxs, dx) on sampled rows and tokens: the oracle recomputes each sampled
    item from the original inputs (slices of x, wi, wo, dy and the oracle's
    own routing), never from GPU outputs;
  * dwi and dwo on sampled entries of the largest, the smallest and a random
    expert, each a sum over all of the expert's rows computed by the oracle.
Floats: |gpu - ref| <= 2e-2*|ref| + 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.block import MoEBlock
from mixture_experts_ffn_histogram_gb300.inputs import WORKLOADS, make_inputs
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu

FULL = ["token_sweep_T1024", "token_sweep_T8192", "long_seq_train", "large_expert_train",
        "zipf_skew_train"]


def _bits(t):
    return to_host(t)


def _sub_problem(rows, row_src, off, K, E):
    """Sampled sorted-order rows -> (rows sorted by expert, their tokens,
    sub-problem group offsets)."""
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    experts = np.searchsorted(off, rows, side="right") - 1
    order = np.lexsort((rows, experts))
    rows, experts = rows[order], experts[order]
    counts = np.bincount(experts, minlength=E)
    sub_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    tokens = row_src[rows] // K
    return rows, tokens, sub_off


@pytest.fixture(scope="module", params=FULL)
def run(request):
    need_gpu()
    wl = WORKLOADS[request.param]
    dev = torch.device("cuda")
    inp = make_inputs(wl, dev, with_grad=wl.train)
    blk = MoEBlock(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=wl.train)
    blk.forward(inp["x"], inp["wi"], inp["wo"], logits=inp["logits"], bias=inp["bias"],
                ids=inp["ids"], w=inp["w"])
    if wl.train:
        blk.backward(inp["dy"], inp["wi"], inp["wo"])
    torch.cuda.synchronize()
    assert int(blk.status.item()) == 0
    # the oracle's routing and histogram, whole
    if wl.score_mode == B.SCORE_GIVEN:
        ids_ref, w_ref = to_host(inp["ids"]), to_host(inp["w"])
    else:
        ids_ref, w_ref = oracle.route(to_host(inp["logits"]),
                                      None if inp["bias"] is None else to_host(inp["bias"]),
                                      wl.score_mode, wl.T, wl.E, wl.K)
    gs, off, pos, row_src, bad = oracle.histogram(ids_ref, wl.E)
    assert bad == 0
    yield dict(wl=wl, inp=inp, blk=blk, ids=ids_ref, w=w_ref, gs=gs, off=off, pos=pos,
               row_src=row_src)
    del blk, inp
    torch.cuda.empty_cache()


def test_routing_and_permutation_whole(run):
    wl, blk = run["wl"], run["blk"]
    assert_exact("ids", to_host(blk.ids), run["ids"])
    assert_close("w", to_host(blk.w), run["w"], rtol=1e-5, atol=1e-6, bf16=False)
    assert_exact("group_sizes", to_host(blk.group_sizes), run["gs"])
    assert_exact("group_offsets", to_host(blk.group_offsets), run["off"])
    assert_exact("pos", to_host(blk.pos), run["pos"])
    assert_exact("row_src", to_host(blk.row_src), run["row_src"])
    # the permutation at full size: xs[r] == x[row_src[r] // K] for every row
    rs = blk.row_src.long()
    assert torch.equal(blk.xs, run["inp"]["x"][rs // wl.K])


def _sample_rows(run, n, rng):
    off, E, R = run["off"], run["wl"].E, run["wl"].R
    sizes = np.diff(off)
    big, small = int(np.argmax(sizes)), int(np.argmin(np.where(sizes > 0, sizes, R + 1)))
    rows = list(rng.integers(0, R, n))
    for e in (big, small, int(rng.integers(0, E))):
        if sizes[e] > 0:
            rows += [int(off[e]), int(off[e + 1] - 1)]
    return rows


def _oracle_rows(run, rows):
    """Oracle forward for sampled sorted-order rows (from the inputs)."""
    wl, inp = run["wl"], run["inp"]
    rows, tokens, sub_off = _sub_problem(rows, run["row_src"], run["off"], wl.K, wl.E)
    xs = to_host(inp["x"][torch.from_numpy(tokens).long().cuda()])
    wi, wo = _bits(inp["wi"]), _bits(inp["wo"])
    h, z = oracle.fc1_swiglu(xs, wi, sub_off)
    ys = oracle.fc2(h, wo, sub_off)
    return dict(rows=rows, tokens=tokens, sub_off=sub_off, xs=xs, h=h, z=z, ys=ys, wi=wi, wo=wo)


def test_gemms_on_sampled_rows(run):
    rng = np.random.Generator(np.random.PCG64(11))
    o = _oracle_rows(run, _sample_rows(run, 24, rng))
    blk = run["blk"]
    idx = torch.from_numpy(o["rows"]).long().cuda()
    assert_close("h", to_host(blk.h[idx]), o["h"])
    if blk.z is not None:
        assert_close("z", to_host(blk.z[idx]), o["z"])
    assert_close("ys", to_host(blk.ys[idx]), o["ys"])


def test_combine_and_backward_on_sampled_tokens(run):
    wl, inp, blk = run["wl"], run["inp"], run["blk"]
    rng = np.random.Generator(np.random.PCG64(12))
    tok = np.sort(rng.choice(wl.T, size=6, replace=False))
    rows = run["pos"][tok].ravel()
    o = _oracle_rows(run, rows)
    # map (token, slot) -> index in the oracle's sorted sub rows
    where = {int(r): i for i, r in enumerate(o["rows"])}
    pos_sub = np.array([[where[int(r)] for r in run["pos"][t]] for t in tok], np.int32)
    w_sub = run["w"][tok]
    out_ref = oracle.combine(o["ys"], w_sub, pos_sub, len(tok), wl.D)
    ti = torch.from_numpy(tok).long().cuda()
    assert_close("out", to_host(blk.out[ti]), out_ref)
    if not wl.train:
        return
    dy = to_host(inp["dy"][ti])
    dys_ref, dw_ref = oracle.combine_bwd(dy, o["ys"], w_sub, pos_sub)
    ri = torch.from_numpy(o["rows"]).long().cuda()
    assert_close("dys", to_host(blk.dys[ri]), dys_ref)
    # dw is a sum over D of dout * ys: end to end it sees the GPU's own ys,
    # whose bf16 roundings may each differ by one ulp (2^-8 relative) from the
    # oracle's; for independent differences the sum moves by about
    # 2^-8 * sqrt(sum_d (dout_d ys_d)^2), so the end-to-end bound adds four
    # times that to the per-element tolerance.
    y64 = (o["ys"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g64 = (dy.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    spread = np.sqrt(np.einsum("td,tkd->tk", g64 ** 2, y64[pos_sub] ** 2))
    err = np.abs(to_host(blk.dw[ti]).astype(np.float64) - dw_ref)
    lim = 2e-2 * np.abs(dw_ref) + 2e-2 + 4 * 2.0 ** -8 * spread
    assert np.all(err <= lim), f"dw end to end: err {err.max():.4g} > bound"
    # the combine backward in isolation, at full width D, on the oracle's ys
    d1 = B.dims(len(tok), wl.D, len(o["rows"]), wl.K, wl.F)
    dys1 = torch.empty((len(o["rows"]), wl.D), dtype=torch.bfloat16, device="cuda")
    dw1 = torch.empty((len(tok), wl.K), dtype=torch.float32, device="cuda")
    B.moe_combine_bwd(inp["dy"][ti].contiguous(), to_dev(o["ys"]), to_dev(w_sub), to_dev(pos_sub),
                      dys1, dw1, d1)
    torch.cuda.synchronize()
    assert_exact("dys (isolated)", to_host(dys1), dys_ref)
    assert_close("dw (isolated)", to_host(dw1), dw_ref, bf16=False)
    dz_ref, _ = oracle.fc2_bwd(dys_ref, o["h"], o["wo"], o["z"], o["sub_off"], want_drhs=False)
    assert_close("dz", to_host(blk.dz[ri]), dz_ref)
    dxs_ref, _ = oracle.fc1_bwd(dz_ref, o["xs"], o["wi"], o["sub_off"], want_drhs=False)
    assert_close("dxs", to_host(blk.dxs[ri]), dxs_ref)
    dx_ref = oracle.permute_bwd(dxs_ref, pos_sub, len(tok), wl.D)
    assert_close("dx", to_host(blk.dx[ti]), dx_ref)


def test_weight_gradients_on_sampled_entries(run):
    wl, inp, blk = run["wl"], run["inp"], run["blk"]
    if not wl.train:
        pytest.skip("forward-only workload")
    rng = np.random.Generator(np.random.PCG64(13))
    off, K, F, D = run["off"], wl.K, wl.F, wl.D
    sizes = np.diff(off)
    experts = {int(np.argmax(sizes)), int(np.argmin(sizes)), int(rng.integers(0, wl.E))}
    wi, wo = blk.dwi, blk.dwo
    for e in sorted(experts):
        r0, r1 = int(off[e]), int(off[e + 1])
        f, d, n = int(rng.integers(0, F)), int(rng.integers(0, D)), int(rng.integers(0, 2 * F))
        if r1 == r0:
            assert float(blk.dwo[e].float().abs().max()) == 0.0
            assert float(blk.dwi[e].float().abs().max()) == 0.0
            continue
        rows = np.arange(r0, r1)
        src = run["row_src"][rows]
        tokens, slots = src // K, src % K
        ti = torch.from_numpy(tokens).long().cuda()
        x_rows = to_host(inp["x"][ti])
        dy_rows = to_host(inp["dy"][ti])
        w_rows = run["w"][tokens, slots].astype(np.float32)
        one = np.array([0, r1 - r0], np.int32)
        # dys rows of this expert: the combine backward per row (unit slot each)
        pos_one = np.arange(r1 - r0, dtype=np.int32)[:, None]
        dys_rows, _ = oracle.combine_bwd(dy_rows, np.zeros((r1 - r0, D), np.uint16),
                                         w_rows[:, None], pos_one)
        wi_e = to_host(inp["wi"][e])          # [D, 2F]
        wo_e = to_host(inp["wo"][e])          # [F, D]
        # h[:, f] and z[:, f], z[:, F+f] from the gate/up columns of wi
        cols = [f, F + f]
        h_f, z_f = oracle.fc1_swiglu(x_rows, wi_e[None][:, :, cols], one)
        # dwo[e, f, d] = sum_r h[r, f] * dys[r, d]
        _, dwo_fd = oracle.fc2_bwd(dys_rows[:, [d]], h_f, wo_e[None][:, [f]][:, :, [d]], None,
                                   one, want_dlhs=False)
        assert_close(f"dwo[{e},{f},{d}]", to_host(blk.dwo[e, f, d].reshape(1)),
                     dwo_fd.reshape(1))
        # dz[:, n]: dh[:, fn] (against all of wo[e, fn, :]) through the SwiGLU backward
        fn = n % F
        cols_n = [fn, F + fn]
        _, z_n = oracle.fc1_swiglu(x_rows, wi_e[None][:, :, cols_n], one)
        dz_n, _ = oracle.fc2_bwd(dys_rows, np.zeros((r1 - r0, 1), np.uint16),
                                 wo_e[None][:, [fn]], z_n, one, want_drhs=False)
        dz_col = dz_n[:, [0 if n < F else 1]]
        # dwi[e, d, n] = sum_r xs[r, d] * dz[r, n]
        _, dwi_dn = oracle.fc1_bwd(np.concatenate([dz_col, dz_col], axis=1), x_rows[:, [d]],
                                   np.zeros((1, 1, 2), np.uint16), one, want_dlhs=False)
        assert_close(f"dwi[{e},{d},{n}]", to_host(blk.dwi[e, d, n].reshape(1)),
                     dwi_dn[0, 0, :1])

"""GPU parity of every libmoe.so entry point against the CPU oracle.

Each step is checked in isolation (the GPU kernel gets the oracle's own
upstream values, so a mismatch points at that kernel) and the whole block is
checked end to end.  Bars: routing ids, group sizes/offsets, pos, row_src
and the permutation bit-exact; combine, permute backward and dys bit-exact
(same operation order as the oracle, no fused multiply-add); every other
float within |gpu - ref| <= 2e-2*|ref| + 2e-2.  Sizes span several 128x256
tiles with ragged group, N and M tails.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.inputs import custom, make_inputs, WORKLOADS
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu

CASES = {
    # F = 192: FC1 gate/up tiles of 128 with a ragged N tail; D = 256: one FC2 N tile
    "ragged_small": custom("ragged_small", T=300, D=256, E=8, K=2, F=192, train=True),
    # D = 320, F = 320: ragged tails against 256-wide tiles; biased router
    "ragged_bias": custom("ragged_bias", T=517, D=320, E=12, K=3, F=320, bias_std=0.5, train=True),
    "sigmoid": custom("sigmoid", T=400, D=384, E=16, K=4, F=128, score_mode=1, train=True),
    "zipf_given": custom("zipf_given", T=640, D=256, E=24, K=4, F=256, score_mode=2, zipf_s=1.2,
                         train=True),
    "tiny_fwd": WORKLOADS["tiny_fwd"],
    # the largest E the ABI takes: 32-lane top-k groups, a full 1024-key sort
    # in the drhs schedule, hundreds of experts with no rows
    "e_max": custom("e_max", T=300, D=128, E=1024, K=8, F=64, bias_std=0.5, train=True),
    # the largest K: 32 slots per token, sigmoid-normalised weights
    "k_max": custom("k_max", T=96, D=192, E=40, K=32, F=128, score_mode=1, train=True),
}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


# The grouped GEMMs run either one CTA per tile or on CTA pairs (a 2-CTA
# cluster sharing one 256-row tile), and drhs pair tiles are 512 or 256
# columns wide; MOE_GEMM_PAIR and MOE_GEMM_WIDE force the path so that every
# one is checked on every shape.
PAIR_MODES = pytest.mark.parametrize("pair", ["0", "1", "1n"], ids=["cta1", "cta2", "cta2narrow"])


@pytest.fixture
def pair_env(monkeypatch, pair):
    monkeypatch.setenv("MOE_GEMM_PAIR", pair[0])
    monkeypatch.setenv("MOE_GEMM_WIDE", "0" if pair.endswith("n") else "1")
    return pair


def _numpy_inputs(wl):
    inp = make_inputs(wl, "cpu", with_grad=True)
    return oracle.to_numpy(inp)


def _oracle(inp):
    fwd = oracle.block_forward(inp)
    bwd = oracle.block_backward(inp, fwd)
    return fwd, bwd


def _dims(wl, T=None):
    return B.dims(wl.T if T is None else T, wl.D, wl.E, wl.K, wl.F)


def _ws(d):
    return torch.empty(max(B.moe_workspace_bytes(d), 256), dtype=torch.uint8, device="cuda")


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    wl = CASES[request.param]
    inp = _numpy_inputs(wl)
    fwd, bwd = _oracle(inp)
    return wl, inp, fwd, bwd


def _route(wl, inp, ids_in=None, w_in=None):
    d = _dims(wl)
    T, E, K = wl.T, wl.E, wl.K
    ids = to_dev(ids_in) if ids_in is not None else torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = to_dev(w_in) if w_in is not None else torch.empty((T, K), dtype=torch.float32, device="cuda")
    gs = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    pos = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    row_src = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_route_histogram(to_dev(inp["logits"]), to_dev(inp["bias"]), wl.score_mode, ids, w, gs,
                          off, pos, row_src, st, _ws(d), d)
    torch.cuda.synchronize()
    return dict(ids=to_host(ids), w=to_host(w), gs=to_host(gs), off=to_host(off),
                pos=to_host(pos), row_src=to_host(row_src), status=int(st.item()))


def test_route_histogram(case):
    wl, inp, fwd, _ = case
    if wl.score_mode == oracle.GIVEN:
        g = _route(wl, inp, inp["ids"], inp["w"])
    else:
        g = _route(wl, inp)
        assert_exact("ids", g["ids"], fwd["ids"])
        assert_close("w", g["w"], fwd["w"], rtol=1e-5, atol=1e-6, bf16=False)
    assert g["status"] == 0
    assert_exact("group_sizes", g["gs"], fwd["group_sizes"])
    assert_exact("group_offsets", g["off"], fwd["group_offsets"])
    assert_exact("pos", g["pos"], fwd["pos"])
    assert_exact("row_src", g["row_src"], fwd["row_src"])


def test_permute_and_combine_exact(case):
    wl, inp, fwd, bwd = case
    d = _dims(wl)
    R = wl.T * wl.K
    xs = torch.full((R, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.moe_permute(to_dev(inp["x"]), to_dev(fwd["pos"]), xs, d)
    out = torch.empty((wl.T, wl.D), dtype=torch.bfloat16, device="cuda")
    B.moe_combine(to_dev(fwd["ys"]), to_dev(fwd["w"]), to_dev(fwd["pos"]), out, d)
    dx = torch.empty((wl.T, wl.D), dtype=torch.bfloat16, device="cuda")
    B.moe_permute_bwd(to_dev(bwd["dxs"]), to_dev(fwd["pos"]), dx, d)
    dys = torch.full((R, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((wl.T, wl.K), dtype=torch.float32, device="cuda")
    B.moe_combine_bwd(to_dev(inp["dy"]), to_dev(fwd["ys"]), to_dev(fwd["w"]), to_dev(fwd["pos"]),
                      dys, dw, d)
    torch.cuda.synchronize()
    assert_exact("xs", to_host(xs), fwd["xs"])       # every row written exactly once
    assert_exact("out", to_host(out), fwd["out"])
    assert_exact("dx", to_host(dx), bwd["dx"])
    assert_exact("dys", to_host(dys), bwd["dys"])
    assert_close("dw", to_host(dw), bwd["dw"], bf16=False)


@PAIR_MODES
def test_fc1_swiglu(case, pair_env):
    wl, inp, fwd, _ = case
    d = _dims(wl)
    R = wl.T * wl.K
    h = torch.full((R, wl.F), float("nan"), dtype=torch.bfloat16, device="cuda")
    z = torch.full((R, 2 * wl.F), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    xs, wi, off = to_dev(fwd["xs"]), to_dev(inp["wi"]), to_dev(fwd["group_offsets"])
    B.moe_grouped_gemm_fc1_swiglu(xs, wi, off, h, z, st, _ws(d), d)
    h2 = torch.empty_like(h)
    B.moe_grouped_gemm_fc1_swiglu(xs, wi, off, h2, None, st, _ws(d), d)   # inference: no z
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close("h", to_host(h), fwd["h"])
    assert_close("z", to_host(z), fwd["z"])
    assert_exact("h (no z)", to_host(h2), to_host(h))


@PAIR_MODES
def test_fc2(case, pair_env):
    wl, inp, fwd, _ = case
    d = _dims(wl)
    R = wl.T * wl.K
    ys = torch.full((R, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_fc2(to_dev(fwd["h"]), to_dev(inp["wo"]), to_dev(fwd["group_offsets"]), ys,
                           st, _ws(d), d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close("ys", to_host(ys), fwd["ys"])


@PAIR_MODES
def test_fc2_bwd(case, pair_env):
    wl, inp, fwd, bwd = case
    d = _dims(wl)
    R, F = wl.T * wl.K, wl.F
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dys, h, wo = to_dev(bwd["dys"]), to_dev(fwd["h"]), to_dev(inp["wo"])
    z, off = to_dev(fwd["z"]), to_dev(fwd["group_offsets"])
    dz = torch.full((R, 2 * F), float("nan"), dtype=torch.bfloat16, device="cuda")
    dwo = torch.full((wl.E, F, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm_fc2_bwd(dys, h, wo, z, off, dz, dwo, st, _ws(d), d)
    dh = torch.full((R, F), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm_fc2_bwd(dys, h, wo, None, off, dh, None, st, _ws(d), d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close("dz (fused SwiGLU bwd)", to_host(dz), bwd["dz"])
    assert_close("dwo", to_host(dwo), bwd["dwo"])
    dh_ref, _ = oracle.fc2_bwd(bwd["dys"], fwd["h"], inp["wo"], None, fwd["group_offsets"],
                               want_drhs=False)
    assert_close("dh", to_host(dh), dh_ref)


@PAIR_MODES
def test_fc1_bwd(case, pair_env):
    wl, inp, fwd, bwd = case
    d = _dims(wl)
    R, F = wl.T * wl.K, wl.F
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    xs, wi, off = to_dev(fwd["xs"]), to_dev(inp["wi"]), to_dev(fwd["group_offsets"])
    dxs = torch.full((R, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    dwi = torch.full((wl.E, wl.D, 2 * F), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm_fc1_swiglu_bwd(to_dev(bwd["dz"]), None, xs, wi, off, dxs, dwi, st,
                                      _ws(d), d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close("dxs", to_host(dxs), bwd["dxs"])
    assert_close("dwi", to_host(dwi), bwd["dwi"])
    # unfused path: grad = dh (bf16), SwiGLU backward inside the call
    dh_ref, _ = oracle.fc2_bwd(bwd["dys"], fwd["h"], inp["wo"], None, fwd["group_offsets"],
                               want_drhs=False)
    dz_ref = oracle.swiglu_bwd(dh_ref, fwd["z"])
    dxs_ref, dwi_ref = oracle.fc1_bwd(dz_ref, fwd["xs"], inp["wi"], fwd["group_offsets"])
    dxs2 = torch.empty_like(dxs)
    dwi2 = torch.empty_like(dwi)
    B.moe_grouped_gemm_fc1_swiglu_bwd(to_dev(dh_ref), to_dev(fwd["z"]), xs, wi, off, dxs2, dwi2,
                                      st, _ws(d), d)
    torch.cuda.synchronize()
    assert_close("dxs (unfused)", to_host(dxs2), dxs_ref)
    assert_close("dwi (unfused)", to_host(dwi2), dwi_ref)


@PAIR_MODES
def test_block_end_to_end(case, pair_env):
    from mixture_experts_ffn_histogram_gb300.block import MoEBlock
    wl, inp, fwd, bwd = case
    blk = MoEBlock(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=True)
    blk.forward(to_dev(inp["x"]), to_dev(inp["wi"]), to_dev(inp["wo"]), logits=to_dev(inp["logits"]),
                bias=to_dev(inp["bias"]), ids=to_dev(inp["ids"]), w=to_dev(inp["w"]))
    blk.backward(to_dev(inp["dy"]), to_dev(inp["wi"]), to_dev(inp["wo"]))
    torch.cuda.synchronize()
    assert int(blk.status.item()) == 0
    assert_exact("pos", to_host(blk.pos), fwd["pos"])
    assert_exact("xs", to_host(blk.xs), fwd["xs"])
    for name in ("h", "z", "ys", "out"):
        assert_close(name, to_host(getattr(blk, name)), fwd[name])
    for name in ("dys", "dz", "dwo", "dxs", "dwi", "dx"):
        assert_close(name, to_host(getattr(blk, name)), bwd[name])
    assert_close("dw", to_host(blk.dw), bwd["dw"], bf16=False)


# ----------------------------------------------------------------- edges
def _given_block(T, D, E, K, F, ids, w, seed=0):
    wl = custom("edge", T=T, D=D, E=E, K=K, F=F, score_mode=2, train=True, seed=seed)
    inp = oracle.to_numpy(make_inputs(wl, "cpu", with_grad=True))
    inp["ids"], inp["w"] = ids.astype(np.int32), w.astype(np.float32)
    return wl, inp


@PAIR_MODES
@pytest.mark.parametrize("kind", ["empty_experts", "one_expert_all", "groups_of_one", "k1", "k_eq_e",
                                  "t1", "e1"])
def test_edge_cases(kind, pair_env):
    rng = np.random.Generator(np.random.PCG64(5))
    if kind == "empty_experts":      # only experts 1, 4, 5 are used
        T, D, E, K, F = 200, 128, 8, 2, 128
        ids = np.stack([rng.choice([1, 4, 5], size=2, replace=False) for _ in range(T)])
    elif kind == "one_expert_all":   # every token's first slot goes to expert 3
        T, D, E, K, F = 300, 192, 6, 2, 64
        ids = np.stack([[3, rng.choice([0, 1, 2, 4, 5])] for _ in range(T)])
    elif kind == "groups_of_one":    # E = R: each expert gets exactly one row
        T, D, E, K, F = 16, 128, 32, 2, 128
        ids = rng.permutation(E).reshape(T, K)
    elif kind == "k1":
        T, D, E, K, F = 257, 128, 5, 1, 192
        ids = rng.integers(0, E, (T, 1))
    elif kind == "k_eq_e":
        T, D, E, K, F = 130, 64, 4, 4, 64
        ids = np.stack([rng.permutation(E) for _ in range(T)])
    elif kind == "t1":
        T, D, E, K, F = 1, 256, 16, 8, 128
        ids = rng.permutation(E)[:K][None]
    else:                            # E = 1: a dense SwiGLU MLP
        T, D, E, K, F = 160, 128, 1, 1, 256
        ids = np.zeros((T, 1))
    w = rng.dirichlet(np.ones(K), size=T)
    wl, inp = _given_block(T, D, E, K, F, ids, w)
    fwd, bwd = _oracle(inp)
    from mixture_experts_ffn_histogram_gb300.block import MoEBlock
    blk = MoEBlock(T, D, E, K, F, B.SCORE_GIVEN, train=True)
    blk.forward(to_dev(inp["x"]), to_dev(inp["wi"]), to_dev(inp["wo"]), ids=to_dev(inp["ids"]),
                w=to_dev(inp["w"]))
    blk.backward(to_dev(inp["dy"]), to_dev(inp["wi"]), to_dev(inp["wo"]))
    torch.cuda.synchronize()
    assert int(blk.status.item()) == 0
    for name in ("group_sizes", "group_offsets", "pos", "row_src", "xs"):
        assert_exact(name, to_host(getattr(blk, name)), fwd[name])
    for name in ("h", "z", "ys", "out"):
        assert_close(name, to_host(getattr(blk, name)), fwd[name])
    assert_exact("dys", to_host(blk.dys), bwd["dys"])
    for name in ("dz", "dwo", "dxs", "dwi", "dx"):
        assert_close(name, to_host(getattr(blk, name)), bwd[name])
    assert_close("dw", to_host(blk.dw), bwd["dw"], bf16=False)
    if kind == "empty_experts":
        dwo, dwi = to_host(blk.dwo), to_host(blk.dwi)
        for e in (0, 2, 3, 6, 7):
            assert not dwo[e].any() and not dwi[e].any()


def test_t0_is_noop():
    d = B.dims(0, 128, 8, 2, 64)
    gs = torch.full((8,), 5, dtype=torch.int32, device="cuda")
    off = torch.full((9,), 5, dtype=torch.int32, device="cuda")
    ws = _ws(d)
    B.moe_route_histogram(None, None, B.SCORE_SOFTMAX_TOPK, None, None, gs, off, None, None, None,
                          ws, d)
    dwo = torch.full((8, 64, 128), 1.0, dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm_fc2_bwd(None, None, None, None, off, None, dwo, None, ws, d)
    torch.cuda.synchronize()
    assert not gs.any() and not off.any() and not dwo.float().abs().sum().item()


def test_bad_ids_reported():
    T, E, K = 64, 8, 2
    d = B.dims(T, 64, E, K, 64)
    rng = np.random.Generator(np.random.PCG64(9))
    ids = rng.integers(0, E, (T, K)).astype(np.int32)
    ids[5, 1] = E
    ids[9, 0] = -3
    w = np.full((T, K), 0.5, np.float32)
    gs = torch.empty(E, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty((T, K), dtype=torch.int32, device="cuda")
    row_src = torch.empty(T * K, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_route_histogram(None, None, B.SCORE_GIVEN, to_dev(ids), to_dev(w), gs, off, pos, row_src,
                          st, _ws(d), d)
    torch.cuda.synchronize()
    assert int(st.item()) == B.MOE_ERR_DEVICE
    gref, oref, pref, rref, bad = oracle.histogram(ids, E)
    assert bad == 2
    assert_exact("group_sizes", to_host(gs), gref)
    assert_exact("pos", to_host(pos), pref)
    assert_exact("row_src", to_host(row_src), rref)


def test_host_side_errors():
    d = B.dims(16, 128, 8, 2, 64)
    x = torch.empty((16, 128), dtype=torch.bfloat16, device="cuda")
    xs = torch.empty((32, 128), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros((16, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as e:
        B.moe_permute(x, pos, None, d)
    assert e.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoeError) as e:
        B.moe_permute(x.data_ptr() + 2, pos, xs, d)           # misaligned
    assert e.value.status == B.MOE_ERR_INVALID_ARG
    for bad in (B.dims(16, 100, 8, 2, 64), B.dims(16, 128, 8, 2, 96), B.dims(16, 128, 8, 9, 64),
                B.dims(16, 128, 64, 33, 64), B.dims(16, 128, 2048, 2, 64)):
        with pytest.raises(B.MoeError) as e:
            B.moe_permute(x, pos, xs, bad)
        assert e.value.status == B.MOE_ERR_UNSUPPORTED


def test_bounded_wait_gives_up_and_context_survives():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_selftest_bounded_wait(st, 2_000_000)       # 2 ms: nothing ever arrives
    torch.cuda.synchronize()
    assert int(st.item()) == B.MOE_ERR_TIMEOUT
    # the context is still usable
    x = torch.arange(16 * 64, device="cuda", dtype=torch.float32).reshape(16, 64).to(torch.bfloat16)
    xs = torch.empty((16, 64), dtype=torch.bfloat16, device="cuda")
    pos = torch.arange(16, dtype=torch.int32, device="cuda").reshape(16, 1)
    B.moe_permute(x, pos, xs, B.dims(16, 64, 1, 1, 64))
    torch.cuda.synchronize()
    assert torch.equal(xs, x)

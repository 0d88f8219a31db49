"""GPU parity of routing at the sizes where moe_route_histogram switches
between its two kernels, and on inputs full of tied scores.  One
thread-block cluster runs given routing and selections over E <= 64 while
every warp has at most two passes (2048 given tokens at K = 8, 4096 tokens
at E = 64, K = 4, when the device holds a 16-block cluster; half that with
8 blocks); a cooperative grid runs the rest.  Bit-exact against the
oracle: ids, group sizes, offsets, pos and row_src; w within 1e-5 relative
(the GPU's exp is not the C library's).

MaxText "Gemma4 26B MoE on TPU v6e: MaxText layer/model optimizations",
Commits table row 6 (top_k_weights and group_size next to the block);
MaxText "MoE: fused TensorCore Pallas permute/combine kernels and
split-expert wi layout for TPU v6e", Commits table row 2 (the group_size
histogram before the gather).
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
    **{f"softmax_bias_e64_T{T}": custom(f"sb{T}", T=T, D=64, E=64, K=4, F=64, bias_std=0.5, seed=T)
       for T in (2048, 2049, 4096, 4097)},
    **{f"given_T{T}": custom(f"g{T}", T=T, D=64, E=128, K=8, F=64, score_mode=2, seed=T)
       for T in (1024, 1025, 2048, 2049)},
    "softmax_bias_e128": custom("sb128", T=1024, D=64, E=128, K=8, F=64, bias_std=0.5, seed=2),
    "sigmoid_e256": custom("s256", T=1500, D=64, E=256, K=8, F=64, score_mode=1, seed=3),
    "one_expert": custom("e1", T=333, D=64, E=1, K=1, F=64, seed=4),
    "two_of_two": custom("e2", T=4097, D=64, E=2, K=2, F=64, seed=5),
    "e_max_k_max": custom("emax", T=700, D=64, E=1024, K=32, F=64, score_mode=1, seed=6),
}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _run(wl, logits, bias, ids_in=None, w_in=None):
    d = B.dims(wl.T, wl.D, wl.E, wl.K, wl.F)
    T, E, K = wl.T, wl.E, wl.K
    ids = to_dev(ids_in) if ids_in is not None else torch.full((T, K), -7, dtype=torch.int32,
                                                                device="cuda")
    w = to_dev(w_in) if w_in is not None else torch.full((T, K), float("nan"),
                                                         dtype=torch.float32, device="cuda")
    gs = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    pos = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    row_src = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(B.moe_workspace_bytes(d), 256), dtype=torch.uint8, device="cuda")
    B.moe_route_histogram(None if logits is None else to_dev(logits),
                          None if bias is None else to_dev(bias), wl.score_mode, ids, w, gs, off,
                          pos, row_src, st, ws, d)
    torch.cuda.synchronize()
    return dict(ids=to_host(ids), w=to_host(w), gs=to_host(gs), off=to_host(off),
                pos=to_host(pos), row_src=to_host(row_src), status=int(st.item()))


def _check(wl, g, logits, bias, ids=None):
    if ids is None:
        ids, w = oracle.route(logits, bias, wl.score_mode, wl.T, wl.E, wl.K)
        assert_exact("ids", g["ids"], ids)
        assert_close("w", g["w"], w, rtol=1e-5, atol=1e-6, bf16=False)
    gs, off, pos, row_src, bad = oracle.histogram(ids, wl.E)
    assert bad == 0 and g["status"] == 0
    assert_exact("group_sizes", g["gs"], gs)
    assert_exact("group_offsets", g["off"], off)
    assert_exact("pos", g["pos"], pos)
    assert_exact("row_src", g["row_src"], row_src)


@pytest.mark.parametrize("name", sorted(CASES))
def test_route_around_kernel_switch(name):
    wl = CASES[name]
    inp = oracle.to_numpy(make_inputs(wl, "cpu"))
    if wl.score_mode == oracle.GIVEN:
        g = _run(wl, None, None, inp["ids"], inp["w"])
        _check(wl, g, None, None, ids=inp["ids"])
    else:
        g = _run(wl, inp["logits"], inp["bias"])
        _check(wl, g, inp["logits"], inp["bias"])


@pytest.mark.parametrize("T", [700, 3000])
def test_route_tied_scores(T):
    """Scores rounded to steps of 0.5: most tokens hold several equal
    scores, which the selection must order by expert id (lower first)."""
    wl = custom("ties", T=T, D=64, E=64, K=6, F=64, bias_std=0.0, seed=7)
    inp = oracle.to_numpy(make_inputs(wl, "cpu"))
    logits = (np.round(inp["logits"] * 2.0) / 2.0).astype(np.float32)
    # the rounding leaves ties within almost every token's top six
    srt = -np.sort(-logits, axis=1)[:, :7]
    assert np.mean(np.any(srt[:, 1:] == srt[:, :-1], axis=1)) > 0.5
    g = _run(wl, logits, None)
    _check(wl, g, logits, None)


@pytest.mark.parametrize("T", [64, 1024, 8192])
def test_bad_ids_on_both_kernels(T):
    """Given routing with ids out of range: MOE_ERR_DEVICE, the bad slots
    dropped (pos -1), the rest placed as the oracle places them, and the
    rows that no valid slot fills set to -1 (64 and 1024 tokens on the
    cluster kernel, 8192 on the cooperative one)."""
    E, K = 16, 4
    d = B.dims(T, 64, E, K, 64)
    rng = np.random.Generator(np.random.PCG64(T))
    ids = rng.integers(0, E, (T, K)).astype(np.int32)
    bad_t = rng.choice(T, size=min(T, 5), replace=False)
    for i, t in enumerate(bad_t):
        ids[t, i % K] = E + i if i % 2 == 0 else -1 - i
    w = np.full((T, K), 0.25, np.float32)
    gs = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    pos = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    row_src = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(B.moe_workspace_bytes(d), 256), dtype=torch.uint8, device="cuda")
    B.moe_route_histogram(None, None, B.SCORE_GIVEN, to_dev(ids), to_dev(w), gs, off, pos,
                          row_src, st, ws, d)
    torch.cuda.synchronize()
    assert int(st.item()) == B.MOE_ERR_DEVICE
    gref, oref, pref, rref, bad = oracle.histogram(ids, E)
    assert bad == len(bad_t)
    assert_exact("group_sizes", to_host(gs), gref)
    assert_exact("group_offsets", to_host(off), oref)
    assert_exact("pos", to_host(pos), pref)
    assert_exact("row_src", to_host(row_src), rref)

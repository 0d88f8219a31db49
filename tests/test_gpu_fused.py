"""GPU parity of the fused inference forward (moe_fused_forward).

After the routing call, the fused forward gathers FC1's rows straight from
the token-major x (no permuted copy) and adds FC2's rows, weighted, into an
fp32 accumulator per token (no ys, no separate combine).  Checks, with every
output buffer first filled with NaN:
  * h equals the unfused FC1's h bit for bit: the same values are summed in
    the same order, only fetched from elsewhere;
  * out against the oracle's block forward, |gpu - ref| <= 2e-2*|ref| + 2e-2
    (whole on ragged small cases and at 1024 tokens; on sampled tokens, each
    recomputed by the oracle from slices of the inputs, at the larger
    token-sweep sizes);
  * out against the unfused GPU forward, within the same tolerance (the
    unfused combine rounds each ys row to bf16 first; the fused one sums fp32
    products in no fixed order, so out is not bitwise reproducible).
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.block import MoEBlock
from mixture_experts_ffn_histogram_gb300.inputs import WORKLOADS, custom, make_inputs
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_host

pytestmark = pytest.mark.gpu

SMALL = {
    # ragged groups spanning several 128-row tiles, F with a 128-wide tail
    "ragged": custom("ragged", T=700, D=256, E=8, K=2, F=192, bias_std=0.5),
    # D = 320: FC2's second N tile is 64 wide; sigmoid-normalised weights
    "narrow_n": custom("narrow_n", T=333, D=320, E=12, K=3, F=320, score_mode=1),
    # given Zipf routing: some groups long, some short
    "zipf": custom("zipf", T=512, D=256, E=24, K=4, F=256, score_mode=2, zipf_s=1.2),
    # many experts without rows
    "sparse_e": custom("sparse_e", T=64, D=128, E=256, K=2, F=128),
    "one_token": custom("one_token", T=1, D=128, E=4, K=1, F=64),
    "tiny_fwd": WORKLOADS["tiny_fwd"],
    "token_sweep_T1024": WORKLOADS["token_sweep_T1024"],
}
SAMPLED = ["token_sweep_T2048", "token_sweep_T4096", "token_sweep_T8192"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _run(wl, inp):
    """The fused and the unfused forward on the same GPU inputs."""
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    fused = MoEBlock(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=False)
    fused.h.fill_(float("nan"))
    fused.out.fill_(float("nan"))
    fused.forward_fused(g["x"], g["wi"], g["wo"], logits=g["logits"], bias=g["bias"],
                        ids=g["ids"], w=g["w"])
    plain = MoEBlock(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=False)
    plain.forward(g["x"], g["wi"], g["wo"], logits=g["logits"], bias=g["bias"], ids=g["ids"],
                  w=g["w"])
    torch.cuda.synchronize()
    assert int(fused.status.item()) == 0 and int(plain.status.item()) == 0
    return fused, plain


@pytest.mark.parametrize("name", sorted(SMALL))
def test_fused_forward_whole(name):
    wl = SMALL[name]
    inp = make_inputs(wl, "cpu", with_grad=False)
    fused, plain = _run(wl, inp)
    R = int(to_host(plain.group_offsets)[-1])
    assert_exact("h (fused vs unfused FC1)", to_host(fused.h)[:R], to_host(plain.h)[:R])
    ref = oracle.block_forward(oracle.to_numpy(inp), want_z=False)
    assert_close("out vs oracle", to_host(fused.out), ref["out"])
    assert_close("out vs unfused", to_host(fused.out), to_host(plain.out))


@pytest.mark.parametrize("name", SAMPLED)
def test_fused_forward_sampled(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda", with_grad=False)
    fused, plain = _run(wl, inp)
    R = wl.R
    assert torch.equal(fused.h[:R], plain.h[:R]), "h differs from the unfused FC1's"
    assert bool(torch.isfinite(fused.out).all()), "out not written everywhere"
    assert_close("out vs unfused", to_host(fused.out), to_host(plain.out))
    # sampled tokens against the oracle, from slices of the inputs
    rng = np.random.Generator(np.random.PCG64(21))
    tok = np.sort(rng.choice(wl.T, size=12, replace=False))
    ids, w = oracle.route(to_host(inp["logits"]), None, wl.score_mode, wl.T, wl.E, wl.K)
    ids_t, w_t = ids[tok], w[tok]
    x_t = to_host(inp["x"][torch.from_numpy(tok).long().cuda()])
    wi_h, wo_h = to_host(inp["wi"]), to_host(inp["wo"])
    # a sub-problem of the sampled tokens with their own routing (given)
    gs, off, pos, _, bad = oracle.histogram(ids_t, wl.E)
    assert bad == 0
    xs = oracle.permute(x_t, pos)
    h, _ = oracle.fc1_swiglu(xs, wi_h, off, want_z=False)
    ys = oracle.fc2(h, wo_h, off)
    ref = oracle.combine(ys, w_t, pos, len(tok), wl.D)
    assert_close("out vs oracle (sampled tokens)",
                 to_host(fused.out[torch.from_numpy(tok).long().cuda()]), ref)

"""GPU check of block.HostPipeline, the block API that takes per-step
activations from pinned host memory and overlaps the copies with the kernels
(the path bench.py's end-to-end number runs).

Each step of the pipeline must give exactly what the plain device-resident
sequence (MoEBlock.forward/backward on the default stream) gives for the same
inputs: the same kernels run on the same data, only on other streams and
interleaved with copies.  Three steps with different inputs catch a step
that reads another step's slot, or a download that reads a buffer before its
step wrote it.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.block import HostPipeline, MoEBlock
from mixture_experts_ffn_histogram_gb300.inputs import custom, make_inputs
from tests.gpu_common import assert_exact, need_gpu, to_host

pytestmark = pytest.mark.gpu

CASES = {
    "train_softmax": dict(T=300, D=256, E=8, K=2, F=192, train=True),
    "train_given": dict(T=260, D=192, E=12, K=4, F=128, score_mode=2, zipf_s=1.2, train=True),
    "forward_only": dict(T=200, D=320, E=6, K=2, F=256, train=False),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_host_pipeline_matches_device_sequence(case):
    need_gpu()
    kw = CASES[case]
    train = kw["train"]
    steps = [make_inputs(custom(case, seed=s, **kw), "cuda", with_grad=train) for s in (1, 2, 3)]
    wi, wo, bias = steps[0]["wi"], steps[0]["wo"], steps[0]["bias"]
    T, D, E, K, F = (kw[k] for k in ("T", "D", "E", "K", "F"))
    mode = kw.get("score_mode", B.SCORE_SOFTMAX_TOPK)

    # reference: the plain sequence, one step after the other
    ref = MoEBlock(T, D, E, K, F, mode, train=train)
    want = []
    for inp in steps:
        ref.forward(inp["x"], wi, wo, logits=inp["logits"], bias=bias, ids=inp["ids"],
                    w=inp["w"])
        o = to_host(ref.out)
        dx = None
        if train:
            ref.backward(inp["dy"], wi, wo)
            dx = to_host(ref.dx)
        want.append((o, dx))
    torch.cuda.synchronize()
    assert int(ref.status.item()) == 0

    blk = MoEBlock(T, D, E, K, F, mode, train=train)
    pipe = HostPipeline(blk, wi, wo, bias)
    pin = lambda t: None if t is None else t.cpu().pin_memory()  # noqa: E731
    outs = []
    for inp in steps:
        out_h = torch.empty((T, D), dtype=torch.bfloat16).pin_memory()
        dx_h = torch.empty((T, D), dtype=torch.bfloat16).pin_memory() if train else None
        pipe.step(pin(inp["x"]), out_h, dy_h=pin(inp.get("dy")), dx_h=dx_h,
                  logits_h=pin(inp["logits"]), ids_h=pin(inp["ids"]), w_h=pin(inp["w"]))
        outs.append((out_h, dx_h))
    pipe.synchronize()
    assert int(blk.status.item()) == 0
    for i, ((o_h, dx_h), (o, dx)) in enumerate(zip(outs, want)):
        assert_exact(f"step {i} out", to_host(o_h), o)
        if train:
            assert_exact(f"step {i} dx", to_host(dx_h), dx)
    # the steps' inputs differ, so their outputs must too
    assert not np.array_equal(want[0][0], want[1][0])

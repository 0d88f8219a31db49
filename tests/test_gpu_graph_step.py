"""GPU check of block.GraphStep: a block step captured into a CUDA graph and
replayed must give exactly what the same calls give when launched one by
one, and must read the input tensors' current contents at every replay (the
graph holds their addresses, not their values)."""
import pytest
import torch

from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.block import GraphStep, MoEBlock
from mixture_experts_ffn_histogram_gb300.inputs import custom, make_inputs
from tests.gpu_common import assert_exact, need_gpu, to_host

pytestmark = pytest.mark.gpu

CASES = {
    "train_bias": dict(T=300, D=256, E=8, K=2, F=192, bias_std=0.5, train=True),
    "train_pairs": dict(T=512, D=256, E=4, K=2, F=128, train=True),   # 256 rows per group: pairs
    "forward_given": dict(T=260, D=192, E=12, K=4, F=128, score_mode=2, zipf_s=1.2, train=False),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_graph_replay_matches_eager(case):
    need_gpu()
    kw = CASES[case]
    train = kw["train"]
    T, D, E, K, F = (kw[k] for k in ("T", "D", "E", "K", "F"))
    mode = kw.get("score_mode", B.SCORE_SOFTMAX_TOPK)
    draws = [make_inputs(custom(case, seed=s, **kw), "cuda", with_grad=train) for s in (1, 2)]
    wi, wo, bias = draws[0]["wi"], draws[0]["wo"], draws[0]["bias"]

    def live(name):  # the tensors the graph reads; refilled in place before each replay
        t = draws[0].get(name)
        return None if t is None else t.clone()

    x, logits, ids, w, dy = (live(n) for n in ("x", "logits", "ids", "w", "dy"))
    blk = MoEBlock(T, D, E, K, F, mode, train=train)
    g = GraphStep(blk, x, wi, wo, logits=logits, bias=bias, ids=ids, w=w, dy=dy)

    ref = MoEBlock(T, D, E, K, F, mode, train=train)
    for inp in draws:
        for dst, name in ((x, "x"), (logits, "logits"), (ids, "ids"), (w, "w"), (dy, "dy")):
            if dst is not None:
                dst.copy_(inp[name])
        g.replay()
        ref.forward(inp["x"], wi, wo, logits=inp["logits"], bias=bias, ids=inp["ids"], w=inp["w"])
        if train:
            ref.backward(inp["dy"], wi, wo)
        torch.cuda.synchronize()
        assert int(blk.status.item()) == 0 and int(ref.status.item()) == 0
        assert_exact("out", to_host(blk.out), to_host(ref.out))
        if train:
            for name in ("dx", "dwi", "dwo", "dw"):
                assert_exact(name, to_host(getattr(blk, name)), to_host(getattr(ref, name)))

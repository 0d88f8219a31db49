"""The routing/histogram call that allocates nothing.

moe_route_histogram_noalloc serves callers that cannot allocate device
memory (code inside another framework's operator or plugin that only gets
the buffers its planner sized, or latency-critical code that must not call
cudaMalloc).  Its scratch is a fixed 1 MiB array inside the library that
every call shares.  These checks call it through the C ABI twice in a row
(and once more after a call with other sizes, so that leftover scratch from
an earlier call would show) and compare every output with the workspace
entry point, moe_route_histogram: integer outputs bit-exact, the routing
weights within the tolerance the parity tests use.  This file is collected
last and also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_histogram_gb300 import binding as B
from mixture_experts_ffn_histogram_gb300.inputs import custom, make_inputs
from tests.gpu_common import assert_close, assert_exact, need_gpu, to_host

pytestmark = pytest.mark.gpu


def _buffers(wl):
    T, E, K = wl.T, wl.E, wl.K
    dev = "cuda"
    return dict(
        ids=torch.full((T, K), -5, dtype=torch.int32, device=dev),
        w=torch.full((T, K), -5.0, dtype=torch.float32, device=dev),
        gs=torch.full((E,), -5, dtype=torch.int32, device=dev),
        off=torch.full((E + 1,), -5, dtype=torch.int32, device=dev),
        pos=torch.full((T, K), -5, dtype=torch.int32, device=dev),
        row_src=torch.full((T * K,), -5, dtype=torch.int32, device=dev),
        st=torch.zeros(1, dtype=torch.int32, device=dev),
    )


def _route(wl, inp, noalloc):
    d = B.dims(wl.T, wl.D, wl.E, wl.K, wl.F)
    b = _buffers(wl)
    if wl.score_mode == B.SCORE_GIVEN:
        b["ids"].copy_(inp["ids"])
        b["w"].copy_(inp["w"])
    args = (inp["logits"], inp["bias"], wl.score_mode, b["ids"], b["w"], b["gs"], b["off"], b["pos"],
            b["row_src"], b["st"])
    if noalloc:
        B.moe_route_histogram_noalloc(*args, d)
    else:
        ws = torch.empty(B.moe_workspace_bytes(d), dtype=torch.uint8, device="cuda")
        B.moe_route_histogram(*args, ws, d)
    torch.cuda.synchronize()
    return {k: to_host(v) for k, v in b.items()}


WORKLOADS = [
    # many chunks and experts: 2*ceil(3000/256)*96 = 2304 int32 of scratch
    custom("noalloc_a", T=3000, D=64, E=96, K=6, F=64, bias_std=0.5),
    # fewer experts and chunks, sigmoid weights: leftovers from the call above would show
    custom("noalloc_b", T=1100, D=64, E=40, K=4, F=64, score_mode=B.SCORE_SIGMOID_NORM, seed=3),
    # given routing with skewed ids
    custom("noalloc_c", T=777, D=64, E=24, K=3, F=64, score_mode=B.SCORE_GIVEN, zipf_s=1.2, seed=4),
]


def test_noalloc_matches_workspace_call_on_calls_in_a_row():
    need_gpu()
    runs = [WORKLOADS[0], WORKLOADS[1], WORKLOADS[2], WORKLOADS[0]]
    for wl in runs:
        inp = make_inputs(wl, "cuda", with_grad=False)
        want = _route(wl, inp, noalloc=False)
        got = _route(wl, inp, noalloc=True)
        assert got["st"][0] == 0 and want["st"][0] == 0
        for name in ("ids", "gs", "off", "pos", "row_src"):
            assert_exact(f"{wl.name}: {name}", got[name], want[name])
        assert_close(f"{wl.name}: w", got["w"], want["w"], bf16=False)
        assert int(got["gs"].sum()) == wl.T * wl.K


def test_noalloc_rejects_sizes_beyond_its_scratch():
    need_gpu()
    # 2 * ceil(262144/256) * 1024 = 2097152 int32 > 262144
    d = B.dims(262144, 64, 1024, 8, 64)
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as e:
        B.moe_route_histogram_noalloc(dummy, None, B.SCORE_SOFTMAX_TOPK, dummy, dummy, dummy, dummy,
                                      dummy, dummy, None, d)
    assert e.value.status == B.MOE_ERR_UNSUPPORTED
    assert "fixed scratch" in str(e.value)

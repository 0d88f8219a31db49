"""Host-side checks of the block API that need no GPU: a weight whose shape
or dtype differs from the block's dims is rejected before any launch (the
library's tensor maps are built from the dims, so such a weight would be read,
and its gradient written, out of bounds)."""
import pytest
import torch

from mixture_experts_ffn_histogram_gb300.block import MoEBlock

T, D, E, K, F = 16, 128, 4, 2, 64


@pytest.fixture(scope="module")
def blk():
    return MoEBlock(T, D, E, K, F, train=True, device="cpu")


def _w(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


@pytest.mark.parametrize("wi,wo", [
    (_w(E, D, F), _w(E, F, D)),                      # wi without its up half
    (_w(E, D, 2 * F), _w(E, D, F)),                  # wo transposed
    (_w(E - 1, D, 2 * F), _w(E, F, D)),              # too few experts
    (_w(E, D, 2 * F, dtype=torch.float32), _w(E, F, D)),
    ([_w(2, D, 2 * F), _w(2, D, F)], _w(E, F, D)),   # a split part of the wrong width
    ([_w(2, D, 2 * F), _w(1, D, 2 * F)], _w(E, F, D)),  # parts covering 3 of 4 experts
    ([_w(2, D, 2 * F), _w(2, D, 2 * F, dtype=torch.float16)], _w(E, F, D)),
])
def test_mis_shaped_weights_are_rejected_before_any_launch(blk, wi, wo):
    x = _w(T, D)
    with pytest.raises(ValueError):
        blk.forward(x, wi, wo, logits=torch.zeros(T, E))
    with pytest.raises(ValueError):
        blk.backward(x, wi, wo)


def test_well_shaped_weights_pass_the_check(blk):
    blk._check_weights(_w(E, D, 2 * F), _w(E, F, D))
    blk._check_weights([_w(1, D, 2 * F), _w(3, D, 2 * F)], _w(E, F, D))

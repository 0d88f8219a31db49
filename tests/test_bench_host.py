"""Host-side logic of bench.py that needs no GPU: which workloads get L2
flushed between timed steps, and the accounting that decides whether a GEMM
is held to the tensor or the HBM peak."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mixture_experts_ffn_histogram_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402


def test_footprint_counts_only_tensors_and_decides_the_flush():
    tiny = make_inputs(WORKLOADS["tiny_fwd"], "cpu", with_grad=False)
    fp = bench.input_footprint(tiny)
    wl = WORKLOADS["tiny_fwd"]
    # x + logits + wi + wo (no bias, no ids/w for softmax routing)
    want = wl.T * wl.D * 2 + wl.T * wl.E * 4 + wl.E * wl.D * 2 * wl.F * 2 + wl.E * wl.F * wl.D * 2
    assert fp == want
    assert fp < bench.L2_BYTES            # small enough to sit in L2: flushed


@pytest.mark.parametrize("name,kernel,bound", [
    ("long_seq_train", "fc1", "tensor"),          # 2048 rows per expert
    ("token_sweep_T1024", "fc1", "hbm"),          # 64 rows per expert: weight streaming
    ("large_expert_train", "fc1_drhs", "hbm"),    # writes 15 GB of dwi
])
def test_binding_resource_of_a_gemm(name, kernel, bound):
    wl = WORKLOADS[name]
    pk = {"hbm": 6791.7, "bf16_sustained": 1698.7}
    t_bytes = bench.gemm_bytes(kernel, wl.R, wl.D, wl.E, wl.F, wl.train) / (pk["hbm"] * 1e9)
    t_flops = bench.gemm_flops(kernel, wl.R, wl.D, wl.F) / (pk["bf16_sustained"] * 1e12)
    assert ("hbm" if t_bytes > t_flops else "tensor") == bound


def test_mx_algorithmic_bytes_match_the_buffers():
    """The MX steps' algorithmic bytes are the sizes of what they must read
    and write, as the library reports its MX buffers (codes plus one scale
    byte per 32 elements; the tile-blocked scale buffers are upper bounds, so
    their 1/32 counts are compared against the exact per-row figure)."""
    wl = WORKLOADS["long_seq_train"]
    T, D, E, K, F, R = wl.T, wl.D, wl.E, wl.K, wl.F, wl.R
    assert bench.mx_bytes("permute_quantize", T, D, E, K, F) == \
        2 * T * D + R * D + R * D // 32 + 4 * T * K
    # FC1 reads xq + scales and wi codes + scales, writes hq + scales
    assert bench.mx_bytes("fc1", T, D, E, K, F) == \
        (R * D + R * D // 32) + (E * 2 * F * D + E * 2 * F * D // 32) + (R * F + R * F // 32)
    # FC2 reads hq + scales and wo codes + scales, writes bf16 ys
    assert bench.mx_bytes("fc2", T, D, E, K, F) == \
        (R * F + R * F // 32) + (E * D * F + E * D * F // 32) + 2 * R * D

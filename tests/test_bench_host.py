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
    and write, taken from the library's own MX buffer sizes (moe_mx_bytes, a
    host-only call): the e4m3 code buffers exactly, plus one scale byte per 32
    codes, which the tile-blocked scale buffers must be able to hold."""
    from mixture_experts_ffn_histogram_gb300 import _build
    from mixture_experts_ffn_histogram_gb300 import binding as B
    _build.build()
    wl = WORKLOADS["long_seq_train"]
    T, D, E, K, F = wl.T, wl.D, wl.E, wl.K, wl.F
    d = B.dims(T, D, E, K, F)
    size = {w: B.moe_mx_bytes(d, w) for w in (B.MX_XQ, B.MX_XSC, B.MX_WIQ, B.MX_WISC, B.MX_WOQ,
                                               B.MX_WOSC, B.MX_HQ, B.MX_HSC)}
    for codes, scales in ((B.MX_XQ, B.MX_XSC), (B.MX_WIQ, B.MX_WISC), (B.MX_WOQ, B.MX_WOSC),
                          (B.MX_HQ, B.MX_HSC)):
        assert 0 < size[codes] // 32 <= size[scales]

    def mx(codes):
        return size[codes] + size[codes] // 32

    # permute + quantize reads bf16 x and pos, writes the token codes and scales
    assert bench.mx_bytes("permute_quantize", T, D, E, K, F) == 2 * T * D + mx(B.MX_XQ) + 4 * T * K
    # FC1 reads the token and wi codes (with scales), writes h's codes and scales
    assert bench.mx_bytes("fc1", T, D, E, K, F) == mx(B.MX_XQ) + mx(B.MX_WIQ) + mx(B.MX_HQ)
    # FC2 reads h's and wo's codes (with scales), writes bf16 ys
    assert bench.mx_bytes("fc2", T, D, E, K, F) == mx(B.MX_HQ) + mx(B.MX_WOQ) + 2 * wl.R * D


def test_tensor_peak_follows_the_sampled_clock():
    pk = {"bf16": 1924.2, "bf16_sustained": 1725.0, "sm_max_mhz": 2070.0, "source": "measured"}
    assert bench.tensor_peak(pk, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})[0] == 1924.2
    half = bench.tensor_peak(pk, {"sm_mhz": 1035.0, "sm_max_mhz": 2070.0})[0]
    assert abs(half - 1924.2 / 2) < 1e-9
    # never above the burst figure, and the sustained one without a clock record
    assert bench.tensor_peak(pk, {"sm_mhz": 2100.0, "sm_max_mhz": 2070.0})[0] == 1924.2
    assert bench.tensor_peak(pk, {"sm_mhz": None})[0] == 1725.0


def test_block_roofline_is_the_sum_of_kernel_rooflines():
    wl = WORKLOADS["long_seq_train"]
    names = ["route", "permute", "fc1", "fc2", "combine"]
    times = {n: [1e-3, 1e-3] for n in names}
    pk = {"hbm": 6688.8}
    kern, roof = bench.kernel_table(wl, names, times, True, pk, 1924.2)
    assert abs(roof * 1e6 - sum(k["roofline_us"] for k in kern.values())) < 1e-6
    fl = bench.gemm_flops("fc1", wl.R, wl.D, wl.F)
    assert kern["fc1"]["bound"] == "tensor"
    assert abs(kern["fc1"]["roofline_us"] - fl / 1924.2e12 * 1e6) < 1e-6
    assert abs(kern["permute"]["roofline_us"] -
               bench.hbm_bytes("permute", wl.T, wl.D, wl.E, wl.K, wl.F) / 6688.8e9 * 1e6) < 1e-6


def test_mx_train_work_with_bf16_weight_gradients():
    """The MX training step with bf16 weight gradients keeps the same six
    GEMMs (two of them on the bf16 tensor peak), drops the four launches
    that quantize along tokens and adds the bf16 permute of xs."""
    wl = WORKLOADS["long_seq_train"]
    mx = bench.mx_train_work(wl)
    bw = bench.mx_train_work(wl, "bf16")
    names_mx = [n for n, _, _ in mx]
    names_bw = [n for n, _, _ in bw]
    assert len(bw) == len(mx) - 3
    assert not any("tokens" in n for n in names_bw)
    assert "permute_xs_bf16" in names_bw and "permute_xs_bf16" not in names_mx
    flops = lambda w: sum(a for _, k, a in w if k.startswith("tensor"))  # noqa: E731
    assert flops(bw) == flops(mx)
    assert [n for n, k, _ in bw if k == "tensor_bf16"] == ["fc2_wgrad_bf16", "fc1_wgrad_bf16"]
    assert dict((n, a) for n, _, a in bw)["fc1_wgrad_bf16"] == dict(
        (n, a) for n, _, a in mx)["fc1_wgrad"]

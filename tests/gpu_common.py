"""Helpers shared by the GPU parity tests (marked ``gpu``)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.refs import bits_to_f64

RTOL = 2e-2   # |gpu - ref| <= RTOL*|ref| + ATOL per element
ATOL = 2e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_histogram_gb300 import _build
    _build.build()


def to_dev(a, dtype=None):
    """numpy (uint16 = bf16 bits, int32, float32) -> CUDA tensor."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t):
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def assert_exact(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{name}: shape {got.shape} vs {want.shape}"
    bad = np.flatnonzero(got.ravel() != want.ravel())
    assert bad.size == 0, (f"{name}: {bad.size} of {got.size} elements differ; first at flat "
                           f"{bad[:5].tolist()}: got {got.ravel()[bad[:5]].tolist()} "
                           f"want {want.ravel()[bad[:5]].tolist()}")


def assert_close(name, got, want, rtol=RTOL, atol=ATOL, bf16=True):
    g = bits_to_f64(got) if bf16 else np.asarray(got, dtype=np.float64)
    w = bits_to_f64(want) if bf16 else np.asarray(want, dtype=np.float64)
    assert g.shape == w.shape, f"{name}: shape {g.shape} vs {w.shape}"
    if g.size == 0:
        return
    err = np.abs(g - w)
    lim = rtol * np.abs(w) + atol
    bad = np.flatnonzero((err > lim).ravel() | ~np.isfinite(g).ravel())
    if bad.size:
        idx = np.unravel_index(bad[:5], g.shape)
        raise AssertionError(
            f"{name}: {bad.size} of {g.size} outside tol (rtol={rtol}, atol={atol}); max err "
            f"{np.nanmax(err):.4g}; first at {list(zip(*[i.tolist() for i in idx]))}: got "
            f"{g.ravel()[bad[:5]].tolist()} want {w.ravel()[bad[:5]].tolist()}")

"""Independent float64 references used to pin the oracle.

Nothing here calls the oracle or the CUDA path.  The central reference is the
brute-force per-token dense loop over each token's top-k experts: for token t,
out[t] = sum_k w[t,k] * (silu(x_t wi_g[e]) * (x_t wi_u[e])) wo[e] with
e = ids[t,k], computed in float64 with torch (so that torch.autograd gives
every gradient), with no sort, no permutation and no grouping.
"""
from __future__ import annotations

import numpy as np
import torch


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits_torch(a) -> np.ndarray:
    """RNE rounding to bf16 with torch's own conversion (a library routine)."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def dense_block(x, wi, wo, ids, w):
    """Per-token dense loop, float64 torch tensors.  x [T,D], wi [E,D,2F],
    wo [E,F,D], ids [T,K] (long), w [T,K].  Returns out [T,D]."""
    T, D = x.shape
    F = wo.shape[1]
    out = torch.zeros(T, D, dtype=torch.float64)
    rows = []
    for t in range(T):
        acc = torch.zeros(D, dtype=torch.float64)
        for k in range(ids.shape[1]):
            e = int(ids[t, k])
            a = x[t] @ wi[e]
            h = torch.nn.functional.silu(a[:F]) * a[F:]
            acc = acc + w[t, k] * (h @ wo[e])
        rows.append(acc)
    if rows:
        out = torch.stack(rows)
    return out


def close(a, b, rtol, atol):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return bool(np.all(np.abs(a - b) <= rtol * np.abs(b) + atol))


def max_excess(a, b, rtol, atol):
    """max over elements of |a-b| - (rtol*|b| + atol); <= 0 means within tolerance."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b) - (rtol * np.abs(b) + atol)))

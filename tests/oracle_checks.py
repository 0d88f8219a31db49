"""Pins of the CPU oracle against things other than itself.

Each ``check_*`` raises AssertionError when the oracle disagrees with a
library routine (numpy sort/bincount/matmul, torch's bf16 conversion, torch
autograd), a brute-force float64 computation (the per-token dense loop over
each token's top-k experts), a closed form or an invariant.  The checks take
the oracle module as an argument so that the mutation test can run the same
battery against deliberately broken builds of the oracle.

Tolerances: bf16 has an 8-bit significand (7 stored bits), so one rounding
costs at most 2^-8 relative; fp32 accumulation adds ~1e-6 relative of the sum of |terms|.
"""
from __future__ import annotations

import numpy as np
import torch

from tests.refs import bits_to_f64, dense_block, f32_to_bf16_bits_torch, max_excess

U = 2.0 ** -7      # one bf16 ulp relative to a value at the bottom of its binade


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _bf16(rng, shape, std=1.0):
    return f32_to_bf16_bits_torch((rng.standard_normal(shape) * std).astype(np.float32))


def _groups_from_ids(ids, E):
    """Reference histogram by library routines: counts, offsets, stable order."""
    flat = ids.ravel()
    gs = np.bincount(flat, minlength=E).astype(np.int32)
    off = np.concatenate([[0], np.cumsum(gs)]).astype(np.int32)
    row_src = np.argsort(flat, kind="stable").astype(np.int32)
    return gs, off, row_src


def _random_grouped_rows(rng, R, E, empty=(1,)):
    """Sorted expert id per row with some experts empty; returns offsets."""
    choices = [e for e in range(E) if e not in empty]
    ids = np.sort(rng.choice(choices, size=R))
    gs = np.bincount(ids, minlength=E)
    return np.concatenate([[0], np.cumsum(gs)]).astype(np.int32), ids


# --------------------------------------------------------------------- bf16
def check_bf16_rounding(orc):
    rng = _rng(1)
    vals = [rng.standard_normal(2000).astype(np.float32) * s for s in (1e-3, 1.0, 1e4, 1e30)]
    # exact halfway cases: low 16 bits = 0x8000 with even and odd kept lsb
    halves = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x40490000 | 0x8000,
                       0x7F7F8000, 0x00008000, 0x00018000], dtype=np.uint32).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, 1e-40, -1e-40], np.float32)
    a = np.concatenate(vals + [halves, special])
    got = orc.f32_to_bf16(a)
    want = f32_to_bf16_bits_torch(a)
    assert np.array_equal(got, want), "f32->bf16 rounding differs from torch's RNE conversion"
    back = orc.bf16_to_f32(want)
    assert np.array_equal(back, torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy())


# -------------------------------------------------------------------- route
def _ref_topk(s, K):
    T, E = s.shape
    eidx = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((eidx, -s.astype(np.float64)), axis=-1)   # score desc, id asc
    return order[:, :K].astype(np.int32)


def check_route(orc):
    rng = _rng(2)
    T, E, K = 48, 12, 4
    cases = [
        (rng.standard_normal((T, E)).astype(np.float32), None),
        (rng.integers(0, 3, (T, E)).astype(np.float32), None),                 # many ties
        (rng.standard_normal((T, E)).astype(np.float32),
         (rng.standard_normal(E) * 0.5).astype(np.float32)),
    ]
    for mode in (orc.SOFTMAX_TOPK, orc.SIGMOID_NORM):
        for logits, bias in cases:
            ids, w = orc.route(logits, bias, mode, T, E, K)
            s = logits + bias[None, :] if bias is not None else logits   # one fp32 add
            want = _ref_topk(s, K)
            assert np.array_equal(ids, want), f"top-k ids differ (mode {mode})"
            sel = np.take_along_axis(s.astype(np.float64), want, axis=1)
            if mode == orc.SOFTMAX_TOPK:
                ex = np.exp(sel - sel.max(axis=1, keepdims=True))
            else:
                ex = 1.0 / (1.0 + np.exp(-sel))
            wref = ex / ex.sum(axis=1, keepdims=True)
            assert max_excess(w, wref, 2e-6, 1e-7) <= 0, f"routing weights differ (mode {mode})"
    # K = 1: a single weight of exactly 1; K = E: every expert, sorted
    lg = rng.standard_normal((5, 6)).astype(np.float32)
    ids, w = orc.route(lg, None, orc.SOFTMAX_TOPK, 5, 6, 1)
    assert np.array_equal(ids[:, 0], lg.argmax(1)) and np.all(w == 1.0)
    ids, w = orc.route(lg, None, orc.SOFTMAX_TOPK, 5, 6, 6)
    assert np.array_equal(ids, _ref_topk(lg, 6))
    # all-equal logits: ids 0..K-1 and uniform weights
    ids, w = orc.route(np.zeros((3, 8), np.float32), None, orc.SOFTMAX_TOPK, 3, 8, 4)
    assert np.array_equal(ids, np.tile(np.arange(4), (3, 1))) and np.allclose(w, 0.25, atol=0)


# ---------------------------------------------------------------- histogram
def check_histogram(orc):
    rng = _rng(3)
    T, K, E = 40, 3, 10
    for ids in (rng.integers(0, 8, (T, K)).astype(np.int32),                  # 8, 9 empty
                np.stack([rng.permutation(8)[:K] for _ in range(T)]).astype(np.int32),
                np.full((T, K), 4, np.int32)):                                  # one expert
        gs, off, pos, row_src, bad = orc.histogram(ids, E)
        gref, oref, rref = _groups_from_ids(ids, E)
        assert bad == 0
        assert np.array_equal(gs, gref) and np.array_equal(off, oref)
        assert np.array_equal(row_src, rref), "row_src is not the stable expert order"
        R = T * K
        assert gs.sum() == R
        assert np.array_equal(np.sort(pos.ravel()), np.arange(R)), "pos is not a bijection"
        assert np.array_equal(row_src[pos.ravel()], np.arange(R)), "row_src o pos != id"
        flat = ids.ravel()
        for e in range(E):
            seg = row_src[off[e]:off[e + 1]]
            assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    bad_ids = rng.integers(0, E, (T, K)).astype(np.int32)
    bad_ids[3, 1], bad_ids[7, 0] = -1, E
    gs, off, pos, row_src, bad = orc.histogram(bad_ids, E)
    assert bad == 2 and pos[3, 1] == -1 and pos[7, 0] == -1 and gs.sum() == T * K - 2
    assert np.all(row_src[T * K - 2:] == -1)


# ------------------------------------------------------- permute / combine
def check_permute_combine(orc):
    rng = _rng(4)
    T, D, E, K = 24, 40, 6, 4
    x = _bf16(rng, (T, D))
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    _, _, pos, row_src, _ = orc.histogram(ids, E)
    xs = orc.permute(x, pos)
    assert np.array_equal(xs, x[row_src // K]), "permute is not x[row_src // K]"
    # combine with unit weights inverts permute up to the factor K (a power of two: exact)
    back = orc.combine(xs, np.ones((T, K), np.float32), pos, T, D)
    assert np.array_equal(back, f32_to_bf16_bits_torch(bits_to_f64(x).astype(np.float32) * K))
    onehot = np.zeros((T, K), np.float32)
    onehot[np.arange(T), rng.integers(0, K, T)] = 1.0
    assert np.array_equal(orc.combine(xs, onehot, pos, T, D), x)
    assert np.array_equal(orc.permute_bwd(xs, pos, T, D), back)
    # weighted combine against float64
    ys = _bf16(rng, (T * K, D))
    w = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
    out = orc.combine(ys, w, pos, T, D)
    y64 = bits_to_f64(ys)
    ref = np.einsum("tk,tkd->td", w.astype(np.float64), y64[pos])
    assert max_excess(bits_to_f64(out), ref, U / 2 + 1e-6, 1e-6) <= 0, "combine differs"
    # dropped slots (pos = -1) contribute nothing
    pos2 = pos.copy()
    pos2[0, 0] = -1
    ref2 = ref.copy()
    ref2[0] -= w[0, 0] * y64[pos[0, 0]]
    assert max_excess(bits_to_f64(orc.combine(ys, w, pos2, T, D)), ref2, U / 2 + 1e-6, 1e-6) <= 0


def check_combine_bwd(orc):
    rng = _rng(5)
    T, D, E, K = 20, 48, 5, 3
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    _, _, pos, _, _ = orc.histogram(ids, E)
    ys = _bf16(rng, (T * K, D))
    dout = _bf16(rng, (T, D))
    w = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
    dys, dw = orc.combine_bwd(dout, ys, w, pos)
    # autograd of out = sum_k w_k ys[pos_k] against L = <out, dout>
    ys_t = torch.tensor(bits_to_f64(ys), requires_grad=True)
    w_t = torch.tensor(w.astype(np.float64), requires_grad=True)
    out = (w_t[:, :, None] * ys_t[torch.from_numpy(pos).long()]).sum(1)
    (out * torch.tensor(bits_to_f64(dout))).sum().backward()
    assert max_excess(bits_to_f64(dys), ys_t.grad.numpy(), U / 2 + 1e-7, 0) <= 0, "dys differs"
    scale = np.abs(bits_to_f64(dout)).sum(1, keepdims=True) * np.abs(bits_to_f64(ys)).max()
    assert max_excess(dw, w_t.grad.numpy(), 0, 1e-6 * scale) <= 0, "dw differs"


# ------------------------------------------------------------------ GEMMs
def _silu(v):
    return v / (1.0 + np.exp(-v))


def check_fc1_fc2(orc):
    rng = _rng(6)
    R, D, E, F = 70, 48, 5, 40
    off, rid = _random_grouped_rows(rng, R, E, empty=(1,))
    xs = _bf16(rng, (R, D))
    wi = _bf16(rng, (E, D, 2 * F), 0.2)
    wo = _bf16(rng, (E, F, D), 0.2)
    h, z = orc.fc1_swiglu(xs, wi, off)
    a = np.einsum("rd,rdn->rn", bits_to_f64(xs), bits_to_f64(wi)[rid])
    atol = 1e-5 * np.abs(a).max()
    assert max_excess(bits_to_f64(z), a, U / 2 + 1e-6, atol) <= 0, "z differs from xs @ wi[e]"
    href = _silu(a[:, :F]) * a[:, F:]
    assert max_excess(bits_to_f64(h), href, U / 2 + 1e-5, atol) <= 0, "h differs from SwiGLU"
    h2, z2 = orc.fc1_swiglu(xs, wi, off, want_z=False)
    assert z2 is None and np.array_equal(h, h2)
    ys = orc.fc2(h, wo, off)
    yref = np.einsum("rf,rfd->rd", bits_to_f64(h), bits_to_f64(wo)[rid])
    assert max_excess(bits_to_f64(ys), yref, U / 2 + 1e-6, 1e-5 * np.abs(yref).max()) <= 0, \
        "ys differs from h @ wo[e]"


def check_swiglu_closed_forms(orc):
    # E=1, one row per special (g, u) pair, xs = unit vectors, wi chosen so a = (g, u)
    g = np.array([0.0, 1.0, -1.0, 8.0, -8.0, 0.5], np.float32)
    u = np.array([3.0, 1.0, 2.0, 0.25, 4.0, 0.0], np.float32)
    n = len(g)
    D, F = n, n
    xs = f32_to_bf16_bits_torch(np.eye(n, dtype=np.float32))
    wi = np.zeros((1, D, 2 * F), np.float32)
    wi[0, np.arange(n), np.arange(n)] = g
    wi[0, np.arange(n), F + np.arange(n)] = u
    h, _ = orc.fc1_swiglu(xs, f32_to_bf16_bits_torch(wi), np.array([0, n], np.int32))
    hd = np.diag(bits_to_f64(h))
    want = np.array([0.0, 0.7310585786300049, -1.0 * 0.2689414213699951 * 2.0,
                     8.0 / (1.0 + np.exp(-8.0)) * 0.25, -8.0 / (1.0 + np.exp(8.0)) * 4.0, 0.0])
    assert max_excess(hd, want, U / 2, 1e-12) <= 0, "SwiGLU closed forms"


def check_dense_special_case(orc):
    """E=1, K=1, w=1: the block is a dense SwiGLU MLP (torch.nn.functional)."""
    rng = _rng(7)
    T, D, F = 16, 32, 24
    x = _bf16(rng, (T, D))
    wi = _bf16(rng, (1, D, 2 * F), 0.2)
    wo = _bf16(rng, (1, F, D), 0.2)
    ids = np.zeros((T, 1), np.int32)
    _, off, pos, _, _ = orc.histogram(ids, 1)
    xs = orc.permute(x, pos)
    h, _ = orc.fc1_swiglu(xs, wi, off)
    ys = orc.fc2(h, wo, off)
    out = orc.combine(ys, np.ones((T, 1), np.float32), pos, T, D)
    X = torch.tensor(bits_to_f64(x))
    Wg = torch.tensor(bits_to_f64(wi[0, :, :F]).T)
    Wu = torch.tensor(bits_to_f64(wi[0, :, F:]).T)
    Wo = torch.tensor(bits_to_f64(wo[0]).T)
    ref = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(X, Wg)) * torch.nn.functional.linear(X, Wu), Wo)
    ref = ref.numpy()
    assert max_excess(bits_to_f64(out), ref, 3 * U, 2e-2 * np.abs(ref).max()) <= 0, "dense MLP"


def check_gemm_backward(orc):
    rng = _rng(8)
    R, D, E, F = 60, 40, 4, 24
    off, rid = _random_grouped_rows(rng, R, E, empty=(2,))
    xs = _bf16(rng, (R, D))
    wi = _bf16(rng, (E, D, 2 * F), 0.2)
    wo = _bf16(rng, (E, F, D), 0.2)
    dys = _bf16(rng, (R, D))
    h, z = orc.fc1_swiglu(xs, wi, off)
    # FC2 backward, fused SwiGLU: autograd through h(a) = silu(a_g) a_u from a = z
    a_t = torch.tensor(bits_to_f64(z), requires_grad=True)
    hh = torch.nn.functional.silu(a_t[:, :F]) * a_t[:, F:]
    wo_r = torch.tensor(bits_to_f64(wo))[torch.from_numpy(rid).long()]
    L = (torch.einsum("rf,rfd->rd", hh, wo_r) * torch.tensor(bits_to_f64(dys))).sum()
    L.backward()
    dz_ref = a_t.grad.numpy()
    dz, dwo = orc.fc2_bwd(dys, h, wo, z, off)
    sc = np.abs(dz_ref).max()
    assert max_excess(bits_to_f64(dz), dz_ref, U / 2 + 1e-4, 1e-5 * sc) <= 0, "fused dz differs"
    dwo_ref = np.zeros((E, F, D))
    for e in range(E):
        dwo_ref[e] = bits_to_f64(h[off[e]:off[e + 1]]).T @ bits_to_f64(dys[off[e]:off[e + 1]])
    assert max_excess(bits_to_f64(dwo), dwo_ref, U / 2 + 1e-5, 1e-5 * np.abs(dwo_ref).max()) <= 0
    assert np.all(dwo[2] == 0), "empty expert must get a zero gradient"
    # unfused: dh = dys @ wo[e]^T, then the SwiGLU backward from bf16 dh
    dh, dwo2 = orc.fc2_bwd(dys, h, wo, None, off)
    dh_ref = np.einsum("rd,rfd->rf", bits_to_f64(dys), bits_to_f64(wo)[rid])
    assert max_excess(bits_to_f64(dh), dh_ref, U / 2 + 1e-5, 1e-5 * np.abs(dh_ref).max()) <= 0
    assert np.array_equal(dwo, dwo2)
    dz2 = orc.swiglu_bwd(dh, z)
    a2 = torch.tensor(bits_to_f64(z), requires_grad=True)
    (torch.nn.functional.silu(a2[:, :F]) * a2[:, F:] * torch.tensor(bits_to_f64(dh))).sum().backward()
    assert max_excess(bits_to_f64(dz2), a2.grad.numpy(), U / 2 + 1e-5,
                      1e-6 * np.abs(a2.grad.numpy()).max()) <= 0, "SwiGLU backward differs"
    # FC1 backward: dxs = dz @ wi[e]^T, dwi[e] = xs_e^T dz_e
    dxs, dwi = orc.fc1_bwd(dz, xs, wi, off)
    dxs_ref = np.einsum("rn,rdn->rd", bits_to_f64(dz), bits_to_f64(wi)[rid])
    assert max_excess(bits_to_f64(dxs), dxs_ref, U / 2 + 1e-5, 1e-5 * np.abs(dxs_ref).max()) <= 0
    dwi_ref = np.zeros((E, D, 2 * F))
    for e in range(E):
        dwi_ref[e] = bits_to_f64(xs[off[e]:off[e + 1]]).T @ bits_to_f64(dz[off[e]:off[e + 1]])
    assert max_excess(bits_to_f64(dwi), dwi_ref, U / 2 + 1e-5, 1e-5 * np.abs(dwi_ref).max()) <= 0
    assert np.all(dwi[2] == 0)


# ----------------------------------------------------- whole block vs dense
def _tiny_block(seed, T=10, D=16, E=4, K=2, F=8, mode=0, bias=False):
    rng = _rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    b = (rng.standard_normal(E) * 0.5).astype(np.float32) if bias else None
    x = _bf16(rng, (T, D))
    wi = _bf16(rng, (E, D, 2 * F), 0.3)
    wo = _bf16(rng, (E, F, D), 0.3)
    dy = _bf16(rng, (T, D))
    return logits, b, x, wi, wo, dy


def _oracle_block(orc, logits, b, x, wi, wo, dy, mode, K):
    T, D = x.shape
    E, F = wo.shape[0], wo.shape[1]
    ids, w = orc.route(logits, b, mode, T, E, K)
    _, off, pos, _, _ = orc.histogram(ids, E)
    xs = orc.permute(x, pos)
    h, z = orc.fc1_swiglu(xs, wi, off)
    ys = orc.fc2(h, wo, off)
    out = orc.combine(ys, w, pos, T, D)
    dys, dw = orc.combine_bwd(dy, ys, w, pos)
    dz, dwo = orc.fc2_bwd(dys, h, wo, z, off)
    dxs, dwi = orc.fc1_bwd(dz, xs, wi, off)
    dx = orc.permute_bwd(dxs, pos, T, D)
    return dict(ids=ids, w=w, out=out, dw=dw, dwo=dwo, dwi=dwi, dx=dx)


def check_block_against_dense(orc):
    for seed, mode, bias in ((9, 0, False), (10, 1, False), (11, 0, True)):
        logits, b, x, wi, wo, dy = _tiny_block(seed, mode=mode, bias=bias)
        K = 2
        o = _oracle_block(orc, logits, b, x, wi, wo, dy, mode, K)
        X = torch.tensor(bits_to_f64(x), requires_grad=True)
        WI = torch.tensor(bits_to_f64(wi), requires_grad=True)
        WO = torch.tensor(bits_to_f64(wo), requires_grad=True)
        W = torch.tensor(o["w"].astype(np.float64), requires_grad=True)
        ref = dense_block(X, WI, WO, torch.from_numpy(o["ids"]), W)
        (ref * torch.tensor(bits_to_f64(dy))).sum().backward()
        r = ref.detach().numpy()
        assert max_excess(bits_to_f64(o["out"]), r, 2e-2, 2e-2 * np.abs(r).max()) <= 0, "out vs dense"
        for name, g in (("dx", X.grad), ("dwi", WI.grad), ("dwo", WO.grad), ("dw", W.grad)):
            got = o[name] if name == "dw" else bits_to_f64(o[name])
            gr = g.numpy()
            assert max_excess(got, gr, 3e-2, 2e-2 * np.abs(gr).max()) <= 0, f"{name} vs autograd"


def check_finite_differences(orc):
    """Directional central differences of the float64 dense loss against the
    oracle's gradients: (L(p + eps v) - L(p - eps v)) / 2eps ~ <grad, v>."""
    logits, b, x, wi, wo, dy = _tiny_block(12)
    K = 2
    o = _oracle_block(orc, logits, b, x, wi, wo, dy, 0, K)
    ids = torch.from_numpy(o["ids"])
    base = dict(x=bits_to_f64(x), wi=bits_to_f64(wi), wo=bits_to_f64(wo), w=o["w"].astype(np.float64))
    dyv = torch.tensor(bits_to_f64(dy))

    def loss(p):
        out = dense_block(torch.tensor(p["x"]), torch.tensor(p["wi"]), torch.tensor(p["wo"]),
                          ids, torch.tensor(p["w"]))
        return float((out * dyv).sum())

    rng = _rng(13)
    grads = dict(x=bits_to_f64(o["dx"]), wi=bits_to_f64(o["dwi"]), wo=bits_to_f64(o["dwo"]), w=o["dw"])
    eps = 1e-3
    for name in ("x", "wi", "wo", "w"):
        v = rng.standard_normal(base[name].shape)
        pp = dict(base)
        pm = dict(base)
        pp[name] = base[name] + eps * v
        pm[name] = base[name] - eps * v
        fd = (loss(pp) - loss(pm)) / (2 * eps)
        an = float((grads[name] * v).sum())
        assert abs(fd - an) <= 2e-2 * abs(fd) + 1e-3 * np.sqrt(np.sum(grads[name] ** 2)), \
            f"finite differences disagree for d{name}: fd={fd} oracle={an}"


# -------------------------------------------------------------------- MXFP8
def _torch_e4m3(values):
    """torch's float32 -> float8_e4m3fn conversion (nearest, ties to even) of
    values already clamped to the finite range; codes as uint8."""
    t = torch.tensor(np.asarray(values, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def check_e4m3_decode(orc):
    """Every code's value equals torch's float8_e4m3fn reading of the same
    byte, and the format's landmarks hold: 1.0 = 0x38, the largest finite
    value 448 = 0x7E, the smallest normal 2^-6 = 0x08, the smallest
    subnormal 2^-9 = 0x01, NaN = 0x7F / 0xFF and no infinities."""
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_to_f64(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan]), \
        "E4M3 decoding differs from torch's float8_e4m3fn"
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6
    assert got[0x01] == 2.0 ** -9 and got[0x07] == 0.875 * 2.0 ** -6 and np.isfinite(got[~nan]).all()


def check_e4m3_encode(orc):
    """Encoding: every finite code round-trips; random values, exact
    midpoints between neighbours and subnormals round like torch's
    conversion (nearest, ties to even); magnitudes beyond 448 saturate."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_to_f64(codes)
    assert np.array_equal(orc.f64_to_e4m3(vals), codes), "finite codes do not round-trip"
    pos = np.sort(vals[(vals > 0)])
    mids = (pos[:-1] + pos[1:]) / 2
    rng = _rng(41)
    rand = np.concatenate([rng.uniform(-448, 448, 3000), rng.uniform(-1, 1, 2000) * 2.0 ** -6,
                           rng.standard_normal(2000)])
    probe = np.concatenate([mids, -mids, rand, mids * (1 + 1e-7), mids * (1 - 1e-7)])
    probe = probe[np.abs(probe) <= 448].astype(np.float32).astype(np.float64)
    assert np.array_equal(orc.f64_to_e4m3(probe), _torch_e4m3(probe)), \
        "E4M3 rounding differs from torch's nearest-even conversion"
    sat = orc.f64_to_e4m3(np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, -1e30, -470.0]))
    assert list(sat) == [0x7E] * 6 + [0xFE, 0xFE], "magnitudes beyond 448 must saturate"


def _mx_quantize_ref(x):
    """Block quantization from library routines: the block's floor(log2(amax))
    from numpy's frexp, the elements by torch's E4M3 conversion."""
    rows, K = x.shape
    blocks = x.astype(np.float64).reshape(rows, K // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    _, ex = np.frexp(amax)
    s = np.where(amax == 0, -127, np.maximum(ex - 1 - 8, -127))
    scaled = np.clip(blocks * np.exp2(-s)[:, :, None], -448, 448)
    q = _torch_e4m3(scaled.reshape(rows, K))
    return q, (s + 127).astype(np.uint8)


def check_mx_quantize(orc):
    """MXFP8 quantization against library routines on random rows (several
    magnitudes, bf16 subnormals included), and its special cases: a zero
    block takes the smallest scale (code 0) and zero codes; a block whose
    amax is 2^k takes scale code k - 8 + 127 and stores amax as 256 (0x78);
    a block of exactly representable values round-trips exactly."""
    rng = _rng(42)
    x = np.concatenate([rng.standard_normal((16, 128)) * m for m in (1e-3, 0.02, 1.0, 300.0)])
    x = np.concatenate([x, rng.standard_normal((2, 128)) * 1e-39]).astype(np.float32)
    q, sc = orc.mx_quantize(x)
    rq, rsc = _mx_quantize_ref(x)
    assert np.array_equal(sc, rsc), "MX scales differ from floor(log2(amax)) - 8"
    assert np.array_equal(q, rq), "MX element codes differ from the library conversion"
    z = np.zeros((1, 64), np.float32)
    q, sc = orc.mx_quantize(z)
    assert (sc == 0).all() and (q == 0).all()
    for k in (-20, -3, 0, 5):
        blk = (rng.uniform(-1, 1, (1, 32)) * 2.0 ** k).astype(np.float32)
        blk[0, 7] = -(2.0 ** k)
        q, sc = orc.mx_quantize(blk)
        assert sc[0, 0] == k - 8 + 127 and q[0, 7] == 0xF8
    exact = (rng.integers(-7, 8, (4, 64)) * 2.0 ** -2).astype(np.float32)
    exact[:, 0] = 1.75      # amax * 2^-s = 448, the largest finite code
    q, sc = orc.mx_quantize(exact)
    assert np.array_equal(orc.mx_dequantize(q, sc), exact.astype(np.float64))


def check_mx_gemms(orc):
    """The MX GEMMs against numpy float64 matmuls of the dequantized operands
    (per group, the expert's own weights), with SwiGLU written out from its
    definition and the bf16 output rounding by torch."""
    rng = _rng(43)
    E, D, F = 3, 64, 32
    offs, ids = _random_grouped_rows(rng, 40, E, empty=(1,))
    R = int(offs[-1])
    xq, xsc = orc.mx_quantize(rng.standard_normal((R, D)).astype(np.float32))
    wq, wsc = orc.mx_quantize((rng.standard_normal((E * 2 * F, D)) * 0.1).astype(np.float32))
    wq, wsc = wq.reshape(E, 2 * F, D), wsc.reshape(E, 2 * F, D // 32)
    h = orc.mx_fc1_swiglu(xq, xsc, wq, wsc, offs)
    xd = orc.mx_dequantize(xq, xsc)
    wd = orc.mx_dequantize(wq, wsc)
    a = np.einsum("rd,rnd->rn", xd, wd[ids])
    g, u = a[:, :F], a[:, F:]
    want = g / (1 + np.exp(-g)) * u
    assert np.abs(h - want).max() <= 1e-6 * np.abs(want).max() + 1e-30, "MX FC1 differs"
    hq, hsc = orc.mx_quantize(h)
    oq, osc = orc.mx_quantize((rng.standard_normal((E * D, F)) * 0.1).astype(np.float32))
    oq, osc = oq.reshape(E, D, F), osc.reshape(E, D, F // 32)
    ys = orc.mx_fc2(hq, hsc, oq, osc, offs)
    y = np.einsum("rf,rdf->rd", orc.mx_dequantize(hq, hsc), orc.mx_dequantize(oq, osc)[ids])
    want_ys = f32_to_bf16_bits_torch(y.astype(np.float32))
    assert np.array_equal(ys, want_ys), "MX FC2 differs from the float64 matmul rounded to bf16"


def _e4m3_decode_torch(q):
    """Values of E4M3 codes as torch's float8_e4m3fn reads them."""
    t = torch.from_numpy(np.ascontiguousarray(q, np.uint8))
    return t.view(torch.float8_e4m3fn).double().numpy()


def _dequant_rows(q, sc):
    """float64 values of row-quantized codes (blocks of 32 along the last axis)."""
    return _e4m3_decode_torch(q) * np.exp2(np.repeat(sc.astype(np.float64) - 127, 32, axis=-1))


def _token_blocks(sizes):
    """Scale row of every row of the groups: group e's rows in blocks of 32
    from its first row, the groups' blocks numbered in order."""
    blk, nb = [], 0
    for s in sizes:
        blk += [nb + i // 32 for i in range(s)]
        nb += -(-s // 32)
    return np.array(blk, np.int64), nb


def check_mx_quantize_tokens(orc):
    """Token-axis MX quantization against the row quantization by library
    routines (frexp, torch's E4M3) of each group's 32-row blocks, transposed
    and padded with zero rows when short; the block index restarts at every
    group (short last blocks, an empty group and an exact multiple of 32)."""
    rng = _rng(44)
    sizes = [33, 0, 64, 1, 70]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R, C = int(offs[-1]), 64
    # row magnitudes spread over 2^-6 .. 2^5, so that a block's scale depends
    # on which rows it holds
    x = (rng.standard_normal((R, C)) * np.exp2(rng.integers(-6, 6, (R, 1)))).astype(np.float32)
    q, sc, boff = orc.mx_quantize_tokens(x, offs)
    blk, nb = _token_blocks(sizes)
    assert np.array_equal(boff, np.concatenate([[0], np.cumsum([-(-s // 32) for s in sizes])])), \
        "token block offsets differ from the prefix of ceil(size / 32)"
    assert sc.shape == (nb, C)
    for b in range(nb):
        rows = np.nonzero(blk == b)[0]
        pad = np.zeros((C, 32), np.float32)
        pad[:, :len(rows)] = x[rows].T
        rq, rsc = _mx_quantize_ref(pad)
        assert np.array_equal(sc[b], rsc[:, 0]), f"token block {b}: scales differ"
        assert np.array_equal(q[rows].T, rq[:, :len(rows)]), f"token block {b}: codes differ"


def check_mx_wgrad(orc):
    """The MX weight gradient against float64 matmuls, per group, of the
    operands dequantized by torch's E4M3 reading and the per-row block
    scales, rounded to bf16 by torch; an empty group gives zeros."""
    rng = _rng(45)
    sizes = [33, 0, 40, 1, 64]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R, Ca, Cb = int(offs[-1]), 64, 96
    a = (rng.standard_normal((R, Ca)) * np.exp2(rng.integers(-4, 4, (R, 1)))).astype(np.float32)
    b = rng.standard_normal((R, Cb)).astype(np.float32)
    at, bt = orc.mx_quantize_tokens(a, offs), orc.mx_quantize_tokens(b, offs)
    out = orc.mx_wgrad(at, bt, offs)
    blk, _ = _token_blocks(sizes)
    A = _e4m3_decode_torch(at[0]) * np.exp2(at[1][blk].astype(np.float64) - 127)
    Bm = _e4m3_decode_torch(bt[0]) * np.exp2(bt[1][blk].astype(np.float64) - 127)
    want = np.stack([A[offs[e]:offs[e + 1]].T @ Bm[offs[e]:offs[e + 1]]
                     for e in range(len(sizes))])
    want = f32_to_bf16_bits_torch(want.astype(np.float32))
    assert np.array_equal(out, want), "MX wgrad differs from the per-group float64 matmul"
    assert not out[1].any(), "an empty group's weight gradient must be zero"


def check_mx_dgrads(orc):
    """The MX dgrads: weights quantized along their last axis (against the
    library-routine row quantization), the FC2 dgrad + SwiGLU backward
    against a float64 matmul and torch autograd of silu(g) * u, and the FC1
    dgrad (the same contraction form as FC2) against a float64 matmul
    rounded to bf16 by torch."""
    rng = _rng(46)
    E, D, F = 3, 64, 32
    offs, ids = _random_grouped_rows(rng, 40, E, empty=(1,))
    R = int(offs[-1])
    wi = _bf16(rng, (E, D, 2 * F), 0.1)
    wo = _bf16(rng, (E, F, D), 0.1)
    iq, isc, oq, osc = orc.mx_weights_bwd(wi, wo)
    rq, rsc = _mx_quantize_ref(bits_to_f64(wo).reshape(E * F, D).astype(np.float32))
    assert np.array_equal(oq.reshape(E * F, D), rq) and np.array_equal(osc.reshape(E * F, -1), rsc)
    rq, rsc = _mx_quantize_ref(bits_to_f64(wi).reshape(E * D, 2 * F).astype(np.float32))
    assert np.array_equal(iq.reshape(E * D, 2 * F), rq) and np.array_equal(isc.reshape(E * D, -1), rsc)
    dq, dsc = orc.mx_quantize(rng.standard_normal((R, D)).astype(np.float32))
    z = _bf16(rng, (R, 2 * F), 2.0)
    dz = orc.mx_fc2_dgrad_swiglu(dq, dsc, oq, osc, z, offs)
    dh = np.einsum("rd,rfd->rf", _dequant_rows(dq, dsc), _dequant_rows(oq, osc)[ids])
    dh = dh.astype(np.float32).astype(np.float64)
    zv = bits_to_f64(z)
    G = torch.tensor(zv[:, :F], requires_grad=True)
    Uu = torch.tensor(zv[:, F:], requires_grad=True)
    (torch.nn.functional.silu(G) * Uu).backward(torch.tensor(dh))
    want = np.concatenate([G.grad.numpy(), Uu.grad.numpy()], axis=1)
    assert max_excess(bits_to_f64(dz), want, U, 1e-6 * np.abs(want).max()) <= 0, \
        "MX FC2 dgrad + SwiGLU backward differs"
    dzq, dzsc = orc.mx_quantize(bits_to_f64(dz).astype(np.float32))
    dxs = orc.mx_fc2(dzq, dzsc, iq, isc, offs)
    want = np.einsum("rn,rdn->rd", _dequant_rows(dzq, dzsc), _dequant_rows(iq, isc)[ids])
    assert np.array_equal(dxs, f32_to_bf16_bits_torch(want.astype(np.float32))), \
        "MX FC1 dgrad differs from the float64 matmul rounded to bf16"


def check_mx_block_backward(orc):
    """The MX forward + backward drivers end to end against torch autograd
    of the float64 dense block (per token, its top-k experts): the MX
    results stay within the format's error in relative norm (E4M3 keeps 3
    significand bits), the routing-weight gradient too; and z is the FC1
    pre-activation whose SwiGLU is h."""
    from types import SimpleNamespace
    logits, b, x, wi, wo, dy = _tiny_block(47, T=100, D=64, E=4, K=2, F=32)
    wl = SimpleNamespace(T=100, D=64, E=4, K=2, F=32, score_mode=0)
    inp = dict(workload=wl, logits=logits, bias=b, x=x, wi=wi, wo=wo, dy=dy)
    f = orc.mx_block_forward(inp)
    g = orc.mx_block_backward(inp, f)
    zv = bits_to_f64(f["z"])
    with np.errstate(over="ignore"):
        hz = zv[:, :32] / (1 + np.exp(-zv[:, :32])) * zv[:, 32:]
    # z is rounded to bf16: silu(g) * u from it is within a few bf16 ulps of h
    assert np.linalg.norm(f["h"] - hz) <= 4 * U * np.linalg.norm(hz), \
        "z is not FC1's pre-activation"
    X = torch.tensor(bits_to_f64(x), requires_grad=True)
    WI = torch.tensor(bits_to_f64(wi), requires_grad=True)
    WO = torch.tensor(bits_to_f64(wo), requires_grad=True)
    W = torch.tensor(f["w"].astype(np.float64), requires_grad=True)
    ref = dense_block(X, WI, WO, torch.from_numpy(f["ids"]), W)
    (ref * torch.tensor(bits_to_f64(dy))).sum().backward()

    def rel(got, want):
        return np.linalg.norm(got - want) / np.linalg.norm(want)

    # measured: 0.07-0.08 for each (several E4M3 roundings compound); a
    # transposed operand, a swapped half or a misplaced block gives ~1
    assert rel(bits_to_f64(f["out"]), ref.detach().numpy()) < 0.12, "MX out vs dense"
    for name, gr in (("dx", X.grad), ("dwi", WI.grad), ("dwo", WO.grad), ("dw", W.grad)):
        got = g[name] if name == "dw" else bits_to_f64(g[name])
        r = rel(got, gr.numpy())
        assert r < 0.12, f"MX {name} vs dense autograd: relative error {r:.3f}"
    # bf16 weight gradients: the dgrads unchanged, dwo = h^T dys and dwi =
    # xs^T dz of the same bf16 operands per expert (float64 products rounded
    # to bf16), and near the dense gradients like the MX ones
    gb = orc.mx_block_backward(inp, f, wgrad="bf16")
    for name in ("dys", "dz", "dxs", "dx", "dw"):
        assert np.array_equal(gb[name], g[name]), f"bf16 weight gradients changed {name}"
    off = f["group_offsets"]
    H, DY, DZ, XS = (bits_to_f64(a) for a in (g["hb"], g["dys"], g["dz"], f["xs"]))
    for e in range(4):
        r0, r1 = off[e], off[e + 1]
        want_o, want_i = H[r0:r1].T @ DY[r0:r1], XS[r0:r1].T @ DZ[r0:r1]
        assert max_excess(bits_to_f64(gb["dwo"][e]), want_o, U / 2 + 1e-5,
                          1e-5 * np.abs(want_o).max()) <= 0, "bf16 dwo differs from h^T dys"
        assert max_excess(bits_to_f64(gb["dwi"][e]), want_i, U / 2 + 1e-5,
                          1e-5 * np.abs(want_i).max()) <= 0, "bf16 dwi differs from xs^T dz"
    for name, gr in (("dwi", WI.grad), ("dwo", WO.grad)):
        r = rel(bits_to_f64(gb[name]), gr.numpy())
        assert r < 0.12, f"bf16 {name} on MX activations vs dense autograd: {r:.3f}"


ALL_CHECKS = [check_bf16_rounding, check_route, check_histogram, check_permute_combine,
              check_combine_bwd, check_fc1_fc2, check_swiglu_closed_forms,
              check_dense_special_case, check_gemm_backward, check_block_against_dense,
              check_finite_differences, check_e4m3_decode, check_e4m3_encode, check_mx_quantize,
              check_mx_gemms, check_mx_quantize_tokens, check_mx_wgrad, check_mx_dgrads,
              check_mx_block_backward]

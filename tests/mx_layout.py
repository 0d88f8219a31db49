"""The byte layouts of libmoe.so's MXFP8 buffers, written out from their
statement in include/moe.h, for the tests: pack the oracle's logical codes
and scales into the library's layouts, and read the library's buffers back
into logical form.  Shares no code with the oracle or the CUDA path.

Logical forms (the oracle's): activation codes [R, k] with scales [R, k/32];
weight codes [E, N, k] (row n = output column n) with scales [E, N, k/32];
token-axis codes [R, C] with scales [NB, C], block b of group e (rows
offs[e] + 32b ..) at scale row boff[e] + b.  A weight quantized along its
last axis has the weight layout without the transpose (unpack_weight with
interleave False).
"""
from __future__ import annotations

import numpy as np


def cdiv(a, b):
    return -(-a // b)


def sf_byte(m, j):
    """Byte of row m (0..127) and 32-element step j (0..3) in a 512-byte block."""
    return (m % 32) * 16 + (m // 32) * 4 + j


def tile_bases(offs):
    """First 128-row tile of each group and the total: prefix of ceil(size/128)."""
    gs = np.diff(np.asarray(offs, np.int64))
    tiles = cdiv(gs, 128)
    return np.concatenate([[0], np.cumsum(tiles)])


def act_scale_index(offs, k):
    """Flat byte index [R_used, k/32] of each row's scales in the tile-blocked
    layout (rows 0 .. offs[E]-1 in expert-sorted order)."""
    offs = np.asarray(offs, np.int64)
    E = len(offs) - 1
    R = int(offs[E])
    tb = tile_bases(offs)
    kb = cdiv(k, 128)
    r = np.arange(R)
    e = np.searchsorted(offs, r, side="right") - 1
    i = r - offs[e]
    g = tb[e] + i // 128
    m = i % 128
    b = np.arange(k // 32)
    return ((g[:, None] * kb + b[None, :] // 4) * 512 + sf_byte(m[:, None], b[None, :] % 4))


# Scale bytes that hold no element's scale (tail blocks past k, rows past a
# group's end in its last 128-row tile, weight rows past N) are packed as 0xFF,
# the E8M0 NaN: a GEMM that used one would produce NaN outputs.
PAD = 0xFF


def pack_act_scales(sc, offs, nbytes):
    buf = np.full(nbytes, PAD, np.uint8)
    idx = act_scale_index(offs, sc.shape[1] * 32)
    buf[idx] = sc[: idx.shape[0]]
    return buf


def unpack_act_scales(buf, offs, k):
    return np.asarray(buf)[act_scale_index(offs, k)]


def weight_rows(N, interleave):
    """Physical row of each logical output column n (FC1: 64-row chunks,
    gate then up)."""
    n = np.arange(N)
    if not interleave:
        return n
    F = N // 2
    f = np.where(n < F, n, n - F)
    return 128 * (f // 64) + 64 * (n >= F) + f % 64


def weight_scale_index(E, N, k, interleave):
    """Flat byte index [E, N, k/32] of each (expert, logical row, block)."""
    kb = cdiv(k, 128)
    nbp = 2 * cdiv(N, 256)
    p = weight_rows(N, interleave)
    e = np.arange(E)[:, None, None]
    b = np.arange(k // 32)[None, None, :]
    pp = p[None, :, None]
    return ((e * kb + b // 4) * nbp + pp // 128) * 512 + sf_byte(pp % 128, b % 4)


def weight_scale_bytes(E, N, k):
    return E * cdiv(k, 128) * 2 * cdiv(N, 256) * 512


def pack_weight(q, sc, interleave):
    """Logical (codes [E,N,k], scales [E,N,k/32]) -> library (codes, scale bytes)."""
    E, N, k = q.shape
    codes = np.empty_like(q)
    codes[:, weight_rows(N, interleave), :] = q
    buf = np.full(weight_scale_bytes(E, N, k), PAD, np.uint8)
    buf[weight_scale_index(E, N, k, interleave)] = sc
    return codes, buf


def unpack_weight(codes, buf, interleave):
    E, N, k = codes.shape
    q = codes[:, weight_rows(N, interleave), :]
    sc = np.asarray(buf)[weight_scale_index(E, N, k, interleave)]
    return q, sc


def act_scale_index_rows(offs, rows, k):
    """act_scale_index for the given sorted-order rows only."""
    offs = np.asarray(offs, np.int64)
    tb = tile_bases(offs)
    kb = cdiv(k, 128)
    r = np.asarray(rows, np.int64)
    e = np.searchsorted(offs, r, side="right") - 1
    i = r - offs[e]
    g = tb[e] + i // 128
    m = i % 128
    b = np.arange(k // 32)
    return ((g[:, None] * kb + b[None, :] // 4) * 512 + sf_byte(m[:, None], b[None, :] % 4))


def unpack_weight_expert(codes_e, buf, e, N, k, interleave):
    """Logical (codes [N,k], scales [N,k/32]) of expert e from the library's
    weight buffers (codes_e = that expert's [N, k] codes)."""
    per = cdiv(k, 128) * 2 * cdiv(N, 256) * 512
    q, sc = unpack_weight(codes_e[None], np.asarray(buf)[e * per:(e + 1) * per], interleave)
    return q[0], sc[0]


def token_cols(R, E):
    """Rp: token columns of the transposed token-axis codes (128 per tile of
    the tile bound ceil(R/128) + E)."""
    return 128 * (cdiv(R, 128) + E)


def token_index(offs):
    """For each sorted row r < offs[E]: its token column (128 tb[e] + i), its
    tile g and its 32-row step j inside the tile; and each group's first
    token block (boff, the prefix of ceil(size/32))."""
    offs = np.asarray(offs, np.int64)
    tb = tile_bases(offs)
    R = int(offs[-1])
    r = np.arange(R)
    e = np.searchsorted(offs, r, side="right") - 1
    i = r - offs[e]
    col = 128 * tb[e] + i
    gs = np.diff(offs)
    boff = np.concatenate([[0], np.cumsum(cdiv(gs, 32))])
    return col, e, i, boff


def token_scale_index(offs, C):
    """Flat byte index [NB, C] of each token block's scales: block b of group
    e lies in tile tb[e] + b // 4 at step b % 4."""
    offs = np.asarray(offs, np.int64)
    tb = tile_bases(offs)
    gs = np.diff(offs)
    nbp = 2 * cdiv(C, 256)
    g, j = [], []
    for e in range(len(gs)):
        b = np.arange(cdiv(int(gs[e]), 32))
        g.append(tb[e] + b // 4)
        j.append(b % 4)
    g = np.concatenate(g).astype(np.int64) if g else np.zeros(0, np.int64)
    j = np.concatenate(j).astype(np.int64) if j else np.zeros(0, np.int64)
    c = np.arange(C)
    return (g[:, None] * nbp + c[None, :] // 128) * 512 + sf_byte(c[None, :] % 128, j[:, None])


def token_scale_bytes(R, E, C):
    return (cdiv(R, 128) + E) * 2 * cdiv(C, 256) * 512


def token_pad_scale_index(offs, C):
    """Flat byte index [n, C] of the scales of the 32-token steps of used
    tiles that hold none of the group's rows (a group's last tile past its
    last block): the quantization of zero rows, scale byte 0."""
    offs = np.asarray(offs, np.int64)
    tb = tile_bases(offs)
    gs = np.diff(offs)
    nbp = 2 * cdiv(C, 256)
    g, j = [], []
    for e in range(len(gs)):
        nb = cdiv(int(gs[e]), 32)
        for b in range(nb, 4 * cdiv(nb, 4)):
            g.append(tb[e] + b // 4)
            j.append(b % 4)
    g = np.array(g, np.int64)
    j = np.array(j, np.int64)
    c = np.arange(C)
    return (g[:, None] * nbp + c[None, :] // 128) * 512 + sf_byte(c[None, :] % 128, j[:, None])


def pack_tokens(q, sc, offs, R, E):
    """Logical (codes [R_used, C], scales [NB, C]) -> library (codes [C, Rp]
    with zero codes in the padding columns and zero-block scales for the
    steps they fill, scale bytes)."""
    C = q.shape[1]
    col, _, _, _ = token_index(offs)
    codes = np.zeros((C, token_cols(R, E)), np.uint8)
    codes[:, col] = q[: len(col)].T
    buf = np.full(token_scale_bytes(R, E, C), PAD, np.uint8)
    buf[token_scale_index(offs, C)] = sc
    buf[token_pad_scale_index(offs, C)] = 0
    return codes, buf


def unpack_tokens(codes, buf, offs):
    """Library (codes [C, Rp], scale bytes) -> logical (codes [R_used, C],
    scales [NB, C]), the codes of the padding columns of used tiles and the
    scales of the steps that hold only padding."""
    C = codes.shape[0]
    col, _, _, _ = token_index(offs)
    q = np.ascontiguousarray(codes[:, col].T)
    sc = np.asarray(buf)[token_scale_index(offs, C)]
    tb = tile_bases(offs)
    used = np.zeros(codes.shape[1], bool)
    used[: 128 * int(tb[-1])] = True
    used[col] = False
    return q, sc, codes[:, used], np.asarray(buf)[token_pad_scale_index(offs, C)]

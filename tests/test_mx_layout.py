"""CPU checks of the test-side statement of the MXFP8 buffer layouts: every
(row, block) scale has its own byte inside the buffer size the library
reports, packing and unpacking are inverse, and FC1's row interleave is a
permutation that puts gate column f and up column F+f 64 rows apart inside
one 128-row half."""
import numpy as np

from tests import mx_layout as L


def test_activation_scale_index_is_injective():
    offs = np.array([0, 0, 130, 131, 400, 400, 655], np.int64)
    E = len(offs) - 1
    for k in (64, 128, 320):
        idx = L.act_scale_index(offs, k)
        assert idx.shape == (offs[-1], k // 32)
        assert len(np.unique(idx)) == idx.size
        bound = (L.cdiv(int(offs[-1]), 128) + E) * L.cdiv(k, 128) * 512
        assert idx.max() < bound
        sc = np.random.default_rng(0).integers(0, 255, idx.shape).astype(np.uint8)
        assert np.array_equal(L.unpack_act_scales(L.pack_act_scales(sc, offs, bound), offs, k), sc)


def test_weight_layout_round_trip_and_interleave():
    rng = np.random.default_rng(1)
    for E, N, k, inter in ((3, 384, 320, True), (2, 320, 192, False), (1, 128, 64, True)):
        q = rng.integers(0, 255, (E, N, k)).astype(np.uint8)
        sc = rng.integers(0, 255, (E, N, k // 32)).astype(np.uint8)
        codes, buf = L.pack_weight(q, sc, inter)
        assert len(np.unique(L.weight_scale_index(E, N, k, inter))) == E * N * (k // 32)
        q2, sc2 = L.unpack_weight(codes, buf, inter)
        assert np.array_equal(q2, q) and np.array_equal(sc2, sc)
    F = 192
    p = L.weight_rows(2 * F, True)
    assert sorted(p.tolist()) == list(range(2 * F))
    f = np.arange(F)
    assert np.all(p[F + f] - p[f] == 64) and np.all(p[f] // 128 == p[F + f] // 128)


def test_token_layout_round_trip():
    """Token-axis layout: every (block, column) scale has its own byte inside
    the library's buffer size, every used row its own token column, padding
    columns lie inside used tiles only, and pack/unpack are inverse."""
    rng = np.random.default_rng(2)
    offs = np.array([0, 0, 130, 131, 400, 400, 655], np.int64)
    E = len(offs) - 1
    R = int(offs[-1]) + 5          # a few dropped slots past the last group
    for C in (64, 192, 320):
        nb = int(sum(L.cdiv(int(s), 32) for s in np.diff(offs)))
        idx = L.token_scale_index(offs, C)
        assert idx.shape == (nb, C) and len(np.unique(idx)) == idx.size
        assert idx.max() < L.token_scale_bytes(R, E, C)
        col, _, _, boff = L.token_index(offs)
        assert len(np.unique(col)) == int(offs[-1]) and col.max() < L.token_cols(R, E)
        assert boff[-1] == nb
        q = rng.integers(0, 255, (int(offs[-1]), C)).astype(np.uint8)
        sc = rng.integers(0, 255, (nb, C)).astype(np.uint8)
        codes, buf = L.pack_tokens(q, sc, offs, R, E)
        q2, sc2, pad, pad_sc = L.unpack_tokens(codes, buf, offs)
        assert np.array_equal(q2, q) and np.array_equal(sc2, sc) and not pad.any()
        assert not pad_sc.any()
        both = np.concatenate([idx.ravel(), L.token_pad_scale_index(offs, C).ravel()])
        assert len(np.unique(both)) == both.size   # padding steps are not block scales
        assert pad.shape[1] == 128 * int(L.tile_bases(offs)[-1]) - int(offs[-1])

"""CPU check of the end-to-end decode tolerance (cases.flip_bound).

The write bar lets a code within BOUNDARY of a rounding boundary round either
way.  The end-to-end decode test therefore widens the decode bar of each
(sequence, query head) by flip_bound: an oracle-side bound of how far the
output can move when the cache holds such alternative codes.  This test
plants exactly those alternatives in the oracle's own cache (on the CPU) and
checks that the oracle's decode moves by no more than the bound.
"""
from __future__ import annotations

import math
import types

import numpy as np
import pytest

import kvq3_inputs as I
from cases import BOUNDARY, flip_bound
from oracle import kvq3_oracle as O


def _case(d=128, hkv=1, hq=4, block=64, scale="f16", page=64, lens=(400,), seed=7, bits=3):
    s, qt = O.rotation_params(d, 42, True, True)
    c = types.SimpleNamespace(d=d, hkv=hkv, hq=hq, block=block, scale=scale, page=page, bits=bits,
                              lens=np.array(lens, np.int32), B=len(lens), U=O.rotation_matrix(s, qt))
    maxp = max(math.ceil(L / page) for L in lens)
    c.layout = O.Layout(d, hkv, block, scale, page, c.B, maxp, c.B * maxp, bits)
    # narrow outlier-free data: many coordinates land near rounding boundaries
    c.spec = I.DataSpec(d, hkv, seed, 0.0, 1.0)
    return c


def _tokens(c):
    ks, vs, si, ps = [], [], [], []
    for b in range(c.B):
        n = int(c.lens[b])
        ks.append(np.stack([I.kv_rows_np(c.spec, 0, b, h, 0, n) for h in range(c.hkv)], 1))
        vs.append(np.stack([I.kv_rows_np(c.spec, 1, b, h, 0, n) for h in range(c.hkv)], 1))
        si.append(np.full(n, b, np.int32))
        ps.append(np.arange(n, dtype=np.int32))
    return np.concatenate(ks), np.concatenate(vs), np.concatenate(si), np.concatenate(ps)


def _flip_near_boundary(c, pool, k, v, si, ps, widen, every=1, differs=None):
    """Moves every `every`-th code within `widen` of a rounding boundary to
    the other side of it, in the oracle's pool (one sequence).  Returns how
    many were moved; records the moved elements in `differs` as
    Case.written_differences would."""
    nb, blk = c.d // c.block, c.block
    qm = O.qmax(c.bits)
    moved = 0
    for which, src in ((0, k), (1, v)):
        for g in range(c.hkv):
            x = src[:, g].astype(np.float64) @ c.U.T
            codes, sq, _ = O.quantize(x, blk, 1e-6, c.scale, c.bits)
            r = x.reshape(-1, nb, blk) / np.where(sq > 0, sq, 1.0)[..., None]
            frac = np.abs(r) - np.floor(np.abs(r))
            near = (np.abs(frac - 0.5) < widen) & (np.abs(r) < qm)
            idx = np.flatnonzero(near)
            near = np.zeros(near.shape, bool)
            near.flat[idx[::every]] = True
            if differs is not None:
                differs[(0, g, which)] = (near.reshape(-1, c.d), np.zeros(sq.shape, bool))
            if not near.any():
                continue
            alt = codes.reshape(-1, nb, blk).astype(np.int64)
            # the other neighbour of the boundary
            other = np.where(np.rint(r) == np.floor(r), np.floor(r) + 1, np.floor(r))
            alt = np.where(near, np.clip(other, -qm, qm), alt).reshape(-1, c.d)
            moved += int(near.sum())
            page, slot, st = O.locate(c.layout, None, si, ps)
            for t in np.nonzero(near.reshape(-1, c.d).any(axis=1))[0]:
                off = c.layout.code_offset(page[t], g, which, slot[t])
                pool[off:off + c.layout.code_bytes] = O.pack_codes(alt[t][None].astype(np.int8), c.bits)[0]
    return moved


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_flip_bound_covers_alternative_codes(bits):
    c = _case(bits=bits)
    k, v, si, ps = _tokens(c)
    pool = np.zeros(c.layout.pool_bytes, np.uint8)
    O.write(pool, c.layout, c.U, k, v, si, ps, None)
    q = I.q_np(c.spec, c.B, c.hq, 0)
    ref = O.decode(pool, c.layout, c.U, q, c.lens, None, 0.0)
    bound = flip_bound(c, k, v, si, ps, q)
    flipped = pool.copy()
    moved = _flip_near_boundary(c, flipped, k, v, si, ps, BOUNDARY)
    got = O.decode(flipped, c.layout, c.U, q, c.lens, None, 0.0)
    delta = np.abs(got - ref).max(axis=-1)
    assert moved > 0, "the case must contain boundary elements"
    assert np.all(delta <= bound * (1 + 1e-9) + 1e-12)
    # the bound is not vacuous: it is within a few orders of the actual move
    assert float(bound.max()) < 1e4 * max(float(delta.max()), 1e-12)


def test_flip_bound_is_zero_without_boundary_elements():
    c = _case(lens=(16,), seed=11)
    k, v, si, ps = _tokens(c)
    q = I.q_np(c.spec, c.B, c.hq, 0)
    bound = flip_bound(c, k, v, si, ps, q)
    # with no element near a boundary the end-to-end bar is the plain decode bar
    nb = c.d // c.block
    near_any = False
    for src in (k, v):
        x = src[:, 0].astype(np.float64) @ c.U.T
        _, sq, _ = O.quantize(x, c.block, 1e-6, c.scale, c.bits)
        r = np.abs(x.reshape(-1, nb, c.block) / sq[..., None])
        near_any |= bool((np.abs(r - np.floor(r) - 0.5) < BOUNDARY).any())
    assert (bound.max() > 0) == near_any


def test_flip_bound_restricted_to_the_elements_that_differ():
    # every third boundary element flipped: the bound over just those covers
    # the move and is far tighter than the bound over the whole band
    c = _case()
    k, v, si, ps = _tokens(c)
    pool = np.zeros(c.layout.pool_bytes, np.uint8)
    O.write(pool, c.layout, c.U, k, v, si, ps, None)
    q = I.q_np(c.spec, c.B, c.hq, 0)
    ref = O.decode(pool, c.layout, c.U, q, c.lens, None, 0.0)
    flipped, differs = pool.copy(), {}
    moved = _flip_near_boundary(c, flipped, k, v, si, ps, BOUNDARY, every=3, differs=differs)
    got = O.decode(flipped, c.layout, c.U, q, c.lens, None, 0.0)
    delta = np.abs(got - ref).max(axis=-1)
    some = flip_bound(c, k, v, si, ps, q, differs=differs)
    band = flip_bound(c, k, v, si, ps, q)
    assert moved > 0
    assert np.all(delta <= some * (1 + 1e-9) + 1e-12)
    assert np.all(some <= band * (1 + 1e-12))


def _flip_near_boundary_asym(c, pool, k, v, si, ps, widen, every=1, differs=None):
    """As _flip_near_boundary for the asymmetric variant: unsigned codes,
    boundaries of (x - z_q)/s_q."""
    nb, blk = c.d // c.block, c.block
    top = (1 << c.bits) - 1
    moved = 0
    for which, src in ((0, k), (1, v)):
        for g in range(c.hkv):
            x = src[:, g].astype(np.float64) @ c.U.T
            u, sz, _ = O.quantize_asym(x, blk, 1e-6, c.bits)
            sq, zq = sz[..., 0], sz[..., 1]
            r = (x.reshape(-1, nb, blk) - zq[..., None]) / np.where(sq > 0, sq, 1.0)[..., None]
            frac = r - np.floor(r)
            near = (np.abs(frac - 0.5) < widen) & (r > 0) & (r < top)
            idx = np.flatnonzero(near)
            near = np.zeros(near.shape, bool)
            near.flat[idx[::every]] = True
            if differs is not None:
                differs[(0, g, which)] = (near.reshape(-1, c.d), np.zeros(sq.shape, bool))
            if not near.any():
                continue
            other = np.where(np.rint(r) == np.floor(r), np.floor(r) + 1, np.floor(r))
            alt = np.where(near, np.clip(other, 0, top), u.reshape(-1, nb, blk)).reshape(-1, c.d)
            moved += int(near.sum())
            page, slot, st = O.locate(c.layout, None, si, ps)
            for t in np.nonzero(near.reshape(-1, c.d).any(axis=1))[0]:
                off = c.layout.code_offset(page[t], g, which, slot[t])
                pool[off:off + c.layout.code_bytes] = O.pack_codes(alt[t][None].astype(np.int64), c.bits)[0]
    return moved


def test_flip_bound_covers_alternative_codes_asym():
    c = _case(scale="e4m3zp")
    k, v, si, ps = _tokens(c)
    pool = np.zeros(c.layout.pool_bytes, np.uint8)
    O.write(pool, c.layout, c.U, k, v, si, ps, None)
    q = I.q_np(c.spec, c.B, c.hq, 0)
    ref = O.decode(pool, c.layout, c.U, q, c.lens, None, 0.0)
    flipped, differs = pool.copy(), {}
    moved = _flip_near_boundary_asym(c, flipped, k, v, si, ps, BOUNDARY, differs=differs)
    got = O.decode(flipped, c.layout, c.U, q, c.lens, None, 0.0)
    delta = np.abs(got - ref).max(axis=-1)
    some = flip_bound(c, k, v, si, ps, q, differs=differs)
    band = flip_bound(c, k, v, si, ps, q)
    assert moved > 0, "the case must contain boundary elements"
    assert np.all(delta <= some * (1 + 1e-9) + 1e-12)
    assert np.all(some <= band * (1 + 1e-12))
    assert float(some.max()) < 1e4 * max(float(delta.max()), 1e-12)

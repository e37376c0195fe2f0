"""Chunked-prefill attention over the packed cache: GPU (kvq3_prefill_attn)
against the oracle (oracle.prefill) on the same oracle-written cache.

Query token i of the chunk sits at position pos0 + i and attends causally to
positions [0, pos0 + i]; the library tiles 16/G query tokens x G heads per kv
head, so the cases cover every group size's tiling, ragged last tiles, a chunk
at the start of a sequence and one in the middle, paged and contiguous caches.
"""
from __future__ import annotations

import numpy as np
import pytest

import kvq3_inputs as I
from cases import TOL_DECODE, Case, rel_err
from oracle import kvq3_oracle as O

pytestmark = pytest.mark.gpu

PREFILL_CASES = [
    # (case kwargs, sequence, pos0, n_q)
    (dict(d=128, block=64, scale="f16", page=64, lens=(300,), hkv=2, hq=8), 0, 200, 100),     # G=4, 25 tiles
    (dict(d=128, block=64, scale="f16", page=16, lens=(90, 257), hkv=2, hq=8, paged=True), 1, 0, 257),
    (dict(d=128, block=64, scale="e4m3", page=64, lens=(520,), hkv=2, hq=16), 0, 450, 70),    # G=8
    (dict(d=128, block=64, scale="f32", page=64, lens=(200,), hkv=4, hq=4), 0, 150, 50),      # G=1, qt=16
    (dict(d=128, block=64, scale="f16", page=16, lens=(130,), hkv=1, hq=16, flags=1), 0, 100, 30),   # G=16
    (dict(d=64, block=32, scale="f16", page=16, lens=(150,), hkv=2, hq=12), 0, 60, 90),       # G=6, qt=2
    (dict(d=256, block=64, scale="f16", page=16, lens=(300, 180), hkv=2, hq=8, paged=True), 1, 100, 80),
    # d = 128, blocks of 64: the tcgen05 kernel (128 rows = 128/G tokens x G heads a CTA, 64-key tiles)
    (dict(d=128, block=64, scale="f16", page=64, lens=(400,), hkv=2, hq=6), 0, 100, 250),      # G=3: 126-row CTAs
    (dict(d=128, block=64, scale="f16", page=48, lens=(700, 90), hkv=2, hq=8, paged=True), 0, 300, 400),  # tiles straddle pages
    (dict(d=128, block=64, scale="f16", page=128, lens=(3000,), hkv=1, hq=4), 0, 2400, 600),   # 47 tiles, stage ring wraps
    (dict(d=128, block=64, scale="e4m3", page=32, lens=(500,), hkv=4, hq=8, paged=True), 0, 499, 1),   # one query
    (dict(d=128, block=64, scale="f32", page=16, lens=(260,), hkv=1, hq=12), 0, 0, 260),      # G=12: 120-row CTAs, from 0
    (dict(d=128, block=64, scale="e4m3", page=64, lens=(1100,), hkv=2, hq=4, flags=7), 0, 1000, 100),  # SO(4) pairs
    # units of eight or more key tiles run as several CTAs over equal shares of their keys (two, or one
    # per 128 tiles), merged in the workspace
    (dict(d=128, block=64, scale="f16", page=16, lens=(40, 900), hkv=2, hq=8, paged=True), 1, 500, 300),  # 4 pages a tile
    (dict(d=128, block=64, scale="f32", page=32, lens=(1300,), hkv=1, hq=16), 0, 1250, 50),    # G=16, 20 tiles
    (dict(d=128, block=64, scale="f16", page=64, lens=(17000,), hkv=1, hq=4), 0, 16992, 8),    # 266 tiles: 3 parts
    (dict(d=128, block=64, scale="e4m3", page=32, lens=(25000, 300), hkv=1, hq=8, paged=True), 0, 24990, 10),  # 4 parts
]


def _ids(c):
    kw, seq, pos0, n = c
    return (f"d{kw['d']}-m{kw['block']}-{kw['scale']}-G{kw['hq'] // kw['hkv']}-"
            f"{'paged' if kw.get('paged') else 'contig'}-pos{pos0}-n{n}")


def _run(c: Case, seq: int, pos0: int, q: np.ndarray, sm_scale: float = 0.0):
    t = c.torch
    qd = t.as_tensor(q, device=c.dev)
    n_out = q.shape[0] * c.hq * c.d * 4
    out_full, out_b = c.guarded(n_out)
    out = out_b.view(t.float32).view(q.shape[0], c.hq, c.d)
    out.fill_(float("nan"))
    n_ws = c.K.kvq3_prefill_workspace_size(c.desc, c.hq, q.shape[0])
    ws_full, ws = c.guarded(n_ws)
    c.K.kvq3_prefill_attn(c.rot.handle, c.desc, c.cache, seq, pos0, qd, out, ws, sm_scale, c.status)
    t.cuda.synchronize()
    c.check_guard(out_full, n_out, "prefill output")
    c.check_guard(ws_full, n_ws, "prefill workspace")
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("cfg", PREFILL_CASES, ids=_ids)
def test_prefill_matches_oracle(cfg):
    kw, seq, pos0, n = cfg
    c = Case(**kw)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = I.q_np(c.spec, n, c.hq, 7)            # [n][Hq][d]: one row per query token
    got = _run(c, seq, pos0, q)
    ref = O.prefill(c.pool_o, c.layout, c.U, q, seq, pos0, c.table)
    assert c.device_status() == 0
    e = rel_err(got, ref)
    print(f"max|err|/rms = {e:.3e}")
    assert e <= TOL_DECODE


def test_prefill_single_query_equals_decode():
    # one query at the last position is a decode step of the whole sequence
    c = Case(d=128, block=64, scale="f16", page=64, lens=(333,), hkv=2, hq=8)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = c.queries(3)                          # [1][Hq][d]
    got_p = _run(c, 0, 332, q)
    got_d = c.gpu_decode(q)
    assert c.device_status() == 0
    assert rel_err(got_p, got_d) <= TOL_DECODE


def test_prefill_custom_scale_and_bounds():
    c = Case(d=128, block=64, scale="f16", page=64, lens=(128,), hkv=2, hq=8)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = I.q_np(c.spec, 40, c.hq, 9)
    for sm in (0.02, 0.3):
        got = _run(c, 0, 88, q, sm)
        ref = O.prefill(c.pool_o, c.layout, c.U, q, 0, 88, c.table, sm)
        assert rel_err(got, ref) <= TOL_DECODE
    t = c.torch
    qd = t.as_tensor(q, device=c.dev)
    out = t.empty((40, c.hq, c.d), dtype=t.float32, device=c.dev)
    ws = t.empty(c.K.kvq3_prefill_workspace_size(c.desc, c.hq, 40), dtype=t.uint8, device=c.dev)
    # past the sequence capacity, or a sequence that does not exist
    for seq, pos0 in ((0, 100), (1, 0), (-1, 0)):
        with pytest.raises(c.K.Kvq3Error):
            c.K.kvq3_prefill_attn(c.rot.handle, c.desc, c.cache, seq, pos0, qd, out, ws)
    # a workspace one byte short
    with pytest.raises(c.K.Kvq3Error):
        c.K.kvq3_prefill_attn(c.rot.handle, c.desc, c.cache, 0, 0, qd, out, ws[:-1])


def test_prefill_bad_page_flags_and_masks():
    # an out-of-range page id in the table: its keys are left out (masked),
    # KVQ3_DEV_BAD_PAGE is flagged, and every output stays finite
    c = Case(d=128, block=64, scale="f16", page=32, lens=(400,), hkv=2, hq=8, paged=True)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    table = c.table.copy()
    table[0, 3] = c.num_pages + 7              # positions 96..127
    c.table_t.copy_(c.torch.as_tensor(table, device=c.dev))
    q = I.q_np(c.spec, 150, c.hq, 9)
    got = _run(c, 0, 250, q)
    assert c.device_status() & 4
    assert np.isfinite(got).all()
    # the masked prefill equals attention over the other positions: compare
    # with the oracle on a cache where those keys can never win (a reference
    # computed from the oracle's dequantised rows without positions 96..127)
    from oracle import kvq3_oracle as Ox
    U = c.U
    ref = np.zeros_like(got)
    keep = np.r_[0:96, 128:400]
    for g in range(c.hkv):
        kh = Ox.read_rotated(c.pool_o, c.layout, 0, g, 0, 0, 400, c.table)[0]
        vh = Ox.read_rotated(c.pool_o, c.layout, 0, g, 1, 0, 400, c.table)[0]
        for i in range(150):
            m = 250 + i + 1
            idx = keep[keep < m]
            for gh in range(c.hq // c.hkv):
                h = g * (c.hq // c.hkv) + gh
                ref[i, h] = Ox.attention_rotated(U, q[i, h], kh[idx], vh[idx], 1.0 / np.sqrt(c.d))
    assert rel_err(got, ref) <= TOL_DECODE


def test_prefill_workspace_covers_split_units():
    import hadamard_rotated_bit_kvq3_gb300 as K
    # d = 128, 3-bit symmetric codes, blocks of 64: the tcgen05 path, whose
    # units (128 (token, head) rows of a kv head) may run as several CTAs
    # that meet in the workspace: a counter per unit, then one partial of
    # 128 rows x 132 floats per CTA of the unit, after the 256-byte aligned
    # counters; a unit runs as at most max(2, ceil(tiles / 128)) CTAs (16 at
    # most), tiles = the 64-key tiles of the longest context the cache holds
    # (the size also covers the decode kernel's plan, which asks the device)
    def desc(**kw):
        base = dict(head_dim=128, num_kv_heads=8, block=64, bits=3, scale_type=1, eps=1e-6,
                    page_size=128, batch=1, max_pages_per_seq=256, reserved=0, num_pages=256)
        base.update(kw)
        return K.CacheDesc(**base)
    for maxp, parts in ((256, 4), (4, 2), (65, 2), (129, 3), (4096, 16)):
        for hq, n in ((32, 2048), (32, 1), (24, 300), (8, 129), (128, 5)):
            g = hq // 8
            units = -(-n // (128 // g)) * 8
            need = -(-units * 4 // 256) * 256 + units * parts * 128 * 132 * 4
            d = desc(max_pages_per_seq=maxp, num_pages=maxp)
            if g > 16:   # more than 16 query heads per kv head: refused
                with pytest.raises(K.Kvq3Error):
                    K.kvq3_prefill_workspace_size(d, hq, n)
                continue
            assert K.kvq3_prefill_workspace_size(d, hq, n) >= need, (maxp, hq, n)
    # other formats run on the decode kernel's prefill variant: no partials,
    # far less than the tcgen05 path would ask for
    small = K.kvq3_prefill_workspace_size(desc(block=32), 32, 2048)
    assert small < 512 * 2 * 128 * 132 * 4

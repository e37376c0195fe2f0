"""Parity at the full workload sizes, in the launch configuration bench.py
times: the GPU writes and decodes the whole workload; the oracle recomputes
sampled (sequence, kv head) units one by one from the same seeded inputs
(codes of sampled positions bit-exact outside rounding boundaries; decode
outputs of the sampled heads within 2e-3 * rms of those outputs; prefill
attention of sampled query tokens within the same bar)."""
import math

import numpy as np
import pytest

import kvq3_inputs as I
from cases import BOUNDARY, MIDPOINT, TOL_DECODE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _oracle_unit(oracle, w, lens, b, kvh, table_row=None):
    """Oracle pool of one (sequence, kv head) unit, its U, k, v."""
    L = int(lens[b])
    P = w.page_size
    maxp = int(math.ceil(L / P))
    lay = oracle.Layout(w.d, 1, w.block, w.scale, P, 1, maxp, maxp, w.bits)
    s, q = oracle.rotation_params(w.d, w.rot_seed, bool(w.rot_flags & 1), bool(w.rot_flags & 2))
    U = oracle.rotation_matrix(s, q)
    k = I.kv_rows_np(w.data, 0, b, kvh, 0, L)
    v = I.kv_rows_np(w.data, 1, b, kvh, 0, L)
    pool = np.zeros(lay.pool_bytes, np.uint8)
    oracle.write(pool, lay, U, k[:, None], v[:, None], np.zeros(L, np.int32), np.arange(L), None, w.eps)
    return lay, pool, U, k, v


def _check_codes(oracle, w, st, gp, lay_full, b, kvh, U, src, which, t0, nt):
    """Stored scales and codes of positions t0..t0+nt-1 (GPU pool bytes gp)
    against the oracle's quantisation of the same input rows."""
    _, cg, sg = oracle.read_rotated(gp, lay_full, b, kvh, which, t0, nt, st.table_np)
    x = src[t0:t0 + nt].astype(np.float64) @ U.T
    if w.scale == "e4m3zp":   # asymmetric variant: (scale, zero point) pairs, unsigned codes
        c, sz, s = oracle.quantize_asym(x, w.block, w.eps, w.bits)
        lo = x.reshape(nt, -1, w.block).min(-1)
        mid = (oracle.scale_midpoint_distance(s, "e4m3") < MIDPOINT) | \
              (oracle.scale_midpoint_distance(np.abs(lo), "e4m3") < MIDPOINT)
        assert np.array_equal(sg[~mid], sz[~mid])
        sq, zq = sz[..., 0], sz[..., 1]
        r = (x.reshape(nt, -1, w.block) - zq[..., None]) / np.where(sq > 0, sq, 1)[..., None]
        top = (1 << w.bits) - 1
    else:
        c, sq, s = oracle.quantize(x, w.block, w.eps, w.scale, w.bits)
        mid = oracle.scale_midpoint_distance(s, w.scale) < MIDPOINT
        assert np.all(np.abs(sg - sq)[~mid] <= 1e-6 * sq[~mid])
        r = np.abs(x.reshape(nt, -1, w.block) / np.where(sq > 0, sq, 1)[..., None])
        top = oracle.qmax(w.bits)
    near = np.zeros(r.shape, bool)
    for kk in range(top):
        near |= np.abs(r - (kk + 0.5)) < BOUNDARY
    near = (near | mid[..., None]).reshape(nt, w.d)
    assert not np.any((cg != c) & ~near)
    return int(near.sum())


@pytest.mark.parametrize("name,samples", [("tiny", [(0, 0), (0, 3)]),
                                          ("llama8b", [(0, 0), (15, 7), (9, 3)]),
                                          ("long70b", [(3, 4), (7, 0)]),
                                          ("ragged", [(0, 0), (63, 3), (17, 2)])])
def test_fullsize_decode_step(oracle, name, samples):
    import bench
    import torch
    st = bench.GpuWorkload(name, torch.device("cuda:0"))
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    out = st.out.cpu().numpy().astype(np.float64)
    w = st.w
    lay_full = oracle.Layout(w.d, w.num_kv_heads, w.block, w.scale, w.page_size, w.batch, st.maxp,
                             st.num_pages, w.bits)
    q = I.q_np(w.data, w.batch, w.num_q_heads)
    gp = st.pool.cpu().numpy()
    got, ref = [], []
    for b, kvh in samples:
        lay, pool, U, k, v = _oracle_unit(oracle, w, st.lens, b, kvh)
        L = int(st.lens[b])
        # codes of the first, a middle and the last (just appended) positions
        for t0 in sorted({0, max(0, L // 2 - 64), max(0, L - 128)}):
            nt = min(128, L - t0)
            _check_codes(oracle, w, st, gp, lay_full, b, kvh, U, k, 0, t0, nt)
            _check_codes(oracle, w, st, gp, lay_full, b, kvh, U, v, 1, t0, nt)
        heads = [(0, g) for g in range(w.group)]
        qs = q[b:b + 1, kvh * w.group:(kvh + 1) * w.group]
        r = oracle.decode(pool, lay, U, qs, np.array([L]), heads=heads)[0]
        ref.append(r)
        got.append(out[b, kvh * w.group:(kvh + 1) * w.group])
    got, ref = np.array(got), np.array(ref)
    rms = math.sqrt(float(np.mean(ref ** 2)))
    err = float(np.abs(got - ref).max())
    print(f"{name}: max|err|/rms = {err / rms:.3e}")
    assert err <= TOL_DECODE * rms


@pytest.mark.parametrize("bits,scale", [(2, ""), (4, ""), (0, "e4m3zp")], ids=["b2", "b4", "asym"])
def test_fullsize_decode_step_other_formats(oracle, bits, scale):
    # the llama8b workload at the other code widths and in the asymmetric
    # variant, as bench.py --bits / --scale runs it
    import bench
    saved = bench.BITS_OVERRIDE, bench.SCALE_OVERRIDE
    bench.BITS_OVERRIDE, bench.SCALE_OVERRIDE = bits, scale
    try:
        test_fullsize_decode_step(oracle, "llama8b", [(0, 0), (15, 7)])
    finally:
        bench.BITS_OVERRIDE, bench.SCALE_OVERRIDE = saved


def test_fullsize_prefill_write(oracle):
    import bench
    import torch
    st = bench.PrefillWorkload(torch.device("cuda:0"))
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    w = st.w
    lay_full = oracle.Layout(w.d, w.num_kv_heads, w.block, w.scale, w.page_size, 1, st.maxp, st.num_pages)
    s, qq = oracle.rotation_params(w.d, w.rot_seed, bool(w.rot_flags & 1), bool(w.rot_flags & 2))
    U = oracle.rotation_matrix(s, qq)
    gp = st.pool.cpu().numpy()
    for kvh in (0, 5, 7):
        for t0 in (0, 77777, w.seq_len - 300):
            k = I.kv_rows_np(w.data, 0, 0, kvh, t0, 300)
            v = I.kv_rows_np(w.data, 1, 0, kvh, t0, 300)
            _check_codes(oracle, w, st, gp, lay_full, 0, kvh, U, _Shift(k, t0), 0, t0, 300)
            _check_codes(oracle, w, st, gp, lay_full, 0, kvh, U, _Shift(v, t0), 1, t0, 300)


class _Shift:
    """Rows t0.. of a tensor presented with absolute indexing."""

    def __init__(self, rows, t0):
        self.rows, self.t0 = rows, t0

    def __getitem__(self, sl):
        return self.rows[sl.start - self.t0:sl.stop - self.t0]


@pytest.mark.parametrize("bits,scale", [(0, ""), (4, ""), (0, "e4m3zp")], ids=["default", "b4", "asym"])
def test_fullsize_prefill_attention(oracle, bits, scale):
    # the prefill-attention step bench.py times (2,048 queries at the end of a
    # 32K-token cache, split units merged in the workspace); the oracle
    # recomputes sampled query tokens -- the first and last rows of query
    # blocks and of the chunk -- over its own cache of the same inputs
    import bench
    import torch
    saved = bench.BITS_OVERRIDE, bench.SCALE_OVERRIDE
    bench.BITS_OVERRIDE, bench.SCALE_OVERRIDE = bits, scale
    try:
        w = bench.workload("prefill_attn")
    finally:
        bench.BITS_OVERRIDE, bench.SCALE_OVERRIDE = saved
    st = bench.PrefillAttnWorkload(torch.device("cuda:0"), w)
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    out = st.out.cpu().numpy().astype(np.float64)
    G = w.num_q_heads // w.num_kv_heads
    q = I.q_np(w.data, w.chunk, w.num_q_heads, 0)
    got, ref = [], []
    for kvh in (0, 6):
        lay, pool, U, _, _ = _oracle_unit(oracle, w, [w.seq_len], 0, kvh)
        for i in (0, 31, 32, 1000, w.chunk - 32, w.chunk - 1):
            qs = q[i:i + 1, kvh * G:(kvh + 1) * G]
            ref.append(oracle.prefill(pool, lay, U, qs, 0, st.pos0 + i)[0])
            got.append(out[i, kvh * G:(kvh + 1) * G])
    got, ref = np.array(got), np.array(ref)
    rms = math.sqrt(float(np.mean(ref ** 2)))
    err = float(np.abs(got - ref).max())
    print(f"prefill attention {w.bits}-bit {w.scale}: max|err|/rms = {err / rms:.3e}")
    assert err <= TOL_DECODE * rms

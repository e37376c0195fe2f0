"""Two-quaternion SO(4) blocks (R_i x = p_i x conj(q_i), the general element of
SO(4); "Orthogonally mixed 3-bit KV cache", Mathematical statement) through
every kernel that rotates: kvq3_rotate, the token-list and chunk writes, the
read-back, decode (isolated and end to end), prefill attention, and the
calibration objective and search -- each against the oracle with the bars of
the one-quaternion tests."""
import math

import numpy as np
import pytest

import kvq3_inputs as I
from cases import TOL_DECODE, Case, flip_bound, rel_err, written_differences
from oracle import kvq3_oracle as O

pytestmark = pytest.mark.gpu

PAIR = 7   # sign flip + SO(4) blocks + pairs


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hadamard_rotated_bit_kvq3_gb300  # noqa: F401


@pytest.mark.parametrize("d", [4, 16, 64, 128, 256])
@pytest.mark.parametrize("flags", [7, 6])
def test_rotate_pair_matches_dense_U(d, flags):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    rot = K.Rotation(d, 42, flags)
    s, q, r = O.rotation_params_pair(d, 42, bool(flags & 1))
    U = O.rotation_matrix(s, q, r)
    rng = np.random.default_rng(d)
    x = rng.standard_normal((333, d)).astype(np.float32)
    xt = torch.as_tensor(x, device="cuda")
    y = torch.empty_like(xt)
    for inverse in (False, True):
        K.kvq3_rotate(rot.handle, xt, y, inverse=inverse)
        ref = x.astype(np.float64) @ (U if inverse else U.T)
        assert np.abs(y.cpu().numpy() - ref).max() < 3e-6 * math.sqrt(d)
    # from explicit parameters: the same rotation
    rot2 = K.kvq3_rotation_create_from_params_pair(d, s, q.astype(np.float32), r.astype(np.float32))
    try:
        K.kvq3_rotate(rot2, xt, y)
        assert np.abs(y.cpu().numpy() - x.astype(np.float64) @ U.T).max() < 3e-6 * math.sqrt(d)
    finally:
        K.kvq3_rotation_destroy(rot2)


WRITE_CASES = [
    dict(d=128, block=64, scale="f16", page=64, lens=(300, 1, 65), hkv=4, hq=16, flags=PAIR),
    dict(d=256, block=64, scale="f16", page=16, lens=(77, 300), hkv=2, hq=8, paged=True, flags=PAIR),
    dict(d=64, block=32, scale="e4m3", page=32, lens=(90,), hkv=2, hq=4, flags=PAIR),
    dict(d=128, block=64, scale="e4m3zp", page=64, lens=(200,), hkv=2, hq=8, flags=PAIR),
]


def _wid(c):
    return f"d{c['d']}-m{c['block']}-{c['scale']}-G{c['hq'] // c['hkv']}"


@pytest.mark.parametrize("cfg", WRITE_CASES, ids=_wid)
def test_write_pair_matches_oracle(cfg):
    c = Case(**cfg)
    k, v, si, ps = c.tokens()
    c.gpu_write(k, v, si, ps)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    stats = c.compare_written(k, v, si, ps)
    if stats["boundary_codes"] == 0 and stats["midpoint_blocks"] == 0:
        assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)


@pytest.mark.parametrize("cfg", [WRITE_CASES[0], WRITE_CASES[2]], ids=_wid)
def test_write_chunk_pair_matches_oracle(cfg):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    c = Case(**dict(cfg, lens=(333,)))
    k, v, si, ps = c.tokens()
    K.kvq3_write_chunk(c.rot.handle, c.desc, c.cache, torch.as_tensor(k, device="cuda"),
                       torch.as_tensor(v, device="cuda"), 0, 0, c.status)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    c.compare_written(k, v, si, ps)


def test_dequant_debug_pair_rotates_back():
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    c = Case(d=256, block=64, scale="f16", page=16, lens=(70,), hkv=2, hq=2, paged=True, flags=PAIR)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    out = torch.empty((50, 256), dtype=torch.float32, device="cuda")
    K.kvq3_dequant_debug(c.rot.handle, c.desc, c.cache, 0, 1, 1, 11, 50, out, None, c.status)
    xh, _, _ = O.read_rotated(c.pool_o, c.layout, 0, 1, 1, 11, 50, c.table)
    ref = xh @ c.U
    assert np.abs(out.cpu().numpy() - ref).max() < 1e-5 * np.abs(ref).max()
    assert c.device_status() == 0


DECODE_CASES = [
    dict(d=128, block=64, scale="f16", page=64, lens=(700, 1, 129, 64), hkv=2, hq=8, flags=PAIR),
    dict(d=256, block=64, scale="f16", page=16, lens=(300, 17, 1000), hkv=2, hq=16, paged=True, flags=PAIR),
    dict(d=128, block=64, scale="e4m3", page=64, lens=(900, 333), hkv=1, hq=16, flags=PAIR),
    dict(d=128, block=64, scale="e4m3zp", page=64, lens=(500,), hkv=2, hq=8, flags=PAIR),
]


@pytest.mark.parametrize("cfg", DECODE_CASES, ids=_wid)
def test_decode_pair_isolated_and_end_to_end(cfg):
    c = Case(**cfg)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = c.queries()
    e_iso = rel_err(c.gpu_decode(q), c.oracle_decode(q))
    assert c.device_status() == 0
    assert e_iso <= TOL_DECODE
    c.pool.zero_()
    c.gpu_write(k, v, si, ps)
    got, ref = c.gpu_decode(q), c.oracle_decode(q)
    assert c.device_status() == 0
    rms = math.sqrt(float(np.mean(ref ** 2)))
    slack = flip_bound(c, k, v, si, ps, q, differs=written_differences(c, k, v, si, ps))
    err = np.abs(got - ref).max(axis=-1)
    print(f"isolated {e_iso:.3e}, end to end {rel_err(got, ref):.3e}")
    assert np.all(err <= TOL_DECODE * rms + slack)


@pytest.mark.parametrize("kw,seq,pos0,n", [
    (dict(d=128, block=64, scale="f16", page=64, lens=(300,), hkv=2, hq=8, flags=PAIR), 0, 200, 100),  # tile kernel
    (dict(d=256, block=64, scale="f16", page=16, lens=(300, 180), hkv=2, hq=8, paged=True, flags=PAIR), 1, 100, 80),
])
def test_prefill_pair_matches_oracle(kw, seq, pos0, n):
    import torch
    c = Case(**kw)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = I.q_np(c.spec, n, c.hq, 7)
    qd = torch.as_tensor(q, device="cuda")
    out = torch.full((n, c.hq, c.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(c.K.kvq3_prefill_workspace_size(c.desc, c.hq, n), dtype=torch.uint8, device="cuda")
    c.K.kvq3_prefill_attn(c.rot.handle, c.desc, c.cache, seq, pos0, qd, out, ws, 0.0, c.status)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref = O.prefill(c.pool_o, c.layout, c.U, q, seq, pos0, c.table)
    assert c.device_status() == 0
    assert rel_err(got, ref) <= TOL_DECODE


def _desc(K, d, block, kind, bits=3):
    return K.CacheDesc(d, 1, block, bits, K.SCALE_TYPES[kind], 1e-6, 16, 1, 1, 0, 1)


def _sample(d, n, seed):
    return I.kv_rows_np(I.DataSpec(d, 1, seed, 0.03, 20.0), 0, 0, 0, 0, n)


@pytest.mark.parametrize("d,block,kind", [(128, 64, "f16"), (256, 64, "e4m3zp"), (64, 32, "f32")])
def test_calib_sse_pair_matches_oracle(d, block, kind):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    rot = K.Rotation(d, 42, PAIR)
    signs, q0, r0 = O.rotation_params_pair(d, 42)
    rng = np.random.default_rng(d)
    P = 4
    cand = rng.standard_normal((P, d // 4, 4))
    cand_r = rng.standard_normal((P, d // 4, 4))
    cand[0], cand_r[0] = q0, r0
    cand /= np.linalg.norm(cand, axis=2, keepdims=True)
    cand_r /= np.linalg.norm(cand_r, axis=2, keepdims=True)
    cand, cand_r = cand.astype(np.float32), cand_r.astype(np.float32)
    x = _sample(d, 300, 9)
    sse = torch.empty((P, d // block), dtype=torch.float64, device="cuda")
    K.kvq3_calib_sse_pair(rot.handle, _desc(K, d, block, kind), torch.as_tensor(cand, device="cuda"),
                          torch.as_tensor(cand_r, device="cuda"), torch.as_tensor(x, device="cuda"), sse)
    got = sse.cpu().numpy()
    for p in range(P):
        ref = O.calib_sse(x.astype(np.float64), signs, cand[p].astype(np.float64), block, kind,
                          quats_r=cand_r[p].astype(np.float64))
        assert np.all(np.abs(got[p] - ref) <= 1e-4 * ref), (p, got[p], ref)


def test_calibrate_so4_pair_lowers_the_error():
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    d, block, n = 128, 64, 1024
    rot = K.Rotation(d, 42, PAIR)
    signs, q0, r0 = O.rotation_params_pair(d, 42)
    desc = _desc(K, d, block, "f16")
    x = _sample(d, n, 21)
    xd = torch.as_tensor(x, device="cuda")
    ws = torch.empty(K.kvq3_calibrate_workspace_size(desc, 32), dtype=torch.uint8, device="cuda")
    q, r, sse = K.kvq3_calibrate_so4_pair(rot.handle, desc, xd, rounds=10, num_candidates=32, step=0.5, seed=7,
                                          workspace=ws)
    for a in (q, r):
        assert a.shape == (d // 4, 4) and np.all(np.abs(np.linalg.norm(a, axis=1) - 1.0) < 1e-6)
    before = O.calib_sse(x.astype(np.float64), signs, q0.astype(np.float32).astype(np.float64), block, "f16",
                         quats_r=r0.astype(np.float32).astype(np.float64))
    after = O.calib_sse(x.astype(np.float64), signs, q.astype(np.float64), block, "f16",
                        quats_r=r.astype(np.float64))
    print(f"pair: reconstruction error {before.sum():.4f} -> {after.sum():.4f}")
    assert np.all(after <= before * (1 + 1e-4))
    assert np.all(np.abs(sse - after) <= 1e-4 * after)
    # zero rounds return the start; a one-quaternion rotation starts from q_i = 1
    q0b, r0b, _ = K.kvq3_calibrate_so4_pair(rot.handle, desc, xd, rounds=0, num_candidates=2, step=0.5, seed=7,
                                            workspace=ws)
    assert np.array_equal(q0b, q0.astype(np.float32)) and np.array_equal(r0b, r0.astype(np.float32))
    rot1 = K.Rotation(d, 42, 3)
    _, r1, _ = K.kvq3_calibrate_so4_pair(rot1.handle, desc, xd, rounds=0, num_candidates=2, step=0.5, seed=7,
                                         workspace=ws)
    assert np.all(r1 == np.array([1, 0, 0, 0], np.float32))
    # the calibrated pair, as a rotation, runs through the write path
    rot2 = K.kvq3_rotation_create_from_params_pair(d, signs, q, r)
    try:
        y = torch.empty((n, d), dtype=torch.float32, device="cuda")
        K.kvq3_rotate(rot2, xd, y)
        U = O.rotation_matrix(signs, q.astype(np.float64), r.astype(np.float64))
        assert np.abs(y.cpu().numpy() - x.astype(np.float64) @ U.T).max() < 1e-4 * np.abs(x).max()
    finally:
        K.kvq3_rotation_destroy(rot2)

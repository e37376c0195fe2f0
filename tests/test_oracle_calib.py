"""Pins of the SO(4) calibration objective (oracle.calib_sse), CPU only.

"Orthogonally mixed 3-bit KV cache", Implementation notes: the rotations are
calibrated by minimising the reconstruction MSE after quantisation, each
SO(4) block a normalised quaternion.  The objective is pinned against the
write / read pipeline of the oracle's cache (an independent path through the
packed bytes), against an exactly representable input, and against its
separation over quantisation blocks, which the library's search relies on."""
import numpy as np
import pytest

import kvq3_inputs as I


def _sample(n=96, seed=5):
    spec = I.DataSpec(128, 1, seed, 0.03, 20.0)
    return I.kv_rows_np(spec, 0, 0, 0, 0, n)          # fp16 [n][128]


@pytest.mark.parametrize("kind,bits", [("f16", 3), ("e4m3", 3), ("f32", 4), ("f16", 2), ("e4m3zp", 3)])
def test_sse_equals_cache_round_trip_error(oracle, kind, bits):
    # sum_j sse_j = sum ||x - U^T x_hat||^2, x_hat read back from the packed cache
    x = _sample()
    signs, quats = oracle.rotation_params(128, 42)
    U = oracle.rotation_matrix(signs, quats)
    sse = oracle.calib_sse(x.astype(np.float64), signs, quats, 64, kind, bits)
    n = x.shape[0]
    L = oracle.Layout(128, 1, 64, kind, 16, 1, n // 16, n // 16, bits)
    pool = np.zeros(L.pool_bytes, np.uint8)
    oracle.write(pool, L, U, x[:, None], x[:, None], np.zeros(n, np.int32), np.arange(n))
    yh = oracle.read_rotated(pool, L, 0, 0, 0, 0, n)[0]
    err = float(((x.astype(np.float64) - yh @ U) ** 2).sum())
    assert sse.shape == (2,) and np.all(sse > 0)
    assert abs(sse.sum() - err) <= 1e-9 * err


def test_sse_zero_for_representable_vectors(oracle):
    # y = s * c per block with max|c| = 3 and eps = 0: the quantiser returns y exactly
    rng = np.random.default_rng(3)
    signs, quats = oracle.rotation_params(128, 7)
    U = oracle.rotation_matrix(signs, quats)
    c = rng.integers(-3, 4, (20, 128)).astype(np.float64)
    c[:, 0] = 3.0
    c[:, 64] = -3.0
    y = c * np.repeat(2.0 ** rng.integers(-4, 4, (20, 2)), 64, axis=1)
    x = y @ U                                            # U^T y, rows
    sse = oracle.calib_sse(x, signs, quats, 64, "f32", 3, eps=0.0)
    assert np.all(sse < 1e-20)


def test_sse_separates_over_quantisation_blocks(oracle):
    # moving the quaternions of the SO(4) blocks inside quantisation block 1
    # (coordinates 64..127: quaternions 16..31) changes sse[1] only
    x = _sample().astype(np.float64)
    signs, quats = oracle.rotation_params(128, 42)
    base = oracle.calib_sse(x, signs, quats, 64, "f16")
    q2 = quats.copy()
    rng = np.random.default_rng(1)
    q2[16:32] += 0.3 * rng.standard_normal((16, 4))
    q2[16:32] /= np.linalg.norm(q2[16:32], axis=1, keepdims=True)
    moved = oracle.calib_sse(x, signs, q2, 64, "f16")
    assert moved[0] == base[0] and moved[1] != base[1]


def test_sse_identity_quaternions_is_hadamard_error(oracle):
    # with identity quaternions B = I: the objective is the error of H D x alone
    x = _sample().astype(np.float64)
    signs, _ = oracle.rotation_params(128, 42)
    ident = np.tile([1.0, 0.0, 0.0, 0.0], (32, 1))
    y = x @ (oracle.hadamard_matrix(128) @ np.diag(signs.astype(np.float64))).T
    c, sq, _ = oracle.quantize(y, 64, float(np.float32(1e-6)), "f16")
    want = ((y - (c.reshape(-1, 2, 64) * sq[..., None]).reshape(y.shape)) ** 2).reshape(-1, 2, 64).sum(axis=(0, 2))
    assert np.allclose(oracle.calib_sse(x, signs, ident, 64, "f16"), want, rtol=1e-12)


def test_sse_pair_equals_cache_round_trip_error(oracle):
    # the two-quaternion blocks R_i = L(p_i) R(conj q_i): the objective still
    # equals the error of the oracle's write -> packed bytes -> read-back -> U^T
    x = _sample()
    signs, quats, quats_r = oracle.rotation_params_pair(128, 42)
    U = oracle.rotation_matrix(signs, quats, quats_r)
    sse = oracle.calib_sse(x.astype(np.float64), signs, quats, 64, "f16", 3, quats_r=quats_r)
    n = x.shape[0]
    L = oracle.Layout(128, 1, 64, "f16", 16, 1, n // 16, n // 16, 3)
    pool = np.zeros(L.pool_bytes, np.uint8)
    oracle.write(pool, L, U, x[:, None], x[:, None], np.zeros(n, np.int32), np.arange(n))
    yh = oracle.read_rotated(pool, L, 0, 0, 0, 0, n)[0]
    err = float(((x.astype(np.float64) - yh @ U) ** 2).sum())
    assert abs(sse.sum() - err) <= 1e-9 * err
    # identity right quaternions give the one-quaternion objective exactly
    ident = np.tile([1.0, 0.0, 0.0, 0.0], (32, 1))
    assert np.array_equal(oracle.calib_sse(x.astype(np.float64), signs, quats, 64, "f16", 3, quats_r=ident),
                          oracle.calib_sse(x.astype(np.float64), signs, quats, 64, "f16", 3))


def test_sse_pair_separates_over_quantisation_blocks(oracle):
    # moving the right quaternions inside quantisation block 0 changes sse[0] only
    x = _sample().astype(np.float64)
    signs, quats, quats_r = oracle.rotation_params_pair(128, 42)
    base = oracle.calib_sse(x, signs, quats, 64, "f16", quats_r=quats_r)
    r2 = quats_r.copy()
    r2[0:16] = np.roll(r2[0:16], 1, axis=1)
    moved = oracle.calib_sse(x, signs, quats, 64, "f16", quats_r=r2)
    assert moved[1] == base[1] and moved[0] != base[0]

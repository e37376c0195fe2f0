"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test targets a mistake the oracle could plausibly contain (a wrong sign,
a transposed operand, a dropped term, a wrong bit order).  CPU only."""
import math
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


# ------------------------------------------------------------- SplitMix64
def test_splitmix64_published_outputs(oracle):
    # First outputs of SplitMix64 seeded with 0 (Steele, Lea & Flood 2014; the
    # values printed with the public reference implementation).
    r = oracle.SplitMix64(0)
    assert [r.next() for _ in range(3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                            0x06C45D188009454F]


def test_uniform_pm1_range(oracle):
    r = oracle.SplitMix64(7)
    u = np.array([r.uniform_pm1() for _ in range(20000)])
    assert u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 0.02 and abs((u ** 2).mean() - 1 / 3) < 0.01


# ------------------------------------------------------------- Hadamard
@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 32, 128, 256])
def test_hadamard_is_normalised_sylvester(oracle, d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = oracle.hadamard_matrix(d)
    # Sylvester construction (scipy) scaled by 1/sqrt(d) -- "Orthogonal
    # Invariance in Activation Space", 3.1: H_d is the normalised Hadamard matrix.
    assert np.array_equal(H * math.sqrt(d), scipy_linalg.hadamard(d).astype(float))
    assert np.allclose(H, H.T, atol=0)
    assert np.abs(H @ H - np.eye(d)).max() < 1e-14     # self-inverse (3.1, item 3)


def test_hadamard_kron_recursion(oracle):
    # H_{2n} = H_2 (x) H_n, built independently of the popcount formula.
    H = np.array([[1.0]])
    h2 = np.array([[1.0, 1.0], [1.0, -1.0]]) / math.sqrt(2)
    for _ in range(6):
        H = np.kron(h2, H)
    assert np.abs(H - oracle.hadamard_matrix(64)).max() < 1e-15


@pytest.mark.parametrize("d", [4, 8, 16])
def test_recursive_fwht_equals_dense_bruteforce(oracle, d):
    # brute force over the whole basis: column j of the transform of e_j
    I = np.eye(d)
    F = np.stack([oracle.fwht_recursive(I[j]) for j in range(d)], axis=1)
    assert np.abs(F - oracle.hadamard_matrix(d)).max() < 1e-15
    x = np.random.default_rng(d).standard_normal((5, d))
    assert np.abs(oracle.fwht_recursive(x) - x @ oracle.hadamard_matrix(d).T).max() < 1e-13


# ------------------------------------------------------------- SO(4) blocks
def test_quaternion_units_follow_hamilton_rules(oracle):
    L = oracle.quat_left_matrix
    one, i, j, k = (1, 0, 0, 0), (0, 1, 0, 0), (0, 0, 1, 0), (0, 0, 0, 1)
    I4 = np.eye(4)
    assert np.array_equal(L(one), I4)
    for u in (i, j, k):
        assert np.array_equal(L(u) @ L(u), -I4)          # i^2 = j^2 = k^2 = -1
    assert np.array_equal(L(i) @ L(j), L(k))              # ij = k
    assert np.array_equal(L(j) @ L(k), L(i))              # jk = i
    assert np.array_equal(L(k) @ L(i), L(j))              # ki = j
    assert np.array_equal(L(i) @ L(j) @ L(k), -I4)        # ijk = -1
    # acting on a vector = quaternion product p*x: i * 1 = i
    assert np.array_equal(L(i) @ np.array([1.0, 0, 0, 0]), np.array([0, 1.0, 0, 0]))


def test_so4_blocks_gram_and_det(oracle):
    # "Orthogonally mixed 3-bit KV cache", Mathematical statement: R_i^T R_i = I_4,
    # det R_i = 1 (the MVP reports a Gram error of 8.9e-16).
    _, quats = oracle.rotation_params(256, 42)
    for p in quats:
        R = oracle.quat_left_matrix(p)
        assert np.abs(R.T @ R - np.eye(4)).max() < 1e-15
        assert abs(np.linalg.det(R) - 1.0) < 1e-14
    rng = np.random.default_rng(1)
    p = rng.standard_normal(4) * 3
    R = oracle.quat_left_matrix(p)
    n2 = float(p @ p)
    assert np.abs(R.T @ R - n2 * np.eye(4)).max() < 1e-12
    assert abs(np.linalg.det(R) - n2 ** 2) < 1e-9 * n2 ** 2


def test_right_multiplication_follows_hamilton_rules(oracle):
    # x -> x (x) u, basis products by Hamilton's rules: i j = k, j i = -k,
    # i k = -j, k j = -i; right multiplications compose in reverse order:
    # (x u) v = x (u v), so R(v) R(u) = R(u v)
    R, L = oracle.quat_right_matrix, oracle.quat_left_matrix
    e = np.eye(4)
    one, i, j, k = (1, 0, 0, 0), (0, 1, 0, 0), (0, 0, 1, 0), (0, 0, 0, 1)
    assert np.array_equal(R(one), e)
    assert np.array_equal(R(j) @ e[1], e[3])        # i j = k
    assert np.array_equal(R(i) @ e[2], -e[3])       # j i = -k
    assert np.array_equal(R(k) @ e[1], -e[2])       # i k = -j
    assert np.array_equal(R(j) @ e[3], -e[1])       # k j = -i
    assert np.array_equal(R(j) @ R(i), R(k))        # (x i) j = x (i j) = x k
    for u in (i, j, k):
        assert np.array_equal(R(u) @ R(u), -e)       # x u u = -x


def test_so4_pair_blocks(oracle):
    # The general rotation of R^4 as x -> p x conj(q) (Orthogonally mixed
    # 3-bit KV cache, Mathematical statement: R_i in SO(4)):
    rng = np.random.default_rng(11)
    L, R = oracle.quat_left_matrix, oracle.quat_right_matrix
    for _ in range(20):
        p = rng.standard_normal(4)
        q = rng.standard_normal(4)
        p /= np.linalg.norm(p)
        q /= np.linalg.norm(q)
        M = oracle.so4_pair_matrix(p, q)
        # orthogonal, det 1
        assert np.abs(M.T @ M - np.eye(4)).max() < 1e-15
        assert abs(np.linalg.det(M) - 1.0) < 1e-14
        # left and right multiplications commute (associativity of the product)
        assert np.abs(L(p) @ R(q) - R(q) @ L(p)).max() < 1e-15
        # (p, q) and (-p, -q) are the same rotation (the double cover)
        assert np.abs(oracle.so4_pair_matrix(-p, -q) - M).max() < 1e-15
        # q = 1 is the one-quaternion block L(p)
        assert np.array_equal(oracle.so4_pair_matrix(p, (1.0, 0, 0, 0)), L(p))
    # a simple rotation by theta in the (e0, e1) plane that fixes e2 and e3:
    # p = (cos t/2, sin t/2, 0, 0), q = conj(p).  No single left
    # multiplication gives it (p' x = x forces p' = 1), so the pair form
    # reaches rotations the one-quaternion blocks cannot.
    t = 0.7
    p = np.array([np.cos(t / 2), np.sin(t / 2), 0.0, 0.0])
    q = np.array([np.cos(t / 2), -np.sin(t / 2), 0.0, 0.0])
    want = np.eye(4)
    want[:2, :2] = [[np.cos(t), -np.sin(t)], [np.sin(t), np.cos(t)]]
    assert np.abs(oracle.so4_pair_matrix(p, q) - want).max() < 1e-15


def test_rotation_params_pair(oracle):
    # the pair rotation keeps the one-quaternion draws (signs, then the left
    # quaternions) and draws one more point of S^3 per block afterwards
    s, q = oracle.rotation_params(128, 42)
    s2, p2, r2 = oracle.rotation_params_pair(128, 42)
    assert np.array_equal(s, s2) and np.array_equal(q, p2)
    assert r2.shape == (32, 4) and np.abs(np.linalg.norm(r2, axis=1) - 1).max() < 1e-15
    rng = oracle.SplitMix64(42)
    for _ in range(128):
        rng.next()
    for _ in range(32):
        oracle.marsaglia_s3(rng)
    assert np.array_equal(np.array(oracle.marsaglia_s3(rng)), r2[0])
    U = oracle.rotation_matrix(s2, p2, r2)
    assert np.abs(U.T @ U - np.eye(128)).max() < 1e-14
    # block i of U is R_i = L(p_i) R(conj q_i) applied after H D
    HD = oracle.hadamard_matrix(128) @ np.diag(s2.astype(np.float64))
    B = U @ HD.T
    assert np.abs(B[4:8, 4:8] - oracle.so4_pair_matrix(p2[1], r2[1])).max() < 1e-14
    assert np.abs(B[4:8, 8:12]).max() < 1e-14


def test_rotation_params_shape_and_flags(oracle):
    s, q = oracle.rotation_params(128, 42)
    assert s.shape == (128,) and set(np.unique(s)) == {-1, 1}
    assert q.shape == (32, 4)
    assert np.abs(np.linalg.norm(q, axis=1) - 1).max() < 1e-15
    s0, q0 = oracle.rotation_params(128, 42, use_sign=False, use_so4=False)
    assert np.all(s0 == 1) and np.all(q0 == [1, 0, 0, 0])
    s1, q1 = oracle.rotation_params(128, 43)
    assert not np.array_equal(s, s1)
    # the first d draws decide the signs: top bit set -> -1
    r = oracle.SplitMix64(42)
    assert [(-1 if r.next() >> 63 else 1) for _ in range(4)] == list(s[:4])


def test_marsaglia_points_uniform_on_s3(oracle):
    r = oracle.SplitMix64(5)
    P = np.array([oracle.marsaglia_s3(r) for _ in range(20000)])
    assert np.abs(np.linalg.norm(P, axis=1) - 1).max() < 1e-15
    # uniform on S^3: every coordinate has mean 0 and second moment 1/4
    assert np.abs(P.mean(0)).max() < 0.02
    assert np.abs((P ** 2).mean(0) - 0.25).max() < 0.01


# ------------------------------------------------------------- U and invariance
@pytest.mark.parametrize("d,flags", [(4, 3), (8, 3), (128, 3), (128, 1), (256, 3), (256, 0)])
def test_U_orthogonal(oracle, d, flags):
    s, q = oracle.rotation_params(d, 42, bool(flags & 1), bool(flags & 2))
    U = oracle.rotation_matrix(s, q)
    assert np.abs(U.T @ U - np.eye(d)).max() < 1e-14     # MVP: inverse error 1.6e-15


def test_U_order_is_B_H_D(oracle):
    # columns: U e_j = B H (sigma_j e_j) -> the sign of column j is sigma_j times
    # the column of B H; with B = I the first row of U is sigma/sqrt(d).
    s, _ = oracle.rotation_params(16, 9)
    U = oracle.rotation_matrix(s, np.tile([1.0, 0, 0, 0], (4, 1)))
    assert np.allclose(U[0], s / 4.0, atol=0)
    s2, q2 = oracle.rotation_params(16, 9)
    U2 = oracle.rotation_matrix(s2, q2)
    B = oracle.block_so4_matrix(q2)
    assert np.abs(U2 - B @ U).max() < 1e-15            # B applied last


def test_dot_product_invariance(oracle):
    # (Uq)^T (Uk) = q^T k ("Orthogonally mixed 3-bit KV cache", Key formulas;
    # the MVP reports 7.1e-15)
    s, q = oracle.rotation_params(128, 42)
    U = oracle.rotation_matrix(s, q)
    rng = np.random.default_rng(0)
    a, b = rng.standard_normal((2, 128))
    assert abs((U @ a) @ (U @ b) - a @ b) < 1e-12


def test_unquantised_rotated_attention_equals_plain(oracle):
    # "Orthogonal Invariance in Activation Space", 2.3: rotating q, k and v by
    # the same orthogonal matrix and v back by U^T leaves attention unchanged.
    s, qq = oracle.rotation_params(128, 3)
    U = oracle.rotation_matrix(s, qq)
    rng = np.random.default_rng(2)
    k = rng.standard_normal((300, 128)) * 4
    v = rng.standard_normal((300, 128))
    q = rng.standard_normal(128)
    ref = oracle.attention_plain(q, k, v, 1 / math.sqrt(128))
    got = oracle.attention_rotated(U, q, k @ U.T, v @ U.T, 1 / math.sqrt(128))
    assert np.abs(got - ref).max() < 1e-13


# ------------------------------------------------------------- scale types
def test_e4m3_against_torch_float8(oracle):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(0, 448, 5000), np.exp(rng.uniform(-14, 6, 5000)),
                           [0.0, 2.0 ** -9, 2.0 ** -10, 2.0 ** -6, 448.0, 447.9, 0.3]])
    mine = oracle.round_e4m3(vals)
    ref = torch.tensor(vals, dtype=torch.float64).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(mine, ref)
    # every finite positive code round-trips through encode/decode
    b = np.arange(1, 127, dtype=np.uint8)
    v = oracle.decode_e4m3(b)
    assert np.array_equal(oracle.encode_e4m3(v), b)
    assert np.array_equal(oracle.round_e4m3(v), v)
    assert oracle.round_e4m3(1e6) == 448.0 and oracle.round_e4m3(464.1) == 448.0
    assert oracle.decode_e4m3(0x7E) == 448.0 and oracle.decode_e4m3(1) == 2.0 ** -9


def test_f16_saturates(oracle):
    assert oracle.round_f16(1e9) == 65504.0
    assert oracle.round_f16(65519.0) == 65504.0
    assert oracle.round_f16(1.0 + 2 ** -11) == 1.0          # tie to even
    assert oracle.round_f16(1.0 + 3 * 2 ** -11) == 1.0 + 2 ** -9


def test_midpoint_distance(oracle):
    q = 2.0 ** -10
    assert oracle.scale_midpoint_distance(1.0 + q / 2, "f16") == 0.0
    assert oracle.scale_midpoint_distance(1.0, "f16") == pytest.approx(q / 2)
    assert oracle.scale_midpoint_distance(1.0 + 1 / 16, "e4m3") == 0.0
    assert np.isinf(oracle.scale_midpoint_distance(3.0, "f32"))


# ------------------------------------------------------------- quantiser
@pytest.mark.parametrize("kind", ["f32", "f16", "e4m3"])
@pytest.mark.parametrize("block", [32, 64])
def test_quantiser_error_bound(oracle, kind, block):
    # |x - s_q c| <= s_q / 2 wherever |x/s_q| <= 3.5, codes in [-3, 3]
    rng = np.random.default_rng(block)
    x = rng.standard_normal((400, 128)) * np.exp(rng.uniform(-3, 3, (400, 1)))
    c, sq, s = oracle.quantize(x, block, 1e-6, kind)
    assert c.min() >= -3 and c.max() <= 3
    xb = x.reshape(400, -1, block)
    err = np.abs(xb - sq[..., None] * c.reshape(xb.shape))
    inside = np.abs(xb) <= 3.5 * sq[..., None]
    assert np.all(err[inside] <= sq[..., None].repeat(block, -1)[inside] / 2 * (1 + 1e-12))
    assert np.allclose(s, (np.abs(xb).max(-1) + 1e-6) / 3, rtol=1e-15)
    if kind == "f32":
        assert np.array_equal(c.reshape(xb.shape).max(-1).clip(0) + (-c.reshape(xb.shape)).max(-1).clip(0) > 0,
                              np.ones(sq.shape, bool))
        # the block's extreme element always lands on +-3 with an fp32 scale
        amax = np.argmax(np.abs(xb), axis=-1)
        cm = np.take_along_axis(c.reshape(xb.shape), amax[..., None], -1)[..., 0]
        assert np.all(np.abs(cm) == 3)


def test_quantiser_quadratic_error_scaling(oracle):
    # with eps = 0, scaling x by 2^k scales the scales by 2^k and leaves the codes
    # unchanged, so MSE/amplitude^2 is constant (the MVP's "quadratic error
    # scaling": MSE/amp^2 varied by 5.4e-12)
    x = np.random.default_rng(4).standard_normal((50, 128))
    c0, s0, _ = oracle.quantize(x, 64, 0.0, "f32")
    ratios = []
    for k in range(-6, 7):
        a = 2.0 ** k
        c, s, _ = oracle.quantize(a * x, 64, 0.0, "f32")
        assert np.array_equal(c, c0) and np.array_equal(s, s0 * a)
        xh = (c.reshape(50, 2, 64) * s[..., None]).reshape(50, 128)
        ratios.append(((xh - a * x) ** 2).mean() / a ** 2)
    assert np.ptp(ratios) < 1e-15


def test_quantiser_zero_and_tiny_blocks(oracle):
    x = np.zeros((1, 64))
    c, sq, _ = oracle.quantize(x, 32, 1e-6, "f32")
    assert np.all(c == 0) and np.allclose(sq, np.float32(1e-6 / 3))
    # an E4M3 scale that underflows to 0 gives zero codes
    c, sq, _ = oracle.quantize(np.full((1, 32), 1e-4), 32, 0.0, "e4m3")
    assert sq[0, 0] == 0.0 and np.all(c == 0)


def test_quantiser_clip_fires_with_rounded_down_scale(oracle):
    # an E4M3 scale rounded down makes |x/s_q| > 3 for the block maximum: the
    # clip keeps the code at 3 (s = 2.0625*... rounds to 2.0)
    x = np.zeros((1, 32))
    x[0, 0] = 3 * 2.0624
    c, sq, s = oracle.quantize(x, 32, 0.0, "e4m3")
    assert sq[0, 0] == 2.0 and c[0, 0] == 3 and x[0, 0] / sq[0, 0] > 3


# ------------------------------------------------------------- packing
def _golden():
    rows = []
    for line in open(os.path.join(HERE, "golden", "pack3_worked_examples.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, d, codes, *hexb = line.split()
        rows.append((name, int(d), [int(t) for t in codes.split(",")], bytes.fromhex("".join(hexb))))
    return rows


def test_pack_worked_examples(oracle):
    for name, d, group, b in _golden():
        codes = np.array(group * (d // 8), dtype=np.int8)[None]
        assert oracle.pack_codes(codes)[0].tobytes() == b * (d // 8), name


def test_unit_vector_writes_all_threes(oracle):
    # end to end through U: k = +-e_0 with D = I, B = I -> every code is +-3
    for sgn, name in ((1, "unit_e0"), (-1, "unit_minus_e0")):
        s, q = oracle.rotation_params(128, 42, False, False)
        U = oracle.rotation_matrix(s, q)
        x = U @ (sgn * np.eye(128)[0])
        c, sq, _ = oracle.quantize(x[None], 64, 1e-6, "f32")
        assert np.all(c == 3 * sgn)
        want = dict((r[0], r[3]) for r in _golden())[name]
        assert oracle.pack_codes(c)[0].tobytes() == want * 16


def test_pack_exhaustive_roundtrip(oracle):
    # all 7^8 = 5,764,801 groups of eight codes in [-3, 3]
    g = np.indices((7,) * 8).reshape(8, -1).T.astype(np.int8) - 3
    b = oracle.pack_codes(g)
    assert b.shape == (7 ** 8, 3)
    assert np.array_equal(oracle.unpack_codes(b, 8), g)
    # distinct groups give distinct byte strings
    key = b[:, 0].astype(np.int64) | (b[:, 1].astype(np.int64) << 8) | (b[:, 2].astype(np.int64) << 16)
    assert len(np.unique(key)) == 7 ** 8


def test_pack_bit_positions_bruteforce(oracle):
    # element j at bits 3j..3j+2: check bit by bit with Python integers
    rng = np.random.default_rng(5)
    for d in (8, 64, 128, 256):
        c = rng.integers(-3, 4, (3, d)).astype(np.int8)
        b = oracle.pack_codes(c)
        for r in range(3):
            acc = int.from_bytes(b[r].tobytes(), "little")
            for j in range(d):
                v = (acc >> (3 * j)) & 7
                assert (v - 8 if v >= 4 else v) == c[r, j]


# ------------------------------------------------------------- storage accounting
def test_storage_accounting(oracle):
    def bits(scale, m, d=128, P=64):
        L = oracle.Layout(d, 1, m, scale, P, 1, 1, 1)
        return 8 * L.record_bytes / (P * d)
    # "Hardware-Fused Fast Hadamard Transforms ...": 3.125 effective bits with an
    # FP8 header per 64 elements, 40 GB (fp16) -> 7.8 GB for a 70B model at 128K
    assert bits("e4m3", 64) == 3.125
    gib = 80 * 8 * 128 * 2 * 2 * 131072 / 2 ** 30          # layers*kvheads*d*K,V*2B*tokens
    assert gib == 40.0 and gib * 3.125 / 16 == 7.8125
    # the MVP's 1.45x with fp32 scales matches one scale per SO(4) block (m = 4)
    assert round(16 / (3 + 32 / 4), 2) == 1.45
    assert bits("f32", 64) == 3.5 and bits("f16", 64) == 3.25 and bits("f32", 32) == 4.0
    # record sizes of the paged layout with 16-token pages, fp16 scales
    assert oracle.Layout(128, 1, 64, "f16", 16, 1, 1, 1).record_bytes == 832
    assert oracle.Layout(256, 1, 64, "f16", 16, 1, 1, 1).record_bytes == 1664


# ------------------------------------------------------------- bit widths 2 and 4
def _golden24():
    rows = []
    for line in open(os.path.join(HERE, "golden", "pack24_worked_examples.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, bits, d, codes, *hexb = line.split()
        rows.append((name, int(bits), int(d), [int(t) for t in codes.split(",")], bytes.fromhex("".join(hexb))))
    return rows


def test_pack24_worked_examples(oracle):
    rows = _golden24()
    assert {r[1] for r in rows} == {2, 4}
    for name, bits, d, group, b in rows:
        codes = np.array(group * (d // 8), dtype=np.int8)[None]
        assert oracle.pack_codes(codes, bits)[0].tobytes() == b * (d // 8), name
        assert np.array_equal(oracle.unpack_codes(np.frombuffer(b * (d // 8), np.uint8)[None], d, bits), codes), name


@pytest.mark.parametrize("bits", [2, 4])
def test_unit_vector_writes_all_qmax(oracle, bits):
    golden = dict((r[0], r[4]) for r in _golden24())
    for sgn, name in ((1, f"unit_e0_{bits}"), (-1, f"unit_minus_e0_{bits}")):
        s, q = oracle.rotation_params(128, 42, False, False)
        U = oracle.rotation_matrix(s, q)
        c, sq, _ = oracle.quantize((U @ (sgn * np.eye(128)[0]))[None], 64, 1e-6, "f32", bits)
        assert np.all(c == sgn * ((1 << (bits - 1)) - 1))
        assert oracle.pack_codes(c, bits)[0].tobytes() == golden[name] * 16


def test_quantiser_b24_hand_examples(oracle):
    # b = 4: block maximum 7 with eps = 0 gives s = 7/7 = 1; 3.5 rounds half to even (4)
    x = np.zeros((1, 32))
    x[0, :5] = [7.0, 3.5, -1.0, 0.0, -2.5]
    c, sq, s = oracle.quantize(x, 32, 0.0, "f32", 4)
    assert s[0, 0] == 1.0 and sq[0, 0] == 1.0
    assert list(c[0, :5]) == [7, 4, -1, 0, -2]
    # b = 2: divisor 1, so s is the block maximum itself: 2 -> x/s = 1, .25, -.75, .5, .2
    x = np.zeros((1, 32))
    x[0, :5] = [2.0, 0.5, -1.5, 1.0, 0.4]
    c, sq, s = oracle.quantize(x, 32, 0.0, "f32", 2)
    assert s[0, 0] == 2.0 and list(c[0, :5]) == [1, 0, -1, 0, 0]
    with pytest.raises(ValueError):
        oracle.quantize(x, 32, 0.0, "f32", 5)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kind", ["f32", "f16", "e4m3"])
def test_quantiser_error_bound_b24(oracle, bits, kind):
    # |x - s_q c| <= s_q / 2 wherever |x/s_q| <= qmax + 1/2, codes in [-qmax, qmax]
    qm = (1 << (bits - 1)) - 1
    rng = np.random.default_rng(bits)
    x = rng.standard_normal((300, 128)) * np.exp(rng.uniform(-3, 3, (300, 1)))
    c, sq, s = oracle.quantize(x, 64, 1e-6, kind, bits)
    assert c.min() >= -qm and c.max() <= qm
    xb = x.reshape(300, -1, 64)
    assert np.allclose(s, (np.abs(xb).max(-1) + 1e-6) / qm, rtol=1e-15)
    err = np.abs(xb - sq[..., None] * c.reshape(xb.shape))
    inside = np.abs(xb) <= (qm + 0.5) * sq[..., None]
    assert np.all(err[inside] <= sq[..., None].repeat(64, -1)[inside] / 2 * (1 + 1e-12))
    if kind == "f32":   # the block's extreme element lands on +-qmax
        amax = np.argmax(np.abs(xb), axis=-1)
        cm = np.take_along_axis(c.reshape(xb.shape), amax[..., None], -1)[..., 0]
        assert np.all(np.abs(cm) == qm)


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_b24_exhaustive_roundtrip(oracle, bits):
    # every b-bit value (including -2^(b-1), which the quantiser never writes)
    # in every position of an 8-element group
    n = 1 << bits
    vals = np.arange(n) - n // 2
    g = np.indices((n,) * (8 if bits == 2 else 4)).reshape(8 if bits == 2 else 4, -1).T
    g = np.concatenate([g, g], axis=1)[:, :8] if bits == 4 else g
    g = vals[g].astype(np.int8)
    b = oracle.pack_codes(g, bits)
    assert b.shape == (len(g), bits)
    assert np.array_equal(oracle.unpack_codes(b, 8, bits), g)


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_b24_bit_positions_bruteforce(oracle, bits):
    qm = (1 << (bits - 1)) - 1
    rng = np.random.default_rng(50 + bits)
    for d in (8, 64, 128, 256):
        c = rng.integers(-qm, qm + 1, (3, d)).astype(np.int8)
        b = oracle.pack_codes(c, bits)
        assert b.shape == (3, bits * d // 8)
        for r in range(3):
            acc = int.from_bytes(b[r].tobytes(), "little")
            for j in range(d):
                v = (acc >> (bits * j)) & ((1 << bits) - 1)
                assert (v - (1 << bits) if v >= (1 << (bits - 1)) else v) == c[r, j]


def test_storage_accounting_b24(oracle):
    # "Orthogonal Invariance in Activation Space", 3.3: d*b bits of codes per
    # vector; 4.2: 48 bytes of data for d = 128 at b = 3 (so 64 at b = 4, 32 at b = 2)
    for bits, cb in ((2, 32), (3, 48), (4, 64)):
        L = oracle.Layout(128, 1, 64, "f16", 16, 1, 1, 1, bits)
        assert L.code_bytes == cb
        assert L.record_bytes == 16 * (2 * 2 + cb)
        assert 8 * L.record_bytes / (16 * 128) == bits + 0.25


# ------------------------------------------------------------- asymmetric variant ("e4m3zp")
def test_asym_hand_example(oracle):
    # "Hardware-Fused Fast Hadamard Transforms ...": unsigned 3-bit codes with
    # an FP8 scale and zero point per block.  min -1, max 2.5 (eps = 0):
    # s = 3.5/7 = 0.5 and z = -1, both exact in E4M3; u = (x + 1)/0.5, half to even
    x = np.zeros((1, 32))
    x[0, :5] = [-1.0, 2.5, 0.0, 0.25, 1.0]
    u, sz, s = oracle.quantize_asym(x, 32, 0.0)
    assert s[0, 0] == 0.5 and tuple(sz[0, 0]) == (0.5, -1.0)
    assert list(u[0, :5]) == [0, 7, 2, 2, 4] and np.all(u[0, 5:] == 2)
    # bytes: scale 0.5 = 0x30, zero point -1 = 0xB8 (sign | exponent 7 << 3)
    assert oracle.encode_scales(sz, "e4m3zp").tobytes() == bytes([0x30, 0xB8])
    # unsigned codes use the same little-endian stream: u = 0,7,2,2,4,2,2,2 sets
    # bits 3-5, 7 | 10, 14 | 16, 19, 22 -> B8 44 49
    assert oracle.pack_codes(u[:, :8], 3)[0].tobytes() == bytes([0xB8, 0x44, 0x49])
    assert np.array_equal(oracle.unpack_codes(oracle.pack_codes(u, 3), 32, 3, signed=False), u)


def test_e4m3_signed_round_trip(oracle):
    b = np.array([v for v in range(256) if (v & 0x7F) != 0x7F], np.uint8)
    vals = oracle.decode_e4m3(b)
    assert np.array_equal(oracle.encode_e4m3_signed(vals)[vals != 0], b[vals != 0])
    assert np.array_equal(oracle.round_e4m3_signed(vals), vals)
    assert oracle.round_e4m3_signed(-3.3) == -oracle.round_e4m3(3.3)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_asym_error_bound(oracle, bits):
    # |x - (s_q u + z_q)| <= s_q/2 wherever (x - z_q)/s_q lies in [-1/2, 2^b - 1/2]
    top = (1 << bits) - 1
    rng = np.random.default_rng(60 + bits)
    x = rng.standard_normal((300, 128)) * np.exp(rng.uniform(-3, 3, (300, 1))) + rng.uniform(-1, 1, (300, 1))
    u, sz, s = oracle.quantize_asym(x, 64, 1e-6, bits)
    assert u.min() >= 0 and u.max() <= top
    xb = x.reshape(300, -1, 64)
    assert np.allclose(s, (xb.max(-1) - xb.min(-1) + 1e-6) / top, rtol=1e-15)
    sq, zq = sz[..., 0:1], sz[..., 1:2]
    xh = u.reshape(xb.shape) * sq + zq
    r = (xb - zq) / sq
    inside = (r >= -0.5) & (r <= top + 0.5)
    err = np.abs(xb - xh)
    assert np.all(err[inside] <= np.broadcast_to(sq, xb.shape)[inside] / 2 * (1 + 1e-12))
    assert inside.mean() > 0.95


def test_asym_storage_and_error_against_symmetric(oracle):
    # 2 header bytes per 64-element block: 3.25 bits per element (the page's
    # 3.125 counts one header byte); on the rotated outlier data the
    # asymmetric codes (8 levels over [min, max]) give a lower error than the
    # symmetric E4M3 ones (7 levels over [-max|x|, max|x|])
    L = oracle.Layout(128, 1, 64, "e4m3zp", 16, 1, 1, 1)
    assert L.record_bytes == 16 * (2 * 2 + 48) and 8 * L.record_bytes / (16 * 128) == 3.25
    import kvq3_inputs as I
    spec = I.DataSpec(128, 1, 79, 0.03, 20.0)
    x = I.kv_rows_np(spec, 0, 0, 0, 0, 512).astype(np.float64)
    s, q = oracle.rotation_params(128, 42)
    U = oracle.rotation_matrix(s, q)
    y = x @ U.T
    c, sq, _ = oracle.quantize(y, 64, 1e-6, "e4m3")
    ys = (c.reshape(-1, 2, 64) * sq[..., None]).reshape(y.shape)
    u, sz, _ = oracle.quantize_asym(y, 64, 1e-6)
    ya = (u.reshape(-1, 2, 64) * sz[..., 0:1] + sz[..., 1:2]).reshape(y.shape)
    mse_s, mse_a = np.mean((ys - y) ** 2), np.mean((ya - y) ** 2)
    assert mse_a < 0.8 * mse_s


def test_asym_edge_cases(oracle):
    # a constant block: s = eps/7 underflows E4M3 to 0, so every code is 0 and
    # x_hat = z_q = E4M3(c) (2.3 -> 2.25: the E4M3 grid near 2 is 0.25)
    x = np.full((1, 32), 2.3)
    u, sz, s = oracle.quantize_asym(x, 32, 1e-6)
    assert sz[0, 0, 0] == 0.0 and sz[0, 0, 1] == 2.25 and np.all(u == 0)
    # an all-positive block: z = min = 1, s = (8 - 1)/7 = 1 (eps = 0), codes x - 1
    x = np.array([[1.0, 8.0, 4.0, 2.0] + [5.0] * 28])
    u, sz, _ = oracle.quantize_asym(x, 32, 0.0)
    assert tuple(sz[0, 0]) == (1.0, 1.0) and list(u[0, :4]) == [0, 7, 3, 1] and np.all(u[0, 4:] == 4)
    # a zero point beyond E4M3's range saturates to -448: the block minimum
    # then lies below z_q and its code clips to 0
    x = np.zeros((1, 32))
    x[0, 0] = -1000.0
    u, sz, s = oracle.quantize_asym(x, 32, 0.0)
    assert sz[0, 0, 1] == -448.0 and u[0, 0] == 0
    assert sz[0, 0, 0] == oracle.round_e4m3(1000.0 / 7)                 # 142.857.. -> 144
    assert np.all(u[0, 1:] == np.clip(np.rint(448.0 / sz[0, 0, 0]), 0, 7))

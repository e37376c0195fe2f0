"""Oracle write/read/decode pins: layout round trips, status bits and the
special cases of attention that have closed forms.  CPU only."""
import math

import numpy as np
import pytest

import kvq3_inputs as I


def _setup(oracle, d=128, H=2, block=64, scale="f16", P=16, B=2, maxp=4, paged=False, seed=42, bits=3):
    s, q = oracle.rotation_params(d, seed)
    U = oracle.rotation_matrix(s, q)
    num_pages = B * maxp + (3 if paged else 0)
    L = oracle.Layout(d, H, block, scale, P, B, maxp, num_pages, bits)
    pool = np.zeros(L.pool_bytes, np.uint8)
    table = None
    if paged:
        ids = I.shuffled_page_ids_np(11, num_pages)
        table = ids[:B * maxp].reshape(B, maxp)
    return U, L, pool, table


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("scale", ["f32", "f16", "e4m3"])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_write_read_roundtrip(oracle, paged, scale, bits):
    U, L, pool, table = _setup(oracle, scale=scale, paged=paged, bits=bits)
    rng = np.random.default_rng(0)
    n = 40
    k = (rng.standard_normal((n, 2, 128)) * 3).astype(np.float16)
    v = rng.standard_normal((n, 2, 128)).astype(np.float16)
    seq = np.repeat([0, 1], n // 2)
    pos = np.concatenate([np.arange(20), np.arange(20) + 17])
    assert oracle.write(pool, L, U, k, v, seq, pos, table) == 0
    for b in (0, 1):
        sel = seq == b
        p0 = int(pos[sel][0])
        for h in (0, 1):
            for which, src in ((0, k), (1, v)):
                xh, c, sc = oracle.read_rotated(pool, L, b, h, which, p0, 20, table)
                x = src[sel, h].astype(np.float64) @ U.T
                c2, sq2, _ = oracle.quantize(x, 64, 1e-6, scale, bits)
                assert np.array_equal(c, c2) and np.array_equal(sc, sq2)


def test_layout_byte_positions(oracle):
    # a single token at position 17 of sequence 1, kv head 1, V record, P = 16:
    # contiguous page id 1*4 + 1 = 5, slot 1
    U, L, pool, _ = _setup(oracle, scale="f32", P=16)
    k = np.zeros((1, 2, 128), np.float16)
    v = np.zeros((1, 2, 128), np.float16)
    v[0, 1, 0] = 1.0
    oracle.write(pool, L, U, k, v, np.array([1]), np.array([17]))
    rec = 5 * L.page_bytes + (1 * 2 + 1) * L.record_bytes
    hdr = rec + 1 * 2 * 4
    codes = rec + 16 * 2 * 4 + 1 * 48
    x = U @ np.eye(128)[0]
    c, sq, _ = oracle.quantize(x[None], 64, 1e-6, "f32")
    assert pool[hdr:hdr + 8].tobytes() == sq.astype("<f4").tobytes()
    assert pool[codes:codes + 48].tobytes() == oracle.pack_codes(c)[0].tobytes()
    # zero vectors (K of both heads, V of head 0) are stored too: scale eps/3,
    # codes 0.  Nothing outside slot 1 of page 5 changes.
    touched = np.zeros(L.pool_bytes, bool)
    for r in range(4):
        h0 = 5 * L.page_bytes + r * L.record_bytes + 1 * 2 * 4
        touched[h0:h0 + 8] = True
        if r != 3:
            assert np.allclose(pool[h0:h0 + 8].view("<f4"), np.float32(np.float32(1e-6) / 3))
    touched[codes:codes + 48] = True
    assert not np.any(pool[~touched])


@pytest.mark.parametrize("paged", [False, True])
def test_write_read_roundtrip_asym(oracle, paged):
    U, L, pool, table = _setup(oracle, scale="e4m3zp", paged=paged)
    rng = np.random.default_rng(2)
    n = 30
    k = (rng.standard_normal((n, 2, 128)) * 3 + 1).astype(np.float16)
    v = rng.standard_normal((n, 2, 128)).astype(np.float16)
    seq = np.repeat([0, 1], n // 2)
    pos = np.concatenate([np.arange(15), np.arange(15) + 9])
    assert oracle.write(pool, L, U, k, v, seq, pos, table) == 0
    for b in (0, 1):
        sel = seq == b
        for h in (0, 1):
            for which, src in ((0, k), (1, v)):
                xh, u, sz = oracle.read_rotated(pool, L, b, h, which, int(pos[sel][0]), 15, table)
                x = src[sel, h].astype(np.float64) @ U.T
                u2, sz2, _ = oracle.quantize_asym(x, 64, 1e-6)
                assert np.array_equal(u, u2) and np.array_equal(sz, sz2)
                assert np.allclose(xh, (u2.reshape(15, 2, 64) * sz2[..., 0:1] + sz2[..., 1:2]).reshape(15, 128))


def test_decode_single_token_returns_value_asym(oracle):
    U, L, pool, _ = _setup(oracle, scale="e4m3zp")
    rng = np.random.default_rng(4)
    _fill(oracle, L, pool, U, None, [1, 1], rng)
    q = rng.standard_normal((2, 4, 128)).astype(np.float16)
    out = oracle.decode(pool, L, U, q, np.array([1, 1]))
    for b in range(2):
        for h in range(4):
            vh = oracle.read_rotated(pool, L, b, h // 2, 1, 0, 1)[0][0]
            assert np.abs(out[b, h] - U.T @ vh).max() < 1e-12


@pytest.mark.parametrize("bits", [2, 4])
def test_layout_byte_positions_b24(oracle, bits):
    # the b-bit code string of slot 1 sits b*d/8 bytes after slot 0's; one
    # token at position 17 of sequence 1, kv head 1, V record, P = 16 (page 5)
    U, L, pool, _ = _setup(oracle, scale="f32", P=16, bits=bits)
    cb = bits * 128 // 8
    assert L.code_bytes == cb and L.record_bytes == 16 * (2 * 4 + cb)
    k = np.zeros((1, 2, 128), np.float16)
    v = np.zeros((1, 2, 128), np.float16)
    v[0, 1, 0] = 1.0
    oracle.write(pool, L, U, k, v, np.array([1]), np.array([17]))
    rec = 5 * L.page_bytes + (1 * 2 + 1) * L.record_bytes
    codes = rec + 16 * 2 * 4 + 1 * cb
    c, _, _ = oracle.quantize((U @ np.eye(128)[0])[None], 64, 1e-6, "f32", bits)
    assert np.abs(c).max() == (1 << (bits - 1)) - 1
    assert pool[codes:codes + cb].tobytes() == oracle.pack_codes(c, bits)[0].tobytes()
    assert not pool[codes + cb:codes + 2 * cb].any() and not pool[codes - cb:codes].any()


def test_write_status_bits(oracle):
    U, L, pool, table = _setup(oracle, paged=True)
    k = np.ones((5, 2, 128), np.float16)
    bad_table = table.copy()
    bad_table[0, 1] = 10 ** 6
    st = oracle.write(pool, L, U, k, k, np.array([0, 5, 0, 1, 0]), np.array([3, 0, 999, -1, 20]),
                      bad_table)
    assert st == oracle.ST_BAD_SEQ | oracle.ST_BAD_POS | oracle.ST_BAD_PAGE
    # only the first token (valid) was written
    assert oracle.read_rotated(pool, L, 0, 0, 0, 3, 1, bad_table)[1].any()


def _fill(oracle, L, pool, U, table, lens, rng, kscale=3.0):
    for b, n in enumerate(lens):
        k = (rng.standard_normal((n, L.num_kv_heads, L.d)) * kscale).astype(np.float16)
        v = rng.standard_normal((n, L.num_kv_heads, L.d)).astype(np.float16)
        oracle.write(pool, L, U, k, v, np.full(n, b), np.arange(n), table)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_decode_single_token_returns_value(oracle, bits):
    # N = 1: softmax weight 1, so o = U^T v_hat
    U, L, pool, _ = _setup(oracle, bits=bits)
    rng = np.random.default_rng(1)
    _fill(oracle, L, pool, U, None, [1, 1], rng)
    q = rng.standard_normal((2, 4, 128)).astype(np.float16)
    out = oracle.decode(pool, L, U, q, np.array([1, 1]))
    for b in range(2):
        for h in range(4):
            vh = oracle.read_rotated(pool, L, b, h // 2, 1, 0, 1)[0][0]
            assert np.abs(out[b, h] - U.T @ vh).max() < 1e-12


@pytest.mark.parametrize("scale,bits", [("f16", 3), ("f16", 2), ("f32", 4), ("e4m3zp", 3)])
def test_decode_zero_query_is_mean(oracle, scale, bits):
    U, L, pool, table = _setup(oracle, paged=True, scale=scale, bits=bits)
    rng = np.random.default_rng(2)
    _fill(oracle, L, pool, U, table, [37, 64], rng)
    q = np.zeros((2, 2, 128), np.float16)
    out = oracle.decode(pool, L, U, q, np.array([37, 64]), table)
    for b, n in enumerate([37, 64]):
        for h in range(2):
            vh = oracle.read_rotated(pool, L, b, h, 1, 0, n, table)[0]
            assert np.abs(out[b, h] - U.T @ vh.mean(0)).max() < 1e-12


def test_decode_gqa_mapping_and_empty(oracle):
    # kv head 1 holds values 10x larger than kv head 0: query heads 0,1 must read
    # kv head 0, heads 2,3 kv head 1 (h // G); an empty sequence gives zeros.
    U, L, pool, _ = _setup(oracle, H=2)
    rng = np.random.default_rng(3)
    n = 20
    k = rng.standard_normal((n, 2, 128)).astype(np.float16)
    v = np.ones((n, 2, 128), np.float16)
    v[:, 1] *= 10
    oracle.write(pool, L, U, k, v, np.zeros(n, int), np.arange(n))
    q = rng.standard_normal((2, 4, 128)).astype(np.float16)
    out = oracle.decode(pool, L, U, q, np.array([n, 0]))
    nrm = np.linalg.norm(out[0], axis=1)
    assert nrm[2] > 5 * nrm[0] and nrm[3] > 5 * nrm[1]
    assert np.all(out[1] == 0)


@pytest.mark.parametrize("scale,bits", [("f16", 3), ("f16", 2), ("f32", 4), ("e4m3zp", 3)])
def test_decode_equal_keys_uniform(oracle, scale, bits):
    U, L, pool, _ = _setup(oracle, scale=scale, bits=bits)
    rng = np.random.default_rng(4)
    n = 33
    k = np.tile(rng.standard_normal((1, 2, 128)), (n, 1, 1)).astype(np.float16)
    v = rng.standard_normal((n, 2, 128)).astype(np.float16)
    oracle.write(pool, L, U, k, v, np.zeros(n, int), np.arange(n))
    q = rng.standard_normal((1, 4, 128)).astype(np.float16)
    out = oracle.decode(pool, L, U, q, np.array([n, 0]), heads=[(0, 0), (0, 3)])
    for h in (0, 3):
        vh = oracle.read_rotated(pool, L, 0, h // 2, 1, 0, n)[0]
        assert np.abs(out[0, h] - U.T @ vh.mean(0)).max() < 1e-12


def test_decode_split_invariance(oracle):
    # softmax attention over [0, N) equals the log-sum-exp combination of the
    # attention over two halves (the identity the split-K kernel relies on)
    U, L, pool, _ = _setup(oracle)
    rng = np.random.default_rng(5)
    _fill(oracle, L, pool, U, None, [50, 1], rng)
    q = rng.standard_normal(128)
    kh = oracle.read_rotated(pool, L, 0, 0, 0, 0, 50)[0]
    vh = oracle.read_rotated(pool, L, 0, 0, 1, 0, 50)[0]
    full = oracle.attention_rotated(U, q, kh, vh, 1 / math.sqrt(128))
    q1 = U @ q
    parts = []
    for sl in (slice(0, 23), slice(23, 50)):
        lg = kh[sl] @ q1 / math.sqrt(128)
        m = lg.max()
        p = np.exp(lg - m)
        parts.append((m, p.sum(), p @ vh[sl]))
    M = max(p[0] for p in parts)
    num = sum(np.exp(m - M) * o for m, l, o in parts)
    den = sum(np.exp(m - M) * l for m, l, o in parts)
    assert np.abs(U.T @ (num / den) - full).max() < 1e-13


def test_rotation_reduces_error_on_outlier_data(oracle):
    # The method's premise ("Orthogonally mixed 3-bit KV cache", Mathematical
    # statement): the transform lowers block maxima and so the quantisation
    # error of outlier-heavy vectors.  Diagnostic on the seeded distribution.
    spec = I.DataSpec(128, 1, 77, 0.03, 20.0)
    x = I.kv_rows_np(spec, 0, 0, 0, 0, 512).astype(np.float64)
    s, q = oracle.rotation_params(128, 42)
    U = oracle.rotation_matrix(s, q)
    errs, bmax = {}, {}
    for name, M in (("none", np.eye(128)), ("hadamard", oracle.hadamard_matrix(128)), ("rotated", U)):
        y = x @ M.T
        c, sq, _ = oracle.quantize(y, 64, 1e-6, "f32")
        yh = (c.reshape(-1, 2, 64) * sq[..., None]).reshape(y.shape)
        errs[name] = np.mean((yh @ M - x) ** 2)
        bmax[name] = np.abs(y).reshape(-1, 2, 64).max(-1).mean()
    assert errs["rotated"] < 0.85 * errs["none"] and errs["hadamard"] < 0.85 * errs["none"]
    assert bmax["hadamard"] < bmax["none"] / 2 and bmax["rotated"] < bmax["none"] / 2


def test_error_falls_with_bit_width(oracle):
    # "Orthogonal Invariance in Activation Space", 5.3: error falls from 2 to 3
    # to 4 bits.  For the quantiser each extra bit roughly halves the step
    # (divisors 1, 3, 7), so the MSE of the rotated outlier data falls by about
    # (7/3)^2 and (3/1)^2 -- diagnostic on the seeded distribution.
    spec = I.DataSpec(128, 1, 78, 0.03, 20.0)
    x = I.kv_rows_np(spec, 0, 0, 0, 0, 512).astype(np.float64)
    s, q = oracle.rotation_params(128, 42)
    U = oracle.rotation_matrix(s, q)
    y = x @ U.T
    mse = {}
    for bits in (2, 3, 4):
        c, sq, _ = oracle.quantize(y, 64, 1e-6, "f32", bits)
        yh = (c.reshape(-1, 2, 64) * sq[..., None]).reshape(y.shape)
        mse[bits] = np.mean((yh @ U - x) ** 2)
    assert mse[4] < mse[3] / 3 and mse[3] < mse[2] / 3


# ---------------------------------------------------------------- prefill pins
def test_prefill_first_position_attends_to_itself(oracle):
    # query at position 0 sees one key: weight 1, so o = U^T v_hat_0
    U, L, pool, table = _setup(oracle, paged=True)
    rng = np.random.default_rng(21)
    _fill(oracle, L, pool, U, table, [30, 50], rng)
    q = rng.standard_normal((5, 4, 128)).astype(np.float16)
    out = oracle.prefill(pool, L, U, q, 1, 0, table)
    for h in range(4):
        vh = oracle.read_rotated(pool, L, 1, h // 2, 1, 0, 1, table)[0][0]
        assert np.abs(out[0, h] - U.T @ vh).max() < 1e-12


@pytest.mark.parametrize("scale,bits", [("f16", 3), ("f16", 2), ("f32", 4), ("e4m3zp", 3)])
def test_prefill_zero_queries_average_their_prefix(oracle, scale, bits):
    # q = 0: uniform weights over positions [0, pos0 + i] (the causal prefix)
    U, L, pool, _ = _setup(oracle, scale=scale, bits=bits)
    rng = np.random.default_rng(22)
    _fill(oracle, L, pool, U, None, [40, 64], rng)
    pos0, n = 17, 23
    q = np.zeros((n, 4, 128), np.float16)
    out = oracle.prefill(pool, L, U, q, 0, pos0)
    for i in (0, 5, n - 1):
        for h in (0, 3):
            vh = oracle.read_rotated(pool, L, 0, h // 2, 1, 0, pos0 + i + 1)[0]
            assert np.abs(out[i, h] - U.T @ vh.mean(0)).max() < 1e-12


@pytest.mark.parametrize("scale,bits", [("f16", 3), ("f16", 2), ("f32", 4), ("e4m3zp", 3)])
def test_prefill_is_causal(oracle, scale, bits):
    # rewriting the key and value at position p changes the outputs of the
    # queries at positions >= p and of none before it
    U, L, pool, _ = _setup(oracle, B=1, maxp=4, scale=scale, bits=bits)
    rng = np.random.default_rng(23)
    _fill(oracle, L, pool, U, None, [60], rng)
    pos0, n, p = 10, 40, 31
    q = rng.standard_normal((n, 4, 128)).astype(np.float16)
    before = oracle.prefill(pool, L, U, q, 0, pos0)
    k = (rng.standard_normal((1, 2, 128)) * 4).astype(np.float16)
    v = (rng.standard_normal((1, 2, 128)) * 4).astype(np.float16)
    oracle.write(pool, L, U, k, v, np.array([0]), np.array([p]))
    after = oracle.prefill(pool, L, U, q, 0, pos0)
    moved = np.abs(after - before).max(axis=(1, 2))
    assert np.all(moved[:p - pos0] == 0.0)
    assert np.all(moved[p - pos0:] > 1e-6)


# ---------------------------------------------------------------- softmax scale
def _two_token_cache(oracle, d=128):
    """A cache whose dequantised rotated keys and values are known in closed
    form.  With the rotation flags off, U = H_d.  Key 0 = e_0 and key 1 = -e_0
    rotate to +-(1/sqrt d) 1, whose blocks all quantise to +-3 (the worked
    example of the packing pins) with the fp32 scale s_q = fl32((1/sqrt d +
    eps)/3); so k_hat_0 = -k_hat_1 = 3 s_q 1.  Value t = e_(t+1) rotates to
    +-(1/sqrt d) entries, all codes +-3 with the same s_q, so
    U^T v_hat_t = 3 s_q sqrt(d) e_(t+1)."""
    signs, quats = oracle.rotation_params(d, 42, False, False)
    U = oracle.rotation_matrix(signs, quats)
    L = oracle.Layout(d, 1, 64, "f32", 16, 1, 1, 1)
    pool = np.zeros(L.pool_bytes, np.uint8)
    k = np.zeros((2, 1, d), np.float16)
    v = np.zeros((2, 1, d), np.float16)
    k[0, 0, 0], k[1, 0, 0] = 1.0, -1.0
    v[0, 0, 1], v[1, 0, 2] = 1.0, 1.0
    assert oracle.write(pool, L, U, k, v, np.zeros(2, np.int32), np.arange(2)) == 0
    s_q = float(np.float32((1.0 / math.sqrt(d) + 1e-6) / 3.0))
    return U, L, pool, s_q


@pytest.mark.parametrize("alpha", [0.5, 3.0, -2.0])
def test_default_softmax_scale_is_one_over_sqrt_d(oracle, alpha):
    # Orthogonally mixed 3-bit KV cache, Key formulas: softmax(Q K^T / sqrt d).
    # Query q = alpha e_0 rotates to q1 = (alpha/sqrt d) 1, so the two logits
    # are +-(q1 . 3 s_q 1) = +-3 alpha s_q sqrt d and, after the 1/sqrt(d)
    # scale, +-z with z = 3 alpha s_q.  Token 0 then weighs
    # w0 = 1/(1 + e^(-2z)) and the output is 3 s_q sqrt(d) (w0 e_1 + w1 e_2).
    # Dropping the scale (z sqrt d) or using 1/d (z / sqrt d) moves w0 by
    # 0.02-0.4 at these alphas.
    d = 128
    U, L, pool, s_q = _two_token_cache(oracle, d)
    q = np.zeros((1, 1, d), np.float16)
    q[0, 0, 0] = alpha
    z = 3.0 * alpha * s_q
    w0 = 1.0 / (1.0 + math.exp(-2.0 * z))
    mag = 3.0 * s_q * math.sqrt(d)
    want = np.zeros(d)
    want[1], want[2] = w0 * mag, (1.0 - w0) * mag
    got = oracle.decode(pool, L, U, q, np.array([2]))[0, 0]
    assert np.abs(got - want).max() < 1e-12
    # the wrong scales are told apart by far more than the tolerance
    for wrong in (1.0, 1.0 / d):
        zw = 3.0 * alpha * s_q * math.sqrt(d) * wrong
        w0w = 1.0 / (1.0 + math.exp(-2.0 * zw))
        assert abs(w0w - w0) * mag > 1e-3
    # an explicit sm_scale replaces the default
    got2 = oracle.decode(pool, L, U, q, np.array([2]), sm_scale=1.0)[0, 0]
    z2 = 3.0 * alpha * s_q * math.sqrt(d)
    w02 = 1.0 / (1.0 + math.exp(-2.0 * z2))
    assert abs(got2[1] - w02 * mag) < 1e-12 and abs(got2[2] - (1.0 - w02) * mag) < 1e-12


def test_prefill_default_softmax_scale(oracle):
    # The prefill chunk's second query (position 1) sees both tokens with the
    # same 1/sqrt(d)-scaled logistic weights; its first query (position 0)
    # sees token 0 alone.
    d = 128
    U, L, pool, s_q = _two_token_cache(oracle, d)
    q = np.zeros((2, 1, d), np.float16)
    q[0, 0, 0], q[1, 0, 0] = 1.5, 1.5
    out = oracle.prefill(pool, L, U, q, 0, 0)
    mag = 3.0 * s_q * math.sqrt(d)
    first = np.zeros(d)
    first[1] = mag
    assert np.abs(out[0, 0] - first).max() < 1e-12
    w0 = 1.0 / (1.0 + math.exp(-2.0 * 3.0 * 1.5 * s_q))
    second = np.zeros(d)
    second[1], second[2] = w0 * mag, (1.0 - w0) * mag
    assert np.abs(out[1, 0] - second).max() < 1e-12

"""The C-ABI library loads, exports every declared entry point, and its
host-only logic (rotation parameters from the seed, sizes, argument checks)
agrees with the oracle.  No GPU needed: nothing here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    lib = os.path.join(ROOT, "hadamard_rotated_bit_kvq3_gb300", "libkvq3.so")
    if not os.path.exists(lib):
        import __graft_entry__
        __graft_entry__.build()
    import hadamard_rotated_bit_kvq3_gb300 as K
    return K


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "kvq3.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq3_[a-z0-9_]+)\s*\(", hdr)))


def test_every_declared_symbol_is_exported(K):
    names = declared_symbols()
    assert "kvq3_write" in names and "kvq3_decode_attn" in names and len(names) >= 12
    for n in names:
        assert hasattr(K.lib, n), n
        assert callable(getattr(K, n)), f"binding lacks {n}"


def test_abi_and_status_strings(K):
    assert K.kvq3_abi_version() == 3
    assert K.kvq3_status_string(0) == "ok"
    assert "workspace" in K.kvq3_status_string(4)


@pytest.mark.parametrize("d", [4, 8, 16, 64, 128, 256])
@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_rotation_params_match_oracle(K, oracle, d, flags):
    h = K.kvq3_rotation_create(d, 42, flags)
    try:
        s, q = K.kvq3_rotation_export(h)
    finally:
        K.kvq3_rotation_destroy(h)
    so, qo = oracle.rotation_params(d, 42, bool(flags & 1), bool(flags & 2))
    assert np.array_equal(s, so)
    assert np.array_equal(q, qo.astype(np.float32))      # fp32 rounding of the fp64 draws


def test_rotation_from_params_normalises(K):
    signs = np.ones(8, np.int8)
    signs[3] = -1
    quats = np.array([[2, 0, 0, 0], [0, 0, 3, 4]], np.float32)
    h = K.kvq3_rotation_create_from_params(8, signs, quats)
    s, q = K.kvq3_rotation_export(h)
    K.kvq3_rotation_destroy(h)
    assert np.array_equal(s, signs)
    assert np.allclose(q, [[1, 0, 0, 0], [0, 0, 0.6, 0.8]], atol=1e-7)
    with pytest.raises(K.Kvq3Error):
        K.kvq3_rotation_create_from_params(8, signs, np.zeros((2, 4), np.float32))
    with pytest.raises(K.Kvq3Error):
        K.kvq3_rotation_create(12, 1)                      # not a power of two


@pytest.mark.parametrize("d", [4, 64, 128, 256])
@pytest.mark.parametrize("flags", [6, 7])
def test_pair_rotation_params_match_oracle(K, oracle, d, flags):
    # reading R20: the signs and left quaternions of the one-quaternion
    # rotation with the same seed, then one right quaternion per block
    h = K.kvq3_rotation_create(d, 42, flags)
    try:
        s, q, r = K.kvq3_rotation_export_pair(h)
    finally:
        K.kvq3_rotation_destroy(h)
    so, qo, ro = oracle.rotation_params_pair(d, 42, bool(flags & 1))
    assert np.array_equal(s, so)
    assert np.array_equal(q, qo.astype(np.float32))
    assert np.array_equal(r, ro.astype(np.float32))
    # one-quaternion rotations export identity right quaternions
    h = K.kvq3_rotation_create(d, 42, 3)
    try:
        _, _, r1 = K.kvq3_rotation_export_pair(h)
    finally:
        K.kvq3_rotation_destroy(h)
    assert np.all(r1 == np.array([1, 0, 0, 0], np.float32))


def test_pair_rotation_flags_and_params(K):
    with pytest.raises(K.Kvq3Error):
        K.kvq3_rotation_create(128, 1, 4)                  # the pair needs the SO(4) blocks
    with pytest.raises(K.Kvq3Error):
        K.kvq3_rotation_create(128, 1, 8)                  # unknown flag
    signs = np.ones(8, np.int8)
    quats = np.array([[2, 0, 0, 0], [0, 0, 3, 4]], np.float32)
    quats_r = np.array([[0, 5, 0, 0], [1, 1, 1, 1]], np.float32)
    h = K.kvq3_rotation_create_from_params_pair(8, signs, quats, quats_r)
    s, q, r = K.kvq3_rotation_export_pair(h)
    K.kvq3_rotation_destroy(h)
    assert np.allclose(q, [[1, 0, 0, 0], [0, 0, 0.6, 0.8]], atol=1e-7)
    assert np.allclose(r, [[0, 1, 0, 0], [0.5, 0.5, 0.5, 0.5]], atol=1e-7)
    with pytest.raises(K.Kvq3Error):
        K.kvq3_rotation_create_from_params_pair(8, signs, quats, np.zeros((2, 4), np.float32))


@pytest.mark.parametrize("d,block,scale,page", [(128, 64, "f16", 16), (256, 64, "f16", 16),
                                                (128, 32, "f32", 64), (128, 64, "e4m3", 64),
                                                (64, 32, "e4m3", 32)])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_cache_sizes_match_oracle_layout(K, oracle, d, block, scale, page, bits):
    desc = K.CacheDesc(d, 3, block, bits, K.SCALE_TYPES[scale], 1e-6, page, 2, 5, 0, 11)
    rb, pb, tb = K.kvq3_cache_sizes(desc)
    L = oracle.Layout(d, 3, block, scale, page, 2, 5, 11, bits)
    assert (rb, pb, tb) == (L.record_bytes, L.page_bytes, L.pool_bytes)
    assert rb % 16 == 0


@pytest.mark.parametrize("d,block,page", [(128, 64, 16), (256, 64, 16), (64, 32, 32)])
def test_cache_sizes_match_oracle_layout_asym(K, oracle, d, block, page):
    # the asymmetric variant: (scale, zero point) byte pairs, 3-bit codes
    desc = K.CacheDesc(d, 2, block, 3, K.SCALE_TYPES["e4m3zp"], 1e-6, page, 2, 5, 0, 11)
    rb, pb, tb = K.kvq3_cache_sizes(desc)
    L = oracle.Layout(d, 2, block, "e4m3zp", page, 2, 5, 11)
    assert (rb, pb, tb) == (L.record_bytes, L.page_bytes, L.pool_bytes)
    assert rb == page * (2 * (d // block) + 3 * d // 8)


def test_invalid_descriptions_rejected_on_host(K):
    def desc(**kw):
        base = dict(head_dim=128, num_kv_heads=2, block=64, bits=3, scale_type=1, eps=1e-6,
                    page_size=16, batch=1, max_pages_per_seq=4, reserved=0, num_pages=4)
        base.update(kw)
        return K.CacheDesc(**base)
    assert K.kvq3_cache_sizes(desc())[0] == 832
    for kw, want in [(dict(head_dim=96), 1), (dict(block=48), 1), (dict(page_size=8), 1),
                     (dict(bits=5), 2), (dict(bits=1), 2), (dict(block=16), 2), (dict(scale_type=7), 1),
                     (dict(scale_type=3, bits=2), 2), (dict(scale_type=3, bits=4), 2), (dict(scale_type=4), 1),
                     (dict(num_kv_heads=0), 1), (dict(eps=float("nan")), 1), (dict(head_dim=32, block=32), 2)]:
        with pytest.raises(K.Kvq3Error) as e:
            K.kvq3_cache_sizes(desc(**kw))
        assert e.value.status == want, kw
    # write: a null pool or a misaligned one is refused before any launch
    d = desc()
    for pool in (0, 8):
        c = K.Cache(pool, None, None)
        st = K.lib.kvq3_write(K.kvq3_rotation_create(128, 1), ctypes.byref(d), ctypes.byref(c),
                              None, None, None, None, 1, None, None)
        assert st == 1
    # decode: query heads must be a multiple of the kv heads
    c = K.Cache(256, None, 256)
    st = K.lib.kvq3_decode_attn(K.kvq3_rotation_create(128, 1), ctypes.byref(d), ctypes.byref(c),
                                ctypes.c_void_p(256), 3, 0.0, ctypes.c_void_p(256), None, 0, None, None)
    assert st == 1


def test_prefill_arguments_checked_on_host(K):
    # q and out are read and written 16 bytes at a time: a null or misaligned
    # pointer is refused before any launch
    d = K.CacheDesc(128, 2, 64, 3, 1, 1e-6, 16, 1, 4, 0, 4)
    c = K.Cache(256, None, 256)
    rot = K.kvq3_rotation_create(128, 1)
    try:
        for q, out in ((258, 256), (264, 256), (256, 260), (256, 264), (0, 256), (256, 0)):
            st = K.lib.kvq3_prefill_attn(rot, ctypes.byref(d), ctypes.byref(c), 0, 0, 4, ctypes.c_void_p(q), 8,
                                         0.0, ctypes.c_void_p(out), ctypes.c_void_p(256), 1 << 20, None, None)
            assert st == 1, (q, out)
    finally:
        K.kvq3_rotation_destroy(rot)


def test_calibration_arguments_checked_on_host(K):
    # workspace: candidate quaternions (rounded up to 256 bytes) + fp64 errors
    d = K.CacheDesc(128, 1, 64, 3, K.SCALE_TYPES["f16"], 1e-6, 16, 1, 1, 0, 1)
    # (left and right quaternions of the two-quaternion search, each rounded)
    assert K.kvq3_calibrate_workspace_size(d, 64) == 2 * ((64 * 128 * 4 + 255) // 256 * 256) + 64 * 2 * 8
    assert K.kvq3_calibrate_workspace_size(d, 3) == 2 * ((3 * 128 * 4 + 255) // 256 * 256) + 3 * 2 * 8
    for p in (1, 0, 70000):
        with pytest.raises(K.Kvq3Error) as e:
            K.kvq3_calibrate_workspace_size(d, p)
        assert e.value.status == 1
    rot = K.kvq3_rotation_create(128, 1)
    sse = ctypes.c_void_p(256)
    # candidates out of range, a null or misaligned candidate array, a misaligned sample
    for p, quats, x in ((0, 256, 256), (1, 0, 256), (1, 264, 256), (1, 256, 258)):
        st = K.lib.kvq3_calib_sse(rot, ctypes.byref(d), ctypes.c_void_p(quats), p, ctypes.c_void_p(x), 16, sse, None)
        assert st == 1, (p, quats, x)
    # a rotation of another dimension
    st = K.lib.kvq3_calib_sse(K.kvq3_rotation_create(64, 1), ctypes.byref(d), ctypes.c_void_p(256), 1,
                              ctypes.c_void_p(256), 16, sse, None)
    assert st == 1
    # the search: a short, missing or misaligned workspace; bad step or rounds
    q = (ctypes.c_float * 128)()
    need = K.kvq3_calibrate_workspace_size(d, 4)
    for ws, nbytes in ((256, need - 8), (0, need), (264, need)):
        st = K.lib.kvq3_calibrate_so4(rot, ctypes.byref(d), ctypes.c_void_p(256), 16, 1, 4, 0.5, 1,
                                      ctypes.c_void_p(ws), nbytes, q, None, None)
        assert st == 4, (ws, nbytes)
    for rounds, step in ((-1, 0.5), (1, -0.5), (1, float("nan"))):
        st = K.lib.kvq3_calibrate_so4(rot, ctypes.byref(d), ctypes.c_void_p(256), 16, rounds, 4, step, 1,
                                      ctypes.c_void_p(256), need, q, None, None)
        assert st == 1, (rounds, step)
    # the two-quaternion search takes the same checks, and needs quats_r_out
    st = K.lib.kvq3_calibrate_so4_pair(rot, ctypes.byref(d), ctypes.c_void_p(256), 16, 1, 4, 0.5, 1,
                                       ctypes.c_void_p(256), need - 8, q, q, None, None)
    assert st == 4
    st = K.lib.kvq3_calibrate_so4_pair(rot, ctypes.byref(d), ctypes.c_void_p(256), 16, 1, 4, 0.5, 1,
                                       ctypes.c_void_p(256), need, q, None, None, None)
    assert st == 1
    for quats, quats_r in ((256, 0), (256, 264), (0, 256)):
        st = K.lib.kvq3_calib_sse_pair(rot, ctypes.byref(d), ctypes.c_void_p(quats), ctypes.c_void_p(quats_r), 1,
                                       ctypes.c_void_p(256), 16, sse, None)
        assert st == 1, (quats, quats_r)


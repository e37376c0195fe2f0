"""GPU path against the CPU oracle through the C ABI, element by element, at
sizes the oracle finishes in seconds that still span several pages and
16-token tiles with ragged tails.

Bars: codes bit-exact except elements within 1e-4 of a rounding boundary of
|x/s_q| (counted), scales within 1e-6 relative except blocks whose fp64 scale
sits within 1e-6 of a storage-type rounding midpoint (counted), decode output
max|err| <= 2e-3 * rms(out)."""
import math

import numpy as np
import pytest

from cases import TOL_DECODE, Case, flip_bound, rel_err, written_differences
from oracle import kvq3_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hadamard_rotated_bit_kvq3_gb300  # noqa: F401


# ------------------------------------------------------------------ rotate
@pytest.mark.parametrize("d", [4, 8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("flags", [3, 1, 0])
def test_rotate_matches_dense_U(oracle, d, flags):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    rot = K.Rotation(d, 42, flags)
    s, q = oracle.rotation_params(d, 42, bool(flags & 1), bool(flags & 2))
    U = oracle.rotation_matrix(s, q)
    rng = np.random.default_rng(d + flags)
    for n in (1, 37, 1000):
        x = rng.standard_normal((n, d)).astype(np.float32)
        xt = torch.as_tensor(x, device="cuda")
        y = torch.empty_like(xt)
        for inverse in (False, True):
            K.kvq3_rotate(rot.handle, xt, y, inverse=inverse)
            ref = x.astype(np.float64) @ (U if inverse else U.T)   # rows: U x or U^T x
            assert np.abs(y.cpu().numpy() - ref).max() < 2e-6 * math.sqrt(d)
        xh = torch.as_tensor(x.astype(np.float16), device="cuda")
        K.kvq3_rotate(rot.handle, xh, y)
        ref = x.astype(np.float16).astype(np.float64) @ U.T
        assert np.abs(y.cpu().numpy() - ref).max() < 2e-6 * math.sqrt(d)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ write
WRITE_CASES = [
    dict(d=128, block=64, scale="f32", page=64, lens=(1024,), hkv=4, hq=4),            # tiny
    dict(d=128, block=64, scale="f16", page=64, lens=(300, 1, 65), hkv=8, hq=32),
    dict(d=128, block=64, scale="e4m3", page=64, lens=(257, 130), hkv=2, hq=16),
    dict(d=128, block=32, scale="f32", page=64, lens=(700,), hkv=3, hq=3, flags=1),     # prefill
    dict(d=256, block=64, scale="f16", page=16, lens=(77, 300, 16), hkv=2, hq=8, paged=True),
    dict(d=64, block=32, scale="e4m3", page=32, lens=(90, 33), hkv=2, hq=4, paged=True),
    dict(d=256, block=32, scale="f32", page=16, lens=(50,), hkv=1, hq=2, flags=0),
    dict(d=64, block=64, scale="f16", page=16, lens=(40,), hkv=1, hq=1, flags=2),
]


@pytest.mark.parametrize("cfg", WRITE_CASES, ids=lambda c: f"d{c['d']}-m{c['block']}-{c['scale']}-P{c['page']}")
def test_write_matches_oracle(cfg):
    c = Case(**cfg)
    k, v, si, ps = c.tokens()
    c.gpu_write(k, v, si, ps)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    stats = c.compare_written(k, v, si, ps)
    print(stats)
    # with nothing excluded the whole pool must be byte-identical
    if stats["boundary_codes"] == 0 and stats["midpoint_blocks"] == 0:
        assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)


def test_write_single_token_appends_and_scatter():
    # decode-style appends: one token per sequence at arbitrary positions
    c = Case(d=128, block=64, scale="f16", page=64, lens=(500, 500, 500, 500), hkv=8, hq=32)
    rng = np.random.default_rng(9)
    k = (rng.standard_normal((4, 8, 128)) * 5).astype(np.float16)
    v = rng.standard_normal((4, 8, 128)).astype(np.float16)
    si = np.array([3, 0, 2, 1], np.int32)
    ps = np.array([499, 0, 63, 64], np.int32)
    c.gpu_write(k, v, si, ps)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    stats = c.compare_written(k, v, si, ps)
    # slots nobody wrote stay zero on both sides; with nothing excluded by the
    # write bar the whole pool is byte-identical
    if stats["boundary_codes"] == 0 and stats["midpoint_blocks"] == 0:
        assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)
    else:
        written = np.zeros(c.layout.pool_bytes, bool)
        page, slot, _ = O.locate(c.layout, c.table, si, ps)
        for pg, sl in zip(page, slot):
            for rec in range(2 * c.hkv):
                base = pg * c.layout.page_bytes + rec * c.layout.record_bytes
                nb_sb = c.layout.nb * c.layout.sb
                written[base + sl * nb_sb: base + (sl + 1) * nb_sb] = True
                co = base + c.page * nb_sb + sl * c.layout.code_bytes
                written[co: co + c.layout.code_bytes] = True
        assert np.array_equal(c.pool.cpu().numpy()[~written], c.pool_o[~written])


def test_write_bad_slots_flag_and_skip():
    c = Case(d=128, block=64, scale="f16", page=16, lens=(40, 40), hkv=2, hq=2, paged=True)
    rng = np.random.default_rng(3)
    k = rng.standard_normal((4, 2, 128)).astype(np.float16)
    si = np.array([0, 7, 1, -1], np.int32)
    ps = np.array([3, 0, 10 ** 6, 0], np.int32)
    c.gpu_write(k, k, si, ps)
    st = c.device_status()
    assert st == (1 | 2)                       # bad sequence, bad position
    assert c.oracle_write(k, k, si, ps) == st
    assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)


def test_write_bad_page_id_flags():
    import torch
    c = Case(d=128, block=64, scale="f16", page=16, lens=(40,), hkv=1, hq=1, paged=True)
    bad = c.table.copy()
    bad[0, 1] = 10 ** 5
    c.table_t.copy_(torch.as_tensor(bad, device="cuda"))
    k = np.ones((2, 1, 128), np.float16)
    c.gpu_write(k, k, np.array([0, 0], np.int32), np.array([0, 20], np.int32))
    assert c.device_status() == 4
    c.table = bad
    c.oracle_write(k, k, np.array([0, 0], np.int32), np.array([0, 20], np.int32))
    assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)


# ------------------------------------------------------------------ read-back
@pytest.mark.parametrize("rotated", [True, False])
def test_dequant_debug_matches_oracle(oracle, rotated):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    c = Case(d=256, block=64, scale="f16", page=16, lens=(70,), hkv=2, hq=2, paged=True)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    for which in (0, 1):
        out = torch.empty((50, 256), dtype=torch.float32, device="cuda")
        codes = torch.empty((50, 256), dtype=torch.int32, device="cuda")
        K.kvq3_dequant_debug(c.rot.handle if not rotated else c.rot.handle, c.desc, c.cache, 0, 1,
                             which, 11, 50, out, codes, c.status)
        xh, co, _ = oracle.read_rotated(c.pool_o, c.layout, 0, 1, which, 11, 50, c.table)
        assert np.array_equal(codes.cpu().numpy(), co)
        ref = xh @ c.U            # rows: U^T x_hat
        assert np.abs(out.cpu().numpy() - ref).max() < 1e-5 * np.abs(ref).max()
        if not rotated:
            K.kvq3_dequant_debug(None, c.desc, c.cache, 0, 1, which, 11, 50, out, None, c.status)
            assert np.array_equal(out.cpu().numpy(), xh.astype(np.float32))
    assert c.device_status() == 0


# ------------------------------------------------------------------ decode
DECODE_CASES = [
    dict(d=128, block=64, scale="f32", page=64, lens=(1024,), hkv=4, hq=4),                       # G=1
    dict(d=128, block=64, scale="f16", page=64, lens=(700, 1, 129, 64), hkv=2, hq=8),              # G=4
    dict(d=128, block=64, scale="e4m3", page=64, lens=(900, 333), hkv=2, hq=16,
         data=None),                                                                                # G=8
    dict(d=256, block=64, scale="f16", page=16, lens=(300, 17, 1000), hkv=2, hq=8, paged=True),    # d256 paged
    dict(d=128, block=32, scale="f32", page=32, lens=(200, 95), hkv=1, hq=2, paged=True),          # G=2, m32
    dict(d=64, block=32, scale="f16", page=16, lens=(150, 40), hkv=2, hq=24),                      # G=12 (pad 16)
    dict(d=128, block=64, scale="f16", page=16, lens=(77,), hkv=1, hq=16, flags=1),                # G=16
    dict(d=256, block=32, scale="e4m3", page=16, lens=(200,), hkv=1, hq=6, flags=0),               # G=6, no rot
]


def _ids(c):
    return f"d{c['d']}-m{c['block']}-{c['scale']}-G{c['hq'] // c['hkv']}-{'paged' if c.get('paged') else 'contig'}"


@pytest.mark.parametrize("cfg", DECODE_CASES, ids=_ids)
def test_decode_isolated_matches_oracle(cfg):
    # GPU decode on the oracle-written cache: isolates the read kernel
    c = Case(**cfg)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = c.queries()
    got = c.gpu_decode(q)
    ref = c.oracle_decode(q)
    assert c.device_status() == 0
    e = rel_err(got, ref)
    print(f"max|err|/rms = {e:.3e}")
    assert e <= TOL_DECODE


@pytest.mark.parametrize("cfg", DECODE_CASES[:4], ids=_ids)
def test_decode_end_to_end(cfg):
    # GPU write + GPU decode against oracle write + oracle decode
    c = Case(**cfg)
    k, v, si, ps = c.tokens()
    c.gpu_write(k, v, si, ps)
    c.oracle_write(k, v, si, ps)
    q = c.queries(1)
    got, ref = c.gpu_decode(q), c.oracle_decode(q)
    assert c.device_status() == 0
    # The GPU write may legitimately hold another code at an element within
    # BOUNDARY of a rounding boundary (or another scale at a midpoint): the
    # write bar allows it.  Each (sequence, head) therefore gets the decode
    # bar plus the oracle-side bound of what the elements that do differ
    # (all checked against the write bar first) can move.
    rms = math.sqrt(float(np.mean(ref ** 2)))
    slack = flip_bound(c, k, v, si, ps, q, differs=written_differences(c, k, v, si, ps))
    err = np.abs(got - ref).max(axis=-1)
    e = rel_err(got, ref)
    print(f"max|err|/rms = {e:.3e}; heads with boundary slack: {int((slack > 0).sum())}; "
          f"worst (err - slack)/rms = {float((err - slack).max()) / rms:.3e}")
    assert np.all(err <= TOL_DECODE * rms + slack)


def test_decode_custom_scale_and_empty_sequences():
    c = Case(d=128, block=64, scale="f16", page=64, lens=(0, 100, 0, 1), hkv=2, hq=4)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = c.queries()
    for sm in (0.0, 0.02, 0.3):
        got = c.gpu_decode(q, sm)
        ref = c.oracle_decode(q, sm)
        assert np.all(got[0] == 0) and np.all(got[2] == 0)
        assert rel_err(got, ref) <= TOL_DECODE


def test_decode_bad_length_and_bad_page():
    import torch
    c = Case(d=128, block=64, scale="f16", page=16, lens=(40, 50), hkv=1, hq=4, paged=True)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = c.queries()
    # length above capacity: that sequence gives zeros, the other is intact
    c.lens_t.copy_(torch.tensor([40, 10 ** 6], dtype=torch.int32, device="cuda"))
    got = c.gpu_decode(q)
    assert c.device_status() & 8
    assert np.all(got[1] == 0)
    ref = c.oracle_decode(q, lens=np.array([40, 0]))
    assert rel_err(got[0], ref[0]) <= TOL_DECODE
    # a bad page id masks that page: equals attention over the other pages
    c.status.zero_()
    c.lens_t.copy_(torch.tensor([40, 50], dtype=torch.int32, device="cuda"))
    bad = c.table.copy()
    bad[0, 1] = -7
    c.table_t.copy_(torch.as_tensor(bad, device="cuda"))
    got = c.gpu_decode(q)
    assert c.device_status() & 4
    assert np.all(np.isfinite(got))


def test_decode_split_count_invariance(oracle):
    # The same sequence decoded alone and inside a large batch.  Alone, its
    # 12 chunks of 256 tokens go to 12 CTAs (a 12-way split merged by the
    # combine kernel); in the batch, 640 units of 2 chunks share the CTAs, so
    # sequence 0's unit lies within one CTA or straddles two.  Both runs must
    # match the oracle (which does not split at all) and each other.
    import hadamard_rotated_bit_kvq3_gb300 as K
    c1 = Case(d=128, block=64, scale="f16", page=64, lens=(3000,), hkv=1, hq=4)
    k, v, si, ps = c1.tokens()
    c1.oracle_write(k, v, si, ps)
    c1.upload_oracle_pool()
    q = c1.queries()
    a = c1.gpu_decode(q)
    ref = c1.oracle_decode(q)
    assert c1.device_status() == 0
    assert rel_err(a, ref) <= TOL_DECODE
    # sequence 0 again (same seeds, so the same keys, values and queries),
    # now with 639 more sequences of 512 tokens after it
    lens = (3000,) + (512,) * 639
    c2 = Case(d=128, block=64, scale="f16", page=64, lens=lens, hkv=1, hq=4)
    k2, v2, si2, ps2 = c2.tokens()
    c2.oracle_write(k2, v2, si2, ps2)
    c2.upload_oracle_pool()
    q2 = c2.queries()
    assert np.array_equal(q2[0], q[0])
    ws_alone = K.kvq3_decode_workspace_size(c1.desc, 4)
    ws_batch = K.kvq3_decode_workspace_size(c2.desc, 4)
    assert ws_batch > ws_alone
    b2 = c2.gpu_decode(q2)
    assert c2.device_status() == 0
    assert rel_err(b2[0], ref[0]) <= TOL_DECODE
    assert rel_err(b2[0], a[0]) <= TOL_DECODE
    # a sample of the other sequences against the oracle as well
    heads = [(b, h) for b in (1, 317, 639) for h in range(4)]
    ref2 = oracle.decode(c2.pool_o, c2.layout, c2.U, q2, c2.lens, heads=heads)
    for b in (1, 317, 639):
        assert rel_err(b2[b], ref2[b]) <= TOL_DECODE


# ------------------------------------------------------------------ write (prefill chunks)
CHUNK_CASES = [
    dict(d=128, block=32, scale="f32", page=64, lens=(700,), hkv=3, hq=3, flags=1, pos0=0),
    dict(d=128, block=64, scale="f16", page=64, lens=(1000, 5), hkv=2, hq=8, flags=3, pos0=37),
    dict(d=128, block=64, scale="e4m3", page=16, lens=(300,), hkv=2, hq=16, paged=True, flags=3, pos0=5),
    dict(d=64, block=32, scale="f16", page=32, lens=(257,), hkv=2, hq=4, paged=True, flags=3, pos0=0),
    dict(d=64, block=64, scale="f32", page=16, lens=(129,), hkv=1, hq=1, flags=0, pos0=16),
    dict(d=128, block=32, scale="e4m3", page=48, lens=(400,), hkv=1, hq=2, flags=2, pos0=1),
]


@pytest.mark.parametrize("cfg", CHUNK_CASES, ids=lambda c: f"d{c['d']}-m{c['block']}-{c['scale']}-P{c['page']}-pos{c['pos0']}")
def test_write_chunk_matches_oracle(cfg):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    cfg = dict(cfg)
    pos0 = cfg.pop("pos0")
    c = Case(**cfg)
    n = int(c.lens[0]) - pos0
    k = np.stack([__import__("kvq3_inputs").kv_rows_np(c.spec, 0, 0, h, pos0, n) for h in range(c.hkv)], 1)
    v = np.stack([__import__("kvq3_inputs").kv_rows_np(c.spec, 1, 0, h, pos0, n) for h in range(c.hkv)], 1)
    si = np.zeros(n, np.int32)
    ps = np.arange(pos0, pos0 + n, dtype=np.int32)
    K.kvq3_write_chunk(c.rot.handle, c.desc, c.cache, torch.as_tensor(k, device="cuda"),
                       torch.as_tensor(v, device="cuda"), 0, pos0, c.status)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    stats = c.compare_written(k, v, si, ps)
    print(stats)
    if stats["boundary_codes"] == 0 and stats["midpoint_blocks"] == 0:
        assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)


def test_write_chunk_equals_token_list_write():
    # the chunk entry point and the token-list entry point store the same bytes
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    c1 = Case(d=128, block=64, scale="f16", page=64, lens=(333,), hkv=4, hq=16)
    c2 = Case(d=128, block=64, scale="f16", page=64, lens=(333,), hkv=4, hq=16)
    k, v, si, ps = c1.tokens()
    K.kvq3_write_chunk(c1.rot.handle, c1.desc, c1.cache, torch.as_tensor(k, device="cuda"),
                       torch.as_tensor(v, device="cuda"), 0, 0, c1.status)
    c2.gpu_write(k, v, si, ps)
    torch.cuda.synchronize()
    assert c1.device_status() == 0 and c2.device_status() == 0
    # Both entry points meet the same write bar against the oracle: codes
    # bit-exact except within 1e-4 of a rounding boundary, scales exact except
    # at a storage midpoint.  Their two fp32 butterflies may round such a
    # boundary element differently, so byte equality between them holds
    # wherever the oracle's bar leaves no choice.
    s1 = c1.compare_written(k, v, si, ps)
    s2 = c2.compare_written(k, v, si, ps)
    a, b = c1.pool.cpu().numpy(), c2.pool.cpu().numpy()
    if s1["boundary_codes"] == 0 and s1["midpoint_blocks"] == 0 and \
            s2["boundary_codes"] == 0 and s2["midpoint_blocks"] == 0:
        assert np.array_equal(a, b)


def test_write_chunk_rejects_out_of_range():
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    c = Case(d=128, block=64, scale="f16", page=64, lens=(100,), hkv=1, hq=1)
    k = torch.zeros((10, 1, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(K.Kvq3Error):
        K.kvq3_write_chunk(c.rot.handle, c.desc, c.cache, k, k, 0, c.maxp * 64 - 5, c.status)
    with pytest.raises(K.Kvq3Error):
        K.kvq3_write_chunk(c.rot.handle, c.desc, c.cache, k, k, 3, 0, c.status)


# ------------------------------------------------------------------ margin at large groups
# At G = 8 and 16 the probabilities-times-value-scales enter PV as one fp16
# rounding (no hi + lo split).  Several data seeds per case, isolated and end
# to end, to see how close the worst case sits to the bar.
SEED_CASES = [
    dict(d=128, block=64, scale="e4m3", page=64, lens=(1500, 400), hkv=2, hq=16),     # G=8, E4M3
    dict(d=128, block=64, scale="f16", page=64, lens=(1500, 400), hkv=2, hq=32),      # G=16
    dict(d=256, block=64, scale="f16", page=16, lens=(900, 33), hkv=1, hq=8, paged=True),   # G=8, d256
]


@pytest.mark.parametrize("seed", [11, 12, 13, 14])
@pytest.mark.parametrize("cfg", SEED_CASES, ids=_ids)
def test_decode_large_group_over_seeds(cfg, seed):
    import kvq3_inputs as I
    cfg = dict(cfg, data=I.DataSpec(cfg["d"], cfg["hkv"], seed, 0.03, 20.0))
    c = Case(**cfg)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = c.queries(seed)
    e_iso = rel_err(c.gpu_decode(q), c.oracle_decode(q))
    assert c.device_status() == 0
    c.pool.zero_()
    c.gpu_write(k, v, si, ps)
    got, ref = c.gpu_decode(q), c.oracle_decode(q)
    assert c.device_status() == 0
    rms = math.sqrt(float(np.mean(ref ** 2)))
    slack = flip_bound(c, k, v, si, ps, q, differs=written_differences(c, k, v, si, ps))
    err = np.abs(got - ref).max(axis=-1)
    print(f"seed {seed}: isolated {e_iso:.3e}, end to end {rel_err(got, ref):.3e} "
          f"(worst (err - slack)/rms {float((err - slack).max()) / rms:.3e})")
    assert e_iso <= TOL_DECODE
    assert np.all(err <= TOL_DECODE * rms + slack)


# ------------------------------------------------------------------ tiny cases
@pytest.mark.parametrize("n", [1, 2, 3])
@pytest.mark.parametrize("d,scale", [(64, "f32"), (128, "f16"), (256, "e4m3")])
def test_tiny_one_page(d, scale, n):
    # one page, 1-3 tokens: write against the oracle byte for byte (when no
    # element sits at a rounding boundary) and decode against the oracle
    c = Case(d=d, block=64 if d >= 128 else 32, scale=scale, page=16, lens=(n,), hkv=1, hq=2)
    k, v, si, ps = c.tokens()
    c.gpu_write(k, v, si, ps)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    stats = c.compare_written(k, v, si, ps)
    # fp16 / E4M3 scales are exact away from a midpoint; an fp32 scale may sit
    # an ulp from the oracle's (the 1e-6 bar), so only its codes are bytewise
    if stats["boundary_codes"] == 0 and stats["midpoint_blocks"] == 0 and scale != "f32":
        assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)
    q = c.queries()
    got, ref = c.gpu_decode(q), c.oracle_decode(q)
    assert c.device_status() == 0
    assert rel_err(got, ref) <= TOL_DECODE

"""2- and 4-bit caches on the GPU against the oracle, through the C ABI.

The quantiser is the method's b-bit one (divisor and clip bound 2^(b-1) - 1,
b-bit two's-complement codes in the same little-endian stream; "Orthogonally
mixed 3-bit KV cache", Key formulas; "Orthogonal Invariance in Activation
Space", 3.3, 4.2, 5.1).  Same bars as the 3-bit tests: codes bit-exact except
elements within 1e-4 of a rounding boundary, scales within 1e-6 relative,
decode and prefill output max|err| <= 2e-3 * rms(out)."""
import math

import numpy as np
import pytest

import kvq3_inputs as I
from cases import TOL_DECODE, Case, flip_bound, rel_err, written_differences
from oracle import kvq3_oracle as O

pytestmark = pytest.mark.gpu

BITS = [2, 4]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hadamard_rotated_bit_kvq3_gb300  # noqa: F401


WRITE_CASES = [
    dict(d=128, block=64, scale="f16", page=64, lens=(300, 1, 65), hkv=8, hq=32),
    dict(d=128, block=32, scale="f32", page=64, lens=(200,), hkv=3, hq=3, flags=1),
    dict(d=256, block=64, scale="e4m3", page=16, lens=(77, 120), hkv=2, hq=8, paged=True),
    dict(d=64, block=32, scale="e4m3", page=32, lens=(90, 33), hkv=2, hq=4, paged=True),
    dict(d=256, block=32, scale="f16", page=16, lens=(50,), hkv=1, hq=2, flags=0),
]


def _wid(c):
    return f"d{c['d']}-m{c['block']}-{c['scale']}-P{c['page']}"


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("cfg", WRITE_CASES, ids=_wid)
def test_write_matches_oracle_b24(cfg, bits):
    c = Case(bits=bits, **cfg)
    k, v, si, ps = c.tokens()
    c.gpu_write(k, v, si, ps)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    stats = c.compare_written(k, v, si, ps)
    print(stats)
    if stats["boundary_codes"] == 0 and stats["midpoint_blocks"] == 0:
        assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)


CHUNK_CASES = [
    dict(d=128, block=64, scale="f16", page=64, lens=(700, 5), hkv=2, hq=8, flags=3, pos0=37),
    dict(d=128, block=32, scale="e4m3", page=16, lens=(300,), hkv=2, hq=16, paged=True, flags=1, pos0=5),
    dict(d=64, block=32, scale="f32", page=32, lens=(257,), hkv=2, hq=4, paged=True, flags=0, pos0=0),
    dict(d=64, block=64, scale="f16", page=48, lens=(200,), hkv=1, hq=1, flags=2, pos0=1),
]


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("cfg", CHUNK_CASES, ids=lambda c: _wid(c) + f"-pos{c['pos0']}")
def test_write_chunk_matches_oracle_b24(cfg, bits):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    cfg = dict(cfg)
    pos0 = cfg.pop("pos0")
    c = Case(bits=bits, **cfg)
    n = int(c.lens[0]) - pos0
    k = np.stack([I.kv_rows_np(c.spec, 0, 0, h, pos0, n) for h in range(c.hkv)], 1)
    v = np.stack([I.kv_rows_np(c.spec, 1, 0, h, pos0, n) for h in range(c.hkv)], 1)
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


@pytest.mark.parametrize("bits", BITS)
def test_dequant_debug_matches_oracle_b24(bits):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    c = Case(d=128, block=32, scale="f16", page=16, lens=(70,), hkv=2, hq=2, paged=True, bits=bits)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    for which in (0, 1):
        out = torch.empty((50, 128), dtype=torch.float32, device="cuda")
        codes = torch.empty((50, 128), dtype=torch.int32, device="cuda")
        K.kvq3_dequant_debug(None, c.desc, c.cache, 0, 1, which, 11, 50, out, codes, c.status)
        xh, co, _ = O.read_rotated(c.pool_o, c.layout, 0, 1, which, 11, 50, c.table)
        assert np.array_equal(codes.cpu().numpy(), co)
        assert np.abs(co).max() == O.qmax(bits)
        assert np.array_equal(out.cpu().numpy(), xh.astype(np.float32))
    assert c.device_status() == 0
    # the one b-bit value the quantiser never writes is flagged and reads as 0
    lay = c.layout
    page, slot, _ = O.locate(lay, c.table, np.array([0]), np.array([3]))
    off = lay.code_offset(int(page[0]), 0, 0, int(slot[0]))
    bad = c.pool_o.copy()
    bad[off] = (int(bad[off]) & (0xFF ^ ((1 << bits) - 1))) | (1 << (bits - 1))   # element 0 := -2^(b-1)
    c.pool.copy_(torch.as_tensor(bad, device="cuda"))
    K.kvq3_dequant_debug(None, c.desc, c.cache, 0, 0, 0, 3, 1, out[:1], codes[:1], c.status)
    assert codes[0, 0].item() == 0 and out[0, 0].item() == 0.0
    assert c.device_status() == 16


DECODE_CASES = [
    dict(d=128, block=64, scale="f32", page=64, lens=(1024,), hkv=4, hq=4),                       # G=1
    dict(d=128, block=64, scale="f16", page=64, lens=(700, 1, 129, 64), hkv=2, hq=8),              # G=4
    dict(d=128, block=64, scale="e4m3", page=64, lens=(900, 333), hkv=2, hq=16),                   # G=8
    dict(d=256, block=64, scale="f16", page=16, lens=(300, 17, 1000), hkv=2, hq=8, paged=True),    # d256 paged
    dict(d=128, block=32, scale="f32", page=32, lens=(200, 95), hkv=1, hq=2, paged=True),          # G=2, m32
    dict(d=64, block=32, scale="f16", page=16, lens=(150, 40), hkv=2, hq=24),                      # G=12
    dict(d=128, block=64, scale="f16", page=16, lens=(77,), hkv=1, hq=16, flags=1),                # G=16
    dict(d=256, block=32, scale="e4m3", page=16, lens=(200,), hkv=1, hq=6, flags=0),               # G=6
]


def _did(c):
    return f"d{c['d']}-m{c['block']}-{c['scale']}-G{c['hq'] // c['hkv']}-{'paged' if c.get('paged') else 'contig'}"


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("cfg", DECODE_CASES, ids=_did)
def test_decode_isolated_matches_oracle_b24(cfg, bits):
    c = Case(bits=bits, **cfg)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = c.queries()
    got, ref = c.gpu_decode(q), c.oracle_decode(q)
    assert c.device_status() == 0
    e = rel_err(got, ref)
    print(f"max|err|/rms = {e:.3e}")
    assert e <= TOL_DECODE


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("cfg", DECODE_CASES[1:4], ids=_did)
def test_decode_end_to_end_b24(cfg, bits):
    c = Case(bits=bits, **cfg)
    k, v, si, ps = c.tokens()
    c.gpu_write(k, v, si, ps)
    c.oracle_write(k, v, si, ps)
    q = c.queries(1)
    got, ref = c.gpu_decode(q), c.oracle_decode(q)
    assert c.device_status() == 0
    rms = math.sqrt(float(np.mean(ref ** 2)))
    slack = flip_bound(c, k, v, si, ps, q, differs=written_differences(c, k, v, si, ps))
    err = np.abs(got - ref).max(axis=-1)
    print(f"max|err|/rms = {rel_err(got, ref):.3e}; heads with slack: {int((slack > 0).sum())}")
    assert np.all(err <= TOL_DECODE * rms + slack)


PREFILL_CASES = [
    (dict(d=128, block=64, scale="f16", page=64, lens=(300,), hkv=2, hq=8), 0, 200, 100),
    (dict(d=128, block=32, scale="e4m3", page=16, lens=(90, 257), hkv=2, hq=16, paged=True), 1, 0, 257),
    (dict(d=64, block=32, scale="f32", page=16, lens=(150,), hkv=2, hq=12), 0, 60, 90),
    # d = 128, blocks of 64: the tcgen05 kernel, here with units split in two key ranges
    (dict(d=128, block=64, scale="e4m3", page=64, lens=(900,), hkv=2, hq=8), 0, 600, 300),
    (dict(d=128, block=64, scale="f32", page=32, lens=(700,), hkv=1, hq=4, paged=True), 0, 500, 200),
    (dict(d=256, block=64, scale="f16", page=16, lens=(300, 180), hkv=2, hq=8, paged=True), 1, 100, 80),
]


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("cfg", PREFILL_CASES, ids=lambda c: _did(c[0]) + f"-pos{c[2]}-n{c[3]}")
def test_prefill_matches_oracle_b24(cfg, bits):
    import torch
    kw, seq, pos0, n = cfg
    c = Case(bits=bits, **kw)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = I.q_np(c.spec, n, c.hq, 7)
    qd = torch.as_tensor(q, device=c.dev)
    out = torch.full((n, c.hq, c.d), float("nan"), dtype=torch.float32, device=c.dev)
    ws = torch.empty(c.K.kvq3_prefill_workspace_size(c.desc, c.hq, n), dtype=torch.uint8, device=c.dev)
    c.K.kvq3_prefill_attn(c.rot.handle, c.desc, c.cache, seq, pos0, qd, out, ws, 0.0, c.status)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref = O.prefill(c.pool_o, c.layout, c.U, q, seq, pos0, c.table)
    assert c.device_status() == 0
    e = rel_err(got, ref)
    print(f"max|err|/rms = {e:.3e}")
    assert e <= TOL_DECODE

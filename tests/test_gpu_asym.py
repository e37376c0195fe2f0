"""The asymmetric variant (scale type "e4m3zp") on the GPU against the oracle.

"Hardware-Fused Fast Hadamard Transforms ...": per 64-element sub-block,
unsigned 3-bit codes plus an FP8 scale and an FP8 zero point; the library's
reading: z = min, s = (max - min + eps)/7, both E4M3, unsigned
codes u = clip(round((x - z_q)/s_q), 0, 7), x_hat = s_q u + z_q.

Bars as for the symmetric codes: codes bit-exact except elements whose
(x - z_q)/s_q lies within 1e-4 of k + 1/2, scale and zero-point bytes exact
except blocks whose fp64 scale or zero point lies within 1e-6 (relative) of
an E4M3 rounding midpoint; decode and prefill output max|err| <= 2e-3 *
rms(out)."""
import numpy as np
import pytest

import kvq3_inputs as I
from cases import TOL_DECODE, Case, flip_bound, rel_err, written_differences
from oracle import kvq3_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hadamard_rotated_bit_kvq3_gb300  # noqa: F401


WRITE_CASES = [
    dict(d=128, block=64, page=64, lens=(300, 1, 65), hkv=8, hq=32),
    dict(d=128, block=32, page=16, lens=(200,), hkv=3, hq=3, flags=1, paged=True),
    dict(d=256, block=64, page=16, lens=(77, 120), hkv=2, hq=8, paged=True),
    dict(d=64, block=32, page=32, lens=(90, 33), hkv=2, hq=4, flags=0),
]


def _wid(c):
    return f"d{c['d']}-m{c['block']}-P{c['page']}{'-paged' if c.get('paged') else ''}"


@pytest.mark.parametrize("cfg", WRITE_CASES, ids=_wid)
def test_write_matches_oracle_asym(cfg):
    c = Case(scale="e4m3zp", **cfg)
    k, v, si, ps = c.tokens()
    c.gpu_write(k, v, si, ps)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    stats = c.compare_written(k, v, si, ps)
    print(stats)
    if stats["boundary_codes"] == 0 and stats["midpoint_blocks"] == 0:
        assert np.array_equal(c.pool.cpu().numpy(), c.pool_o)


@pytest.mark.parametrize("cfg", [dict(d=128, block=64, page=64, lens=(700, 5), hkv=2, hq=8, flags=3, pos0=37),
                                 dict(d=64, block=32, page=16, lens=(257,), hkv=2, hq=4, paged=True, flags=1, pos0=0)],
                         ids=lambda c: _wid(c) + f"-pos{c['pos0']}")
def test_write_chunk_matches_oracle_asym(cfg):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    cfg = dict(cfg)
    pos0 = cfg.pop("pos0")
    c = Case(scale="e4m3zp", **cfg)
    n = int(c.lens[0]) - pos0
    k = np.stack([I.kv_rows_np(c.spec, 0, 0, h, pos0, n) for h in range(c.hkv)], 1)
    v = np.stack([I.kv_rows_np(c.spec, 1, 0, h, pos0, n) for h in range(c.hkv)], 1)
    si = np.zeros(n, np.int32)
    ps = np.arange(pos0, pos0 + n, dtype=np.int32)
    K.kvq3_write_chunk(c.rot.handle, c.desc, c.cache, torch.as_tensor(k, device="cuda"),
                       torch.as_tensor(v, device="cuda"), 0, pos0, c.status)
    assert c.oracle_write(k, v, si, ps) == 0
    assert c.device_status() == 0
    print(c.compare_written(k, v, si, ps))


def test_dequant_debug_matches_oracle_asym():
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    c = Case(d=128, block=64, scale="e4m3zp", page=16, lens=(70,), hkv=2, hq=2, paged=True)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    for which in (0, 1):
        out = torch.empty((50, 128), dtype=torch.float32, device="cuda")
        codes = torch.empty((50, 128), dtype=torch.int32, device="cuda")
        K.kvq3_dequant_debug(None, c.desc, c.cache, 0, 1, which, 11, 50, out, codes, c.status)
        xh, u, _ = O.read_rotated(c.pool_o, c.layout, 0, 1, which, 11, 50, c.table)
        assert np.array_equal(codes.cpu().numpy(), u)
        assert u.min() == 0 and u.max() == 7
        assert np.abs(out.cpu().numpy() - xh).max() <= 1e-6 * np.abs(xh).max()
    assert c.device_status() == 0


DECODE_CASES = [
    dict(d=128, block=64, page=64, lens=(1024,), hkv=4, hq=4),                        # G=1
    dict(d=128, block=64, page=64, lens=(700, 1, 129, 64), hkv=2, hq=8),               # G=4
    dict(d=128, block=64, page=64, lens=(900, 333), hkv=2, hq=16),                     # G=8
    dict(d=256, block=64, page=16, lens=(300, 17, 1000), hkv=2, hq=8, paged=True),     # d256 paged
    dict(d=128, block=32, page=32, lens=(200, 95), hkv=1, hq=2, paged=True),           # G=2, m32
    dict(d=64, block=32, page=16, lens=(150, 40), hkv=2, hq=24),                       # G=12
]


def _did(c):
    return f"d{c['d']}-m{c['block']}-G{c['hq'] // c['hkv']}-{'paged' if c.get('paged') else 'contig'}"


@pytest.mark.parametrize("cfg", DECODE_CASES, ids=_did)
def test_decode_isolated_matches_oracle_asym(cfg):
    c = Case(scale="e4m3zp", **cfg)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    for step in (0, 1):
        q = c.queries(step)
        got, ref = c.gpu_decode(q), c.oracle_decode(q)
        assert c.device_status() == 0
        e = rel_err(got, ref)
        print(f"max|err|/rms = {e:.3e}")
        assert e <= TOL_DECODE


@pytest.mark.parametrize("cfg", [(dict(d=128, block=64, page=64, lens=(300,), hkv=2, hq=8), 0, 200, 100),
                                 (dict(d=256, block=64, page=16, lens=(300, 180), hkv=2, hq=8, paged=True), 1, 100, 80),
                                 # the tcgen05 kernel with units split in two key ranges, and G = 16
                                 (dict(d=128, block=64, page=32, lens=(900,), hkv=2, hq=8, paged=True), 0, 600, 300),
                                 (dict(d=128, block=64, page=64, lens=(600,), hkv=1, hq=16), 0, 550, 50)],
                         ids=lambda c: _did(c[0]) + f"-pos{c[2]}-n{c[3]}")
def test_prefill_matches_oracle_asym(cfg):
    import torch
    kw, seq, pos0, n = cfg
    c = Case(scale="e4m3zp", **kw)
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


def test_asym_rejects_other_widths():
    import hadamard_rotated_bit_kvq3_gb300 as K
    for bits in (2, 4):
        d = K.CacheDesc(128, 2, 64, bits, K.SCALE_TYPES["e4m3zp"], 1e-6, 16, 1, 4, 0, 4)
        with pytest.raises(K.Kvq3Error) as e:
            K.kvq3_cache_sizes(d)
        assert e.value.status == 2


@pytest.mark.parametrize("cfg", DECODE_CASES[1:4], ids=_did)
def test_decode_end_to_end_asym(cfg):
    # GPU write + GPU decode against oracle write + oracle decode; elements the
    # write bar lets differ widen each head's bar by the oracle-side bound of
    # what they can move (cases.flip_bound)
    import math
    c = Case(scale="e4m3zp", **cfg)
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

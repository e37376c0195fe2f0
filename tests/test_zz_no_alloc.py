"""kvq3_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory when they call (its workspace is a fixed array inside
the library).  It must give what kvq3_decode_attn gives with a
caller-allocated workspace and what the oracle gives, on repeated calls that
reuse the same array with different shapes, and refuse work that would not
fit.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from cases import TOL_DECODE, Case, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


NOALLOC_CASES = [
    dict(d=128, block=64, scale="f16", page=64, lens=(700, 1, 129, 64), hkv=2, hq=8),        # G=4
    dict(d=256, block=64, scale="e4m3zp", page=16, lens=(300, 17, 450), hkv=2, hq=32,
         paged=True),                                                                          # G=16
]


def _noalloc(c, q):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    out = torch.full((c.B, c.hq, c.d), float("nan"), dtype=torch.float32, device="cuda")
    K.kvq3_decode_attn_noalloc(c.rot.handle, c.desc, c.cache, torch.as_tensor(q, device="cuda"), out,
                               0.0, c.status)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def test_noalloc_matches_oracle_and_workspace_entry_point_twice():
    import hadamard_rotated_bit_kvq3_gb300 as K
    cases = [Case(**cfg) for cfg in NOALLOC_CASES]
    for c in cases:
        assert K.kvq3_decode_workspace_size(c.desc, c.hq) <= 8 << 20   # fits the array
        k, v, si, ps = c.tokens()
        c.oracle_write(k, v, si, ps)
        c.upload_oracle_pool()
    # calls alternate between the two shapes (partial slots of G*(d+2) floats
    # and the unit ranges move between calls that share the array), two rounds
    for step in (0, 1):
        for c in cases:
            q = c.queries(step)
            got = _noalloc(c, q)
            assert c.device_status() == 0
            assert np.all(np.isfinite(got))
            assert rel_err(got, c.oracle_decode(q)) <= TOL_DECODE
            # the entry point with a caller-provided workspace on the same cache
            assert rel_err(got, c.gpu_decode(q)) <= TOL_DECODE


def test_noalloc_rejects_work_beyond_its_array():
    import hadamard_rotated_bit_kvq3_gb300 as K
    # 4096 sequences x 8 kv heads x 16 query heads each need far more than 8 MiB
    desc = K.CacheDesc(128, 8, 64, 3, 1, 1e-6, 64, 4096, 1, 0, 4096)
    need = K.kvq3_decode_workspace_size(desc, 128)
    assert need > (8 << 20)
    cache = K.Cache(256, None, 256)          # never dereferenced: refused before any launch
    rot = K.kvq3_rotation_create(128, 1)
    try:
        st = K.lib.kvq3_decode_attn_noalloc(rot, ctypes.byref(desc), ctypes.byref(cache),
                                            ctypes.c_void_p(256), 128, 0.0, ctypes.c_void_p(256), None, None)
    finally:
        K.kvq3_rotation_destroy(rot)
    assert st == 4                           # KVQ3_ERR_WORKSPACE

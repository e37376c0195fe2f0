"""kvq3_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory (its workspace is a fixed array inside the library).
It must give what kvq3_decode_attn gives with a caller-allocated workspace,
on repeated calls that reuse the same array, and refuse work that would not
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


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    c = Case(d=128, block=64, scale="f16", page=64, lens=(700, 1, 129, 64), hkv=2, hq=8)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    for step in (0, 1):                        # two calls in a row, different queries
        q = torch.as_tensor(c.queries(step), device="cuda")
        ref = c.gpu_decode(c.queries(step))    # kvq3_decode_attn with its own workspace
        out = torch.full((c.B, c.hq, c.d), float("nan"), dtype=torch.float32, device="cuda")
        K.kvq3_decode_attn_noalloc(c.rot.handle, c.desc, c.cache, q, out, 0.0, c.status)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert c.device_status() == 0
        assert np.all(np.isfinite(got))
        assert rel_err(got, ref) <= TOL_DECODE


def test_noalloc_rejects_work_beyond_its_array():
    import hadamard_rotated_bit_kvq3_gb300 as K
    # 4096 sequences x 8 kv heads x 16 query heads each need far more than 8 MiB
    desc = K.CacheDesc(128, 8, 64, 3, 1, 1e-6, 64, 4096, 1, 0, 4096)
    need = K.kvq3_decode_workspace_size(desc, 128)
    assert need > (8 << 20)
    cache = K.Cache(256, None, 256)          # never dereferenced: refused before any launch
    st = K.lib.kvq3_decode_attn_noalloc(K.kvq3_rotation_create(128, 1), ctypes.byref(desc),
                                        ctypes.byref(cache), ctypes.c_void_p(256), 128, 0.0,
                                        ctypes.c_void_p(256), None, None)
    assert st == 4                           # KVQ3_ERR_WORKSPACE

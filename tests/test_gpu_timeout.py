"""The decode kernel's bounded waits: when a stage's copy has not arrived
within the bound, the CTA flags KVQ3_DEV_TIMEOUT in the status word, waits
for its own copies still in flight and returns; the context stays usable.

The library's test hook kvq3_test_decode_attn_polls sets the bound; with 0
polls no wait can succeed, so every CTA takes that path while every copy it
issued still targets valid memory (nothing faults and nothing hangs).  A
normal call on the same buffers afterwards must still match the oracle."""
import ctypes

import numpy as np
import pytest

from cases import TOL_DECODE, Case, rel_err

pytestmark = pytest.mark.gpu

TIMEOUT = 32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _hook():
    import hadamard_rotated_bit_kvq3_gb300 as K
    fn = K.lib.kvq3_test_decode_attn_polls
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(K.CacheDesc), ctypes.POINTER(K.Cache), ctypes.c_void_p,
                   ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32]
    return fn


TIMEOUT_CASES = [
    dict(d=128, block=64, scale="f16", page=64, lens=(700, 1, 129, 64), hkv=2, hq=8),
    dict(d=256, block=64, scale="f16", page=16, lens=(300, 17, 1000), hkv=2, hq=8, paged=True),
    dict(d=128, block=64, scale="e4m3", page=64, lens=(2000, 333), hkv=2, hq=16),
]


@pytest.mark.parametrize("cfg", TIMEOUT_CASES, ids=lambda c: f"d{c['d']}-{c['scale']}-G{c['hq'] // c['hkv']}")
def test_wait_that_runs_out_flags_and_returns(cfg):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    fn = _hook()
    c = Case(**cfg)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    q = torch.as_tensor(c.queries(), device="cuda")
    ws = torch.empty(K.kvq3_decode_workspace_size(c.desc, c.hq), dtype=torch.uint8, device="cuda")
    out = torch.zeros((c.B, c.hq, c.d), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):   # twice: the context and the buffers stay usable
        st = fn(c.rot.handle, ctypes.byref(c.desc), ctypes.byref(c.cache), ctypes.c_void_p(q.data_ptr()), c.hq,
                0.0, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                ctypes.c_void_p(c.status.data_ptr()), stream, 0)
        assert st == 0
        torch.cuda.synchronize()
        assert c.device_status() & TIMEOUT
        c.status.zero_()
    # the default bound on the same buffers: no time-out, the oracle's result
    got = c.gpu_decode(c.queries())
    assert c.device_status() == 0
    assert rel_err(got, c.oracle_decode(c.queries())) <= TOL_DECODE
    # the hook with a generous bound behaves like the public entry point
    st = fn(c.rot.handle, ctypes.byref(c.desc), ctypes.byref(c.cache), ctypes.c_void_p(q.data_ptr()), c.hq,
            0.0, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
            ctypes.c_void_p(c.status.data_ptr()), stream, 1 << 22)
    assert st == 0
    torch.cuda.synchronize()
    assert c.device_status() == 0
    assert rel_err(out.cpu().numpy().astype(np.float64), got) <= TOL_DECODE


def _prefill_hook():
    import hadamard_rotated_bit_kvq3_gb300 as K
    fn = K.lib.kvq3_test_prefill_attn_polls
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(K.CacheDesc), ctypes.POINTER(K.Cache), ctypes.c_int32,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_uint32]
    return fn


PREFILL_TIMEOUT_CASES = [
    # (case, pos0, n): the tcgen05 kernel (d = 128, blocks of 64) and the decode kernel's prefill variant
    (dict(d=128, block=64, scale="f16", page=64, lens=(900,), hkv=2, hq=8), 500, 400),
    (dict(d=128, block=64, scale="e4m3", page=16, lens=(300,), hkv=1, hq=16, paged=True), 100, 200),
    (dict(d=256, block=64, scale="f16", page=16, lens=(400,), hkv=2, hq=8), 300, 100),
]


@pytest.mark.parametrize("cfg", PREFILL_TIMEOUT_CASES,
                         ids=lambda c: f"d{c[0]['d']}-{c[0]['scale']}-G{c[0]['hq'] // c[0]['hkv']}")
def test_prefill_wait_that_runs_out_flags_and_returns(cfg):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    import kvq3_inputs as I
    from oracle import kvq3_oracle as O
    fn = _prefill_hook()
    kw, pos0, n = cfg
    c = Case(**kw)
    k, v, si, ps = c.tokens()
    c.oracle_write(k, v, si, ps)
    c.upload_oracle_pool()
    qn = I.q_np(c.spec, n, c.hq, 5)
    q = torch.as_tensor(qn, device="cuda")
    ws = torch.empty(max(1, K.kvq3_prefill_workspace_size(c.desc, c.hq, n)), dtype=torch.uint8, device="cuda")
    out = torch.zeros((n, c.hq, c.d), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(polls):
        st = fn(c.rot.handle, ctypes.byref(c.desc), ctypes.byref(c.cache), 0, pos0, n,
                ctypes.c_void_p(q.data_ptr()), c.hq, 0.0, ctypes.c_void_p(out.data_ptr()),
                ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(c.status.data_ptr()), stream, polls)
        assert st == 0
        torch.cuda.synchronize()

    for _ in range(2):   # twice: the context, the tensor memory and the buffers stay usable
        call(0)
        assert c.device_status() & TIMEOUT
        c.status.zero_()
    call(1 << 22)        # a generous bound: the oracle's result
    assert c.device_status() == 0
    ref = O.prefill(c.pool_o, c.layout, c.U, qn, 0, pos0, c.table)
    assert rel_err(out.cpu().numpy().astype(np.float64), ref) <= TOL_DECODE

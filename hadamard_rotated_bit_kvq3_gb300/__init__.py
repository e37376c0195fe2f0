"""Python binding of the rotated 3-bit KV cache library (libkvq3.so).

Argument marshalling only: every step of the write and read paths runs in
the CUDA kernels behind the C ABI declared in include/kvq3.h.  Tensors are
torch tensors on a CUDA device (PyTorch supplies device memory and streams);
the functions take the C names.  There is no CPU fallback: importing this
module fails loudly when the compiled library is missing.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "KVQ3_OK", "KVQ3_ROT_SIGN", "KVQ3_ROT_SO4", "SCALE_TYPES", "CacheDesc", "Cache", "Kvq3Error",
    "lib", "kvq3_abi_version", "kvq3_status_string", "kvq3_rotation_create",
    "kvq3_rotation_create_from_params", "kvq3_rotation_create_from_params_pair", "kvq3_rotation_destroy",
    "kvq3_rotation_export", "kvq3_rotation_export_pair", "KVQ3_ROT_SO4_PAIR", "kvq3_calib_sse_pair",
    "kvq3_calibrate_so4_pair",
    "kvq3_cache_sizes", "kvq3_rotate", "kvq3_write", "kvq3_write_chunk", "kvq3_decode_workspace_size",
    "kvq3_decode_attn", "kvq3_decode_attn_noalloc", "kvq3_prefill_workspace_size", "kvq3_prefill_attn",
    "kvq3_dequant_debug", "kvq3_calib_sse", "kvq3_calibrate_workspace_size", "kvq3_calibrate_so4", "Rotation",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVQ3_LIBRARY selects another build of the library (e.g. libkvq3_checked.so,
# the build with in-kernel bounds checks); the default is the in-tree build
LIB_PATH = os.environ.get("KVQ3_LIBRARY") or os.path.join(_HERE, "libkvq3.so")

KVQ3_OK = 0
KVQ3_ROT_SIGN = 1
KVQ3_ROT_SO4 = 2
KVQ3_ROT_SO4_PAIR = 4
SCALE_TYPES = {"f32": 0, "f16": 1, "e4m3": 2, "e4m3zp": 3}
DEV_BITS = {"bad_seq": 1, "bad_pos": 2, "bad_page": 4, "bad_len": 8, "bad_code": 16, "timeout": 32,
            "check": 64}

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
lib = ctypes.CDLL(LIB_PATH)


class CacheDesc(ctypes.Structure):
    """Mirror of kvq3_cache_desc."""
    _fields_ = [("head_dim", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("block", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("scale_type", ctypes.c_int32), ("eps", ctypes.c_float),
                ("page_size", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("num_pages", ctypes.c_int64)]


class Cache(ctypes.Structure):
    """Mirror of kvq3_cache (device pointers)."""
    _fields_ = [("pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p)]


_p = ctypes.c_void_p
_i32, _i64, _u32, _u64, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float
_sz = ctypes.c_size_t
_D, _C = ctypes.POINTER(CacheDesc), ctypes.POINTER(Cache)

_SIGS = {
    "kvq3_abi_version": (_i32, []),
    "kvq3_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kvq3_rotation_create": (ctypes.c_int, [_i32, _u64, _u32, ctypes.POINTER(_p)]),
    "kvq3_rotation_create_from_params": (ctypes.c_int, [_i32, _p, _p, ctypes.POINTER(_p)]),
    "kvq3_rotation_create_from_params_pair": (ctypes.c_int, [_i32, _p, _p, _p, ctypes.POINTER(_p)]),
    "kvq3_rotation_destroy": (ctypes.c_int, [_p]),
    "kvq3_rotation_export": (ctypes.c_int, [_p, _p, _p, _p]),
    "kvq3_rotation_export_pair": (ctypes.c_int, [_p, _p, _p, _p, _p]),
    "kvq3_cache_sizes": (ctypes.c_int, [_D, ctypes.POINTER(_sz), ctypes.POINTER(_sz), ctypes.POINTER(_sz)]),
    "kvq3_rotate": (ctypes.c_int, [_p, _p, _i32, _p, _i64, _i32, _p]),
    "kvq3_write": (ctypes.c_int, [_p, _D, _C, _p, _p, _p, _p, _i64, _p, _p]),
    "kvq3_write_chunk": (ctypes.c_int, [_p, _D, _C, _p, _p, _i32, _i64, _i64, _p, _p]),
    "kvq3_decode_workspace_size": (ctypes.c_int, [_D, _i32, ctypes.POINTER(_sz)]),
    "kvq3_decode_attn": (ctypes.c_int, [_p, _D, _C, _p, _i32, _f32, _p, _p, _sz, _p, _p]),
    "kvq3_decode_attn_noalloc": (ctypes.c_int, [_p, _D, _C, _p, _i32, _f32, _p, _p, _p]),
    "kvq3_prefill_workspace_size": (ctypes.c_int, [_D, _i32, _i64, ctypes.POINTER(_sz)]),
    "kvq3_prefill_attn": (ctypes.c_int, [_p, _D, _C, _i32, _i64, _i64, _p, _i32, _f32, _p, _p, _sz, _p, _p]),
    "kvq3_dequant_debug": (ctypes.c_int, [_p, _D, _C, _i32, _i32, _i32, _i64, _i64, _p, _p, _p, _p]),
    "kvq3_calib_sse": (ctypes.c_int, [_p, _D, _p, _i32, _p, _i64, _p, _p]),
    "kvq3_calib_sse_pair": (ctypes.c_int, [_p, _D, _p, _p, _i32, _p, _i64, _p, _p]),
    "kvq3_calibrate_so4_pair": (ctypes.c_int, [_p, _D, _p, _i64, _i32, _i32, _f32, _u64, _p, _sz, _p, _p, _p,
                                               _p]),
    "kvq3_calibrate_workspace_size": (ctypes.c_int, [_D, _i32, ctypes.POINTER(_sz)]),
    "kvq3_calibrate_so4": (ctypes.c_int, [_p, _D, _p, _i64, _i32, _i32, _f32, _u64, _p, _sz, _p, _p, _p]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class Kvq3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvq3_status_string(status)} (status {status})")


def _check(status: int, where: str) -> None:
    if status != KVQ3_OK:
        raise Kvq3Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------------ C names
def kvq3_abi_version() -> int:
    return lib.kvq3_abi_version()


def kvq3_status_string(status: int) -> str:
    return lib.kvq3_status_string(status).decode()


def kvq3_rotation_create(d: int, seed: int, flags: int = KVQ3_ROT_SIGN | KVQ3_ROT_SO4):
    """Returns an opaque handle (ctypes.c_void_p)."""
    h = ctypes.c_void_p()
    _check(lib.kvq3_rotation_create(d, seed & ((1 << 64) - 1), flags, ctypes.byref(h)),
           "kvq3_rotation_create")
    return h


def kvq3_rotation_create_from_params(d: int, signs, quats):
    """signs: int8 host array [d]; quats: float32 host array [d/4][4] (numpy)."""
    import numpy as np
    s = np.ascontiguousarray(signs, dtype=np.int8)
    q = np.ascontiguousarray(quats, dtype=np.float32)
    h = ctypes.c_void_p()
    _check(lib.kvq3_rotation_create_from_params(d, s.ctypes.data_as(_p), q.ctypes.data_as(_p),
                                                ctypes.byref(h)), "kvq3_rotation_create_from_params")
    return h


def kvq3_rotation_create_from_params_pair(d: int, signs, quats, quats_r):
    """Two-quaternion blocks: signs int8 [d]; quats, quats_r float32 [d/4][4] (numpy)."""
    import numpy as np
    s = np.ascontiguousarray(signs, dtype=np.int8)
    q = np.ascontiguousarray(quats, dtype=np.float32)
    r = np.ascontiguousarray(quats_r, dtype=np.float32)
    h = ctypes.c_void_p()
    _check(lib.kvq3_rotation_create_from_params_pair(d, s.ctypes.data_as(_p), q.ctypes.data_as(_p),
                                                     r.ctypes.data_as(_p), ctypes.byref(h)),
           "kvq3_rotation_create_from_params_pair")
    return h


def kvq3_rotation_destroy(h) -> None:
    _check(lib.kvq3_rotation_destroy(h), "kvq3_rotation_destroy")


def kvq3_rotation_export(h):
    """(signs int8 [d], quats float32 [d/4][4]) as numpy arrays."""
    import numpy as np
    d = ctypes.c_int32()
    _check(lib.kvq3_rotation_export(h, None, None, ctypes.byref(d)), "kvq3_rotation_export")
    s = np.zeros(d.value, np.int8)
    q = np.zeros((d.value // 4, 4), np.float32)
    _check(lib.kvq3_rotation_export(h, s.ctypes.data_as(_p), q.ctypes.data_as(_p), None),
           "kvq3_rotation_export")
    return s, q


def kvq3_rotation_export_pair(h):
    """(signs int8 [d], quats float32 [d/4][4], quats_r float32 [d/4][4])."""
    import numpy as np
    d = ctypes.c_int32()
    _check(lib.kvq3_rotation_export_pair(h, None, None, None, ctypes.byref(d)), "kvq3_rotation_export_pair")
    s = np.zeros(d.value, np.int8)
    q = np.zeros((d.value // 4, 4), np.float32)
    r = np.zeros((d.value // 4, 4), np.float32)
    _check(lib.kvq3_rotation_export_pair(h, s.ctypes.data_as(_p), q.ctypes.data_as(_p), r.ctypes.data_as(_p),
                                         None), "kvq3_rotation_export_pair")
    return s, q, r


def kvq3_cache_sizes(desc: CacheDesc):
    rb, pb, tb = _sz(), _sz(), _sz()
    _check(lib.kvq3_cache_sizes(ctypes.byref(desc), ctypes.byref(rb), ctypes.byref(pb),
                                ctypes.byref(tb)), "kvq3_cache_sizes")
    return rb.value, pb.value, tb.value


def kvq3_rotate(h, x, y, inverse: bool = False, stream=None) -> None:
    """y[n][d] (fp32) = U x or U^T x; x fp32 or fp16 [n][d] (CUDA tensors)."""
    import torch
    n = x.shape[0] if x.numel() else 0
    _check(lib.kvq3_rotate(h, _ptr(x), 1 if x.dtype == torch.float16 else 0, _ptr(y), n,
                           1 if inverse else 0, _stream(stream)), "kvq3_rotate")


def kvq3_write(h, desc: CacheDesc, cache: Cache, k, v, seq_idx, pos, dev_status=None,
               stream=None) -> None:
    """k, v: fp16 [n_tok][Hkv][d]; seq_idx, pos: int32 [n_tok] (CUDA tensors)."""
    _check(lib.kvq3_write(h, ctypes.byref(desc), ctypes.byref(cache), _ptr(k), _ptr(v),
                          _ptr(seq_idx), _ptr(pos), int(k.shape[0]), _ptr(dev_status),
                          _stream(stream)), "kvq3_write")


def kvq3_write_chunk(h, desc: CacheDesc, cache: Cache, k, v, seq: int, pos0: int, dev_status=None,
                     stream=None) -> None:
    """k, v: fp16 [n_tok][Hkv][d] for positions pos0.. of sequence seq (CUDA tensors)."""
    _check(lib.kvq3_write_chunk(h, ctypes.byref(desc), ctypes.byref(cache), _ptr(k), _ptr(v), seq,
                                pos0, int(k.shape[0]), _ptr(dev_status), _stream(stream)),
           "kvq3_write_chunk")


def kvq3_decode_workspace_size(desc: CacheDesc, num_q_heads: int) -> int:
    n = _sz()
    _check(lib.kvq3_decode_workspace_size(ctypes.byref(desc), num_q_heads, ctypes.byref(n)),
           "kvq3_decode_workspace_size")
    return n.value


def kvq3_decode_attn(h, desc: CacheDesc, cache: Cache, q, out, workspace, sm_scale: float = 0.0,
                     dev_status=None, stream=None) -> None:
    """q: fp16 [B][Hq][d]; out: fp32 [B][Hq][d]; workspace: uint8 CUDA tensor."""
    _check(lib.kvq3_decode_attn(h, ctypes.byref(desc), ctypes.byref(cache), _ptr(q),
                                int(q.shape[1]), float(sm_scale), _ptr(out), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                _stream(stream)), "kvq3_decode_attn")


def kvq3_decode_attn_noalloc(h, desc: CacheDesc, cache: Cache, q, out, sm_scale: float = 0.0,
                             dev_status=None, stream=None) -> None:
    """kvq3_decode_attn for callers that cannot allocate device memory: the
    workspace is a fixed array inside the library (KVQ3_DECODE_NOALLOC_MAX_BYTES);
    calls sharing it must not overlap on the GPU."""
    _check(lib.kvq3_decode_attn_noalloc(h, ctypes.byref(desc), ctypes.byref(cache), _ptr(q),
                                        int(q.shape[1]), float(sm_scale), _ptr(out), _ptr(dev_status),
                                        _stream(stream)), "kvq3_decode_attn_noalloc")


def kvq3_prefill_workspace_size(desc: CacheDesc, num_q_heads: int, n_q: int) -> int:
    n = _sz()
    _check(lib.kvq3_prefill_workspace_size(ctypes.byref(desc), num_q_heads, n_q, ctypes.byref(n)),
           "kvq3_prefill_workspace_size")
    return n.value


def kvq3_prefill_attn(h, desc: CacheDesc, cache: Cache, seq: int, pos0: int, q, out, workspace,
                      sm_scale: float = 0.0, dev_status=None, stream=None) -> None:
    """q: fp16 [n_q][Hq][d] at positions pos0.. of sequence seq; out: fp32 [n_q][Hq][d];
    workspace: uint8 CUDA tensor (kvq3_prefill_workspace_size bytes)."""
    _check(lib.kvq3_prefill_attn(h, ctypes.byref(desc), ctypes.byref(cache), seq, pos0,
                                 int(q.shape[0]), _ptr(q), int(q.shape[1]), float(sm_scale),
                                 _ptr(out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                 _stream(stream)), "kvq3_prefill_attn")


def kvq3_calib_sse(h, desc: CacheDesc, quats, x, sse, stream=None) -> None:
    """quats: fp32 CUDA [P][d/4][4] candidate quaternion sets; x: fp16 CUDA
    [n][d] sample vectors; sse: fp64 CUDA [P][d/m] (overwritten)."""
    _check(lib.kvq3_calib_sse(h, ctypes.byref(desc), _ptr(quats), int(quats.shape[0]), _ptr(x),
                              int(x.shape[0]), _ptr(sse), _stream(stream)), "kvq3_calib_sse")


def kvq3_calib_sse_pair(h, desc: CacheDesc, quats, quats_r, x, sse, stream=None) -> None:
    """quats, quats_r: fp32 CUDA [P][d/4][4] candidate two-quaternion blocks;
    x: fp16 CUDA [n][d]; sse: fp64 CUDA [P][d/m] (overwritten)."""
    _check(lib.kvq3_calib_sse_pair(h, ctypes.byref(desc), _ptr(quats), _ptr(quats_r), int(quats.shape[0]),
                                   _ptr(x), int(x.shape[0]), _ptr(sse), _stream(stream)), "kvq3_calib_sse_pair")


def kvq3_calibrate_workspace_size(desc: CacheDesc, num_candidates: int) -> int:
    n = _sz()
    _check(lib.kvq3_calibrate_workspace_size(ctypes.byref(desc), num_candidates, ctypes.byref(n)),
           "kvq3_calibrate_workspace_size")
    return n.value


def kvq3_calibrate_so4(h, desc: CacheDesc, x, rounds: int, num_candidates: int, step: float, seed: int,
                       workspace, stream=None):
    """Returns (quats float32 [d/4][4], sse float64 [d/m]) as numpy arrays; x:
    fp16 CUDA [n][d]; workspace: uint8 CUDA tensor of
    kvq3_calibrate_workspace_size bytes.  Synchronises the stream."""
    import numpy as np
    d = desc.head_dim
    q = np.zeros((d // 4, 4), np.float32)
    e = np.zeros(d // desc.block, np.float64)
    _check(lib.kvq3_calibrate_so4(h, ctypes.byref(desc), _ptr(x), int(x.shape[0]), rounds, num_candidates,
                                  float(step), seed & ((1 << 64) - 1), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), q.ctypes.data_as(_p),
                                  e.ctypes.data_as(_p), _stream(stream)), "kvq3_calibrate_so4")
    return q, e


def kvq3_calibrate_so4_pair(h, desc: CacheDesc, x, rounds: int, num_candidates: int, step: float, seed: int,
                            workspace, stream=None):
    """Returns (quats, quats_r float32 [d/4][4], sse float64 [d/m]) as numpy
    arrays: the search over two-quaternion blocks.  Synchronises the stream."""
    import numpy as np
    d = desc.head_dim
    q = np.zeros((d // 4, 4), np.float32)
    r = np.zeros((d // 4, 4), np.float32)
    e = np.zeros(d // desc.block, np.float64)
    _check(lib.kvq3_calibrate_so4_pair(h, ctypes.byref(desc), _ptr(x), int(x.shape[0]), rounds, num_candidates,
                                       float(step), seed & ((1 << 64) - 1), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), q.ctypes.data_as(_p),
                                       r.ctypes.data_as(_p), e.ctypes.data_as(_p), _stream(stream)),
           "kvq3_calibrate_so4_pair")
    return q, r, e


def kvq3_dequant_debug(h, desc: CacheDesc, cache: Cache, seq: int, kv_head: int, which: int,
                       t0: int, nt: int, out, codes_out=None, dev_status=None, stream=None) -> None:
    """out: fp32 [nt][d]; codes_out: int32 [nt][d] or None; h None = rotated domain."""
    _check(lib.kvq3_dequant_debug(h, ctypes.byref(desc), ctypes.byref(cache), seq, kv_head, which,
                                  t0, nt, _ptr(out), _ptr(codes_out), _ptr(dev_status),
                                  _stream(stream)), "kvq3_dequant_debug")


class Rotation:
    """Owning wrapper of a rotation handle."""

    def __init__(self, d: int, seed: int, flags: int = KVQ3_ROT_SIGN | KVQ3_ROT_SO4):
        self.d = d
        self.handle = kvq3_rotation_create(d, seed, flags)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and lib is not None:
            lib.kvq3_rotation_destroy(h)
            self.handle = None

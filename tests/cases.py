"""Shared set-up for the GPU parity tests: one cache description built twice,
once for the library (device buffers) and once for the CPU oracle, fed with
the same seeded inputs (kvq3_inputs).  Expected values come from the oracle
only; the comparisons below parse the library's output bytes."""
from __future__ import annotations

import math

import numpy as np

import kvq3_inputs as I
from oracle import kvq3_oracle as O

CANARY = 256             # guard bytes after every device buffer a kernel writes
CANARY_BYTE = 0xA5

TOL_DECODE = 2e-3        # max|err| <= TOL_DECODE * rms(out)
TOL_SCALE = 1e-6         # relative
BOUNDARY = 1e-4          # |x/s_q| within this of k + 1/2: code may round either way
MIDPOINT = 1e-6          # fp64 scale within this (relative) of a storage midpoint


class Case:
    def __init__(self, d=128, hkv=2, hq=8, block=64, scale="f16", page=16, lens=(37, 100),
                 maxp=None, paged=False, flags=3, rot_seed=42, data=None, spare_pages=0, bits=3):
        import torch
        import hadamard_rotated_bit_kvq3_gb300 as K
        self.K, self.torch = K, torch
        self.dev = torch.device("cuda:0")
        self.d, self.hkv, self.hq, self.block, self.scale, self.page = d, hkv, hq, block, scale, page
        self.bits = bits
        self.lens = np.array(lens, np.int32)
        self.B = len(lens)
        need = [max(1, math.ceil(int(L) / page)) for L in lens]
        self.maxp = maxp or max(need)
        self.paged = paged
        if paged:
            self.table, n = I.page_table_np(rot_seed + 5, np.maximum(self.lens, 1), page, self.maxp)
            self.num_pages = n + spare_pages
        else:
            self.table = None
            self.num_pages = self.B * self.maxp + spare_pages
        self.desc = K.CacheDesc(d, hkv, block, bits, K.SCALE_TYPES[scale], 1e-6, page, self.B, self.maxp,
                                0, self.num_pages)
        self.layout = O.Layout(d, hkv, block, scale, page, self.B, self.maxp, self.num_pages, bits)
        self.rot = K.Rotation(d, rot_seed, flags)
        if flags & 4:   # two-quaternion SO(4) blocks
            s, q, qr = O.rotation_params_pair(d, rot_seed, bool(flags & 1))
            self.U = O.rotation_matrix(s, q, qr)
        else:
            s, q = O.rotation_params(d, rot_seed, bool(flags & 1), bool(flags & 2))
            self.U = O.rotation_matrix(s, q)
        self.spec = data or I.DataSpec(d, hkv, 1234, 0.03, 20.0)
        # the pool, then CANARY guard bytes that no kernel may touch
        self._pool_full = torch.zeros(self.layout.pool_bytes + CANARY, dtype=torch.uint8, device=self.dev)
        self._pool_full[self.layout.pool_bytes:] = CANARY_BYTE
        self.pool = self._pool_full[:self.layout.pool_bytes]
        self.pool_o = np.zeros(self.layout.pool_bytes, np.uint8)
        self.table_t = None if self.table is None else torch.as_tensor(self.table, device=self.dev)
        self.lens_t = torch.as_tensor(self.lens, device=self.dev)
        self.cache = K.Cache(self.pool.data_ptr(),
                             None if self.table_t is None else self.table_t.data_ptr(),
                             self.lens_t.data_ptr())
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)

    # ------------------------------------------------------------ inputs
    def tokens(self, upto=None):
        """(k, v, seq_idx, pos) of every position [0, L_b) of every sequence."""
        ks, vs, si, ps = [], [], [], []
        for b in range(self.B):
            n = int(self.lens[b]) if upto is None else min(int(self.lens[b]), upto)
            if n == 0:
                continue
            ks.append(np.stack([I.kv_rows_np(self.spec, 0, b, h, 0, n) for h in range(self.hkv)], 1))
            vs.append(np.stack([I.kv_rows_np(self.spec, 1, b, h, 0, n) for h in range(self.hkv)], 1))
            si.append(np.full(n, b, np.int32))
            ps.append(np.arange(n, dtype=np.int32))
        return (np.concatenate(ks), np.concatenate(vs), np.concatenate(si), np.concatenate(ps))

    def queries(self, step=0):
        return I.q_np(self.spec, self.B, self.hq, step)

    # ------------------------------------------------------------ runs
    def gpu_write(self, k, v, si, ps):
        t = self.torch
        self.K.kvq3_write(self.rot.handle, self.desc, self.cache, t.as_tensor(k, device=self.dev),
                          t.as_tensor(v, device=self.dev), t.as_tensor(si, device=self.dev),
                          t.as_tensor(ps, device=self.dev), self.status)

    def oracle_write(self, k, v, si, ps):
        return O.write(self.pool_o, self.layout, self.U, k, v, si, ps, self.table)

    def guarded(self, nbytes):
        """A uint8 device buffer of nbytes followed by CANARY guard bytes:
        (full, view); check_guard(full, nbytes) after the kernels ran."""
        t = self.torch
        full = t.empty(nbytes + CANARY, dtype=t.uint8, device=self.dev)
        full[nbytes:] = CANARY_BYTE
        return full, full[:nbytes]

    @staticmethod
    def check_guard(full, nbytes, what):
        tail = full[nbytes:].cpu().numpy()
        assert np.all(tail == CANARY_BYTE), f"{what}: a kernel wrote past the end of the buffer"

    def gpu_decode(self, q, sm_scale=0.0):
        t = self.torch
        n_out = self.B * self.hq * self.d * 4
        out_full, out_b = self.guarded(n_out)
        out = out_b.view(t.float32).view(self.B, self.hq, self.d)
        out.fill_(float("nan"))
        n_ws = self.K.kvq3_decode_workspace_size(self.desc, self.hq)
        ws_full, ws = self.guarded(n_ws)
        self.K.kvq3_decode_attn(self.rot.handle, self.desc, self.cache, t.as_tensor(q, device=self.dev),
                                out, ws, sm_scale, self.status)
        t.cuda.synchronize()
        self.check_guard(out_full, n_out, "decode output")
        self.check_guard(ws_full, n_ws, "decode workspace")
        self.check_pool_guard()
        return out.cpu().numpy().astype(np.float64)

    def check_pool_guard(self):
        self.check_guard(self._pool_full, self.layout.pool_bytes, "cache pool")

    def oracle_decode(self, q, sm_scale=0.0, lens=None):
        return O.decode(self.pool_o, self.layout, self.U, q, self.lens if lens is None else lens,
                        self.table, sm_scale)

    def upload_oracle_pool(self):
        self.pool.copy_(self.torch.as_tensor(self.pool_o, device=self.dev))

    def device_status(self):
        self.torch.cuda.synchronize()
        self.check_pool_guard()
        return int(self.status.item())

    # ------------------------------------------------------------ comparisons
    def compare_written(self, k, v, si, ps):
        """Compares the library's stored scales and codes with the oracle's
        for every written token.  Returns counts of excluded boundary
        elements and scale-midpoint blocks."""
        if self.scale == "e4m3zp":
            return self._compare_written_asym(k, v, si, ps)
        gp = self.pool.cpu().numpy()
        nb = self.d // self.block
        excl_codes = excl_blocks = checked = 0
        for which, src in ((0, k), (1, v)):
            x = src.astype(np.float64).reshape(-1, self.d) @ self.U.T
            c_o, sq_o, s_o = O.quantize(x, self.block, 1e-6, self.scale, self.bits)
            page, slot, st = O.locate(self.layout, self.table, np.repeat(si, self.hkv),
                                      np.repeat(ps, self.hkv))
            ok = st == 0
            heads = np.tile(np.arange(self.hkv), len(si))
            rec = page * self.layout.page_bytes + (heads * 2 + which) * self.layout.record_bytes
            so = rec + slot * nb * self.layout.sb
            co = rec + self.page * nb * self.layout.sb + slot * self.layout.code_bytes
            idx_s = so[ok][:, None] + np.arange(nb * self.layout.sb)[None]
            idx_c = co[ok][:, None] + np.arange(self.layout.code_bytes)[None]
            sg = O.decode_scales(gp[idx_s], self.scale)
            cg = O.unpack_codes(gp[idx_c], self.d, self.bits)
            sq_o, s_o, c_o, xo = sq_o[ok], s_o[ok], c_o[ok], x[ok]
            mid = O.scale_midpoint_distance(s_o, self.scale) < MIDPOINT          # [n, nb]
            good_blk = ~mid
            assert np.all(np.abs(sg - sq_o)[good_blk] <= TOL_SCALE * sq_o[good_blk]), "scale mismatch"
            r = np.abs(xo.reshape(-1, nb, self.block) / np.where(sq_o > 0, sq_o, 1)[..., None])
            near = np.zeros(r.shape, bool)
            for kk in range(O.qmax(self.bits)):
                near |= np.abs(r - (kk + 0.5)) < BOUNDARY
            near |= mid[..., None]
            near = near.reshape(-1, self.d)
            bad = (cg != c_o) & ~near
            assert not bad.any(), f"{int(bad.sum())} codes differ outside rounding boundaries"
            excl_codes += int(near.sum())
            excl_blocks += int(mid.sum())
            checked += cg.size
        return dict(checked=checked, boundary_codes=excl_codes, midpoint_blocks=excl_blocks)


def _asym_sets(case, x):
    """Asymmetric variant: oracle codes, (scale, zero point), fp64 scale,
    (x - z_q)/s_q and the blocks whose scale or zero point sits within
    MIDPOINT of an E4M3 rounding midpoint."""
    nb, blk = case.d // case.block, case.block
    u, sz, s = O.quantize_asym(x, blk, 1e-6, case.bits)
    lo = x.reshape(-1, nb, blk).min(-1)
    mid_s = O.scale_midpoint_distance(s, "e4m3") < MIDPOINT
    mid_z = O.scale_midpoint_distance(np.abs(lo), "e4m3") < MIDPOINT
    sq, zq = sz[..., 0], sz[..., 1]
    r = (x.reshape(-1, nb, blk) - zq[..., None]) / np.where(sq > 0, sq, 1)[..., None]
    return u, sz, r, mid_s, mid_z


def _compare_written_asym(self, k, v, si, ps):
    gp = self.pool.cpu().numpy()
    lay, nb = self.layout, self.d // self.block
    top = (1 << self.bits) - 1
    checked = excluded = mids = 0
    for which, src in ((0, k), (1, v)):
        x = src.astype(np.float64).reshape(-1, self.d) @ self.U.T
        u_o, sz_o, r, mid_s, mid_z = _asym_sets(self, x)
        page, slot, st = O.locate(lay, self.table, np.repeat(si, self.hkv), np.repeat(ps, self.hkv))
        ok = st == 0
        heads = np.tile(np.arange(self.hkv), len(si))
        rec = page * lay.page_bytes + (heads * 2 + which) * lay.record_bytes
        so = rec + slot * nb * lay.sb
        co = rec + self.page * nb * lay.sb + slot * lay.code_bytes
        sz_g = O.decode_scales(gp[so[ok][:, None] + np.arange(nb * lay.sb)[None]], "e4m3zp")
        u_g = O.unpack_codes(gp[co[ok][:, None] + np.arange(lay.code_bytes)[None]], self.d, self.bits, signed=False)
        mid = (mid_s | mid_z)[ok]
        assert np.array_equal(sz_g[~mid], sz_o[ok][~mid]), "scale / zero point mismatch"
        near = np.zeros(r[ok].shape, bool)
        for kk in range(top):
            near |= np.abs(r[ok] - (kk + 0.5)) < BOUNDARY
        near = (near | mid[..., None]).reshape(-1, self.d)
        bad = (u_g != u_o[ok]) & ~near
        assert not bad.any(), f"{int(bad.sum())} codes differ outside rounding boundaries"
        checked += u_g.size
        excluded += int(near.sum())
        mids += int(mid.sum())
    return dict(checked=checked, boundary_codes=excluded, midpoint_blocks=mids)


Case._compare_written_asym = _compare_written_asym


def flip_bound(case, k, v, si, ps, q, sm_scale=0.0, differs=None):
    """Upper bound, per (sequence, query head), on how far the decode output
    may move when the cache holds any of the codes and scales that the write
    bar allows besides the oracle's own: elements whose |x/s_q| lies within
    BOUNDARY of a rounding boundary may be one code step off, and blocks whose
    fp64 scale lies within MIDPOINT of a storage midpoint may hold the
    neighbouring scale.  Computed from the oracle's data.  `differs`
    (optional, from Case.written_differences) restricts the bound to the
    elements and blocks that do differ in a given cache.

    A value change dv at token t shifts the rotated output by w_t dv (w the
    softmax weights).  A key change dk in coordinate i shifts logit t by
    delta = sm |q1_i| dk; the output then moves by at most
    sum_t w_t (e^|delta_t| - 1) (|v_t - o| + max_s |v_s - o|).  Both bound the
    L2 change of the rotated output, hence every element after U^T."""
    d, blk, nb = case.d, case.block, case.d // case.block
    G = case.hq // case.hkv
    sm = sm_scale if sm_scale > 0 else 1.0 / math.sqrt(d)
    # relative spacing of neighbouring stored scales (upper bound)
    ulp_rel = {"f32": 2.0 ** -23, "f16": 2.0 ** -10, "e4m3": 2.0 ** -3, "e4m3zp": 2.0 ** -3}[case.scale]
    out = np.zeros((case.B, case.hq))
    for b in range(case.B):
        sel = np.nonzero(si == b)[0]
        if sel.size == 0:
            continue
        sel = sel[np.argsort(ps[sel])]
        for g in range(case.hkv):
            deq, slack = [], []
            for which, src in enumerate((k, v)):
                x = src[sel, g].astype(np.float64) @ case.U.T
                if case.scale == "e4m3zp":
                    # asymmetric variant: a code within reach of a boundary of
                    # (x - z_q)/s_q may be one step s_q off; a neighbouring
                    # scale moves every value s_q u by u * ulp * s_q and shifts
                    # (x - z_q)/s_q by up to (2^b - 1/2) * ulp, a neighbouring
                    # zero point moves every value by ulp * |z_q| and shifts
                    # (x - z_q)/s_q by that over s_q
                    top = (1 << case.bits) - 1
                    u, sz, r, mid_s, mid_z = _asym_sets(case, x)
                    sq, zq = sz[..., 0], sz[..., 1]
                    reach = BOUNDARY + np.where(mid_s, (top + 0.5) * ulp_rel, 0.0) + \
                        np.where(mid_z, ulp_rel * np.abs(zq) / np.where(sq > 0, sq, 1), 0.0)
                    near = np.zeros(r.shape, bool)
                    for kk in range(top):
                        near |= np.abs(r - (kk + 0.5)) < reach[..., None]
                    mid = mid_s | mid_z
                    if differs is not None:
                        code_d, blk_d = differs[(b, g, which)]
                        near &= code_d.reshape(r.shape)
                        mid &= blk_d
                        mid_s, mid_z = mid_s & blk_d, mid_z & blk_d
                    step = np.where(near, 1.0 + ulp_rel, 0.0) * sq[..., None]
                    step += np.where(mid_s[..., None], u.reshape(r.shape) * ulp_rel, 0.0) * sq[..., None]
                    step += np.where(mid_z[..., None], ulp_rel * np.abs(zq)[..., None], 0.0)
                    deq.append((u.reshape(r.shape) * sq[..., None] + zq[..., None]).reshape(-1, d))
                    slack.append(step.reshape(-1, d))
                    continue
                qm = O.qmax(case.bits)
                c, sq, s = O.quantize(x, blk, 1e-6, case.scale, case.bits)
                r = np.abs(x.reshape(-1, nb, blk) / np.where(sq > 0, sq, 1.0)[..., None])
                mid = O.scale_midpoint_distance(s, case.scale) < MIDPOINT
                # a neighbouring scale moves every x/s by up to (qmax + 1/2) * ulp_rel:
                # codes that close to a boundary may flip, and every value
                # c * s_q moves by |c| * ulp_rel * s_q
                reach = np.where(mid, BOUNDARY + (qm + 0.5) * ulp_rel, BOUNDARY)[..., None]
                near = np.zeros(r.shape, bool)
                for kk in range(qm):
                    near |= np.abs(r - (kk + 0.5)) < reach
                if differs is not None:
                    code_d, blk_d = differs[(b, g, which)]
                    near &= code_d.reshape(r.shape)
                    mid &= blk_d
                step = np.where(near, 1.0 + ulp_rel, 0.0) * sq[..., None]
                step += np.where(mid[..., None], np.abs(c.reshape(r.shape)) * ulp_rel, 0.0) * sq[..., None]
                deq.append((c.reshape(-1, nb, blk) * sq[..., None]).reshape(-1, d))
                slack.append(step.reshape(-1, d))
            k_hat, v_hat = deq
            dk, dv = slack
            for gh in range(G):
                h = g * G + gh
                q1 = case.U @ q[b, h].astype(np.float64)
                z = sm * (k_hat @ q1)
                w = np.exp(z - z.max())
                w /= w.sum()
                o = w @ v_hat
                bound_v = float(w @ dv.sum(axis=1))
                delta = sm * (dk @ np.abs(q1))
                dist = np.linalg.norm(v_hat - o, axis=1)
                bound_k = float((w * np.expm1(delta)) @ (dist + dist.max()))
                out[b, h] = bound_v + bound_k
    return out


def written_differences(case, k, v, si, ps):
    """Where the library's stored codes and scales differ from the oracle's,
    per (sequence, kv head, K|V), in position order: (code mask [n][d], block
    mask [n][d/m]).  Every difference must be one the write bar allows
    (compare_written checks that first)."""
    case.compare_written(k, v, si, ps)
    gp = case.pool.cpu().numpy()
    nb = case.d // case.block
    out = {}
    for b in range(case.B):
        sel = np.nonzero(si == b)[0]
        if sel.size == 0:
            continue
        sel = sel[np.argsort(ps[sel])]
        page, slot, st = O.locate(case.layout, case.table, si[sel], ps[sel])
        for g in range(case.hkv):
            for which, src in ((0, k), (1, v)):
                x = src[sel, g].astype(np.float64) @ case.U.T
                if case.scale == "e4m3zp":
                    u_o, sz_o, _ = O.quantize_asym(x, case.block, 1e-6, case.bits)
                    rec = page * case.layout.page_bytes + (g * 2 + which) * case.layout.record_bytes
                    so = rec + slot * nb * case.layout.sb
                    co = rec + case.page * nb * case.layout.sb + slot * case.layout.code_bytes
                    sz_g = O.decode_scales(gp[so[:, None] + np.arange(nb * case.layout.sb)[None]], "e4m3zp")
                    u_g = O.unpack_codes(gp[co[:, None] + np.arange(case.layout.code_bytes)[None]], case.d,
                                         case.bits, signed=False)
                    out[(b, g, which)] = (u_g != u_o, (sz_g != sz_o).any(-1))
                    continue
                c_o, sq_o, _ = O.quantize(x, case.block, 1e-6, case.scale, case.bits)
                rec = page * case.layout.page_bytes + (g * 2 + which) * case.layout.record_bytes
                so = rec + slot * nb * case.layout.sb
                co = rec + case.page * nb * case.layout.sb + slot * case.layout.code_bytes
                sg = O.decode_scales(gp[so[:, None] + np.arange(nb * case.layout.sb)[None]], case.scale)
                cg = O.unpack_codes(gp[co[:, None] + np.arange(case.layout.code_bytes)[None]], case.d, case.bits)
                out[(b, g, which)] = (cg != c_o, sg != sq_o)
    return out


def rel_err(got, ref):
    rms = math.sqrt(float(np.mean(ref ** 2)))
    return float(np.abs(got - ref).max()) / rms if rms > 0 else float(np.abs(got).max())

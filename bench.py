"""Benchmark of the rotated 3-bit KV cache on GB300.

Decode workloads: one step = one decode step of one layer for every sequence
of the workload -- kvq3_write appends the current token's K and V (one per
sequence, position N-1) and kvq3_decode_attn attends over the N cached
tokens.  The write-path workload: one step rotates, quantises and packs the
whole prefill (131,072 tokens x 8 kv heads, K and V) with kvq3_write_chunk.
Inputs are seeded synthetic data (kvq3_inputs).

The default run measures every single-GPU workload in one process and prints
one JSON line.  Its headline is the largest decode workload, ragged (batch 64,
lengths drawn from [1,024, 65,536], d = 256, paged); the 70B-shaped 128K
decode (long70b), the Llama-3-8B-shaped decode (llama8b) and the prefill
write path (prefill) ride along under "configs", each with its own roofline,
end-to-end figure and CPU-oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W]
  python bench.py --workload NAME ...     (one workload only; --profile for ncu)
  python bench.py --impl reference ...    (the CPU oracle, bounded sample)

Multi-GPU: every rank serves its own batch of sequences (data parallel over
(sequence, kv head) units, no exchange on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import kvq3_inputs as I  # noqa: E402

# ---------------------------------------------------------------------- helpers
def algorithmic_bytes(w: I.Workload, lens) -> dict:
    """Algorithmic bytes of one step: packed K/V codes and scales of every
    attended token (read once), q (fp16) and out (fp32) of the decode; fp16
    input and packed output of the write."""
    nb = w.d // w.block
    sb = {"f32": 4, "f16": 2, "e4m3": 1, "e4m3zp": 2}[w.scale]
    per_tok_head = 2 * (w.bits * w.d // 8 + nb * sb)
    kv = int(sum(int(L) for L in lens)) * w.num_kv_heads * per_tok_head
    qo = w.batch * w.num_q_heads * w.d * (2 + 4)
    write_in = w.batch * w.num_kv_heads * 2 * w.d * 2
    write_out = w.batch * w.num_kv_heads * per_tok_head
    return dict(decode=kv + qo, write=write_in + write_out, per_token_head=per_tok_head)


# code width, scale format and page size overrides (--bits, --scale, --page): 0 / "" keep each
# workload's own
BITS_OVERRIDE = 0
SCALE_OVERRIDE = ""
PAGE_OVERRIDE = 0


def workload(name: str) -> I.Workload:
    """The named workload, with the code width of --bits and the scale
    format of --scale when given."""
    import dataclasses
    w = I.workloads()[name]
    if BITS_OVERRIDE:
        w = dataclasses.replace(w, bits=BITS_OVERRIDE)
    if SCALE_OVERRIDE:
        w = dataclasses.replace(w, scale=SCALE_OVERRIDE)
    if PAGE_OVERRIDE and w.decode and not w.paged:
        w = dataclasses.replace(w, page_size=PAGE_OVERRIDE)
    return w


def workload_lens(w: I.Workload) -> np.ndarray:
    if w.len_range:
        return I.seq_lens_np(w.data.seed, w.batch, *w.len_range)
    return np.full(w.batch, w.seq_len, np.int32)


# the source files each profiled kernel is built from (headers included)
KERNEL_SOURCES = {
    "decode": ("kvq3_decode.cuh", "kvq3_decode.cu", "kvq3_decode_d*.cu"),
    "write_chunk": ("kvq3_write_chunk.cu",),
    "prefill_tc": ("kvq3_prefill_tc.cu", "kvq3_tc.cuh"),
}


def source_hash(kernel: str) -> str:
    """Hash of the sources of `kernel`: its own files, the shared device and
    internal headers and the public header."""
    import fnmatch
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hadamard_rotated_bit_kvq3_gb300", "csrc")
    pats = KERNEL_SOURCES[kernel] + ("kvq3_common.cuh", "kvq3_internal.h")
    for f in sorted(os.listdir(csrc)):
        if any(fnmatch.fnmatch(f, pt) for pt in pats):
            h.update(open(os.path.join(csrc, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "kvq3.h"), "rb").read())
    return h.hexdigest()[:16]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d.get("bf16_tflops", 1900.0)), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, src="fallback")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.rows and time.time() - t0 < 5.0:   # first sample before timing
                time.sleep(0.02)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([t.strip() for t in line.split(",")])

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm = [float(r[0]) for r in self.rows if len(r) >= 8 and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if len(r) >= 8 and r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows if len(r) >= 8
                          for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(sm)}


# ---------------------------------------------------------------------- GPU state
class GpuWorkload:
    """Device buffers of one workload, its cache prefilled with N-1 tokens per
    sequence through kvq3_write."""

    def __init__(self, name: str, device, rank: int = 0, batch: int = 0):
        import dataclasses

        import torch
        import hadamard_rotated_bit_kvq3_gb300 as K
        self.K, self.torch = K, torch
        self.w = w = workload(name)
        if batch:
            self.w = w = dataclasses.replace(w, batch=batch)
        self.dev = device
        self.lens = workload_lens(w)
        P = w.page_size
        self.maxp = int(math.ceil(int(self.lens.max()) / P))
        if w.paged:
            self.table_np, self.num_pages = I.page_table_np(w.data.seed, self.lens, P, self.maxp)
            self.table = torch.as_tensor(self.table_np, device=device)
        else:
            self.table_np, self.table = None, None
            self.num_pages = w.batch * self.maxp
        self.desc = K.CacheDesc(w.d, w.num_kv_heads, w.block, w.bits, K.SCALE_TYPES[w.scale], w.eps, P,
                                w.batch, self.maxp, 0, self.num_pages)
        _, _, pool_bytes = K.kvq3_cache_sizes(self.desc)
        self.pool = torch.zeros(pool_bytes, dtype=torch.uint8, device=device)
        self.lens_t = torch.as_tensor(self.lens, device=device)
        self.cache = K.Cache(self.pool.data_ptr(), None if self.table is None else self.table.data_ptr(),
                             self.lens_t.data_ptr())
        self.rot = K.Rotation(w.d, w.rot_seed, w.rot_flags)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws = torch.empty(K.kvq3_decode_workspace_size(self.desc, w.num_q_heads), dtype=torch.uint8,
                              device=device)
        self.out = torch.empty((w.batch, w.num_q_heads, w.d), dtype=torch.float32, device=device)
        # prefill positions [0, L_b - 1) of every sequence
        for b in range(w.batch):
            n = int(self.lens[b]) - 1
            for t0 in range(0, n, 65536):
                m = min(65536, n - t0)
                k, v = self.kv_rows(b, t0, m)
                if w.d <= 128:
                    K.kvq3_write_chunk(self.rot.handle, self.desc, self.cache, k, v, b, t0, self.status)
                else:
                    self.write(k, v, torch.full((m,), b, dtype=torch.int32, device=device),
                               torch.arange(t0, t0 + m, dtype=torch.int32, device=device))
        # the decode step's own token: position L_b - 1 of every sequence
        rows = [self.kv_rows(b, int(self.lens[b]) - 1, 1) for b in range(w.batch)]
        self.k_new = torch.cat([r[0] for r in rows])
        self.v_new = torch.cat([r[1] for r in rows])
        self.seq_new = torch.arange(w.batch, dtype=torch.int32, device=device)
        self.pos_new = torch.as_tensor(self.lens - 1, device=device)
        self.q = torch.as_tensor(I.q_np(w.data, w.batch, w.num_q_heads), device=device)
        torch.cuda.synchronize()

    def kv_rows(self, b, t0, m):
        torch = self.torch
        w = self.w
        k = torch.stack([I.kv_rows_torch(w.data, 0, b, h, t0, m, self.dev) for h in range(w.num_kv_heads)], 1)
        v = torch.stack([I.kv_rows_torch(w.data, 1, b, h, t0, m, self.dev) for h in range(w.num_kv_heads)], 1)
        return k.contiguous(), v.contiguous()

    def write(self, k, v, seq, pos):
        self.K.kvq3_write(self.rot.handle, self.desc, self.cache, k, v, seq, pos, self.status)

    def decode(self, q=None, out=None):
        self.K.kvq3_decode_attn(self.rot.handle, self.desc, self.cache, self.q if q is None else q,
                                self.out if out is None else out, self.ws, 0.0, self.status)

    def step(self):
        self.write(self.k_new, self.v_new, self.seq_new, self.pos_new)
        self.decode()


class PrefillWorkload:
    """The prefill write workload: 131,072 tokens x 8 kv heads x d = 128, K and
    V fp16 resident on the device; one step writes all of them (rotate,
    quantise, pack) into a contiguous cache."""

    def __init__(self, device, tokens: int = 0):
        import dataclasses

        import torch
        import hadamard_rotated_bit_kvq3_gb300 as K
        self.K, self.torch = K, torch
        self.w = w = workload("prefill")
        if tokens:
            self.w = w = dataclasses.replace(w, seq_len=tokens)
        self.dev = device
        n, P = w.seq_len, w.page_size
        self.maxp = n // P
        self.num_pages = self.maxp
        self.table_np = None
        self.desc = K.CacheDesc(w.d, w.num_kv_heads, w.block, w.bits, K.SCALE_TYPES[w.scale], w.eps, P, 1,
                                self.maxp, 0, self.num_pages)
        _, _, pool_bytes = K.kvq3_cache_sizes(self.desc)
        self.pool = torch.zeros(pool_bytes, dtype=torch.uint8, device=device)
        self.lens_t = torch.tensor([n], dtype=torch.int32, device=device)
        self.cache = K.Cache(self.pool.data_ptr(), None, self.lens_t.data_ptr())
        self.rot = K.Rotation(w.d, w.rot_seed, w.rot_flags)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        ks, vs = [], []
        for t0 in range(0, n, 32768):
            m = min(32768, n - t0)
            ks.append(torch.stack([I.kv_rows_torch(w.data, 0, 0, h, t0, m, device)
                                   for h in range(w.num_kv_heads)], 1))
            vs.append(torch.stack([I.kv_rows_torch(w.data, 1, 0, h, t0, m, device)
                                   for h in range(w.num_kv_heads)], 1))
        self.k = torch.cat(ks).contiguous()
        self.v = torch.cat(vs).contiguous()
        self.seq = torch.zeros(n, dtype=torch.int32, device=device)
        self.pos = torch.arange(n, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    def step(self):
        self.K.kvq3_write_chunk(self.rot.handle, self.desc, self.cache, self.k, self.v, 0, 0,
                                self.status)

    def bytes(self):
        w = self.w
        rec_tok = w.bits * w.d // 8 + (w.d // w.block) * {"f32": 4, "f16": 2, "e4m3": 1, "e4m3zp": 2}[w.scale]
        n = w.seq_len * w.num_kv_heads * 2
        return n * w.d * 2 + n * rec_tok


# ---------------------------------------------------------------------- CPU oracle
def oracle_sample(w: I.Workload, lens, unit: int):
    """Builds the oracle's pool for one (sequence, kv head) unit of the
    workload (setup, untimed) and returns a closure that runs the oracle on
    that unit: write of the step's token and decode of its G query heads."""
    from oracle import kvq3_oracle as O
    b, h = divmod(unit, w.num_kv_heads)
    L = int(lens[b])
    P = w.page_size
    maxp = int(math.ceil(L / P))
    lay = O.Layout(w.d, 1, w.block, w.scale, P, 1, maxp, maxp, w.bits)
    signs, quats = O.rotation_params(w.d, w.rot_seed, bool(w.rot_flags & 1), bool(w.rot_flags & 2))
    U = O.rotation_matrix(signs, quats)
    pool = np.zeros(lay.pool_bytes, np.uint8)
    k = I.kv_rows_np(w.data, 0, b, h, 0, L)[:, None]
    v = I.kv_rows_np(w.data, 1, b, h, 0, L)[:, None]
    O.write(pool, lay, U, k[:-1], v[:-1], np.zeros(L - 1, np.int32), np.arange(L - 1), None, w.eps)
    q = I.q_np(w.data, w.batch, w.num_q_heads)[b:b + 1, h * w.group:(h + 1) * w.group]

    def run():
        O.write(pool, lay, U, k[-1:], v[-1:], np.zeros(1, np.int32), np.array([L - 1]), None, w.eps)
        return O.decode(pool, lay, U, q, np.array([L]))
    return run


def cpu_baseline(w: I.Workload, lens, budget_s: float = 15.0) -> dict:
    """Times the oracle on a bounded sample of (sequence, kv head) units and
    scales to the workload's tokens/s."""
    units = w.batch * w.num_kv_heads
    run = oracle_sample(w, lens, 0)
    t0 = time.perf_counter()
    run()
    per_unit = time.perf_counter() - t0
    n = max(1, min(units, int(budget_s / max(per_unit, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(n):
        run()
    per_unit = (time.perf_counter() - t0) / n
    step_s = per_unit * units * float(np.mean(lens)) / int(lens[0])
    return {"value": w.batch / step_s, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"unit (b=0, kv head 0): write 1 token + decode {w.group} heads over "
                      f"{int(lens[0])} tokens, x{n} runs; scaled to {units} units"}


# ---------------------------------------------------------------------- main
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.init_process_group("nccl")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units per second of the whole job: every rank processes units_per_rank
    units per step and ms is the slowest rank's time per step (max over ranks)."""
    return units_per_rank * world / (ms * 1e-3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def timed_cpu_baseline(run, to_value, unit: str, what: str, budget_s: float = 15.0) -> dict:
    """The oracle as it stands, timed on a bounded sample (about budget_s of
    CPU work after one untimed run)."""
    t0 = time.perf_counter()
    run()
    per = time.perf_counter() - t0
    n = max(1, min(16, int(budget_s / max(per, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(n):
        run()
    per = (time.perf_counter() - t0) / n
    return {"value": to_value(per), "unit": unit, "cores": blas_threads(), "kind": "oracle",
            "sample": f"{what}; x{n} runs"}


def oracle_write_sample(w: I.Workload, n_tok: int):
    """Oracle leg of the write-path workload: a closure writing the first
    n_tok positions (all kv heads, K and V) into a fresh oracle pool."""
    from oracle import kvq3_oracle as O
    P = w.page_size
    maxp = int(math.ceil(n_tok / P))
    lay = O.Layout(w.d, w.num_kv_heads, w.block, w.scale, P, 1, maxp, maxp, w.bits)
    signs, quats = O.rotation_params(w.d, w.rot_seed, bool(w.rot_flags & 1), bool(w.rot_flags & 2))
    U = O.rotation_matrix(signs, quats)
    k = np.stack([I.kv_rows_np(w.data, 0, 0, h, 0, n_tok) for h in range(w.num_kv_heads)], 1)
    v = np.stack([I.kv_rows_np(w.data, 1, 0, h, 0, n_tok) for h in range(w.num_kv_heads)], 1)
    pool = np.zeros(lay.pool_bytes, np.uint8)

    def run():
        O.write(pool, lay, U, k, v, np.zeros(n_tok, np.int32), np.arange(n_tok), None, w.eps)
    return run


def oracle_prefill_sample(w: I.Workload, n_q: int):
    """Oracle leg of the prefill-attention workload: the cache of the whole
    context written once (untimed); a closure answering the last n_q queries
    of the chunk (all query heads)."""
    from oracle import kvq3_oracle as O
    n, P = w.seq_len, w.page_size
    maxp = int(math.ceil(n / P))
    lay = O.Layout(w.d, w.num_kv_heads, w.block, w.scale, P, 1, maxp, maxp, w.bits)
    signs, quats = O.rotation_params(w.d, w.rot_seed, bool(w.rot_flags & 1), bool(w.rot_flags & 2))
    U = O.rotation_matrix(signs, quats)
    pool = np.zeros(lay.pool_bytes, np.uint8)
    step = 4096
    for t0 in range(0, n, step):
        m = min(step, n - t0)
        k = np.stack([I.kv_rows_np(w.data, 0, 0, h, t0, m) for h in range(w.num_kv_heads)], 1)
        v = np.stack([I.kv_rows_np(w.data, 1, 0, h, t0, m) for h in range(w.num_kv_heads)], 1)
        O.write(pool, lay, U, k, v, np.zeros(m, np.int32), np.arange(t0, t0 + m), None, w.eps)
    q = I.q_np(w.data, n_q, w.num_q_heads, 3)

    def run():
        return O.prefill(pool, lay, U, q, 0, n - n_q)
    return run


DECODE_METRIC = "decode tokens/s (one layer, all heads)"
WRITE_METRIC = "write-path GB/s (fp16 in + packed out)"
PREFILL_ATTN_METRIC = "prefill-attention query tokens/s (one layer, all heads)"
PRIMARY = "ragged"                                 # the largest single-GPU decode workload
EXTRAS = ("long70b", "llama8b", "prefill", "prefill_attn")   # measured in the same run, under "configs"
NOMINAL_HBM_GBS = 8000.0                           # the HBM peak the method's target is quoted against


def sbytes(w: I.Workload) -> int:
    return {"f32": 4, "f16": 2, "e4m3": 1, "e4m3zp": 2}[w.scale]


def blas_threads() -> int:
    """Threads numpy's BLAS may use (the oracle's matrix products); its other
    steps run on one Python thread."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count() or 1


def workload_config(w: I.Workload, lens, world: int) -> dict:
    """The "config" object of a workload's JSON record (the same for both arms)."""
    if w.decode:
        ab = algorithmic_bytes(w, lens)
        return {"workload": workload_desc(w),
                "l2": f"inputs larger than L2 (packed cache {ab['decode'] / 1e6:.0f} MB per step)",
                "parallelism": f"replicas x{world} (dp over sequences)"}
    if w.chunk > 0:
        return {"workload": f"{w.name}: chunk of {w.chunk} queries at positions {w.seq_len - w.chunk}.."
                            f"{w.seq_len - 1} of a {w.seq_len}-token cache, Hkv{w.num_kv_heads} "
                            f"Hq{w.num_q_heads} d{w.d} m{w.block} {w.scale} scales, {w.bits}-bit codes, contiguous "
                            f"P{w.page_size}, causal", "l2": "cache 3.4 MB per kv head",
                "parallelism": f"replicas x{world}"}
    return {"workload": f"prefill: {w.seq_len} tokens x Hkv{w.num_kv_heads} x d{w.d}, K+V fp16, "
                        f"sign flip + FWHT, m{w.block} {w.scale} scales, {w.bits}-bit codes",
            "l2": "inputs larger than L2 (537 MB fp16 in, 134 MB packed out per step)",
            "parallelism": f"replicas x{world}"}


def recorded_traffic_of(kernel: str, name: str):
    """DRAM bytes per launch from the committed ncu summary of `kernel` on
    workload `name`, if it was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{name}_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    fam = "decode" if kernel.startswith("decode") else kernel
    return d["dram_bytes_per_launch"] if d.get("source_hash") == source_hash(fam) else None


def _median(xs):
    return statistics.median(xs) if xs else float("nan")


def time_decode(st, steps: int, warmup: int, world: int, stream) -> dict:
    """Device-timed steps of a decode workload, inputs resident: first K steps
    with nothing between the calls (the step time, between barriers, max over
    ranks; the decode may then start under the token write), then K steps
    with an event before the write, between write and decode and after the
    decode (the per-call times)."""
    import torch
    for _ in range(warmup):
        st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0, f"device status {int(st.status.item())}"
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(steps):
        st.write(st.k_new, st.v_new, st.seq_new, st.pos_new)
        st.decode()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        st.write(st.k_new, st.v_new, st.seq_new, st.pos_new)
        ev[i][1].record(stream)
        st.decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    dec = [e[1].elapsed_time(e[2]) for e in ev]
    wr = [e[0].elapsed_time(e[1]) for e in ev]
    step = [e[0].elapsed_time(e[2]) for e in ev]
    assert int(st.status.item()) == 0
    return dict(ms_step=total_ms / steps, ms_step_median=_median(step), dec_median=_median(dec),
                dec_mean=statistics.mean(dec), wr_median=_median(wr), wr_mean=statistics.mean(wr))


def time_decode_e2e(st, steps: int, warmup: int, world: int, stream, dev) -> dict:
    """The same step through pinned host buffers with the copies inside the
    timed region: the step's inputs (new k, v, the queries, positions,
    sequence ids) sit in one pinned host buffer and go over in one copy; the
    output comes back."""
    import torch
    srcs = (st.k_new, st.v_new, st.q, st.pos_new, st.seq_new)
    offs, total = [], 0
    for t in srcs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    inp_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    inp_d = torch.empty(total, dtype=torch.uint8, device=dev)
    views_d = []
    for t, o in zip(srcs, offs):
        nb = t.numel() * t.element_size()
        inp_h[o:o + nb].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        views_d.append(inp_d[o:o + nb].view(t.dtype).view(t.shape))
    k_d, v_d, q_d, pos_d, seq_d = views_d
    out_h = torch.empty(st.out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in srcs)
    d2h = out_h.numel() * out_h.element_size()

    def e2e_step():
        inp_d.copy_(inp_h, non_blocking=True)
        st.write(k_d, v_d, seq_d, pos_d)
        st.decode(q_d, st.out)
        out_h.copy_(st.out, non_blocking=True)

    for _ in range(warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    return dict(ms=max_over_ranks(a.elapsed_time(b), world) / steps, h2d=h2d, d2h=d2h)


def decode_record(name: str, args, world: int, rank: int, dev, peaks: dict, cpu: bool) -> dict:
    """Builds, times and tears down one decode workload; returns its record."""
    import torch
    st = GpuWorkload(name, dev, rank, args.batch)
    w = st.w
    stream = torch.cuda.current_stream()
    t = time_decode(st, args.steps, args.warmup, world, stream)
    e = time_decode_e2e(st, args.steps, args.warmup, world, stream, dev)
    ab = algorithmic_bytes(w, st.lens)
    gbs = ab["decode"] / (t["dec_median"] * 1e-3) / 1e9
    rec = {
        "metric": DECODE_METRIC, "value": whole_job_rate(w.batch, world, t["ms_step"]), "unit": "tokens/s",
        "ms_per_step": t["ms_step"], "ms_per_step_median": t["ms_step_median"],
        "dtype": f"f16 mma / f32 accumulate ({w.bits}-bit packed cache)",
        "config": workload_config(w, st.lens, world),
        "decode": {"ms_median": t["dec_median"], "ms_mean": t["dec_mean"], "hbm_gbs": gbs,
                   "frac_of_peak": gbs / peaks["hbm"], "frac_of_nominal": gbs / NOMINAL_HBM_GBS,
                   "bytes": ab["decode"], "bytes_per_token_head": ab["per_token_head"]},
        "write": {"ms_median": t["wr_median"], "gbs": ab["write"] / (t["wr_median"] * 1e-3) / 1e9,
                  "bytes": ab["write"]},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm"], "frac_of_nominal": gbs / NOMINAL_HBM_GBS,
                     "traffic": recorded_traffic_of("decode", name) if w.bits == 3 and not args.batch else None,
                     "kernel": "kvq3_decode_attn (decode_split_kernel + decode_combine_kernel)",
                     "timing": "median over steps of CUDA events around the kvq3_decode_attn call",
                     "peak_source": peaks["src"]},
        "e2e": {"value": whole_job_rate(w.batch, world, e["ms"]), "unit": "tokens/s",
                "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"]},
        "gpu_launches": 3 * args.steps,
    }
    if cpu:
        rec["cpu_baseline"] = cpu_baseline(w, st.lens)
    del st
    torch.cuda.empty_cache()
    return rec


def prefill_record(args, world: int, rank: int, dev, peaks: dict, cpu: bool) -> dict:
    """The write-path workload: device-timed steps (inputs resident), then
    the same step with the fp16 input copied from pinned host memory and the
    packed cache read back inside the timed region."""
    import torch
    st = PrefillWorkload(dev, args.tokens)
    w = st.w
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        st.step()
        ev[i][1].record(stream)
    b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    assert int(st.status.item()) == 0
    ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
    med = _median([x.elapsed_time(y) for x, y in ev])
    nbytes = st.bytes()
    gbs_med = nbytes / (med * 1e-3) / 1e9
    # end to end: fp16 K, V from pinned host memory, packed pool back
    k_h = st.k.cpu().pin_memory()
    v_h = st.v.cpu().pin_memory()
    pool_h = torch.empty(st.pool.shape, dtype=torch.uint8).pin_memory()

    def e2e_step():
        st.k.copy_(k_h, non_blocking=True)
        st.v.copy_(v_h, non_blocking=True)
        st.step()
        pool_h.copy_(st.pool, non_blocking=True)

    for _ in range(min(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    a.record(stream)
    n_e2e = max(3, min(args.steps, 20))
    for _ in range(n_e2e):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b), world) / n_e2e
    rec = {
        "metric": WRITE_METRIC, "value": whole_job_rate(nbytes, world, ms) / 1e9, "unit": "GB/s",
        "ms_per_step": ms, "ms_per_step_median": med, "dtype": "f32",
        "config": workload_config(w, None, world),
        "roofline": {"bound": "hbm", "achieved": gbs_med, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": gbs_med / peaks["hbm"], "frac_of_nominal": gbs_med / NOMINAL_HBM_GBS,
                     "traffic": recorded_traffic_of("write_chunk", "prefill") if not args.tokens else None,
                     "kernel": "write_chunk_kernel", "bytes": nbytes,
                     "timing": "median over steps of CUDA events around the kvq3_write_chunk call",
                     "peak_source": peaks["src"]},
        "tokens_per_s": whole_job_rate(w.seq_len, world, ms),
        "e2e": {"value": whole_job_rate(nbytes, world, e2e_ms) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": (k_h.numel() + v_h.numel()) * 2, "d2h_bytes_per_step": pool_h.numel(),
                "steps": n_e2e},
        "gpu_launches": args.steps,
    }
    if cpu:
        n_tok = 256
        nb = n_tok * w.num_kv_heads * 2 * (2 * w.d + w.bits * w.d // 8 + (w.d // w.block) * sbytes(w))
        rec["cpu_baseline"] = timed_cpu_baseline(
            oracle_write_sample(w, n_tok), lambda per: nb / per / 1e9, "GB/s",
            f"oracle write of {n_tok} tokens x {w.num_kv_heads} kv heads, K and V")
    del st
    torch.cuda.empty_cache()
    return rec


def single_thread_oracle(names=("tiny", "llama8b")) -> dict:
    """The oracle's decode step timed with every BLAS pool at one thread, in
    a child process (the thread count of a BLAS library is fixed when it
    loads)."""
    out = {}
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    for n in names:
        try:
            p = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-leg", n], env=env,
                               capture_output=True, text=True, timeout=300)
            out[n] = json.loads(p.stdout.strip().splitlines()[-1]) if p.returncode == 0 else \
                {"error": p.stderr.strip()[-300:]}
        except (subprocess.TimeoutExpired, ValueError, IndexError) as e:
            out[n] = {"error": str(e)[:300]}
    return out


def run_suite(args, world, rank, dev):
    """The default run (every workload, one JSON line), or one named
    workload."""
    import torch
    peaks = load_peaks()
    cpu = not args.no_cpu_baseline and world == 1 and rank == 0
    names = [args.workload] if args.workload else [PRIMARY, *EXTRAS]
    if args.profile:
        for name in names:
            profile_steps(name, args, rank, dev)
        return
    records = {}
    with ClockSampler(dev.index or 0) as clk:
        for name in names:
            if name == "prefill":
                records[name] = prefill_record(args, world, rank, dev, peaks, False)
            elif name == "prefill_attn":
                records[name] = prefill_attn_record(args, world, rank, dev, peaks)
            else:
                records[name] = decode_record(name, args, world, rank, dev, peaks, False)
            torch.cuda.synchronize()
    clocks = clk.summary()
    if rank != 0:
        return
    if cpu:   # after the GPU work: the oracle legs run on the host alone
        for name in names:
            w = workload(name)
            if name == "prefill":
                n_tok = 256
                nb = n_tok * w.num_kv_heads * 2 * (2 * w.d + w.bits * w.d // 8 + (w.d // w.block) * sbytes(w))
                records[name]["cpu_baseline"] = timed_cpu_baseline(
                    oracle_write_sample(w, n_tok), lambda per, nb=nb: nb / per / 1e9, "GB/s",
                    f"oracle write of {n_tok} tokens x {w.num_kv_heads} kv heads, K and V",
                    budget_s=10.0 if name != names[0] else 15.0)
            elif name == "prefill_attn":
                records[name]["cpu_baseline"] = prefill_attn_cpu_baseline(w, budget_s=10.0)
            else:
                if args.batch:
                    import dataclasses
                    w = dataclasses.replace(w, batch=args.batch)
                records[name]["cpu_baseline"] = cpu_baseline(
                    w, workload_lens(w), budget_s=10.0 if name != names[0] else 15.0)
    head = records[names[0]]
    line = {"metric": head["metric"], "value": head["value"], "unit": head["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
            "data": "synthetic", "config": head["config"]}
    for key in ("ms_per_step_median", "decode", "write", "roofline", "e2e", "gpu_launches", "cpu_baseline",
                "tokens_per_s"):
        if key in head:
            line[key] = head[key]
    line["clocks"] = clocks
    if len(names) > 1:
        line["configs"] = {n: records[n] for n in names[1:]}
        line["gpu_launches_all"] = sum(r["gpu_launches"] for r in records.values())
    if cpu and not args.workload:
        line["cpu_baseline_single_thread"] = single_thread_oracle()
    print(json.dumps(line))


def profile_steps(name, args, rank, dev):
    """Plain steps only, for ncu captures (kernel order per decode step:
    write, decode split, decode combine)."""
    import torch
    if name == "prefill":
        st = PrefillWorkload(dev, args.tokens)
    elif name == "prefill_attn":
        import dataclasses
        w = workload(name)
        if args.tokens:
            w = dataclasses.replace(w, seq_len=args.tokens, chunk=min(w.chunk, max(1, args.tokens // 4)))
        st = PrefillAttnWorkload(dev, w)
    else:
        st = GpuWorkload(name, dev, rank, args.batch)
    for _ in range(args.warmup + args.steps):
        st.step()
    torch.cuda.synchronize()
    print(json.dumps({"profile": name, "status": int(st.status.item())}))
    del st
    torch.cuda.empty_cache()


def oracle_leg(name: str) -> None:
    """One oracle timing (for single_thread_oracle): prints a cpu_baseline
    record of workload `name` (decode step)."""
    w = workload(name)
    rec = cpu_baseline(w, workload_lens(w), budget_s=8.0)
    rec["cores"] = blas_threads()
    print(json.dumps(rec))


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, timed as it stands on a bounded
    sample of the workload (rank 0 only; about 120 s of timed work at most).
    Each timed step runs one sample (one (sequence, kv head) unit, or a slice
    of the write or of the prefill chunk); ms_per_step is that measured time,
    and value scales it to the whole workload by the factor in "sample"."""
    w = workload(args.workload or PRIMARY)
    lens = workload_lens(w)
    if rank != 0:
        return
    if w.chunk > 0:            # prefill attention: query tokens/s
        n_q = 2
        run = oracle_prefill_sample(w, n_q)
        metric, unit = PREFILL_ATTN_METRIC, "tokens/s"
        what = (f"oracle prefill attention of the last {n_q} queries of the chunk (all "
                f"{w.num_q_heads} heads) over the {w.seq_len}-token cache")
        scale = w.chunk / n_q
        to_value = lambda per: n_q / per                                   # noqa: E731
    elif not w.decode:         # write path: GB/s of fp16 in + packed out
        n_tok = 256
        run = oracle_write_sample(w, n_tok)
        nbytes = n_tok * w.num_kv_heads * 2 * (2 * w.d + w.bits * w.d // 8 + (w.d // w.block) * sbytes(w))
        metric, unit = WRITE_METRIC, "GB/s"
        what = f"oracle write of {n_tok} tokens x {w.num_kv_heads} kv heads, K and V"
        scale = w.seq_len / n_tok
        to_value = lambda per: nbytes / per / 1e9                          # noqa: E731
    else:                      # decode: tokens/s of the whole batch
        units = w.batch * w.num_kv_heads
        run = oracle_sample(w, lens, 0)
        metric, unit = DECODE_METRIC, "tokens/s"
        what = (f"oracle write of 1 token + decode of the {w.group} query heads of one (sequence, kv head) "
                f"unit over {int(lens[0])} tokens")
        scale = units * float(np.mean(lens)) / int(lens[0])
        to_value = lambda per: w.batch / (per * scale)                     # noqa: E731
    for _ in range(min(args.warmup, 3)):
        run()
    # bounded: the timed samples stop after ~120 s of CPU work (at least one)
    t0 = time.perf_counter()
    done = 0
    while done < args.steps and (done == 0 or time.perf_counter() - t0 < 120.0):
        run()
        done += 1
    per = (time.perf_counter() - t0) / done
    value = to_value(per)
    sample = (f"each step: {what}; the workload is {scale:.4g} such samples (value = the sample rate "
              f"scaled by that factor); {done} of {args.steps} steps timed (120 s cap)")
    line = {
        "impl": "reference", "metric": metric, "value": value,
        "unit": unit, "n_gpus": args.gpus, "steps": done, "warmup": min(args.warmup, 3),
        "ms_per_step": per * 1e3, "sample_scale": scale, "ms_per_workload_step": per * scale * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": workload_config(w, lens, world),
        "cpu_baseline": {"value": value, "unit": unit, "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


class PrefillAttnWorkload:
    """Chunked-prefill attention: one sequence whose cache holds seq_len
    tokens (written once with kvq3_write_chunk); one step runs
    kvq3_prefill_attn for its last `chunk` positions (queries resident)."""

    def __init__(self, device, w: I.Workload):
        import torch
        import hadamard_rotated_bit_kvq3_gb300 as K
        self.K, self.torch, self.w, self.dev = K, torch, w, device
        n, P = w.seq_len, w.page_size
        self.maxp = (n + P - 1) // P
        self.desc = K.CacheDesc(w.d, w.num_kv_heads, w.block, w.bits, K.SCALE_TYPES[w.scale], w.eps, P, 1,
                                self.maxp, 0, self.maxp)
        _, _, pool_bytes = K.kvq3_cache_sizes(self.desc)
        self.pool = torch.zeros(pool_bytes, dtype=torch.uint8, device=device)
        self.lens_t = torch.tensor([n], dtype=torch.int32, device=device)
        self.cache = K.Cache(self.pool.data_ptr(), None, self.lens_t.data_ptr())
        self.rot = K.Rotation(w.d, w.rot_seed, w.rot_flags)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        for t0 in range(0, n, 8192):
            m = min(8192, n - t0)
            k = torch.stack([I.kv_rows_torch(w.data, 0, 0, h, t0, m, device) for h in range(w.num_kv_heads)], 1)
            v = torch.stack([I.kv_rows_torch(w.data, 1, 0, h, t0, m, device) for h in range(w.num_kv_heads)], 1)
            K.kvq3_write_chunk(self.rot.handle, self.desc, self.cache, k.contiguous(), v.contiguous(), 0, t0,
                               self.status)
        self.pos0 = n - w.chunk
        self.q = torch.as_tensor(I.q_np(w.data, w.chunk, w.num_q_heads, 0), device=device)
        self.out = torch.empty((w.chunk, w.num_q_heads, w.d), dtype=torch.float32, device=device)
        self.ws = torch.empty(K.kvq3_prefill_workspace_size(self.desc, w.num_q_heads, w.chunk),
                              dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

    def step(self):
        self.K.kvq3_prefill_attn(self.rot.handle, self.desc, self.cache, 0, self.pos0, self.q, self.out,
                                 self.ws, 0.0, self.status)

    def flops(self) -> float:
        """QK^T and PV multiply-adds of the causal chunk: 4 d flops per (query
        head, attended key)."""
        w = self.w
        keys = sum(self.pos0 + i + 1 for i in range(w.chunk))
        return 4.0 * w.d * w.num_q_heads * keys


def prefill_attn_record(args, world: int, rank: int, dev, peaks: dict) -> dict:
    """The prefill-attention workload: device-timed steps (queries and cache
    resident), then the same step with the fp16 queries copied from pinned
    host memory and the fp32 outputs read back inside the timed region."""
    import dataclasses

    import torch
    w = workload("prefill_attn")
    if args.tokens:   # a shorter context (profiling): the chunk is at most a quarter of it
        w = dataclasses.replace(w, seq_len=args.tokens, chunk=min(w.chunk, max(1, args.tokens // 4)))
    st = PrefillAttnWorkload(dev, w)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        st.step()
        ev[i][1].record(stream)
    b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    assert int(st.status.item()) == 0
    ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
    med = _median([x.elapsed_time(y) for x, y in ev])
    tflops = st.flops() / (med * 1e-3) / 1e12
    # end to end: queries from pinned host memory, outputs back
    q_h = st.q.cpu().pin_memory()
    out_h = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()

    def e2e_step():
        st.q.copy_(q_h, non_blocking=True)
        st.step()
        out_h.copy_(st.out, non_blocking=True)

    for _ in range(min(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    a.record(stream)
    n_e2e = max(3, min(args.steps, 20))
    for _ in range(n_e2e):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b), world) / n_e2e
    # d = 128 runs a tile kernel (one launch): the tcgen05 one with blocks of
    # 64 (symmetric codes of 2-4 bits, asymmetric 3-bit codes), the mma.sync
    # one with blocks of 32 (symmetric 3-bit codes); the other formats the
    # decode kernel's prefill variant and the combine
    tc = w.d == 128 and w.block == 64 and (w.scale != "e4m3zp" or w.bits == 3)
    tile = tc or (w.d == 128 and w.bits == 3 and w.scale != "e4m3zp")
    tile_kernel = "prefill_tc_kernel" if tc else "prefill_tile_kernel"
    rec = {
        "metric": PREFILL_ATTN_METRIC, "value": whole_job_rate(w.chunk, world, ms), "unit": "tokens/s",
        "ms_per_step": ms, "ms_per_step_median": med,
        "dtype": f"f16 mma / f32 accumulate ({w.bits}-bit packed cache)",
        "config": workload_config(w, None, world),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": tflops / peaks["bf16"],
                     "traffic": recorded_traffic_of("prefill_tc", "prefill_attn")
                     if tc and w.bits == 3 and w.scale == "f16" and not args.tokens else None,
                     "flops": st.flops(),
                     "kernel": "kvq3_prefill_attn (" + (tile_kernel if tile else
                               "decode_split_kernel<..., prefill> + decode_combine_kernel") + ")",
                     "timing": "median over steps of CUDA events around the kvq3_prefill_attn call",
                     "peak_source": ("measured bf16 (fp16 MMAs have the same nominal rate)"
                                     if peaks["src"] == "measured" else "fallback")},
        "e2e": {"value": whole_job_rate(w.chunk, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": q_h.numel() * q_h.element_size(),
                "d2h_bytes_per_step": out_h.numel() * out_h.element_size(), "steps": n_e2e},
        "gpu_launches": (1 if tile else 2) * args.steps,
    }
    del st
    torch.cuda.empty_cache()
    return rec


def prefill_attn_cpu_baseline(w: I.Workload, budget_s: float = 15.0) -> dict:
    return timed_cpu_baseline(oracle_prefill_sample(w, 1), lambda per: 1.0 / per, "tokens/s",
                              f"oracle prefill attention of the chunk's last query (all {w.num_q_heads} "
                              f"heads) over the {w.seq_len}-token cache (cache written once, untimed)",
                              budget_s=budget_s)


def run_prefill_attn(args, world, rank, dev):
    import torch
    if args.profile:
        import dataclasses
        w = workload(args.workload)
        if args.tokens:
            w = dataclasses.replace(w, seq_len=args.tokens, chunk=min(w.chunk, max(1, args.tokens // 4)))
        st = PrefillAttnWorkload(dev, w)
        for _ in range(args.warmup + args.steps):
            st.step()
        torch.cuda.synchronize()
        print(json.dumps({"profile": w.name, "status": int(st.status.item())}))
        return
    peaks = load_peaks()
    with ClockSampler(dev.index or 0) as clk:
        rec = prefill_attn_record(args, world, rank, dev, peaks)
    if rank == 0:
        line = {"metric": rec["metric"], "value": rec["value"], "unit": rec["unit"], "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": rec["dtype"],
                "data": "synthetic", "config": rec["config"]}
        for key in ("ms_per_step_median", "roofline", "e2e", "gpu_launches"):
            line[key] = rec[key]
        line["clocks"] = clk.summary()
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = prefill_attn_cpu_baseline(workload(args.workload))
        print(json.dumps(line))


def workload_desc(w: I.Workload) -> str:
    lens = f"N={w.seq_len}" if not w.len_range else f"N~U[{w.len_range[0]},{w.len_range[1]}]"
    return (f"{w.name}: B{w.batch} Hkv{w.num_kv_heads} Hq{w.num_q_heads} d{w.d} {lens} m{w.block} "
            f"{w.scale} scales, {w.bits}-bit codes, {'paged' if w.paged else 'contiguous'} P{w.page_size}, "
            f"rot flags {w.rot_flags}; step = kvq3_write(1 token/seq) + kvq3_decode_attn")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="", choices=[""] + sorted(I.workloads()),
                    help="one workload only (default: all, ragged first)")
    ap.add_argument("--impl", default="kvq3", choices=["kvq3", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (smaller profiling cases)")
    ap.add_argument("--tokens", type=int, default=0, help="override the prefill token count")
    ap.add_argument("--profile", action="store_true", help="plain steps only, for ncu captures")
    ap.add_argument("--bits", type=int, default=0, choices=[0, 2, 3, 4],
                    help="code width of the cache (0: the workload's own, 3)")
    ap.add_argument("--scale", default="", choices=["", "f32", "f16", "e4m3", "e4m3zp"],
                    help="scale format (e4m3zp: the asymmetric variant, E4M3 scale and zero point)")
    ap.add_argument("--page", type=int, default=0,
                    help="tokens per page of the contiguous decode caches (0: the workload's own, 128)")
    ap.add_argument("--oracle-leg", default="", help=argparse.SUPPRESS)
    args = ap.parse_args()
    global BITS_OVERRIDE, SCALE_OVERRIDE, PAGE_OVERRIDE
    BITS_OVERRIDE = args.bits
    SCALE_OVERRIDE = args.scale
    PAGE_OVERRIDE = args.page
    if args.oracle_leg:
        oracle_leg(args.oracle_leg)
        return
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.workload and workload(args.workload).chunk > 0:
        run_prefill_attn(args, world, rank, dev)
    else:
        run_suite(args, world, rank, dev)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

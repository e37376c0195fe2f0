"""Benchmark of the rotated 3-bit KV cache on GB300.

One step = one decode step of one layer for every sequence of the workload:
kvq3_write appends the current token's K and V (one per sequence, position
N-1) and kvq3_decode_attn attends over the N cached tokens.  The default
workload is the Llama-3-8B-shaped layer (batch 16, 32 query heads over 8 kv
heads, d = 128, 32,768-token contiguous cache, blocks of 64 with fp16
scales).  Inputs are seeded synthetic data (kvq3_inputs).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle, bounded sample)

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

DEFAULT_WORKLOAD = "llama8b"


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


# code width and scale format overrides (--bits, --scale): 0 / "" keep each workload's own
BITS_OVERRIDE = 0
SCALE_OVERRIDE = ""


def workload(name: str) -> I.Workload:
    """The named workload, with the code width of --bits and the scale
    format of --scale when given."""
    import dataclasses
    w = I.workloads()[name]
    if BITS_OVERRIDE:
        w = dataclasses.replace(w, bits=BITS_OVERRIDE)
    if SCALE_OVERRIDE:
        w = dataclasses.replace(w, scale=SCALE_OVERRIDE)
    return w


def workload_lens(w: I.Workload) -> np.ndarray:
    if w.len_range:
        return I.seq_lens_np(w.data.seed, w.batch, *w.len_range)
    return np.full(w.batch, w.seq_len, np.int32)


def source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hadamard_rotated_bit_kvq3_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), src="measured")
    return dict(hbm=6800.0, src="fallback")


def recorded_traffic(name: str, bits: int = 3):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel sources (3-bit codes)."""
    p = os.path.join(ROOT, "profiles", f"decode_{name}_traffic.json")
    if bits != 3:
        return None
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    return d["dram_bytes_per_launch"] if d.get("source_hash") == source_hash() else None


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
    return {"value": w.batch / step_s, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
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
    return {"value": to_value(per), "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
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


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, timed as it stands on a bounded
    sample of the workload (rank 0 only; about 120 s of timed work at most),
    scaled to the workload's metric."""
    w = workload(args.workload)
    lens = workload_lens(w)
    if rank != 0:
        return
    if w.chunk > 0:            # prefill attention: query tokens/s
        n_q = 2
        run = oracle_prefill_sample(w, n_q)
        metric, unit = "prefill-attention query tokens/s (one layer, all heads)", "tokens/s"
        what = (f"each step: oracle prefill attention of the last {n_q} queries of the chunk (all "
                f"{w.num_q_heads} heads) over the {w.seq_len}-token cache")
        to_value = lambda per: n_q / per                                   # noqa: E731
        to_step_s = lambda per: per * w.chunk / n_q                        # noqa: E731
    elif not w.decode:         # write path: GB/s of fp16 in + packed out
        n_tok = 256
        run = oracle_write_sample(w, n_tok)
        sb = {"f32": 4, "f16": 2, "e4m3": 1, "e4m3zp": 2}[w.scale]
        nbytes = n_tok * w.num_kv_heads * 2 * (2 * w.d + w.bits * w.d // 8 + (w.d // w.block) * sb)
        metric, unit = "write-path GB/s (fp16 in + packed out)", "GB/s"
        what = f"each step: oracle write of {n_tok} tokens x {w.num_kv_heads} kv heads, K and V"
        to_value = lambda per: nbytes / per / 1e9                          # noqa: E731
        to_step_s = lambda per: per * w.seq_len / n_tok                    # noqa: E731
    else:                      # decode: tokens/s of the whole batch
        units = w.batch * w.num_kv_heads
        run = oracle_sample(w, lens, 0)
        metric, unit = "decode tokens/s (one layer, all heads)", "tokens/s"
        what = (f"each step: oracle write 1 token + decode {w.group} query heads of one (sequence, "
                f"kv head) unit over {int(lens[0])} tokens; scaled by {units} units")
        to_step_s = lambda per: per * units * float(np.mean(lens)) / int(lens[0])   # noqa: E731
        to_value = lambda per: w.batch / to_step_s(per)                    # noqa: E731
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
    line = {
        "impl": "reference", "metric": metric, "value": value,
        "unit": unit, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": to_step_s(per) * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w)},
        "cpu_baseline": {"value": value, "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{what}; {done} steps timed (120 s cap)"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_prefill(args, world, rank, dev):
    """Write-path throughput: one step writes the whole prefill workload."""
    import torch
    st = PrefillWorkload(dev, args.tokens)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    if args.profile:
        for _ in range(args.steps):
            st.step()
        torch.cuda.synchronize()
        print(json.dumps({"profile": "prefill", "tokens": st.w.seq_len, "status": int(st.status.item())}))
        return
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index or 0) as clk:
        a.record(stream)
        for _ in range(args.steps):
            st.step()
        b.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
    assert int(st.status.item()) == 0
    peaks = load_peaks()
    gbs = whole_job_rate(st.bytes(), world, ms) / 1e9
    if rank == 0:
        w = st.w
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            n_tok = 256
            sb = {"f32": 4, "f16": 2, "e4m3": 1, "e4m3zp": 2}[w.scale]
            nbytes = n_tok * w.num_kv_heads * 2 * (2 * w.d + w.bits * w.d // 8 + (w.d // w.block) * sb)
            cpu = timed_cpu_baseline(oracle_write_sample(w, n_tok), lambda per: nbytes / per / 1e9, "GB/s",
                                     f"oracle write of {n_tok} tokens x {w.num_kv_heads} kv heads, K and V")
        print(json.dumps({
            "metric": "write-path GB/s (fp16 in + packed out)", "value": gbs, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"prefill: {w.seq_len} tokens x Hkv{w.num_kv_heads} x d{w.d}, K+V fp16, "
                                   f"sign flip + FWHT, m{w.block} {w.scale} scales, {w.bits}-bit codes",
                       "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / world / peaks["hbm"], "traffic": None,
                         "kernel": "write_chunk_kernel", "peak_source": peaks["src"]},
            "tokens_per_s": whole_job_rate(w.seq_len, world, ms),
            "gpu_launches": args.steps, "clocks": clk.summary(),
            **({"cpu_baseline": cpu} if cpu else {})}))


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


def run_prefill_attn(args, world, rank, dev):
    import dataclasses

    import torch
    w = workload(args.workload)
    if args.tokens:   # a shorter context (profiling): the chunk is at most a quarter of it
        w = dataclasses.replace(w, seq_len=args.tokens, chunk=min(w.chunk, max(1, args.tokens // 4)))
    st = PrefillAttnWorkload(dev, w)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    if args.profile:
        for _ in range(args.steps):
            st.step()
        torch.cuda.synchronize()
        print(json.dumps({"profile": w.name, "status": int(st.status.item())}))
        return
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index or 0) as clk:
        a.record(stream)
        for _ in range(args.steps):
            st.step()
        b.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
    assert int(st.status.item()) == 0
    pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(pk.get("bf16_tflops", 1900.0))
    tflops = st.flops() / (ms * 1e-3) / 1e12
    # d = 128 with 3-bit symmetric codes runs the tile kernel (one launch);
    # the other formats the decode kernel's prefill variant and the combine
    tile = w.d == 128 and w.bits == 3 and w.scale != "e4m3zp"
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = timed_cpu_baseline(oracle_prefill_sample(w, 1), lambda per: 1.0 / per, "tokens/s",
                                     f"oracle prefill attention of the chunk's last query (all {w.num_q_heads} "
                                     f"heads) over the {w.seq_len}-token cache (cache written once, untimed)")
        print(json.dumps({
            "metric": "prefill-attention query tokens/s (one layer, all heads)",
            "value": whole_job_rate(w.chunk, world, ms), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": f"f16 mma / f32 accumulate ({w.bits}-bit packed cache)",
            "data": "synthetic",
            "config": {"workload": f"{w.name}: chunk of {w.chunk} queries at positions {w.seq_len - w.chunk}.."
                                   f"{w.seq_len - 1} of a {w.seq_len}-token cache, Hkv{w.num_kv_heads} "
                                   f"Hq{w.num_q_heads} d{w.d} m{w.block} {w.scale} scales, {w.bits}-bit codes, contiguous "
                                   f"P{w.page_size}, causal", "l2": "cache 3.4 MB per kv head"},
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "traffic": None,
                         "kernel": "kvq3_prefill_attn (" + ("prefill_tile_kernel" if tile else
                                   "decode_split_kernel<..., prefill> + decode_combine_kernel") + ")",
                         "peak_source": "measured bf16 (fp16 mma has the same nominal rate)"
                         if pk else "fallback"},
            "gpu_launches": (1 if tile else 2) * args.steps, "clocks": clk.summary(),
            **({"cpu_baseline": cpu} if cpu else {})}))


def workload_desc(w: I.Workload) -> str:
    lens = f"N={w.seq_len}" if not w.len_range else f"N~U[{w.len_range[0]},{w.len_range[1]}]"
    return (f"{w.name}: B{w.batch} Hkv{w.num_kv_heads} Hq{w.num_q_heads} d{w.d} {lens} m{w.block} "
            f"{w.scale} scales, {w.bits}-bit codes, {'paged' if w.paged else 'contiguous'} P{w.page_size}, "
            f"rot flags {w.rot_flags}; step = kvq3_write(1 token/seq) + kvq3_decode_attn")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.workloads()))
    ap.add_argument("--impl", default="kvq3", choices=["kvq3", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (smaller profiling cases)")
    ap.add_argument("--tokens", type=int, default=0, help="override the prefill token count")
    ap.add_argument("--profile", action="store_true", help="plain steps only, for ncu captures")
    ap.add_argument("--bits", type=int, default=0, choices=[0, 2, 3, 4],
                    help="code width of the cache (0: the workload's own, 3)")
    ap.add_argument("--scale", default="", choices=["", "f32", "f16", "e4m3", "e4m3zp"],
                    help="scale format (e4m3zp: the asymmetric variant, E4M3 scale and zero point)")
    args = ap.parse_args()
    global BITS_OVERRIDE, SCALE_OVERRIDE
    BITS_OVERRIDE = args.bits
    SCALE_OVERRIDE = args.scale
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload(args.workload)
    if w.chunk > 0:
        run_prefill_attn(args, world, rank, dev)
        return
    if not w.decode:
        run_prefill(args, world, rank, dev)
        return
    st = GpuWorkload(args.workload, dev, rank, args.batch)
    w = st.w
    stream = torch.cuda.current_stream()
    clk = ClockSampler(local)
    if not args.profile:
        clk.__enter__()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0, f"device status {int(st.status.item())}"
    if args.profile:
        # plain steps only (kernel order per step: write, decode split, decode combine)
        for _ in range(args.steps):
            st.step()
        torch.cuda.synchronize()
        print(json.dumps({"profile": w.name, "batch": w.batch, "status": int(st.status.item())}))
        return

    # ---- device-timed steps (inputs resident; cache > L2 so every step streams it from HBM)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        st.write(st.k_new, st.v_new, st.seq_new, st.pos_new)
        ev[i][1].record(stream)
        st.decode()
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_step = total_ms / args.steps
    dec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    wr_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)

    # ---- end to end through host buffers (pinned), copies inside the timed region:
    # the step's inputs (new k, v, the queries, positions, sequence ids) sit in
    # one pinned host buffer and go over in one copy; the output comes back
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

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
    clk.__exit__(None, None, None)
    assert int(st.status.item()) == 0

    ab = algorithmic_bytes(w, st.lens)
    peaks = load_peaks()
    dec_gbs = ab["decode"] / (dec_ms * 1e-3) / 1e9
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(w, st.lens)
        line = {
            "metric": "decode tokens/s (one layer, all heads)", "value": whole_job_rate(w.batch, world, ms_step),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": f"f16 mma / f32 accumulate ({w.bits}-bit packed cache)", "data": "synthetic",
            "config": {"workload": workload_desc(w), "l2": "inputs larger than L2 (packed cache "
                       f"{ab['decode'] / 1e6:.0f} MB per step)", "parallelism": f"replicas x{world} (dp over sequences)"},
            "decode": {"ms": dec_ms, "hbm_gbs": dec_gbs, "frac_of_peak": dec_gbs / peaks["hbm"],
                       "bytes": ab["decode"]},
            "write": {"ms": wr_ms, "gbs": ab["write"] / (wr_ms * 1e-3) / 1e9, "bytes": ab["write"]},
            "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": dec_gbs / peaks["hbm"], "traffic": recorded_traffic(args.workload, w.bits),
                         "kernel": "kvq3_decode_attn (decode_split_kernel + decode_combine_kernel)",
                         "peak_source": peaks["src"]},
            "e2e": {"value": whole_job_rate(w.batch, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": 3 * args.steps,
            "clocks": clk.summary(),
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

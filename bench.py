"""Benchmark of the paged-KV attention hot path on GB300.

Headline: a serving decode step on the Qwen2.5-7B-shaped workload (batch 32,
8,192-token contexts, Hq=28, Hkv=4, D=128, 16-token pages in a 16,384-page
pool): the eager writeback of each sequence's newest K/V row
(``kv_write_paged``) followed by split-K decode (``attn_decode_paged``).
``value`` is decode KV bytes read per second (sum of seq_len * Hkv * D * 2 * 2
bytes per step / step time).  Extra measurements on the same line: the
varlen causal prefill (TFLOP/s over visible pairs) and the mixed
prefill+decode step, each against its roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: every rank runs an independent replica on its own batch (the path
has no exchange step), so scaling is weak and ``value`` sums all ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402
from paged_kv_decode_17_gb300 import roofline  # noqa: E402

METRIC = "paged decode KV-read GB/s (% of HBM peak); varlen prefill TFLOPS (% peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def profile_traffic(name: str, source_files):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source (sha256 of the listed files); else None."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in source_files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    want = h.hexdigest()
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "kernel_source_sha256")):
                k, v = line.strip().split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != want:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (ctypes) every
    few ms while running; read-only."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, interval_s=0.002):
        self.interval = interval_s
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            got = False
            try:
                props = torch.cuda.get_device_properties(torch.cuda.current_device())
                bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
                got = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            except Exception:
                got = False
            if not got and nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                return
            self.nv, self.h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            pass

    def _run(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        getr = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                rs = int(r.value) if getr(self.h, ctypes.byref(r)) == 0 else 0
                self.samples.append((int(c.value), rs))
            time.sleep(self.interval)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": "NVML unavailable" if not self.ok else "no samples"}
        mhz = [s[0] for s in self.samples]
        reasons = set()
        for _, rs in self.samples:
            for bit, name in self.REASONS.items():
                if rs & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, pg


def barrier(pg):
    if pg is not None:
        if torch.cuda.is_available():
            pg.barrier(device_ids=[torch.cuda.current_device()])
        else:
            pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle baseline
def _compact_numpy(case, seqs):
    """Pages of `seqs` copied to host numpy, table renumbered (input movement only)."""
    import numpy as np
    ps = case.page_size
    idx, tables, lens, cu, rows = [], [], [], [0], []
    cu_full = case.cu_seqlens_q.cpu().tolist()
    nxt = 0
    maxp = 1
    for b in seqs:
        L = case.seq_lens_host[b]
        n = -(-L // ps)
        idx.append(case.block_table[b, :n].long())
        tables.append(list(range(nxt, nxt + n)))
        nxt += n
        maxp = max(maxp, n)
        lens.append(L)
        rows.extend(range(cu_full[b], cu_full[b + 1]))
        cu.append(cu[-1] + cu_full[b + 1] - cu_full[b])
    ii = torch.cat(idx)

    def bits(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    bt = np.full((len(seqs), maxp), -1, dtype=np.int64)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    rr = torch.tensor(rows, dtype=torch.long, device=case.q.device)
    return dict(q_bits=bits(case.q[rr]), k_pool_bits=bits(case.k_pool[ii]), v_pool_bits=bits(case.v_pool[ii]),
                block_table=bt, seq_lens=lens, cu_seqlens_q=np.array(cu), num_q_heads=case.num_q_heads,
                num_kv_heads=case.num_kv_heads, page_size=ps, scale=case.softmax_scale)


def oracle_decode_rate(case, time_limit_s=12.0, max_seqs=None):
    """Time the fp64 CPU oracle on whole sequences of `case` until `time_limit_s`
    of CPU work; returns (GB/s of KV, seconds, sequences done)."""
    import oracle  # test infrastructure: only the CPU-baseline legs use it
    done, t_total, nbytes = 0, 0.0, 0
    B = case.batch
    for b in range(B if max_seqs is None else min(B, max_seqs)):
        args = _compact_numpy(case, [b])
        t0 = time.perf_counter()
        oracle.paged_attention(**args)
        t_total += time.perf_counter() - t0
        nbytes += roofline.decode_kv_bytes([case.seq_lens_host[b]], case.num_kv_heads, case.head_dim)
        done += 1
        if t_total >= time_limit_s:
            break
    return nbytes / t_total / 1e9, t_total, done


def cpu_baseline_subprocess(time_limit_s=12.0):
    """Run the oracle in a fresh single-threaded process (BLAS pinned to one
    thread, so `cores` is exact)."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ("import sys, json; sys.path.insert(0, %r); import bench, workloads; "
            "c = workloads.qwen7b_decode(device='cpu'); "
            "r = bench.oracle_decode_rate(c, %r); print('CPU_BASELINE', json.dumps(r))" % (ROOT, time_limit_s))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        for line in out.stdout.splitlines():
            if line.startswith("CPU_BASELINE"):
                gbs, secs, n = json.loads(line.split(" ", 1)[1])
                return {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                        "sample": "%d of 32 sequences (x 28 heads x 8192 tokens) of the qwen7b_decode batch, "
                                  "fp64 numpy oracle, %.1f s" % (n, secs)}
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": "failed: %s" % (out.stderr.strip().splitlines()[-1:] or ["?"])[0]}
    except Exception as e:  # pragma: no cover
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "failed: %s" % e}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, rank, world, pg):
    """The oracle as it stands, on the host cores, on the same workload and
    metric; each step decodes a bounded sample (one sequence of the batch)."""
    if rank != 0:
        return
    case = workloads.qwen7b_decode(device="cpu")
    import oracle
    times = []
    nbytes = 0
    for i in range(args.warmup + args.steps):
        b = i % case.batch
        a = _compact_numpy(case, [b])
        t0 = time.perf_counter()
        oracle.paged_attention(**a)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            nbytes += roofline.decode_kv_bytes([case.seq_lens_host[b]], case.num_kv_heads, case.head_dim)
    tot = sum(times)
    val = nbytes / tot / 1e9
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "qwen7b_decode (one sequence per step: 28 heads x 8192 tokens)",
                       "batch": 32, "ctx": 8192, "Hq": 28, "Hkv": 4, "head_dim": 128, "page_size": 16},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "one whole sequence of the batch per step"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
def _events(stream, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def measure_decode(pa, case, steps, warmup, pg):
    """Decode step = split-K decode with each sequence's newest K/V row written
    back by the same kernel (attn_decode_paged_append: decode + merge
    kernels).  The K timed steps run back to back (each launch a programmatic
    dependent of the one before); a second pass with events around each call
    gives the per-call time for the roofline."""
    dev = case.q.device
    stream = torch.cuda.current_stream()
    B, Hq, D = case.q.shape
    ws = pa.Workspace(pa.decode_workspace_bytes(B, Hq, case.num_kv_heads, D), dev)
    out = torch.empty_like(case.q)

    def step():
        pa.attn_decode_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                             case.softmax_scale, max_seq_len=case.max_seq_len, out=out, workspace=ws,
                             k_new=case.k_new, v_new=case.v_new)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    sampler = ClockSampler()
    with sampler:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    ev = _events(stream, 2 * steps)
    for i in range(steps):
        ev[2 * i].record(stream)
        step()
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    dec_ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)]
    return total_ms, dec_ms, sampler.summary(), 2 * steps


def measure_decode_e2e(pa, case, steps, warmup):
    """Same step through the public API with the step's inputs and result in
    pinned host memory: the kernels read q, the new K/V rows and seq_lens,
    and write the attention output, in place over the CPU-GPU link
    (NVLink-C2C on GB300), as a serving loop on this machine would pass them;
    no copy-engine copies."""
    dev = case.q.device
    B, Hq, D = case.q.shape
    ws = pa.Workspace(pa.decode_workspace_bytes(B, Hq, case.num_kv_heads, D), dev)
    h_q, h_k, h_v, h_len = (t.cpu().pin_memory() for t in (case.q, case.k_new, case.v_new, case.seq_lens))
    h_out = torch.empty(case.q.shape, dtype=case.q.dtype).pin_memory()
    stream = torch.cuda.current_stream()

    def step():
        pa.attn_decode_paged(h_q, case.k_pool, case.v_pool, case.block_table, h_len, case.softmax_scale,
                             max_seq_len=case.max_seq_len, out=h_out, workspace=ws, k_new=h_k, v_new=h_v)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_len))
    return ms, h2d, h_out.numel() * h_out.element_size()


def _flush_l2(buf):
    """Evict L2 between timed iterations: write the first half of `buf` (256 MiB, twice
    the L2), then read the second half.  The read evicts the dirty lines the write
    leaves behind, so their write-back to HBM happens here and not inside the next
    timed kernel; the kernel's own inputs are not in L2 either way."""
    h = buf.numel() // 2
    buf[:h].zero_()
    buf[h:].view(torch.int32).sum()


class _prefill_path:
    """Select how attn_prefill_varlen_causal runs a call with prefill entries (the
    library reads PAGEDATTN_PREFILL_PATH at every call): "fused" = one persistent
    kernel for the decode rows and the prefill tiles, then the merge of split decode
    rows; "separate" = split-K decode + merge, plan and prefill kernels."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        self.old = os.environ.get("PAGEDATTN_PREFILL_PATH")
        os.environ["PAGEDATTN_PREFILL_PATH"] = self.path
        return self

    def __exit__(self, *a):
        if self.old is None:
            os.environ.pop("PAGEDATTN_PREFILL_PATH", None)
        else:
            os.environ["PAGEDATTN_PREFILL_PATH"] = self.old


def measure_prefill(pa, steps, warmup, peaks):
    """Varlen causal prefill step: writeback of every new row, then prefill.
    16 sequences of 512..4096 tokens, Hq=28, Hkv=4, D=128.  L2 is flushed
    (256 MiB write, then 256 MiB read) between iterations, outside the timed events."""
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workloads.varlen_prefill(device=dev)
    stream = torch.cuda.current_stream()
    B = case.batch
    ws = pa.Workspace(pa.prefill_workspace_bytes(B, case.total_q, case.num_q_heads, case.num_kv_heads,
                                                 case.head_dim), dev)
    out = torch.empty_like(case.q)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def write():
        pa.kv_write_paged(case.k_pool, case.v_pool, case.k_new, case.v_new, case.cu_seqlens_q, case.seq_lens,
                          case.block_table)

    def attn():
        pa.attn_prefill_varlen_causal(case.q, case.k_pool, case.v_pool, case.block_table, case.cu_seqlens_q,
                                      case.seq_lens, case.softmax_scale, max_q_len=case.max_q_len,
                                      max_seq_len=case.max_seq_len, out=out, workspace=ws)

    def run(path):
        with _prefill_path(path):
            for _ in range(warmup):
                write()
                attn()
            torch.cuda.synchronize()
            w_ms, a_ms = [], []
            for _ in range(steps):
                _flush_l2(flush)
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record(stream)
                write()
                e[1].record(stream)
                attn()
                e[2].record(stream)
                torch.cuda.synchronize()
                w_ms.append(e[0].elapsed_time(e[1]))
                a_ms.append(e[1].elapsed_time(e[2]))
        return statistics.median(w_ms), statistics.median(a_ms)

    w, a = run("fused")
    _, a_sep = run("separate")
    flops = roofline.prefill_flops(case.q_lens_host, case.seq_lens_host, case.num_q_heads, case.head_dim)
    wbytes = roofline.kv_write_bytes(case.total_q, case.num_kv_heads, case.head_dim)
    tflops = flops / (a * 1e-3) / 1e12
    res = {"workload": "varlen_prefill: 16 sequences, lengths uniform 512..4096 (seeded), no prior tokens, "
                       "Hq=28, Hkv=4, head_dim 128, 16-token pages; step = writeback of all new rows + prefill",
           "tokens": case.total_q, "flops_visible_pairs": flops, "prefill_ms": a, "tflops": tflops,
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": tflops / peaks["bf16_tflops"], "peak_source": peaks["source"] + " (burst)"},
           "tokens_per_s": case.total_q / ((a + w) * 1e-3),
           "kv_write": {"ms": w, "bytes": wbytes, "gbs": wbytes / (w * 1e-3) / 1e9,
                        "frac_hbm": wbytes / (w * 1e-3) / 1e9 / peaks["hbm_gbs"]},
           "l2": "flushed (256 MiB write, then 256 MiB read) between iterations", "steps": steps,
           "path": "fused: one persistent kernel (decode rows, none here, then prefill tiles) + merge",
           "launches_per_step": 3,  # writeback, fused kernel, merge
           "separate_kernels": {"prefill_ms": a_sep, "tflops": flops / (a_sep * 1e-3) / 1e12,
                                "launches_per_step": 5}}  # writeback, decode + merge, plan, prefill
    del case, flush
    torch.cuda.empty_cache()
    return res


def measure_fp8_decode(pa, steps, warmup, peaks):
    """Decode over an FP8 (e4m3) KV cache on the qwen7b_decode shape (batch 32
    x 8192, Hq=28, Hkv=4, D=128): 256 MiB of K/V codes per step (half the bf16
    bytes), random finite codes, per-KV-head scales.  L2 is flushed between
    iterations (the codes are only twice the size of L2)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workloads.qwen7b_decode(device=dev)
    P, Hkv, ps, D = case.k_pool.shape
    g = torch.Generator(device=dev).manual_seed(11)
    kc = torch.randint(0, 256, (P, Hkv, ps, D), dtype=torch.uint8, device=dev, generator=g)
    vc = torch.randint(0, 256, (P, Hkv, D, ps), dtype=torch.uint8, device=dev, generator=g)
    kc[(kc & 0x7F) == 0x7F] = 0  # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0
    case.k_pool = case.v_pool = None
    torch.cuda.empty_cache()
    ks = torch.full((Hkv,), 0.01, dtype=torch.float32, device=dev)
    vs = torch.full((Hkv,), 0.01, dtype=torch.float32, device=dev)
    B, Hq, _ = case.q.shape
    ws = pa.Workspace(pa.decode_workspace_bytes(B, Hq, Hkv, D), dev)
    out = torch.empty_like(case.q)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def attn():
        pa.attn_decode_paged_fp8(case.q, kc, vc, ks, vs, case.block_table, case.seq_lens, case.softmax_scale,
                                 max_seq_len=case.max_seq_len, out=out, workspace=ws)

    for _ in range(warmup):
        attn()
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        _flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        attn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    t = statistics.median(ms)
    kv = roofline.decode_kv_bytes(case.seq_lens_host, Hkv, D, elem_bytes=1)
    gbs = kv / (t * 1e-3) / 1e9
    res = {"workload": "qwen7b_decode on an FP8 (e4m3) cache: batch 32 x 8192-token contexts, Hq=28, Hkv=4, "
                       "head_dim 128, 16-token pages, per-KV-head scales",
           "ms": t, "kv_bytes": kv,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"]},
           "tokens_per_s": B / (t * 1e-3), "l2": "flushed (256 MiB write, then 256 MiB read) between iterations", "steps": steps,
           "launches_per_step": 2}  # decode + merge
    del case, kc, vc, flush
    torch.cuda.empty_cache()
    return res


def measure_rope_writeback(pa, steps, warmup, peaks):
    """Fused Q/K RMS norm + rotary embedding + KV writeback of the
    varlen_prefill rows (34k tokens: K and V into their pages, the queries
    rotated in place), L2 flushed between iterations; HBM-bound."""
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workloads.varlen_prefill(device=dev)
    stream = torch.cuda.current_stream()
    g = torch.Generator().manual_seed(7)
    kw = (0.5 + torch.rand(case.head_dim, generator=g)).to(torch.bfloat16).to(dev)
    qw = (0.5 + torch.rand(case.head_dim, generator=g)).to(torch.bfloat16).to(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def write():
        pa.kv_write_paged_rope(case.k_pool, case.v_pool, case.k_new, case.v_new, case.cu_seqlens_q, case.seq_lens,
                               case.block_table, 1e6, q=case.q, q_norm_weight=qw, k_norm_weight=kw)

    for _ in range(warmup):
        write()
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        _flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        write()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    t = statistics.median(ms)
    nbytes = roofline.kv_write_rope_bytes(case.total_q, case.num_kv_heads, case.num_q_heads, case.head_dim)
    gbs = nbytes / (t * 1e-3) / 1e9
    res = {"workload": "varlen_prefill rows (16 sequences, 512..4096 tokens; Hq=28, Hkv=4, head_dim 128): K/V "
                       "RMS norm + rotary embedding (base 1e6) + writeback, queries rotated in place",
           "tokens": case.total_q, "ms": t, "bytes": nbytes,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"]},
           "l2": "flushed (256 MiB write, then 256 MiB read) between iterations", "steps": steps, "launches_per_step": 1}
    del case, flush
    torch.cuda.empty_cache()
    return res


def measure_mixed(pa, steps, warmup, peaks, small=False):
    """Mixed serving step in one call: 4 prefill chunks of 2048 tokens after
    0..8192 cached tokens + 60 decodes (1k..64k context) + one 131,072-token
    decode; Hq=32, Hkv=8, D=128.  Inputs (about 9 GB of KV) exceed L2."""
    dev = torch.device("cuda", torch.cuda.current_device())
    case = (workloads.mixed_step_small if small else workloads.mixed_step)(device=dev)
    stream = torch.cuda.current_stream()
    ws = pa.Workspace(pa.prefill_workspace_bytes(case.batch, case.total_q, case.num_q_heads, case.num_kv_heads,
                                                 case.head_dim), dev)
    out = torch.empty_like(case.q)

    def attn():
        pa.attn_prefill_varlen_causal(case.q, case.k_pool, case.v_pool, case.block_table, case.cu_seqlens_q,
                                      case.seq_lens, case.softmax_scale, max_q_len=case.max_q_len,
                                      max_seq_len=case.max_seq_len, out=out, workspace=ws)

    def run(path):
        with _prefill_path(path):
            for _ in range(warmup):
                attn()
            torch.cuda.synchronize()
            ms = []
            for _ in range(steps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                attn()
                e1.record(stream)
                torch.cuda.synchronize()
                ms.append(e0.elapsed_time(e1))
        return statistics.median(ms)

    t = run("fused")
    t_sep = run("separate")
    # entries with up to 8 query rows run on the split-K decode path (HBM-bound), longer ones on the prefill kernel
    dec = [(L, q) for L, q in zip(case.seq_lens_host, case.q_lens_host) if q <= 8]
    pre_q = [q for q in case.q_lens_host if q > 8]
    pre_L = [L for L, q in zip(case.seq_lens_host, case.q_lens_host) if q > 8]
    dbytes = roofline.decode_kv_bytes([L for L, _ in dec], case.num_kv_heads, case.head_dim)
    flops = roofline.prefill_flops(pre_q, pre_L, case.num_q_heads, case.head_dim)
    t_bytes = dbytes / (peaks["hbm_gbs"] * 1e9)
    t_flops = flops / (peaks["bf16_tflops"] * 1e12)
    res = {"workload": ("mixed_step_small: 4 prefill chunks x 2048 tokens (0..8192 prior) + 60 decodes (1k..4k) "
                        "+ 1 decode at 16384" if small else
                        "mixed_step: 4 prefill chunks x 2048 tokens (0..8192 prior) + 60 decodes (1k..64k) + "
                        "1 decode at 131072") + "; Hq=32, Hkv=8, head_dim 128, 16-token pages",
           "step_ms": t, "decode_kv_bytes": dbytes, "prefill_flops": flops,
           "t_roofline_ms": 1e3 * max(t_bytes, t_flops), "t_serial_roofline_ms": 1e3 * (t_bytes + t_flops),
           "frac_of_roofline": max(t_bytes, t_flops) / (t * 1e-3),
           "tokens_per_s": case.total_q / (t * 1e-3), "steps": steps,
           "path": "fused: one persistent kernel (split-K decode rows, then prefill tiles) + merge",
           "launches_per_step": 2,
           "separate_kernels": {"step_ms": t_sep, "frac_of_roofline": max(t_bytes, t_flops) / (t_sep * 1e-3),
                                "launches_per_step": 4},  # decode + merge, plan, prefill
           "l2": "inputs larger than L2 (about 9 GB of KV)"}
    del case
    torch.cuda.empty_cache()
    return res


def measure_ragged_decode(pa, steps, warmup, peaks, small=False):
    """Ragged Llama-3-8B-shaped decode step: batch 64, contexts uniform on
    [1, 32768] (seeded), Hq=32, Hkv=8, D=128, 16-token pages scattered over a
    131,072-page pool; the same call as the headline step (split-K decode with
    each sequence's newest row written back in the kernel).  About 4.3 GB of
    KV per step, far above L2, so no flush; K calls back to back, then K calls
    with an event on each side."""
    dev = torch.device("cuda", torch.cuda.current_device())
    case = (workloads.llama8b_ragged_small if small else workloads.llama8b_ragged_decode)(device=dev)
    stream = torch.cuda.current_stream()
    B, Hq, D = case.q.shape
    ws = pa.Workspace(pa.decode_workspace_bytes(B, Hq, case.num_kv_heads, D), dev)
    out = torch.empty_like(case.q)

    def step():
        pa.attn_decode_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                             case.softmax_scale, max_seq_len=case.max_seq_len, out=out, workspace=ws,
                             k_new=case.k_new, v_new=case.v_new)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / steps
    ev = _events(stream, 2 * steps)
    for i in range(steps):
        ev[2 * i].record(stream)
        step()
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    t_iso = statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps))
    kv = roofline.decode_kv_bytes(case.seq_lens_host, case.num_kv_heads, D)
    gbs = kv / (t * 1e-3) / 1e9
    res = {"workload": ("llama8b_ragged_small: the first 16 sequences of the batch-64 draw, pool = pages needed"
                        if small else "llama8b_ragged_decode: batch 64, contexts uniform on [1, 32768] (seeded), "
                        "Hq=32, Hkv=8, head_dim 128, 16-token pages in a 131072-page pool") +
                       "; step = split-K decode with the newest row of each sequence written back in the same "
                       "kernel (attn_decode_paged_append)",
           "tokens_in_context": int(sum(case.seq_lens_host)), "ms": t, "ms_isolated": t_iso, "kv_bytes": kv,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "frac_isolated": kv / (t_iso * 1e-3) / 1e9 / peaks["hbm_gbs"],
                        "peak_source": peaks["source"]},
           "tokens_per_s": B / (t * 1e-3), "steps": steps, "launches_per_step": 2,
           "l2": "inputs larger than L2 (%.2f GB of KV), no flush" % (kv / 1e9)}
    del case
    torch.cuda.empty_cache()
    return res


def measure_multiquery(pa, steps, warmup, peaks, q_len=4):
    """Multi-query decode (speculative-decode verification): the qwen7b_decode
    shape with q_len query rows per sequence, causal inside the block; the
    KV (512 MiB) exceeds L2, so no flush is needed."""
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workloads.qwen7b_multiquery(device=dev, q_len=q_len)
    stream = torch.cuda.current_stream()
    B, Hq, D = case.batch, case.num_q_heads, case.head_dim
    ws = pa.Workspace(pa.decode_multiquery_workspace_bytes(B, q_len, Hq, case.num_kv_heads, D), dev)
    out = torch.empty_like(case.q)

    def attn():
        pa.attn_decode_multiquery_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.cu_seqlens_q,
                                        case.seq_lens, case.softmax_scale, max_q_len=q_len,
                                        max_seq_len=case.max_seq_len, out=out, workspace=ws)

    for _ in range(warmup):
        attn()
    torch.cuda.synchronize()
    # K calls back to back, as the decode step: average duration over the timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        attn()
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / steps
    kv = roofline.decode_kv_bytes(case.seq_lens_host, case.num_kv_heads, D)
    gbs = kv / (t * 1e-3) / 1e9
    res = {"workload": "qwen7b_multiquery: batch 32 x 8192-token contexts, %d query rows per sequence (causal "
                       "inside the block), Hq=28, Hkv=4, head_dim 128, 16-token pages" % q_len,
           "q_len": q_len, "ms": t, "kv_bytes": kv,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"]},
           "tokens_per_s": B * q_len / (t * 1e-3), "steps": steps, "launches_per_step": 2,
           "l2": "inputs larger than L2 (512 MiB of KV), no flush"}
    del case
    torch.cuda.empty_cache()
    return res


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-only", action="store_true", help="skip the prefill and mixed-step measurements")
    ap.add_argument("--small", action="store_true",
                    help="with --only mixed / llama8b_ragged: the profiling-size workload (about 1 GB of KV)")
    ap.add_argument("--only", choices=["prefill", "mixed", "multiquery", "rope_writeback", "fp8_decode",
                                       "llama8b_ragged"],
                    default=None,
                    help="run just this extra measurement (for profiling); prints its object only")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    rank, world, pg = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world, pg)
        return 0

    import paged_kv_decode_17_gb300 as pa
    pa.load_library(build_if_missing=True)
    peaks = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    if args.only is not None:
        fn = {"prefill": measure_prefill, "mixed": measure_mixed, "multiquery": measure_multiquery,
              "rope_writeback": measure_rope_writeback, "fp8_decode": measure_fp8_decode,
              "llama8b_ragged": measure_ragged_decode}[args.only]
        kw = {"small": True} if args.small and args.only in ("mixed", "llama8b_ragged") else {}
        res = fn(pa, args.steps, args.warmup, peaks, **kw)
        if rank == 0:
            print(json.dumps({"only": args.only, args.only: res}), flush=True)
        return 0

    case = workloads.qwen7b_decode(device=dev, seed=1 + rank)
    kv_bytes = roofline.decode_kv_bytes(case.seq_lens_host, case.num_kv_heads, case.head_dim)
    total_ms, dec_ms, clocks, launches = measure_decode(pa, case, args.steps, args.warmup, pg)
    total_ms = max_over_ranks(pg, total_ms)
    ms_per_step = total_ms / args.steps
    all_bytes = sum_over_ranks(pg, kv_bytes * args.steps)
    value = all_bytes / (total_ms * 1e-3) / 1e9

    # the step is this one call (decode + merge kernels): its average duration over the timed
    # region is the step time; the same call with an event on each side (no overlap with the
    # neighbouring calls) is reported beside it
    dec_avg = statistics.mean(dec_ms)
    launch_ms = ms_per_step
    achieved = kv_bytes / (launch_ms * 1e-3) / 1e9
    traffic = profile_traffic("attn_decode_qwen7b_ncu.md", ["paged_kv_decode_17_gb300/csrc/decode_dev.cuh",
                                                            "paged_kv_decode_17_gb300/csrc/pa_common.cuh"])
    e2e_ms, h2d, d2h = measure_decode_e2e(pa, case, args.steps, args.warmup)
    e2e_ms = max_over_ranks(pg, e2e_ms)
    e2e_val = sum_over_ranks(pg, kv_bytes) / (e2e_ms * 1e-3) / 1e9
    del case
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "qwen7b_decode: batch 32 x 8192-token contexts, Hq=28, Hkv=4, head_dim 128, "
                               "16-token pages, 16384-page pool (seeded permutation); step = split-K decode with "
                               "the KV writeback of each sequence's newest row in the same kernel "
                               "(attn_decode_paged_append)",
                   "batch": 32, "ctx": 8192, "Hq": 28, "Hkv": 4, "head_dim": 128, "page_size": 16,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2: 512 MiB of KV read per step vs 129 MB L2, no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "attn_decode_paged_append (decode_kernel<128> + merge_kernel<128>)",
                     "algorithmic_bytes_per_launch": kv_bytes, "launch_ms": launch_ms,
                     "launch_ms_isolated": dec_avg,
                     "peak_source": peaks["source"]},
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "transfer": "step inputs and output in pinned host memory, read and written in place by the "
                            "kernels over NVLink-C2C (no copy-engine copies)"},
        "gpu_launches": launches * world,
        "clocks": clocks,
    }
    if not args.decode_only:
        psteps = max(3, min(args.steps, 20))
        line["llama8b_ragged"] = measure_ragged_decode(pa, psteps, 3, peaks)
        line["prefill"] = measure_prefill(pa, psteps, 3, peaks)
        line["mixed"] = measure_mixed(pa, psteps, 3, peaks)
        line["multiquery"] = measure_multiquery(pa, psteps, 3, peaks)
        line["rope_writeback"] = measure_rope_writeback(pa, psteps, 3, peaks)
        line["fp8_decode"] = measure_fp8_decode(pa, psteps, 3, peaks)
        line["gpu_launches"] += world * psteps * (2 * 2 + (3 + 5) + (2 + 4) + 2 + 1 + 2)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess()
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(pg)
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the fused FP8 DSA indexer + exact top-2048 on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

One step = one complete operator call (plan, sampled thresholds, fused
tcgen05 scoring + candidate filter, exact selection of the candidates,
repair) over the causal-prefill workload Q=4096 query rows x N=131072 keys,
K=2048 (the "128K" chunk of the indexer study), inputs resident in HBM.
--config 4 runs the paged decode batch through the paged entry point.  The metric is
scored row-keys per second (sum over rows of the valid range length); the
effective FP8 rate is 2*64*128 FLOP per row-key ("Fusing Indexer Scoring and
Exact Top-k for DeepSeek-V3.2", section 5.1 equation).

L2 is flushed (a 512 MiB write) before every timed step, outside the timed
events.  With --gpus N under torchrun each rank runs an independent replica
(no collective on the data path; weak scaling); rank 0 prints one JSON line.
--impl reference times the CPU oracle (exact FP64 scores, full sort) on a
bounded sample of rows of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADS, DIM = 64, 128
FLOP_PER_ROW_KEY = 2 * HEADS * DIM          # 16384
BYTES_PER_KEY = DIM + 4                     # FP8 vector + fp32 scale = 132
FP8_OVER_BF16 = 2.0                         # nominal dense ratio (4.5 / 2.25 PFLOP/s)
CORE_OPS_PER_ROW_KEY = 2 * HEADS + 4        # ReLU + FMA per head, ~4 per key (scale, mask, compare)
CPU_BASELINE_SECONDS = 10.0                 # CPU work of the oracle's timed sample
MAX_ORACLE_ROWS = 2048                      # cap on that sample (rows)
METRIC = "fused indexer+top-2048 row-keys/s and FP8 TFLOP/s (% of GB300 FP8 roofline), 1 GPU"


# ------------------------------------------------------------- accounting --
def algorithmic_bytes(Q: int, N: int, K: int) -> int:
    """Bytes the operator must move at least once: q codes + q scale + weights,
    every key once (codes + scale), the int32 output."""
    return Q * HEADS * DIM + Q * 4 + Q * HEADS * 4 + N * BYTES_PER_KEY + Q * K * 4


def algorithmic_bytes_of(inp) -> int:
    """algorithmic_bytes for a dense or a paged problem (paged: every
    sequence's keys once, its rows share them)."""
    if hasattr(inp, "block_table"):
        R = inp.B * inp.next_n
        keys = int(inp.seq_lens.astype(np.int64).sum())
        return R * HEADS * DIM + R * 4 + R * HEADS * 4 + keys * BYTES_PER_KEY + R * inp.K * 4
    return algorithmic_bytes(inp.Q, inp.N, inp.K)


def score_matrix_bytes(Q: int, N: int) -> int:
    """FP32 [Q, N] score matrix of the unfused pipeline (written once, read once)."""
    return Q * N * 4


def measured_traffic(config: int, rows: int, keys: int):
    """DRAM bytes per launch of the main kernel from the committed ncu record,
    or None when the workload differs or the kernel sources changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "score_kernel_traffic_c2.json")
    if config != 2 or rows or keys or not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return rec["dram_bytes_per_launch"] if h.hexdigest() == rec["sources_sha256"] else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "sm_max_mhz": float(pk.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0, "source": "fallback"}


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------- workload --
def make_workload(config: int, rows: int = 0, keys: int = 0):
    """The indexed workload, or a causal prefill chunk of `rows` x `keys`
    drawn like it (for profiling smaller cases of the same kernels)."""
    from fp8_scoring_exact_gb300 import synthetic
    if rows and keys:
        return synthetic.make_dense(rows, keys, seed=config, name=f"causal_q{rows}_n{keys}")
    return synthetic.make_config(config)


def describe(inp, config):
    if hasattr(inp, "block_table"):
        return {"workload": f"{inp.name} (paged decode: B={inp.B} sequences x next_n={inp.next_n} rows, "
                            f"64-token pages, seq_len {int(inp.seq_lens.min())}..{int(inp.seq_lens.max())}, "
                            f"K={inp.K})",
                "B": inp.B, "next_n": inp.next_n, "K": inp.K, "row_keys": inp.row_keys(),
                "config_index": config,
                "l2": "flushed by a 512 MiB write before each timed step (outside the timed events)",
                "parallelism": "replicas (one independent problem per GPU)"}
    Q, N = inp.Q, inp.N
    return {"workload": f"{inp.name} (Q={Q} rows x N={N} keys, causal, K={inp.K})", "Q": Q, "N": N,
            "K": inp.K, "row_keys": inp.row_keys(), "config_index": config,
            "l2": "flushed by a 512 MiB write before each timed step (outside the timed events)",
            "parallelism": "replicas (one independent problem per GPU)"}


# ------------------------------------------------------------ CPU oracle --
def oracle_rows(inp, n_rows, seed=123):
    rng = np.random.default_rng(seed)
    return sorted(rng.choice(inp.Q, size=min(n_rows, inp.Q), replace=False).tolist())


def oracle_subset(inp, rows):
    """The same workload restricted to `rows` (all keys kept)."""
    from fp8_scoring_exact_gb300.synthetic import DenseInputs
    r = np.asarray(rows)
    return DenseInputs(q=inp.q[r], q_scale=inp.q_scale[r], k=inp.k, k_scale=inp.k_scale, w=inp.w[r],
                       row_begin=inp.row_begin[r], row_end=inp.row_end[r], K=inp.K, name=inp.name)


def paged_subset(inp, n_seq, seed=123):
    """`n_seq` seeded sequences of a paged problem with their pages gathered
    into a compact cache (block tables renumbered), and the (b, i) rows of
    the subset."""
    from fp8_scoring_exact_gb300.synthetic import PagedInputs
    rng = np.random.default_rng(seed)
    bs = sorted(rng.choice(inp.B, size=min(n_seq, inp.B), replace=False).tolist())
    pages, tables = [], []
    for b in bs:
        n = (int(inp.seq_lens[b]) + 63) // 64
        pages.append(inp.block_table[b, :n])
    maxp = max(len(x) for x in pages)
    base = 0
    for x in pages:
        t = np.full(maxp, -1, np.int32)
        t[:len(x)] = np.arange(base, base + len(x), dtype=np.int32)
        tables.append(t)
        base += len(x)
    allp = np.concatenate(pages)
    sub = PagedInputs(q=inp.q[bs], q_scale=inp.q_scale[bs], k_cache=inp.k_cache[allp],
                      k_cache_scale=inp.k_cache_scale[allp], w=inp.w[bs], block_table=np.stack(tables),
                      seq_lens=inp.seq_lens[bs], K=inp.K, name=inp.name)
    rows = [(b, i) for b in range(len(bs)) for i in range(inp.next_n)]
    return sub, rows


def cpu_procs():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def time_oracle(inp, n_rows, procs, reps=1):
    """(row-keys/s, seconds, rows) of the oracle over a seeded row sample."""
    from oracle.indexer import OraclePool
    if hasattr(inp, "block_table"):
        sub, rows = paged_subset(inp, max(1, n_rows // inp.next_n))
        rk = int(sub.row_lengths().sum())
        kind = "paged"
    else:
        rows = oracle_rows(inp, n_rows)
        sub = oracle_subset(inp, rows)
        rk = int((sub.row_end.astype(np.int64) - sub.row_begin).sum())
        rows = range(len(rows))
        kind = "dense"
    with OraclePool(sub, procs, kind) as pool:
        t0 = time.perf_counter()
        for _ in range(reps):
            pool.topk(rows)
        dt = time.perf_counter() - t0
    return rk * reps / dt, dt, list(rows)


# ------------------------------------------------------ other workloads --
def other_configs_leg(args, binding, device, flush, skip):
    """The fused call on the indexed workloads other than the timed one (same
    protocol: warm-up, L2 flushed before every step, CUDA events; the main
    kernel timed by the library's events), so that every workload has a
    number measured in the same run."""
    import torch
    from fp8_scoring_exact_gb300 import synthetic
    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    out_rec = {}
    for cid in range(len(synthetic.CONFIG_NAMES)):
        if cid == skip:
            continue
        inp = synthetic.make_config(cid)
        host, shape, call, _ = problem(inp, binding)
        dev = [torch.from_numpy(a).to(device) for a in host]
        out = torch.empty(shape, dtype=torch.int32, device=device)
        binding.set_option("profile", 1)
        for _ in range(max(3, args.warmup)):
            call(dev, out)
        torch.cuda.synchronize(device)
        stream = torch.cuda.current_stream(device)
        ms, main = [], []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call(dev, out)
            e1.record(stream)
            main.append(binding.profiled_main_ms())
            torch.cuda.synchronize(device)
            ms.append(e0.elapsed_time(e1))
        binding.set_option("profile", 0)
        rc, counters = binding.last_device_status()
        if rc != 0:
            raise RuntimeError(f"device status {rc} on workload {cid}")
        R = inp.row_keys()
        m, k = statistics.mean(ms), statistics.mean(main)
        t_tensor = FLOP_PER_ROW_KEY * R / (fp8_peak * 1e12) * 1e3
        t_core = CORE_OPS_PER_ROW_KEY * R / (sms * 128 * peaks["sm_max_mhz"] * 1e6) * 1e3
        t_hbm = algorithmic_bytes_of(inp) / (peaks["hbm_gbs"] * 1e9) * 1e3
        rec = {"workload": inp.name, "ms_per_call": m, "row_keys_per_s": R / (m * 1e-3), "main_kernel_ms": k,
               "call_frac_of_roofline": max(t_tensor, t_core, t_hbm) / m, "failures": counters}
        if t_hbm > t_tensor:
            rec["main_kernel_frac_of_hbm"] = algorithmic_bytes_of(inp) / (k * 1e-3) / 1e9 / peaks["hbm_gbs"]
        else:
            rec["main_kernel_frac_of_fp8_peak"] = FLOP_PER_ROW_KEY * R / (k * 1e-3) / 1e12 / fp8_peak
        out_rec[synthetic.CONFIG_NAMES[cid]] = rec
        del dev, out
    return out_rec


# --------------------------------------------------------- FP8 peak probe --
def fp8_peak_probe(device, seconds=2.0, n=8192):
    """Dense e4m3 x e4m3 GEMM throughput of the library GEMM (torch._scaled_mm,
    cuBLASLt), n^3 with fp32 accumulation, bf16 output: best of 10 (burst) and
    back to back for `seconds` (sustained), with the SM clock sampled during
    the sustained loop.  Evidence for the FP8 roofline denominator, which stays
    the measured bf16 peak times the nominal fp8/bf16 ratio."""
    import torch
    try:
        a = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        one = torch.ones((), device=device, dtype=torch.float32)

        def mm():
            return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(3):
            mm()
        torch.cuda.synchronize(device)
        flop = 2.0 * n ** 3
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize(device)
            best = min(best, e0.elapsed_time(e1))
        with ClockSampler(device.index) as clk:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(1, int(seconds * 1e3 / best))
            e0.record()
            for _ in range(reps):
                mm()
            e1.record()
            torch.cuda.synchronize(device)
        sus_ms = e0.elapsed_time(e1) / reps
        return {"burst_tflops": flop / (best * 1e-3) / 1e12, "sustained_tflops": flop / (sus_ms * 1e-3) / 1e12,
                "sustained_clocks": clk.summary(), "n": n,
                "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, per-tensor scales 1: best of 10 and back to back "
                       f"for {seconds:.0f} s"}
    except Exception as e:  # the probe is evidence only; the bench line stands without it
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


# ------------------------------------------------ sparse-attention decode --
def sparse_attention_leg(args, binding, device, flush, heads=16):
    """The step downstream of the indexer (contest write-up, "DSA Sparse
    Attention"): the paged decode batch's top-2048 slots (the paged indexer's
    own result on that workload) feed the sparse-attention decode over a bf16
    latent cache (512 + 64 dims per slot) with the same page layout, `heads`
    heads per token.  The cache and queries are seeded Gaussian values drawn
    on the device.  Bytes = every valid slot's 1152-byte row once per token
    (tokens do not share their gathers) + queries + output."""
    import torch
    from fp8_scoring_exact_gb300 import synthetic
    g = torch.Generator(device=device)
    g.manual_seed(4)
    if args.sparse_slots > 0:
        # a smaller case of the same kernel for profiling: 128 tokens x 2048
        # uniformly random slots of a cache of `sparse_slots` slots
        K, T, slots = 2048, 128, args.sparse_slots
        idx = torch.randint(0, slots, (T, K), generator=g, device=device, dtype=torch.int32)
    else:
        ip = synthetic.make_config(4)
        host = [np.ascontiguousarray(a) for a in (ip.q, ip.q_scale, ip.k_cache, ip.k_cache_scale, ip.w,
                                                  ip.block_table, ip.seq_lens)]
        dev = [torch.from_numpy(a).to(device) for a in host]
        idx = binding.indexer_topk_paged(*dev, K=ip.K).reshape(-1, ip.K)
        rc, _ = binding.last_device_status()
        if rc != 0:
            raise RuntimeError(f"device status {rc} from the indexer feeding the sparse attention")
        del dev
        K, T, slots = ip.K, idx.shape[0], ip.k_cache.shape[0] * 64
    ckv = torch.randn((slots, 512), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    kpe = torch.randn((slots, 64), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    qn = torch.randn((T, heads, 512), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    qp = torch.randn((T, heads, 64), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    out = torch.empty((T, heads, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((T, heads), dtype=torch.float32, device=device)
    scale = synthetic.sm_scale_default()
    for _ in range(max(1, args.warmup)):
        binding.sparse_attention(qn, qp, ckv, kpe, idx, scale, out=out, lse=lse)
    torch.cuda.synchronize(device)
    if binding.sparse_attention_last_status() != 0:
        raise RuntimeError("sparse attention status")
    stream = torch.cuda.current_stream(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        binding.sparse_attention(qn, qp, ckv, kpe, idx, scale, out=out, lse=lse)
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    ms = statistics.mean([a.elapsed_time(b) for a, b in ev])
    valid = int((idx >= 0).sum().item())
    nbytes = valid * (512 + 64) * 2 + T * heads * 576 * 2 + T * heads * (512 * 2 + 4) + T * K * 4
    flop = valid * heads * 2 * (576 + 512)
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm = load_peaks()["hbm_gbs"]
    del ckv, kpe
    return {"ms_per_step": ms, "tokens": T, "heads": heads, "K": K, "valid_slots": valid, "cache_slots": slots,
            "bytes_per_step": nbytes, "achieved_gbs": gbs, "frac_of_hbm": gbs / hbm,
            "tflops": flop / (ms * 1e-3) / 1e12,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm},
            "note": ("dsa_sparse_attention over " + (f"uniformly random slots of a {slots}-slot cache"
                                                     if args.sparse_slots > 0 else
                                                     "the paged decode batch's own top-2048 slots (64 sequences x 2 tokens)")
                     + ", bf16 latent cache 512+64 per slot, L2 flushed before each step")}


# ------------------------------------------------------------ GPU arm -------
def _e2e(args, dev, host, out, stream, world, device, call, R, host_call=None):
    """Same metric through the public API with host buffers: every step copies
    the inputs from pinned host memory and reads the indices back.  Dense
    workloads go through the host-buffer entry point (the library stages the
    copies and overlaps them with the scoring, row chunk by row chunk); paged
    ones copy with torch and call the device entry."""
    import torch
    pinned = [torch.from_numpy(a).pin_memory() for a in host]
    out_h = torch.empty(tuple(out.shape), dtype=torch.int32).pin_memory()
    h2d = sum(a.nbytes for a in host)
    d2h = out_h.numel() * 4

    def one_step():
        if host_call is not None:
            host_call(pinned, out_h)
            return
        for d, h in zip(dev, pinned):
            d.copy_(h, non_blocking=True)
        call(dev, out)
        out_h.copy_(out, non_blocking=True)

    for i in range(args.steps + 1):
        if i == 1:
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        one_step()
    e1 = torch.cuda.Event(enable_timing=True)
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device) / args.steps
    # the host link alone: one plain 64 MiB copy each way between pinned host
    # memory and the device (torch issues a cudaMemcpyAsync), best of 5
    probe_h = torch.empty(64 << 20, dtype=torch.uint8).pin_memory()
    probe_d = torch.empty(64 << 20, dtype=torch.uint8, device=device)
    link = {}
    for name, dst, src in (("h2d_gbs", probe_d, probe_h), ("d2h_gbs", probe_h, probe_d)):
        best = float("inf")
        for _ in range(5):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            dst.copy_(src, non_blocking=True)
            c1.record(stream)
            torch.cuda.synchronize(device)
            best = min(best, c0.elapsed_time(c1))
        link[name] = (64 << 20) / (best * 1e-3) / 1e9
    return {"value": world * R / (e2e_ms * 1e-3), "unit": "row-keys/s", "pinned_copy_64mib": link,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "api": ("dsa_indexer_topk_host (host buffers; copies inside the library)" if host_call is not None
                    else "torch copies + dsa_indexer_topk_paged")}


def problem(inp, binding):
    """(host arrays, output shape, fused call, unfused call or None) of a
    dense or a paged workload."""
    K = inp.K
    if hasattr(inp, "block_table"):
        host = [np.ascontiguousarray(a) for a in (inp.q, inp.q_scale, inp.k_cache, inp.k_cache_scale, inp.w,
                                                   inp.block_table, inp.seq_lens)]
        return (host, (inp.B, inp.next_n, K),
                lambda dev, out: binding.indexer_topk_paged(*dev, K=K, out=out), None)
    host = [np.ascontiguousarray(a) for a in (inp.q, inp.q_scale, inp.k, inp.k_scale, inp.w, inp.row_begin,
                                               inp.row_end)]
    return (host, (inp.Q, K), lambda dev, out: binding.indexer_topk(*dev, K=K, out=out),
            lambda dev, out: binding.indexer_topk_unfused(*dev, K=K, out=out))


def host_problem(inp, binding):
    """The host-buffer call of a dense workload (None for paged ones)."""
    if hasattr(inp, "block_table"):
        return None
    return lambda pinned, out_h: binding.indexer_topk_host(*pinned, K=inp.K, out=out_h)


def run_ours(args, rank, world, device):
    import torch

    from fp8_scoring_exact_gb300 import binding

    inp = make_workload(args.config, args.rows, args.keys)
    R = inp.row_keys()
    legs = set(args.legs.split(","))
    host, out_shape, call, call_unfused = problem(inp, binding)
    dev = [torch.from_numpy(a).to(device) for a in host]
    out = torch.empty(out_shape, dtype=torch.int32, device=device)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        call(dev, out)

    binding.set_option("profile", 1)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    rc, counters = binding.last_device_status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} after warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    main_ms = []
    l0 = binding.launch_count()
    barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(device.index) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
            main_ms.append(binding.profiled_main_ms())  # waits for this step's main kernel
        torch.cuda.synchronize(device)
    barrier(world)
    launches = binding.launch_count() - l0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, device)
    ms_per_step = total_ms / args.steps
    rc, counters = binding.last_device_status()
    binding.set_option("profile", 0)

    # unfused attribution baseline, same protocol
    unf_ms = None
    if call_unfused is None:
        legs.discard("unfused")
    for _ in range(max(1, args.warmup // 2) if "unfused" in legs else 0):
        call_unfused(dev, out)
    if "unfused" in legs:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            call_unfused(dev, out)
            ev[i][1].record(stream)
        torch.cuda.synchronize(device)
        unf_ms = statistics.mean([a.elapsed_time(b) for a, b in ev])

    # the same call captured once into a CUDA graph and replayed (no host
    # launch work per call); the capture runs on a side stream whose library
    # scratch the warm-up calls have already sized, so nothing allocates
    graph = None
    if "graph" in legs:
        gs = torch.cuda.Stream(device)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            for _ in range(max(1, args.warmup)):
                step()
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            step()
        torch.cuda.synchronize(device)
        with torch.cuda.stream(gs):
            for i in range(args.steps):
                flush.zero_()
                ev[i][0].record(gs)
                g.replay()
                ev[i][1].record(gs)
        torch.cuda.synchronize(device)
        grc, _ = binding.last_device_status(gs)
        if grc != 0:
            raise RuntimeError(f"device status {grc} after graph replays")
        graph = {"ms_per_step": statistics.mean([a.elapsed_time(b) for a, b in ev]),
                 "note": "one fused call captured into a CUDA graph, replayed; L2 flushed before each replay"}
        del g

    # the standalone exact top-K over this workload's fp32 score matrix
    # (dsa_indexer_topk_from_scores; the pages' standalone top-K table): the
    # matrix is computed once outside the timed region, each timed step
    # reads every valid score once after an L2 flush
    select = None
    if "select" in legs and call_unfused is not None:
        scores = binding.indexer_scores(*dev)
        N = inp.N
        for _ in range(max(1, args.warmup)):
            binding.topk_from_scores(scores, dev[5], dev[6], K=inp.K, N=N, out=out)
        torch.cuda.synchronize(device)
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            binding.topk_from_scores(scores, dev[5], dev[6], K=inp.K, N=N, out=out)
            ev[i][1].record(stream)
        torch.cuda.synchronize(device)
        srec, _ = binding.last_device_status()
        if srec != 0:
            raise RuntimeError(f"device status {srec} after the standalone select")
        sel_ms = statistics.mean([a.elapsed_time(b) for a, b in ev])
        sel_bytes = 4 * R + 4 * inp.Q * inp.K + 8 * inp.Q
        sel_gbs = sel_bytes / (sel_ms * 1e-3) / 1e9
        hbm = load_peaks()["hbm_gbs"]
        select = {"ms_per_step": sel_ms, "rows": inp.Q, "achieved_gbs": sel_gbs, "frac_of_hbm": sel_gbs / hbm,
                  "bytes_per_step": sel_bytes,
                  "note": "standalone exact top-K (dsa_indexer_topk_from_scores) over this workload's fp32 score "
                          "matrix; bytes = every valid score once + output; L2 flushed before each step"}
        del scores

    # the math-only control ("Fusing Indexer Scoring and Exact Top-k for
    # DeepSeek-V3.2", section 5.2): the main scorer with its score reduction
    # and candidate filter removed, timed alternately with the real call in
    # the same rounds; exposed = the share of the main kernel's time they add
    control = None
    if "control" in legs and call_unfused is not None:
        checksum = torch.zeros(1, dtype=torch.float32, device=device)
        binding.set_option("profile", 1)
        ctl_args = (*dev[:7],)
        for _ in range(max(1, args.warmup)):
            binding.math_control(*ctl_args, K=inp.K, checksum=checksum)
        torch.cuda.synchronize(device)
        f_ms, c_ms = [], []
        for i in range(args.steps):
            flush.zero_()
            step()
            f_ms.append(binding.profiled_main_ms())
            flush.zero_()
            binding.math_control(*ctl_args, K=inp.K, checksum=checksum)
            c_ms.append(binding.profiled_main_ms())
        binding.set_option("profile", 0)
        fm, cm = statistics.mean(f_ms), statistics.mean(c_ms)
        control = {"main_kernel_ms": fm, "control_kernel_ms": cm, "exposed_frac": (fm - cm) / fm,
                   "control_tflops": FLOP_PER_ROW_KEY * R / (cm * 1e-3) / 1e12,
                   "call_ms": ms_per_step, "exposed_call_frac": (ms_per_step - cm) / ms_per_step,
                   "note": "math-only control (dsa_indexer_math_control): same units, TMA loads, tcgen05 MMAs and "
                           "barriers; the epilogue folds one accumulator column per warp and tile into a checksum. "
                           "exposed_frac = (main - control) / main, alternating rounds; exposed_call_frac = "
                           "(whole call - control) / whole call"}

    fp8_probe = fp8_peak_probe(device) if "fp8peak" in legs else None
    others = (other_configs_leg(args, binding, device, flush, args.config)
              if "configs" in legs and not (args.rows or args.keys) else None)
    sparse = sparse_attention_leg(args, binding, device, flush) if "sparse" in legs else None

    # end to end through the public API from pinned host buffers
    e2e = None
    if "e2e" in legs:
        e2e = _e2e(args, dev, host, out, stream, world, device, call, R, host_problem(inp, binding))
    peaks = load_peaks()
    main_avg = statistics.mean(main_ms)
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    achieved = FLOP_PER_ROW_KEY * R / (main_avg * 1e-3) / 1e12
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    clocks = clk.summary()
    f_sm = (clocks.get("sm_max_mhz") or peaks["sm_max_mhz"]) * 1e6
    t_tensor = FLOP_PER_ROW_KEY * R / (fp8_peak * 1e12) * 1e3
    t_core = CORE_OPS_PER_ROW_KEY * R / (sms * 128 * f_sm) * 1e3
    t_hbm = algorithmic_bytes_of(inp) / (peaks["hbm_gbs"] * 1e9) * 1e3
    t_roof = max(t_tensor, t_core, t_hbm)
    kernel_name = "score_kernel (filter mode: tcgen05 scoring + candidate filter)"
    peak_note = f"{peaks['source']} bf16 {peaks['bf16_tflops']} TFLOP/s x {FP8_OVER_BF16} (nominal fp8/bf16 ratio), burst"
    if t_hbm > t_tensor:
        # paged decode: every row reads its own keys, the HBM term dominates
        gbs = algorithmic_bytes_of(inp) / (main_avg * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": kernel_name, "kernel_ms": main_avg,
                    "peak_source": f"{peaks['source']} HBM copy bandwidth"}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                    "frac": achieved / fp8_peak, "traffic": measured_traffic(args.config, args.rows, args.keys),
                    "kernel": kernel_name, "kernel_ms": main_avg, "peak_source": peak_note}
        if fp8_probe is not None:
            roofline["fp8_probe"] = fp8_probe

    res = {
        "metric": METRIC,
        "value": world * R / (ms_per_step * 1e-3),
        "unit": "row-keys/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8e4m3 x fp8e4m3 -> f32",
        "data": "synthetic (seeded Gaussian activations quantised to FP8 e4m3 per token)",
        "config": describe(inp, args.config),
        "tflops_effective": world * FLOP_PER_ROW_KEY * R / (ms_per_step * 1e-3) / 1e12,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "roofline": roofline,
        "roofline_terms": {"t_tensor_ms": t_tensor, "t_core_ms": t_core, "t_hbm_ms": t_hbm, "t_roof_ms": t_roof,
                           "frac_of_roofline": t_roof / ms_per_step, "sm_count": sms,
                           "sm_clock_for_core_term_mhz": f_sm / 1e6},
        "unfused": ({"ms_per_step": unf_ms, "fused_speedup": unf_ms / ms_per_step} if unf_ms else None),
        "graph": graph,
        "select": select,
        "math_control": control,
        "sparse_attention": sparse,
        "other_workloads": others,
        "failures": counters,
    }
    if rank == 0 and not args.no_cpu_baseline:
        procs = cpu_procs()
        # a short pass sizes the sample so that the timed pass is ~10 s of CPU work
        rate, secs, rows = time_oracle(inp, 2 * procs, procs)
        if secs < CPU_BASELINE_SECONDS:
            n_rows = int(min(MAX_ORACLE_ROWS, 2 * procs * CPU_BASELINE_SECONDS / max(secs, 1e-3)))
            rate, secs, rows = time_oracle(inp, max(n_rows, 2 * procs), procs)
        res["cpu_baseline"] = {"value": rate, "unit": "row-keys/s", "cores": procs, "kind": "oracle",
                               "sample": f"{len(rows)} seeded rows of the same workload (all their keys), "
                                         f"{secs:.1f} s on {procs} spawned single-thread processes"}
    return res


def run_reference(args, rank, world):
    """CPU oracle as the reference arm: rank 0 only."""
    if rank != 0:
        return None
    inp = make_workload(args.config, args.rows, args.keys)
    procs = cpu_procs()
    from oracle.indexer import OraclePool
    per = procs
    if hasattr(inp, "block_table"):
        n_seq = max(1, per // inp.next_n)
        sub, allrows = paged_subset(inp, n_seq * (args.steps + args.warmup), seed=321)
        kind = "paged"
        per = n_seq * inp.next_n
        lens_all = sub.row_lengths().reshape(-1)
    else:
        rows = oracle_rows(inp, procs * (args.steps + args.warmup), seed=321)
        sub = oracle_subset(inp, rows)
        allrows = list(range(len(rows)))
        kind = "dense"
        lens_all = sub.row_end.astype(np.int64) - sub.row_begin
    n_all = len(allrows)
    per = min(per, n_all)

    def window(i):  # step i's rows, cycling when the sample is short
        return [(i * per + j) % n_all for j in range(per)]

    with OraclePool(sub, procs, kind) as pool:
        for i in range(args.warmup):
            pool.topk([allrows[j] for j in window(i)])
        t0 = time.perf_counter()
        for i in range(args.warmup, args.warmup + args.steps):
            pool.topk([allrows[j] for j in window(i)])
        dt = time.perf_counter() - t0
    lens = np.concatenate([lens_all[window(i)] for i in range(args.warmup, args.warmup + args.steps)])
    rate = float(lens.sum()) / dt
    res = {
        "impl": "reference",
        "metric": METRIC,
        "value": rate,
        "unit": "row-keys/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (exact integer dots, fp64 combination)",
        "data": "synthetic (seeded Gaussian activations quantised to FP8 e4m3 per token)",
        "config": describe(inp, args.config),
        "cpu_baseline": {"value": rate, "unit": "row-keys/s", "cores": procs, "kind": "oracle",
                         "sample": f"{per} seeded rows per step (all their keys), {args.steps} timed steps"},
        "e2e": {"value": rate, "unit": "row-keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return res


# ------------------------------------------------------------ distributed --
def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, help="workload index (2 = causal Q4096 x N131072)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", type=int, default=0, help="override: causal workload with this many query rows")
    ap.add_argument("--keys", type=int, default=0, help="override: causal workload with this many keys")
    ap.add_argument("--sparse-slots", type=int, default=0,
                    help="sparse leg on random slots of a cache of this many slots (a smaller profiling case) "
                         "instead of the paged decode batch's own top-2048 result")
    ap.add_argument("--legs", default="fused,unfused,graph,select,control,fp8peak,sparse,configs,e2e",
                    help="comma list of legs to run besides the timed fused leg "
                         "(unfused, graph, select, control, fp8peak, sparse, configs, e2e)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world = init_dist()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        import torch
        local = int(os.environ.get("LOCAL_RANK", "0"))
        device = torch.device("cuda", local)
        torch.cuda.set_device(device)
        if rank == 0:
            import __graft_entry__
            __graft_entry__.build()
        barrier(world)
        res = run_ours(args, rank, world, device)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

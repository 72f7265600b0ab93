"""Batch-1 decode throughput of the persistent megakernel on one GB300.

A step is one mk_decode launch of the workload's full decode (the 1B bf16
workload: 256 greedy tokens after a 128-token prompt), rewound to the end of
the prompt before every step, with weights (2.2 GB, larger than L2) and KV
cache resident in HBM.  `value` is decode tokens/s from CUDA events on the
launching stream; `e2e` is the same metric through the host-buffer C-ABI calls
(mk_set_state with the step's pending token and position, then mk_decode:
launch, device->host copy of the ids and status, stream sync) on the host
clock.  `roofline` reports algorithmic bytes per launch (GEMV weights incl.
quantisation scales, embedding row, norm gains, KV reads and writes at each
step's position) over the launch time, against the measured HBM copy
bandwidth.  `cpu_baseline` times the float64 CPU oracle on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
"""
import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

# The CPU oracle's BLAS threads are set before NumPy loads its BLAS: all host
# cores unless the caller fixed a count.
ORACLE_THREADS = int(os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
                     or os.cpu_count() or 1)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(ORACLE_THREADS))

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "batch-1 decode tokens/s"
UNIT = "tokens/s"


def algorithmic_bytes(w, pos0, n_steps):
    """Bytes the decode path must move per launch (see the module docstring)."""
    def rb(K):
        return {"bf16": 2 * K, "fp16": 2 * K, "int8": K + 2, "int4": K // 2 + 2 * (K // 128),
                "fp8": K + 2 * (K // 128)}[w.wdtype]
    d, qd, kd, F, V, L = w.d_model, w.q_dim, w.kv_dim, w.d_ffn, w.vocab, w.n_layers
    gemv = L * ((qd + 2 * kd) * rb(d) + d * rb(qd) + 2 * F * rb(d) + d * rb(F)) + V * rb(d)
    fixed = gemv + 2 * d + (2 * L + 1) * 2 * d
    kv_pos = 2 * L * kd * 2  # K and V bytes of one position over all layers
    total = 0
    for s in range(n_steps):
        pos = pos0 + s
        total += fixed + kv_pos * (pos + 1) + kv_pos
    return total, gemv


def max_over_ranks(value, device):
    """The largest value over all ranks of the default process group (every
    rank gets it): the job's time is its slowest replica's."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, seconds):
    """Whole-job throughput of `world` replicas that each processed
    units_per_rank units, over the slowest replica's time."""
    return world * units_per_rank / seconds


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


KERNEL_SOURCES = ("decode_megakernel_02_gb300/csrc/mk_vm.cuh", "decode_megakernel_02_gb300/csrc/mk_internal.h",
                  "decode_megakernel_02_gb300/csrc/mk_schedule.cpp")


def code_only(text):
    """The source text without comments, blank lines and trailing spaces: an
    edit of the comments leaves the kernel, and so this form, unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash(read=None):
    """Hash of the decode kernel's code (the kernel, its internal header and the
    schedule lowering), ignoring comments.  `read(path)` returns a file's text
    (default: the working tree)."""
    read = read or (lambda f: open(os.path.join(ROOT, f)).read())
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(code_only(read(f)).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", f"vm_kernel_{workload}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def blas_info():
    """BLAS library NumPy uses and its thread count, as far as this NumPy reports them."""
    vendor, threads = "unknown", ORACLE_THREADS
    try:
        cfg = np.show_config(mode="dicts")
        b = cfg.get("Build Dependencies", {}).get("blas", {})
        vendor = f"{b.get('name', 'unknown')} {b.get('version', '')}".strip()
    except Exception:
        pass
    try:
        from threadpoolctl import threadpool_info
        pools = [p for p in threadpool_info() if p.get("user_api") == "blas"]
        if pools:
            threads = int(pools[0]["num_threads"])
            vendor = f"{pools[0].get('internal_api', vendor)} {pools[0].get('version', '')}".strip()
    except Exception:
        pass
    return vendor, threads


def oracle_rate(w, weights, budget_s=12.0, min_steps=2, max_steps=64):
    """Tokens/s of the float64 oracle decoding from the end of the prompt."""
    from oracle import llama as L
    from oracle import quant as Q
    deq = None
    if w.wdtype in ("int8", "int4", "fp8"):
        deq, _ = Q.quantised_model_weights(w, weights, w.wdtype)
    m = L.Model(w, weights, w.base_dtype, dequantised=deq)
    prompt = synthetic.generate_prompt(w)
    kv = m.new_cache(w.max_seq)
    # The prompt's cache entries stay zero (untimed prefill skipped): the
    # sample keeps the attention lengths of the workload, which is what the
    # time depends on.
    tok, pos = int(prompt[-1]), len(prompt) - 1
    L.decode_step(m, kv, tok, pos)  # widen the weights once (untimed)
    n, t0 = 0, time.perf_counter()
    while n < max_steps:
        lg = L.decode_step(m, kv, tok, pos + n)
        tok = L.argmax_lowest(lg)
        n += 1
        if n >= min_steps and time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama-1b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sms", type=int, default=0)
    ap.add_argument("--rows-in-flight", type=int, default=0)
    ap.add_argument("--chunks", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0, help="decode tokens per step (default: the workload's)")
    ap.add_argument("--prefill-chunk", type=int, default=-1,
                    help="tensor-core prefill chunk (tokens); 0: the decode kernel walks the prompt; "
                         "-1 (default): 1024 for 16-bit weights, else 0")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    w = synthetic.get_workload(args.workload)
    n_tok = args.tokens or w.decode_steps
    pos0 = w.prompt_len - 1
    config = {"workload": w.name, "prompt_len": w.prompt_len, "decode_tokens": n_tok, "batch": 1,
              "weights": w.wdtype, "l2": "inputs larger than L2 (weights streamed every token)",
              "parallelism": "replicas" if world > 1 else "single-gpu"}

    if args.impl == "reference":
        if rank != 0:
            return
        weights = synthetic.generate_weights(w)
        rates = []
        for s in range(args.warmup + args.steps):
            r, n, dt = oracle_rate(w, weights, budget_s=2.0, min_steps=1, max_steps=4)
            if s >= args.warmup:
                rates.append(r)
        v = float(np.mean(rates))
        vendor, cores = blas_info()
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * 4 / v,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "blas": vendor,
                                 "host_cpus": os.cpu_count(),
                                 "sample": f"up to 4 greedy decode steps from position {pos0} per step"},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import torch.distributed as dist
    from decode_megakernel_02_gb300 import build
    build.build()
    import decode_megakernel_02_gb300 as mk

    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev_index = torch.cuda.current_device()

    weights = synthetic.generate_weights(w)
    desc = mk.make_desc(w)
    blob = mk.pack_model(desc, weights)
    chunk = args.prefill_chunk if args.prefill_chunk >= 0 else (1024 if w.wdtype == w.base_dtype else 0)
    cfg = mk.make_config(sms=args.sms, rows_in_flight=args.rows_in_flight, attn_chunks=args.chunks,
                         prefill_chunk=chunk)
    dec = mk.Decoder(desc, blob, cfg)
    del blob
    prompt = synthetic.generate_prompt(w)
    torch.cuda.synchronize()
    t_pf = time.perf_counter()
    dec.prefill(prompt)  # synchronous
    prefill_ms = (time.perf_counter() - t_pf) * 1e3
    pending = int(prompt[-1])
    ids_dev = torch.empty(n_tok, dtype=torch.int32, device="cuda")
    stream = dec.stream

    def step():
        dec.set_state(pos0, pending)
        dec.decode_async(n_tok, out_ids=ids_dev)

    for _ in range(args.warmup):
        step()
    dec.finish()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = dec.launch_count()
    per_launch = []
    with ClockSampler(dev_index) as clk:
        ev0.record(stream)
        evs = []
        for _ in range(args.steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            evs.append((a, b))
        ev1.record(stream)
        torch.cuda.synchronize()
    dec.finish()
    launches = dec.launch_count() - launches0
    total_ms = ev0.elapsed_time(ev1)
    per_launch = [a.elapsed_time(b) for a, b in evs]
    if world > 1:
        total_ms = max_over_ranks(total_ms, "cuda")
        dist.barrier()
    ms_per_step = total_ms / args.steps
    value = job_rate(world, n_tok * args.steps, total_ms / 1000.0)

    # end to end through the host-buffer call (ids copied to host, stream synced)
    host_ids = np.empty(n_tok, np.int32)
    e2e_t = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        dec.set_state(pos0, pending)  # the step's input: the pending token and its position
        dec.decode(n_tok, out=host_ids)
        if i >= args.warmup:
            e2e_t.append(time.perf_counter() - t0)
    e2e_rate = world * n_tok * len(e2e_t) / sum(e2e_t)

    alg_bytes, gemv_bytes = algorithmic_bytes(w, pos0, n_tok)
    launch_ms = float(np.mean(per_launch))
    achieved = alg_bytes / (launch_ms / 1000.0) / 1e9
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    traffic = profiled_traffic(w.name)
    info = dec.launch_info()

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": {"bf16": "bf16", "fp16": "fp16", "int8": "int8w-f32acc",
                                           "int4": "int4w-f32acc", "fp8": "fp8e4m3w-f32acc"}[w.wdtype],
            "data": "synthetic", "config": config,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "frac_of_8tbs": achieved / 8000.0},
            "e2e": {"value": e2e_rate, "unit": UNIT, "h2d_bytes_per_step": 8, "d2h_bytes_per_step": 4 * n_tok + 16,
                    "inputs": "pending token and position (2 x int32), passed by value in the launch parameters"},
            "gpu_launches": int(launches), "launch": info, "kernel_source": kernel_source_hash(),
            "prefill": {"positions": len(prompt) - 1, "ms": prefill_ms,
                        "path": f"tensor cores, chunks of {chunk}" if chunk else "decode kernel, one position per step",
                        "timed": "host clock around the synchronous mk_prefill, outside the decode timing"}}
    clocks = clk.summary()
    if clocks:
        line["clocks"] = clocks
    if rank == 0 and not args.no_cpu_baseline:
        r, n, dt = oracle_rate(w, weights)
        vendor, threads = blas_info()
        line["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": threads, "kind": "oracle", "blas": vendor,
                                "host_cpus": os.cpu_count(),
                                "sample": f"{n} greedy decode steps from position {pos0} ({dt:.1f} s; prompt cache "
                                          f"zero-filled, untimed), float64 NumPy, {threads} BLAS threads"}
    if rank == 0:
        print(json.dumps(line))
    dec.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

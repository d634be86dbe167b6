"""Benchmark: batch-1 greedy decode of the 2B fp16 workload through the persistent
megakernel, all K timed steps in ONE launch of mk_decode_steps (the monokernel runs the whole
generation; --steps-per-launch C: C chained steps per launch instead, 1 = one launch per
step, measured ~1.4 % slower: the launch boundary costs a little more than the in-kernel
step boundary).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Workload: 24 layers, d 2048, 16/8 heads of 128, FFN 8192, vocab 128256, fp16 weights
and KV cache (seeded synthetic weights), batch 1, a 512-token prompt (mk_prefill), then
W warm-up and K timed greedy decode steps.  One step streams all weights but the
embedding (3.545 GB) plus the KV cache -- far above the 129 MB L2, so no flush is needed
between steps.  Prints one JSON line (rank 0).

value: tok/s with everything resident in HBM: K chained steps (each step embeds the
token the previous step chose on the device), CUDA events on the context's stream
around every launch (one launch by default).
e2e: the same metric through mk_decode_step with host token buffers (token and position
travel as kernel parameters; the step's tokens and status come back through an 80-byte
mapped host mailbox the kernel writes), host loop included.
roofline: algorithmic bytes per step / (mean launch duration / steps per launch) against
the measured HBM copy bandwidth; traffic: the profiled DRAM bytes of one step.  cpu_baseline / --impl reference: the fp64 oracle on the host cores.
Multi-GPU (torchrun, N > 1): independent replicas, one per GPU; max time over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "2b"
METRIC = "batch-1 decode tok/s (2B fp16) + weight-stream HBM GB/s vs GB300 peak"
UNIT = "tok/s"
PROMPT = 512
WORKLOAD_DESC = ("2b-fp16 decode: 24 layers, d 2048, 16/8 heads x 128, FFN 8192, vocab 128256; "
                 "batch 1, 512-token prompt, greedy decode (synthetic seeded weights)")
NOMINAL_HBM_GBS = 7900.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "mk_step_kernel_2b_b1.txt")
KERNEL_SOURCES = ["mk_kernel.cuh", "mk_device.cuh", "mk_internal.h"]


def kernel_source_hash(sync="sentinel"):
    """Hash of the sources the timed kernel instance is compiled from."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES + [f"mk_k_f16_{sync}.cu", f"mk_k_f16_{sync}_ms.cu"]:
        with open(os.path.join(ROOT, "persistent_sm_decode_megakernel_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(sync="sentinel"):
    """(DRAM bytes, algorithmic bytes) of one decode step from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    try:
        with open(PROFILE_SUMMARY) as f:
            kv = dict(l.split(":", 1) for l in f.read().splitlines() if ":" in l)
        if kv.get("kernel_source_sha", "").strip() != kernel_source_hash(sync):
            return None
        dram = float(kv["dram_bytes_per_step"].strip())
        return dram, float(kv["algorithmic_bytes_per_step"].split()[0])

    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("MK_BENCH_BACKEND", "") != "gloo" else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def aggregate_max(seconds, world, device=None):
    """Max of a per-rank duration over all ranks (the job ends with its slowest rank)."""
    if world == 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units, seconds, world, device=None):
    """Whole-job throughput of `world` replicas that each processed `units` in their own
    `seconds`: all units over the slowest rank's time.  Returns (rate, max seconds)."""
    t = aggregate_max(seconds, world, device)
    return world * units / t, t


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def algorithmic_bytes(cfg, positions):
    """Bytes one decode step must read: weights (all but the embedding table), the cached
    keys/values below each sequence's position, the embedding row; plus the new k,v."""
    w = cfg.streamed_weight_bytes()
    per_pos = cfg.kv_bytes_per_position()
    return w + sum(per_pos * p for p in positions) + len(positions) * (2 * cfg.d_model + per_pos)


def cpu_oracle_rate(cfg, weights, budget_s=20.0, max_steps=64, ctx0=PROMPT + 8, n_warm=1):
    """Oracle decode steps (fp64, host cores) at the GPU's context: the cache holds ctx0
    positions (seeded synthetic keys and values, as a prompt would leave them) and the
    steps run at positions ctx0, ctx0 + 1, ...  Returns (tok/s, steps, seconds)."""
    import numpy as np
    import oracle
    import synth
    m = oracle.Model(cfg, weights)
    for name in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "attn_norm", "mlp_norm"):
        for l in range(cfg.n_layers):
            m.w(name, l)
    m.w("lm_head")
    m.w("final_norm")
    cache = oracle.KVCache(cfg, 1, ctx0 + n_warm + max_steps + 2)
    for l in range(cfg.n_layers):
        cache.k[l][0, :, :ctx0] = oracle.upcast(synth.gen_kv(cfg, l, 0, 0, ctx0), cfg.dtype)
        cache.v[l][0, :, :ctx0] = oracle.upcast(synth.gen_kv(cfg, l, 0, 1, ctx0), cfg.dtype)
    tok = int(synth_prompt(cfg)[0, -1])
    for k in range(n_warm):                               # warm-up, untimed
        z = oracle.decode_step(m, cache, [tok], [ctx0 + k])
        tok = int(np.argmax(z[0]))
    n, t0 = 0, time.perf_counter()
    while n < max_steps and time.perf_counter() - t0 < budget_s:
        z = oracle.decode_step(m, cache, [tok], [ctx0 + n_warm + n])
        tok = int(np.argmax(z[0]))
        n += 1
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def synth_prompt(cfg):
    import synth
    return synth.gen_prompts(cfg, 1, PROMPT)


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max((i.get("num_threads", 1) for i in info), default=os.cpu_count())
    except Exception:
        return os.cpu_count()


def run_reference(args):
    """The fp64 oracle as the reference arm: same workload, metric and unit."""
    rank, world, _ = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0
    if rank != 0:
        return 0
    import synth
    cfg = synth.CONFIGS[WORKLOAD]
    weights = synth.gen_weights(cfg)
    steps = max(1, min(args.steps, 16))
    warm = max(1, min(args.warmup, 8))
    rate, n, dt = cpu_oracle_rate(cfg, weights, budget_s=120.0, max_steps=steps, n_warm=warm)
    ctx0 = PROMPT + 8
    sample = (f"{n} fp64 oracle decode steps of the 2B model at positions {ctx0 + warm + 1}..{ctx0 + warm + n} "
              f"(the cache holds {ctx0} seeded synthetic positions, the GPU's context), after {warm} untimed "
              f"steps; {args.steps} timed and {args.warmup} warm-up steps requested, capped to bound the run")
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
            "steps": n, "warmup": warm, "ms_per_step": 1000.0 * dt / max(n, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC, "batch": 1, "prompt_len": PROMPT,
                       "note": "the oracle's sample steps run at the GPU's context (see cpu_baseline.sample)"},
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sync", default="sentinel", choices=["counter", "sentinel"])
    ap.add_argument("--exec", default="persistent", choices=["persistent", "multilaunch", "graph"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--steps-per-launch", type=int, default=0,
                    help="decode steps per launch (0: all K in one; persistent control only)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import numpy as np
    import torch

    import synth
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = synth.CONFIGS[WORKLOAD]
    B = args.batch
    weights = synth.gen_weights(cfg)
    K, W = args.steps, args.warmup
    max_ctx = PROMPT + W + K + args.e2e_steps + 4
    dm = DeviceModel(cfg, weights, max_batch=B, max_ctx=max_ctx, device=device)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        dec = Decoder(dm, sync_mode=0 if args.sync == "counter" else 1,
                      exec_mode={"persistent": 0, "multilaunch": 1, "graph": 2}[args.exec], stream=stream)
        info = dec.info()
        prompt = synth.gen_prompts(cfg, B, PROMPT)
        first = dec.prefill(prompt)
        pos = PROMPT
        # warm-up: chained greedy steps
        dec.decode_steps(first, [pos] * B, W)
        pos += W
        dec.synchronize()

        # ---- timed region: K chained steps in launches of C steps, events around every launch
        C = K if args.steps_per_launch <= 0 else min(args.steps_per_launch, K)
        if args.exec != "persistent":
            C = 1
        chunks = [min(C, K - k0) for k0 in range(0, K, C)]
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(chunks) + 1)]
        positions = []
        barrier(world, device)
        torch.cuda.synchronize(device)
        with ClockSampler(local) as clocks:
            ev[0].record(stream)
            for i, n in enumerate(chunks):
                dec.decode_steps(None, [pos] * B, n)
                positions += list(range(pos, pos + n))
                pos += n
                ev[i + 1].record(stream)
            dec.synchronize()
            torch.cuda.synchronize(device)
        barrier(world, device)
        per_step_ms = [ev[i].elapsed_time(ev[i + 1]) / n for i, n in enumerate(chunks)]
        total_s = ev[0].elapsed_time(ev[len(chunks)]) / 1000.0
        value, total_s = job_rate(B * K, total_s, world, device)
        mean_step_s = statistics.mean(per_step_ms) / 1000.0

        # ---- e2e: host buffers through mk_decode_step, host loop timed
        K2 = min(args.e2e_steps, K)
        tok = np.array(first, dtype=np.int32)
        barrier(world, device)
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        for k in range(K2):
            tok = dec.decode_step(tok, [pos] * B)
            pos += 1
        e2e_value, e2e_s = job_rate(B * K2, time.perf_counter() - t0, world, device)
        dec.close()

    if rank != 0:
        return 0
    peak, peak_kind = measured_peaks()
    bytes_per_step = statistics.mean(algorithmic_bytes(cfg, [p] * B) for p in positions)
    achieved_gbs = bytes_per_step / mean_step_s / 1e9
    t_min = bytes_per_step / (peak * 1e9)
    cpu = None
    if not args.no_cpu_baseline and world >= 1:
        rate, n, dt = cpu_oracle_rate(cfg, weights)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{n} fp64 oracle decode steps of the same 2B model, batch 1, at positions "
                         f"{PROMPT + 9}..{PROMPT + 8 + n} (cache of {PROMPT + 8} seeded synthetic positions, the "
                         f"GPU's context), {dt:.1f} s after 1 untimed step"}
    prof = profiled_traffic(args.sync)
    # the capture ran at a shorter context: scale its DRAM bytes by the algorithmic bytes (K/V grows with it)
    traffic = None if prof is None else prof[0] * bytes_per_step / prof[1]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": 1000.0 * total_s / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC,
                   "batch": B, "prompt_len": PROMPT, "context": [positions[0], positions[-1]],
                   "l2": "inputs larger than L2: 3.6 GB streamed per step vs 129 MB L2, no flush",
                   "sync": args.sync, "exec": args.exec, "parallelism": f"replicas x{world}"},
        "gpu_launches": len(chunks) * info["launches_per_step"],
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak, "traffic": traffic,
                     "traffic_source": None if traffic is None else
                     "ncu DRAM read+write of a 64-step launch of this command at a shorter context, per step, "
                     "scaled by the algorithmic bytes (profiles/mk_step_kernel_2b_b1.txt)",
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs, copy)",
                     "per": "decode step (a launch runs steps_per_launch of them)",
                     "steps_per_launch": C, "bytes_per_step": bytes_per_step, "mean_step_us": mean_step_s * 1e6,
                     "frac_of_nominal_7900": achieved_gbs / NOMINAL_HBM_GBS},
        "overhead_fraction": (total_s / K - t_min) / (total_s / K),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 8 * B, "d2h_bytes_per_step": 80,
                "steps": K2, "note": "token+position as kernel parameters; tokens and status posted by the "
                                     "kernel to an 80-byte mapped host mailbox"},
        "cpu_baseline": cpu,
        "clocks": clocks.summary(),
        "launch": {"ctas": info["n_ctas"], "threads": info["threads_per_cta"], "smem": info["smem_bytes"],
                   "pages": info["n_pages"], "page_bytes": info["page_bytes"], "kv_splits": info["kv_splits"],
                   "instructions": info["n_instructions"]},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())

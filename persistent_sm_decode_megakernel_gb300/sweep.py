"""Measurements beside the headline bench: the pages' secondary figures redone on one GPU.

    python -m persistent_sm_decode_megakernel_gb300.sweep [--only NAME ...] [--json FILE]

Each part prints one JSON object (and all of them go to --json):
  barrier   all-CTA barrier latency, atomic counters vs NaN sentinels ("7 · AMD et le
            monokernel", §7.3 measures 7.59-7.88 us vs 0.80-0.93 us on MI300X)
  launch    one 2b decode step (batch 1, 512 cached positions) as one persistent launch,
            as the multi-launch control and as its CUDA graph; the per-launch cost is the
            step-time difference over the launch-count difference (§7.2: ~4.5 us per HIP
            launch); and the waiting share of each CTA's step from the journal (§7.2:
            grid synchronisation ~35 % of a token's time)
  batch512  the 2b model at 512 cached positions (the benchmark's context), batch 1/2/4/8/16,
            persistent with counters and with sentinels: us per step, aggregate tok/s and the
            fraction of the HBM roofline (batches 3..16 run the tensor-core GEMV)
  ctx32k    the 2b model at 32768 cached positions, batch 1/2/4/8/16, persistent with
            counters, persistent with sentinels and the multi-launch control: us per step,
            aggregate tok/s, and the fraction of the HBM roofline (weights + KV per step)
  ragged    batches of 8 and 16 at 32768 cached positions for all sequences against
            positions spread evenly over 8192..32767: step time, and from the journal the
            attention phase's tail per layer (the last CTA's attention end minus the median
            CTA's), with the attention units dealt to fixed queues and claimed from a pool
  ctx8k     the 8b model at 8192 cached positions, batch 1, both sync modes
  prefill   mk_prefill wall time of the 2b model: 512- and 32768-token prompts in chunks,
            and the 512-token prompt fed one position per mk_decode_step launch
  dies      the SM -> die map and the address -> die interleave (§7.4): L2 latency of every
            256-byte line of an 8 MB buffer from an SM of each group; near / far medians
            and how often the four lines of a 1 KB block share a home
The caches of the long-context parts hold synthetic keys and values (normal, std 0.9),
drawn on the device: the timings do not depend on the values.
"""
import argparse
import ctypes
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return 6800.0


def _fill_kv(dm, cfg, B, T, seed=0):
    import torch
    g = torch.Generator(device=dm.device)
    g.manual_seed(seed)
    dt = torch.float16 if cfg.dtype == "f16" else torch.bfloat16
    for l in range(cfg.n_layers):
        for cache in (dm.k_cache[l], dm.v_cache[l]):
            for b in range(B):
                x = torch.randn((cfg.n_kv_heads, T, cfg.head_dim), generator=g, device=dm.device, dtype=torch.float32)
                cache[b, :, :T] = (x * 0.9).to(dt).view(torch.int16)


def _time_steps(dec, tok, pos, n_warm=2, n=6, trace=False):
    """Median us of n decode steps at positions pos (+k), after n_warm untimed ones."""
    import torch
    times = []
    p = list(pos)
    for k in range(n_warm + n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(dec.stream)
        tok = dec.decode_step(tok, p)
        e1.record(dec.stream)
        e1.synchronize()
        if k >= n_warm:
            times.append(e0.elapsed_time(e1) * 1e3)
        p = [x + 1 for x in p]
    return statistics.median(times), tok, p


def _algo_bytes(cfg, positions):
    per_pos = cfg.kv_bytes_per_position()
    return cfg.streamed_weight_bytes() + sum(per_pos * p for p in positions) + len(positions) * (2 * cfg.d_model + per_pos)


def part_barrier():
    import persistent_sm_decode_megakernel_gb300 as mk
    out = {}
    for mode, name in ((0, "counter_us"), (1, "sentinel_us")):
        us = ctypes.c_double()
        mk.check(mk.mk_barrier_bench(mode, 2000, ctypes.byref(us)), "mk_barrier_bench")
        out[name] = us.value
    return out


def part_launch():
    import synth
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel
    from persistent_sm_decode_megakernel_gb300.profile_step import summarize
    cfg = synth.CONFIGS["2b"]
    w = synth.gen_weights(cfg)
    P = 512
    dm = DeviceModel(cfg, w, max_batch=1, max_ctx=P + 64)
    _fill_kv(dm, cfg, 1, P)
    out = {}
    for name, sync, ex in (("persistent_sentinel", 1, 0), ("persistent_counter", 0, 0),
                           ("multilaunch", 0, 1), ("graph", 0, 2)):
        dec = Decoder(dm, sync_mode=sync, exec_mode=ex)
        us, _, _ = _time_steps(dec, [1], [P])
        out[name] = {"us_per_step": us, "launches_per_step": dec.info()["launches_per_step"]}
        dec.close()
    base = out["persistent_counter"]
    for name in ("multilaunch", "graph"):
        d = out[name]
        d["us_per_extra_launch"] = (d["us_per_step"] - base["us_per_step"]) / max(1, d["launches_per_step"] - 1)
    for name, sync in (("persistent_sentinel", 1), ("persistent_counter", 0)):
        dec = Decoder(dm, sync_mode=sync, trace=1)
        _time_steps(dec, [1], [P], n_warm=2, n=1)
        out[name]["wait_share_of_step"] = summarize(dec.trace())["wait_share_mean"]
        dec.close()
    return out


def part_batch512():
    import synth
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel
    cfg = synth.CONFIGS["2b"]
    T = cfg.prompt_len
    w = synth.gen_weights(cfg)
    peak = _peak()
    out = {}
    for B in (1, 2, 4, 8, 16):
        dm = DeviceModel(cfg, w, max_batch=B, max_ctx=T + 16)
        _fill_kv(dm, cfg, B, T)
        for name, sync in (("counter", 0), ("sentinel", 1)):
            dec = Decoder(dm, sync_mode=sync)
            us, _, _ = _time_steps(dec, [1] * B, [T] * B, n_warm=2, n=6)
            dec.close()
            gbs = _algo_bytes(cfg, [T + 4] * B) / (us * 1e-6) / 1e9
            out[f"B{B}_{name}"] = {"us_per_step": us, "tok_s": B / (us * 1e-6), "roofline_frac": gbs / peak}
            print(json.dumps({f"B{B}_{name}": out[f"B{B}_{name}"]}), flush=True)
        del dm
    return out


def part_ctx32k():
    import synth
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel
    import torch
    cfg = synth.CONFIGS["2b-32k"]
    T = cfg.prompt_len
    w = synth.gen_weights(cfg)
    peak = _peak()
    out = {}
    for B in (1, 2, 4, 8, 16):
        # a context of max_batch B, as a user serving B sequences creates it (batches of 1..2
        # run the kernel variant without the tensor-core GEMV)
        dm = DeviceModel(cfg, w, max_batch=B, max_ctx=T + 16)
        _fill_kv(dm, cfg, B, T)
        for name, sync, ex in (("persistent_counter", 0, 0), ("persistent_sentinel", 1, 0), ("multilaunch", 0, 1)):
            dec = Decoder(dm, sync_mode=sync, exec_mode=ex)
            us, _, _ = _time_steps(dec, [1] * B, [T] * B, n_warm=2, n=4)
            dec.close()
            gbs = _algo_bytes(cfg, [T + 3] * B) / (us * 1e-6) / 1e9
            out[f"B{B}_{name}"] = {"us_per_step": us, "tok_s": B / (us * 1e-6), "roofline_frac": gbs / peak}
            print(json.dumps({f"B{B}_{name}": out[f"B{B}_{name}"]}), flush=True)
        del dm
        torch.cuda.empty_cache()
    return out


def _attn_tail(trace):
    """Per layer, over the CTAs: the end of each CTA's last attention unit; the tail is the
    latest of those minus their median (what a CTA that finishes early could still take
    over from the others), against the layer's span (previous layer's last down-projection
    end to this layer's).  Medians over layers."""
    last, downs = {}, {}
    for r in trace:
        cta, op, layer, t_end = r[0], r[2], r[3], r[6]
        if op in (3, 9):
            k = (layer, cta)
            last[k] = max(last.get(k, 0), t_end)
        elif op == 7:
            downs[layer] = max(downs.get(layer, 0), t_end)
    per_layer = {}
    for (l, cta), t in last.items():
        per_layer.setdefault(l, []).append(t)
    tails, spans = [], []
    for l, ends in per_layer.items():
        if l - 1 not in downs or l not in downs:
            continue
        tails.append((max(ends) - statistics.median(ends)) / 1e3)
        spans.append((downs[l] - downs[l - 1]) / 1e3)
    return statistics.median(tails), statistics.median(spans)


def part_ragged():
    import synth
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel
    cfg = synth.CONFIGS["2b-32k"]
    T = cfg.prompt_len
    w = synth.gen_weights(cfg)
    dm = DeviceModel(cfg, w, max_batch=16, max_ctx=T + 16)
    _fill_kv(dm, cfg, 16, T)
    out = {}
    for B in (1, 8, 16):
        for kind in ("uniform", "ragged"):
            if B == 1 and kind == "ragged":
                continue
            pos = [T] * B if kind == "uniform" else [8192 + (T - 8192) * b // B for b in range(B)]
            for pool in (0, 1):
                dec = Decoder(dm, sync_mode=1, attn_pool=pool)
                us, _, _ = _time_steps(dec, [1] * B, pos, n_warm=2, n=4)
                dec.close()
                dec = Decoder(dm, sync_mode=1, trace=1, attn_pool=pool)
                _time_steps(dec, [1] * B, pos, n_warm=1, n=1)
                tail, span = _attn_tail(dec.trace())
                dec.close()
                key = f"B{B}_{kind}{'_pool' if pool else ''}"
                out[key] = {"us_per_step": us, "attn_tail_us": tail, "layer_us": span,
                            "tail_share_of_layer": tail / span, "positions": [min(pos), max(pos)]}
                print(json.dumps({key: out[key]}), flush=True)
    return out


def part_ctx8k():
    import synth
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel
    cfg = synth.CONFIGS["8b"]
    T = cfg.prompt_len
    w = synth.gen_weights(cfg)
    dm = DeviceModel(cfg, w, max_batch=1, max_ctx=T + 16)
    _fill_kv(dm, cfg, 1, T)
    peak = _peak()
    out = {}
    for name, sync in (("persistent_counter", 0), ("persistent_sentinel", 1)):
        dec = Decoder(dm, sync_mode=sync)
        us, _, _ = _time_steps(dec, [1], [T])
        dec.close()
        gbs = _algo_bytes(cfg, [T + 3]) / (us * 1e-6) / 1e9
        out[name] = {"us_per_step": us, "tok_s": 1e6 / us, "roofline_frac": gbs / peak}
    return out


def part_prefill():
    import torch
    import synth
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel
    cfg = synth.CONFIGS["2b"]
    w = synth.gen_weights(cfg)
    out = {}
    for P, chunks in ((512, True), (512, False), (32768, True)):
        dm = DeviceModel(cfg, w, max_batch=1, max_ctx=P + 8)
        prompt = synth.gen_prompts(cfg, 1, P)
        dec = Decoder(dm, sync_mode=1)

        def run():
            if chunks:
                dec.prefill(prompt)
            else:
                for t in range(P):
                    dec.decode_step(prompt[:, t], [t])
        if P <= 512:
            run()  # warm-up
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run()
        dt = time.perf_counter() - t0
        dec.close()
        del dm
        torch.cuda.empty_cache()
        key = f"P{P}_{'chunks' if chunks else 'per_position'}"
        out[key] = {"seconds": dt, "prompt_tok_s": P / dt}
        print(json.dumps({key: out[key]}), flush=True)
    return out


def part_dies():
    import numpy as np
    import persistent_sm_decode_megakernel_gb300 as mk
    n_max = 512
    die = (ctypes.c_int * n_max)()
    rtt = (ctypes.c_float * n_max)()
    nsm = ctypes.c_int()
    mk.check(mk.mk_die_map(6, n_max, die, rtt, ctypes.byref(nsm)), "mk_die_map")
    groups = [[i for i in range(nsm.value) if die[i] == g] for g in (0, 1)]
    offs = np.arange(0, 8 << 20, 256, dtype=np.int64)
    la = (ctypes.c_float * len(offs))()
    lb = (ctypes.c_float * len(offs))()
    mk.check(mk.mk_line_latency(8 << 20, offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(offs),
                                groups[0][1], groups[1][1], 8, la, lb), "mk_line_latency")
    a, b = np.array(la[:]), np.array(lb[:])
    d = a - b
    near_a = d < 0
    blocks = near_a.reshape(-1, 4).sum(axis=1)
    return {"sm_groups": [len(g) for g in groups], "probe_sms": [groups[0][1], groups[1][1]],
            "rtt_cycles_med_per_group": [float(np.median([rtt[i] for i in g if rtt[i] > 0])) for g in groups],
            "line_cycles_near_med": float(np.median(np.where(near_a, a, b))),
            "line_cycles_far_med": float(np.median(np.where(near_a, b, a))),
            "lines_near_first_sm": float(np.mean(near_a)),
            "kb_blocks_one_home": float(np.mean((blocks == 0) | (blocks == 4)))}


PARTS = {"barrier": part_barrier, "launch": part_launch, "batch512": part_batch512, "ctx32k": part_ctx32k, "ragged": part_ragged,
         "ctx8k": part_ctx8k, "prefill": part_prefill, "dies": part_dies}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", nargs="*", default=list(PARTS))
    ap.add_argument("--json", default="")
    args = ap.parse_args()
    import torch
    res = {}
    for name in args.only:
        res[name] = PARTS[name]()
        print(json.dumps({name: res[name]}), flush=True)
        torch.cuda.empty_cache()
    if args.json:
        with open(args.json, "w") as f:
            json.dump(res, f, indent=1)


if __name__ == "__main__":
    main()

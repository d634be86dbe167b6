"""Run a few decode steps of a workload for timing, tracing or an ncu capture.

    python -m persistent_sm_decode_megakernel_gb300.profile_step --workload 2b \
        [--layers L] [--prompt P] [--steps N] [--batch B] [--trace] [--sync counter|sentinel]
        [--exec persistent|multilaunch] [--page-bytes X] [--n-pages N] [--backoff NS]

Prints the per-step time (CUDA events on the context stream) and, with --trace, a
summary of the last step's instruction journal: per op, the mean time from fetch to
dependency-satisfied (waiting) and from there to the end (working), the per-CTA
waiting share of the step, the first op groups' start/end on the step's timeline, and
the per-layer dependency chain (chain_us: when each op's inputs were staged and when it
ended, after the previous layer's end, and the hop between consecutive ops).
The decode steps are preceded by exactly `prompt` launches of the same kernel (one per
prompt position), which is the count an ncu capture skips with -s.
"""
import argparse
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

OPS = {1: "embed", 2: "qkv", 3: "attn", 4: "reduce", 5: "oproj", 6: "upgate", 7: "down", 8: "lmhead", 9: "attn_pool"}


GEMV_OPS = (2, 5, 6, 7, 8)


def summarize(trace):
    """Per-op means of the journal's phases.  GEMV: stage (dependency satisfied -> inputs
    staged), pages (-> last page consumed; page_wait = the part spent waiting for pages to
    land), epi (-> outputs written), tail (-> end, the closing barrier).  Attention: stage,
    pages (page_wait: the part spent waiting for K, V pages), write (partial written), then
    arrive (the arrival) or merge (last arriver)."""
    t0 = min(r[4] for r in trace)
    t1 = max(r[6] for r in trace)
    span = (t1 - t0) / 1e3
    ctas = {r[0] for r in trace}
    by = {}
    per_cta_wait = {}
    groups = {}
    keys = ("stage", "pages", "page_wait", "page_work", "epi", "epi_cycles", "tail", "write", "arrive", "merge")
    for cta, pc, op, layer, tf, tr, te, m0, m1, m2, m3, m4, m5 in trace:
        d = by.setdefault(OPS.get(op, str(op)), {k: [] for k in ("wait", "work") + keys})
        d["wait"].append((tr - tf) / 1e3)
        d["work"].append((te - tr) / 1e3)
        if op in GEMV_OPS and m0 and m1:
            d["stage"].append((m0 - tr) / 1e3)
            d["pages"].append((m1 - m0) / 1e3)
            d["page_wait"].append(m2 / 1e3)
            d["page_work"].append(m4 / 1e3)
            if m3:
                d["epi"].append((m3 - m1) / 1e3)
                d["epi_cycles"].append(m5)         # SM clock cycles (the clock varies; not converted)
                d["tail"].append((te - m3) / 1e3)
        elif op == 3 and m0 and m1:
            d["stage"].append((m0 - tr) / 1e3)
            d["pages"].append((m1 - m0) / 1e3)
            d["page_wait"].append(m4 / 1e3)
            if m2:
                d["write"].append((m2 - m1) / 1e3)
                if m3:
                    d["merge"].append((m3 - m2) / 1e3)
                else:
                    d["arrive"].append((te - m2) / 1e3)
            else:
                d["epi"].append((te - m1) / 1e3)
        per_cta_wait[cta] = per_cta_wait.get(cta, 0.0) + (tr - tf) / 1e3
        g = groups.setdefault((layer, op), [tf, te])
        g[0] = min(g[0], tf)
        g[1] = max(g[1], te)
    out = {"span_us": span, "ops": {}}
    for k, d in by.items():
        out["ops"][k] = {"n": len(d["work"]), "wait_us_mean": statistics.mean(d["wait"]),
                         "work_us_mean": statistics.mean(d["work"]), "work_us_max": max(d["work"]),
                         "wait_us_per_cta": sum(d["wait"]) / len(ctas)}
        for key in keys:
            if d[key]:
                out["ops"][k][key if key.endswith("cycles") else key + "_us"] = statistics.mean(d[key])
    out["wait_share_mean"] = statistics.mean(v / span for v in per_cta_wait.values())
    items = sorted(groups.items(), key=lambda kv: kv[1][0])
    out["timeline_us"] = {f"L{l}:{OPS.get(o, o)}": [round((a - t0) / 1e3, 2), round((b - t0) / 1e3, 2)]
                          for (l, o), (a, b) in items[:20]}
    return out


CHAIN = (2, 3, 4, 5, 6, 7)  # one layer's ops in dependency order


def chain(trace):
    """The per-layer dependency chain from the journal: for each op of a layer, the time
    (us) after the previous layer's last down-projection CTA ended at which its CTAs had
    their inputs staged (median over CTAs; mark 0) and ended (median and max), and the hop
    -- the first CTA's staging done minus the previous op's last end.  Medians over the
    layers that have a previous layer.  Ops without a staging mark (the split merge) report
    ends only."""
    by = {}
    for r in trace:
        by.setdefault((r[3], r[2]), []).append(r)
    layers = sorted({l for (l, op) in by if op == 7})
    acc = {}
    for L in layers:
        if (L - 1, 7) not in by:
            continue
        ref = max(r[6] for r in by[(L - 1, 7)])
        prev_max = ref
        for op in CHAIN:
            rs = by.get((L, op))
            if not rs:
                continue
            ends = sorted(r[6] for r in rs)
            marks = sorted(r[7] for r in rs if r[7])
            d = acc.setdefault(OPS[op], {"staged": [], "end_med": [], "end_max": [], "hop": []})
            d["end_med"].append((statistics.median(ends) - ref) / 1e3)
            d["end_max"].append((ends[-1] - ref) / 1e3)
            if marks:
                d["staged"].append((statistics.median(marks) - ref) / 1e3)
                d["hop"].append((marks[0] - prev_max) / 1e3)
            prev_max = ends[-1]
    return {op: {k: round(statistics.median(v), 3) for k, v in d.items() if v} for op, d in acc.items()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="2b")
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--prompt", type=int, default=32)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--trace", action="store_true")
    ap.add_argument("--sync", default="counter", choices=["counter", "sentinel"])
    ap.add_argument("--exec", default="persistent", choices=["persistent", "multilaunch", "graph"])
    ap.add_argument("--page-bytes", type=int, default=0)
    ap.add_argument("--n-pages", type=int, default=0)
    ap.add_argument("--backoff", type=int, default=0)
    ap.add_argument("--merge", type=int, default=0, help="KV-split merge: 0 auto, 1 separate step, 2 in O-proj, 3 last-arriving split")
    ap.add_argument("--inflight", type=int, default=0, help="page copies in flight per CTA (0: default, <0: pool)")
    ap.add_argument("--split-min", type=int, default=0)
    ap.add_argument("--pool", type=int, default=0, help="attention units claimed from a per-layer pool")
    ap.add_argument("--kv-splits", type=int, default=0, help="KV splits per (sequence, kv head) in the schedule")
    ap.add_argument("--attn-tc", type=int, default=0,
                    help="tensor-core attention: 0 where it pays, 1 in every context, -1 never")
    ap.add_argument("--max-ctx", type=int, default=0, help="KV capacity (default: prompt + steps + 2)")
    ap.add_argument("--synthetic-kv", action="store_true",
                    help="fill the first --prompt cache positions with seeded synthetic keys/values instead of a prefill")
    ap.add_argument("--json", default="")
    args = ap.parse_args()

    import torch

    import synth
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel

    cfg = synth.CONFIGS[args.workload]
    if args.layers:
        cfg = synth.with_overrides(cfg, n_layers=args.layers)
    w = synth.gen_weights(cfg)
    B = args.batch
    dm = DeviceModel(cfg, w, max_batch=B, max_ctx=max(args.max_ctx, args.prompt + args.steps + 2))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dec = Decoder(dm, sync_mode=0 if args.sync == "counter" else 1,
                      exec_mode={"persistent": 0, "multilaunch": 1, "graph": 2}[args.exec], trace=1 if args.trace else 0,
                      page_bytes=args.page_bytes, n_pages=args.n_pages, backoff_max_ns=args.backoff,
                      kv_splits=args.kv_splits,
                      split_min_positions=args.split_min, attn_merge=args.merge,
                      inflight_pages=args.inflight, attn_pool=args.pool, attn_tensor_cores=args.attn_tc,
                      stream=stream)
        prompt = synth.gen_prompts(cfg, B, args.prompt)
        if args.synthetic_kv:
            for l in range(cfg.n_layers):
                for b in range(B):
                    dm.set_kv(l, b, synth.gen_kv(cfg, l, b, 0, args.prompt), synth.gen_kv(cfg, l, b, 1, args.prompt))
            tok = prompt[:, -1]
        else:
            tok = dec.prefill(prompt)
        pos = args.prompt
        times = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            tok = dec.decode_step(tok, [pos] * B)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
            pos += 1
        res = {"workload": args.workload, "layers": cfg.n_layers, "step_us": times, "info": dec.info()}
        if args.trace:
            tr = dec.trace()
            res["trace"] = summarize(tr)
            res["chain_us"] = chain(tr)
        dec.close()
    print(json.dumps(res, indent=1))
    if args.json:
        with open(args.json, "w") as f:
            json.dump(res, f, indent=1)


if __name__ == "__main__":
    main()

"""Writes tests/golden/tiny_greedy.json from the fp64 oracle alone.

Fixture: the tiny workload (2 layers, d 256, 4/2 heads of 64, FFN 768, vocab 1024,
bf16, seed 0), batch 1, its 16-token seeded prompt, 32 greedy tokens.  The pages print
no worked example, so this fixture pins the oracle against accidental change only.
Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
import synth  # noqa: E402


def main():
    cfg = synth.CONFIGS["tiny"]
    m = O.Model(cfg, synth.gen_weights(cfg))
    P, n_new = cfg.prompt_len, cfg.decode_len
    p = synth.gen_prompts(cfg, 1, P)
    toks, logits = O.greedy_generate(m, p, n_new)
    out = {
        "source": "oracle/decoder.py greedy_generate on the tiny workload (seed 0)",
        "prompt_len": P, "n_new": n_new,
        "prompt": p[0].tolist(),
        "tokens": toks[0].tolist(),
        "logits_head": [[float(x) for x in row] for row in logits[0, :, :8]],
        "margin": [float(x) for x in O.top2_margin(logits[0])],
    }
    with open(os.path.join(HERE, "tiny_greedy.json"), "w") as f:
        json.dump(out, f, indent=0)


if __name__ == "__main__":
    main()

"""Shared helpers of the GPU parity tests: oracle runs under teacher forcing and the
parity criteria (per-step logits within 1e-2 of the oracle's largest |logit|; greedy
tokens identical wherever the oracle's top-2 margin exceeds that tolerance)."""
import numpy as np

import oracle

LOGIT_RTOL = 1e-2


def oracle_run(cfg, weights, prompt, n_new, model=None):
    """Oracle prefill of the prompt, then n_new - 1 greedy decode steps.
    Returns tokens [B, P + n_new] and logits [B, n_new, V] where logits[:, k] is the step
    that consumed the token at position P - 1 + k."""
    m = model or oracle.Model(cfg, weights)
    B, P = prompt.shape
    cache = oracle.KVCache(cfg, B, P + n_new)
    zp = oracle.prefill(m, prompt, cache)
    toks = np.zeros((B, P + n_new), dtype=np.int64)
    toks[:, :P] = prompt
    logits = [zp[:, -1]]
    toks[:, P] = oracle.argmax_lowest(zp[:, -1])
    for t in range(P, P + n_new - 1):
        z = oracle.decode_step(m, cache, toks[:, t], [t] * B)
        logits.append(z)
        toks[:, t + 1] = oracle.argmax_lowest(z)
    return toks, np.stack(logits, axis=1)


def gpu_teacher_forced(dec, prompt, toks, n_new, vocab):
    """GPU prefill of the prompt, then decode steps fed the oracle's tokens.
    Returns logits [B, n_new, V] and the GPU's greedy tokens [B, n_new]."""
    import torch
    B, P = prompt.shape
    logits = torch.zeros((B, vocab), dtype=torch.float32, device=dec.dm.device)
    out = [dec.prefill(prompt, logits=logits)]
    z = [logits.cpu().numpy()]
    for t in range(P, P + n_new - 1):
        out.append(dec.decode_step(toks[:, t], [t] * B, logits=logits))
        z.append(logits.cpu().numpy())
    return np.stack(z, axis=1), np.stack(out, axis=1)


def assert_parity(z_gpu, tok_gpu, z_ref, toks_ref, P):
    """Logits within LOGIT_RTOL of the oracle's largest |logit| and the greedy token equal
    to the oracle's wherever its top-2 margin exceeds that tolerance, step by step and
    sequence by sequence."""
    B, n, V = z_ref.shape
    worst = 0.0
    for b in range(B):
        for k in range(n):
            tol = LOGIT_RTOL * np.abs(z_ref[b, k]).max()
            err = np.abs(z_gpu[b, k] - z_ref[b, k]).max()
            worst = max(worst, err / np.abs(z_ref[b, k]).max())
            assert err <= tol, f"seq {b} step {k}: max |dlogit| {err:.3e} > {tol:.3e}"
            if oracle.top2_margin(z_ref[b, k]) > tol:
                assert tok_gpu[b, k] == toks_ref[b, P + k], f"seq {b} step {k}: token {tok_gpu[b, k]} != {toks_ref[b, P + k]}"
    return worst

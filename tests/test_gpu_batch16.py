"""Batches of 3 to 16 sequences on the tensor-core GEMV path, against the oracle.

Every GEMV of a 3..16-sequence step runs with
mma.sync on 16-row weight blocks, its inputs split into hi/lo 16-bit halves (both the
fp16 and the bf16 instances); batches of 1 and 2 in the same context keep the CUDA-core
path.  Teacher forcing, per-step logits within 1e-2 of the oracle's largest |logit|.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_parity, gpu_teacher_forced, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from persistent_sm_decode_megakernel_gb300 import model
    return model


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_weights(cfg)
    return cfg, w, oracle.Model(cfg, w)


@pytest.mark.parametrize("B", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_tiny_batches_in_a_batch16_context(lib, tiny, B, sync):
    cfg, w, m = tiny
    P, n_new = 12, 6
    prompt = synth.gen_prompts(cfg, B, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    dm = lib.DeviceModel(cfg, w, max_batch=16, max_ctx=P + n_new)
    dec = lib.Decoder(dm, sync_mode=sync)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


def test_tiny_ragged_batch16(lib, tiny):
    """16 sequences at different positions: each continues its own prompt."""
    cfg, w, m = tiny
    B, P = 16, 14
    prompt = synth.gen_prompts(cfg, B, P)
    dm = lib.DeviceModel(cfg, w, max_batch=16, max_ctx=P + 2)
    dec = lib.Decoder(dm)
    # sequence b has consumed P - (b % 5) prompt tokens before the step
    lens = [P - (b % 5) for b in range(B)]
    import torch
    logits = torch.zeros((B, cfg.vocab), dtype=torch.float32, device=dm.device)
    for t in range(max(lens)):
        active = [b for b in range(B) if t < lens[b]]
        # steps run for the whole batch; sequences past their length repeat their last
        # position with the same token (the cache entry is rewritten with the same value)
        toks = [int(prompt[b, min(t, lens[b] - 1)]) for b in range(B)]
        pos = [min(t, lens[b] - 1) for b in range(B)]
        dec.decode_step(toks, pos, logits=logits)
    z = logits.cpu().numpy()
    dec.close()
    for b in (0, 3, 9, 15):
        cache = oracle.KVCache(cfg, 1, P + 2)
        zr = None
        for t in range(lens[b]):
            zr = oracle.decode_step(m, cache, [prompt[b, t]], [t])[0]
        scale = np.abs(zr).max()
        assert np.abs(z[b] - zr).max() <= 1e-2 * scale, f"seq {b}"


def test_2b_batch8_short_prompt(lib):
    cfg = synth.CONFIGS["2b"]
    w = synth.gen_weights(cfg)
    B, P, n_new = 8, 16, 3
    prompt = synth.gen_prompts(cfg, B, P)
    m = oracle.Model(cfg, w)
    toks, zref = oracle_run(cfg, w, prompt[[0, 7]], n_new, model=m)
    # the GPU runs all 8; sequences 0 and 7 are teacher-forced with the oracle's tokens,
    # the others with their own prompt continuation (any valid token stream)
    full = np.zeros((B, P + n_new), dtype=np.int64)
    full[:, :P] = prompt
    full[0], full[7] = toks[0], toks[1]
    for b in range(1, 7):
        full[b, P:] = synth.gen_prompt(cfg, 100 + b, n_new)
    dm = lib.DeviceModel(cfg, w, max_batch=8, max_ctx=P + n_new)
    dec = lib.Decoder(dm)
    z, tg = gpu_teacher_forced(dec, prompt, full, n_new, cfg.vocab)
    dec.close()
    assert_parity(z[[0, 7]], tg[[0, 7]], zref, toks, P)

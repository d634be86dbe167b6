"""Parity on the two largest workloads, at their full model dimensions.

* 8b: the bf16 model with 32 layers, d 4096, 32/8 heads, FFN 14336 and vocab 128256.
  (a) A 32-token prompt goes through mk_prefill, then teacher-forced decode steps follow;
  the same at batch 4 (the tensor-core GEMV) under both syncs.
  (b) The workload's own context: 8192 cached positions per sequence (seeded synthetic
  keys and values, synth.gen_kv, the same bytes on both sides -- an 8192-token fp64
  prefill of the 8b model would take the oracle hours), then two teacher-forced decode
  steps at batch 1 and 2 under counter and sentinel sync.  With four query heads per kv
  head and ~431 positions per split, every split runs the grouped attention instance's
  four-pass chunks.
* 2b at 32k context: the 2b fp16 model with 32768 cached positions per sequence, at
  batch 1, 2, 4, 8 and 16 (3..16 on the tensor-core GEMV).  The cache holds seeded synthetic keys and values (synth.gen_kv, the
  same bytes on both sides) instead of a 32k-token prefill, which the oracle cannot run
  in test time.  The oracle checks sequences 0, 1, 3, 7 and 15 one at a time.  Every sequence
  of a batch must also match that sequence at the smallest batch that holds it
  (batch invariance).  The same cache is decoded by the persistent kernel with counter
  sync (every batch), with NaN-sentinel sync and by the multi-launch control (batches 1
  and 8), and with the attention units claimed from a pool (batches 8 and 16); the token
  mk_decode_step returns is checked against the oracle's argmax.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import LOGIT_RTOL, assert_parity, gpu_teacher_forced, oracle_run

pytestmark = pytest.mark.gpu


class _UncachedModel(oracle.Model):
    """The oracle model without its fp64 weight cache (the 8b model's fp64 weights
    would take 64 GB of host memory); each lookup upcasts again."""

    def w(self, name, layer=-1):
        src = self._bits[name] if layer < 0 else self._bits["layers"][layer][name]
        return oracle.upcast(src, self.dtype)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from persistent_sm_decode_megakernel_gb300 import model
    return model


def test_8b_teacher_forced(lib):
    cfg = synth.CONFIGS["8b"]
    w = synth.gen_weights(cfg)
    P, n_new = 32, 3
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=_UncachedModel(cfg, w))
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + n_new)
    dec = lib.Decoder(dm)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


@pytest.fixture(scope="module")
def b4_8b(lib):
    """The 8b model at batch 4: an 8-token prompt per sequence, three teacher-forced steps."""
    cfg = synth.CONFIGS["8b"]
    w = synth.gen_weights(cfg)
    P, n_new = 8, 3
    prompt = synth.gen_prompts(cfg, 4, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=_UncachedModel(cfg, w))
    return cfg, w, prompt, toks, zref, P, n_new


@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_8b_batch4_teacher_forced(b4_8b, lib, sync):
    """bf16 on the tensor-core GEMV at the 8b widths: d 4096 does not fit the x buffer whole,
    so every GEMV stages window by window (double-buffered bulk copies with counters, three
    windows per polled staging with sentinels) and the down projection walks 14 windows."""
    cfg, w, prompt, toks, zref, P, n_new = b4_8b
    dm = lib.DeviceModel(cfg, w, max_batch=4, max_ctx=P + n_new)
    dec = lib.Decoder(dm, sync_mode=sync)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    del dm
    assert_parity(z, tg, zref, toks, P)


T8K = synth.CONFIGS["8b"].prompt_len          # 8192 cached positions
N8 = 2                                         # decode steps per sequence


@pytest.fixture(scope="module")
def ctx_8k(lib):
    """Device model for two sequences with 8192 cached positions each, the teacher-forced
    tokens, and the oracle's logits [2, N8, V] (both sequences in one oracle call per step)."""
    cfg = synth.CONFIGS["8b"]
    w = synth.gen_weights(cfg)
    m = _UncachedModel(cfg, w)
    dm = lib.DeviceModel(cfg, w, max_batch=2, max_ctx=T8K + N8 + 1)
    cache = oracle.KVCache(cfg, 2, T8K + N8)
    for b in range(2):
        for l in range(cfg.n_layers):
            kb = synth.gen_kv(cfg, l, b, 0, T8K)
            vb = synth.gen_kv(cfg, l, b, 1, T8K)
            dm.set_kv(l, b, kb, vb)
            cache.k[l][b, :, :T8K] = oracle.upcast(kb, cfg.dtype)
            cache.v[l][b, :, :T8K] = oracle.upcast(vb, cfg.dtype)
    toks = np.stack([synth.gen_prompt(cfg, b, N8) for b in range(2)])
    zref = np.stack([oracle.decode_step(m, cache, toks[:, t], [T8K + t] * 2) for t in range(N8)], axis=1)
    del cache
    return cfg, dm, toks, zref


@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
@pytest.mark.parametrize("B", [1, 2])
def test_8b_at_8k_context(ctx_8k, lib, B, sync):
    cfg, dm, toks, zref = ctx_8k
    dec = lib.Decoder(dm, sync_mode=sync)
    logits = torch.zeros((B, cfg.vocab), dtype=torch.float32, device=dm.device)
    for t in range(N8):
        # every run rewrites positions T8K + t of its sequences with the same values
        got = dec.decode_step(toks[:B, t], [T8K + t] * B, logits=logits)
        z = logits.cpu().numpy()
        for b in range(B):
            zr = zref[b, t]
            scale = np.abs(zr).max()
            err = np.abs(z[b] - zr).max()
            assert err <= LOGIT_RTOL * scale, f"seq {b} step {t}: max |dlogit| {err:.3e}"
            if oracle.top2_margin(zr) > LOGIT_RTOL * scale:
                assert got[b] == int(np.argmax(zr)), f"seq {b} step {t}: token {got[b]} != {int(np.argmax(zr))}"
    dec.close()


T32K = synth.CONFIGS["2b-32k"].prompt_len     # 32768 cached positions
N_STEPS = 2
CHECKED = (0, 1, 3, 7, 15)                     # sequences the oracle decodes
MAXB = 16


@pytest.fixture(scope="module")
def long_ctx(lib):
    """Device model for 16 sequences with every sequence's 32k cache filled, the
    teacher-forced tokens, and the oracle's logits [N_STEPS, V] for the checked sequences."""
    cfg = synth.CONFIGS["2b-32k"]
    w = synth.gen_weights(cfg)
    m = oracle.Model(cfg, w)
    dm = lib.DeviceModel(cfg, w, max_batch=MAXB, max_ctx=T32K + N_STEPS + 1)
    toks = np.stack([synth.gen_prompt(cfg, b, N_STEPS) for b in range(MAXB)])
    zref = {}
    for b in range(MAXB):
        cache = oracle.KVCache(cfg, 1, T32K + N_STEPS) if b in CHECKED else None
        for l in range(cfg.n_layers):
            kb = synth.gen_kv(cfg, l, b, 0, T32K)
            vb = synth.gen_kv(cfg, l, b, 1, T32K)
            dm.set_kv(l, b, kb, vb)
            if cache is not None:
                cache.k[l][0, :, :T32K] = oracle.upcast(kb, cfg.dtype)
                cache.v[l][0, :, :T32K] = oracle.upcast(vb, cfg.dtype)
        if cache is not None:
            zref[b] = np.stack([oracle.decode_step(m, cache, [toks[b, t]], [T32K + t])[0] for t in range(N_STEPS)])
            del cache
    return cfg, dm, toks, zref, {}


# (batch, sync, exec, attention pool)
ARMS = [(B, 0, 0, 0) for B in (1, 2, 4, 8, 16)] + [(1, 1, 0, 0), (8, 1, 0, 0), (1, 0, 1, 0), (8, 0, 1, 0),
                                                   (8, 0, 0, 1), (16, 1, 0, 1)]


@pytest.mark.parametrize("B,sync,execm,pool", ARMS,
                         ids=[f"B{b}-{'sentinel' if s else 'counter'}-{'multilaunch' if e else 'persistent'}"
                              f"{'-pool' if q else ''}" for b, s, e, q in ARMS])
def test_2b_32k_context_batches(long_ctx, lib, B, sync, execm, pool):
    cfg, dm, toks, zref, seen = long_ctx
    dec = lib.Decoder(dm, sync_mode=sync, exec_mode=execm, attn_pool=pool)
    logits = torch.zeros((B, cfg.vocab), dtype=torch.float32, device=dm.device)
    z, tk = [], []
    for t in range(N_STEPS):
        # every run rewrites positions T32K + t of its sequences with the same values
        tk.append(dec.decode_step(toks[:B, t], [T32K + t] * B, logits=logits))
        z.append(logits.cpu().numpy().copy())
    dec.close()
    z = np.stack(z, axis=1)                                   # [B, N_STEPS, V]
    tk = np.stack(tk, axis=1)                                 # [B, N_STEPS] returned tokens
    for b in range(B):
        if b in zref:
            for t in range(N_STEPS):
                zr = zref[b][t]
                scale = np.abs(zr).max()
                err = np.abs(z[b, t] - zr).max()
                assert err <= LOGIT_RTOL * scale, f"seq {b} step {t}: max |dlogit| {err:.3e}"
                if oracle.top2_margin(zr) > LOGIT_RTOL * scale:
                    assert tk[b, t] == np.argmax(zr), f"seq {b} step {t}: token {tk[b, t]} != {np.argmax(zr)}"
        if b in seen:      # the same sequence at a smaller batch
            assert np.abs(z[b] - seen[b]).max() <= 1e-3 * np.abs(seen[b]).max(), f"seq {b}: batch variance"
        else:
            seen[b] = z[b]

"""Parity of the CUDA decode path with the fp64 oracle, through the C ABI.

Ladder steps 5-7 of "8 · Écrire son megakernel", §8.6: one real instruction (RMSNorm
inside RMSNORM_QKV_ROPE, checked through q), every instruction of a layer (per-layer
intermediates), and the whole model under teacher forcing.  Logits must stay within
1e-2 of the oracle's largest |logit| per step; greedy tokens must match wherever the
oracle's top-2 margin exceeds that.  Intermediates are held to a tighter bound,
2e-3 of the tensor's largest magnitude: fp32 accumulation against fp64 differs by
~1e-6 relative, and a cached key/value that falls on the other side of a bf16/fp16
rounding boundary moves one entry by one storage ulp (2^-8 relative for bf16), which
shifts an attention output by far less than that bound."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, gpu_teacher_forced, oracle_run

pytestmark = pytest.mark.gpu
INTER_RTOL = 2e-3


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


def _close(got, want, rtol=INTER_RTOL, what=""):
    scale = np.abs(want).max()
    err = np.abs(got - want).max()
    assert err <= rtol * scale, f"{what}: max err {err:.3e} > {rtol:.0e} * {scale:.3e}"
    return err / scale


@pytest.mark.parametrize("sync,execm", [(0, 0), (1, 0), (0, 1), (0, 2), (1, 2)],
                         ids=["counter", "sentinel", "multilaunch", "graph", "graph-sentinel"])
def test_tiny_full_model_teacher_forced(lib, tiny, sync, execm):
    cfg, w, m = tiny
    P, n_new = cfg.prompt_len, cfg.decode_len
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + n_new)
    dec = lib.Decoder(dm, sync_mode=sync, exec_mode=execm)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    worst = assert_parity(z, tg, zref, toks, P)
    assert worst < 1e-3


def test_tiny_layer_intermediates(lib, tiny):
    """Ladder steps 5 and 6: the RMSNorm-QKV-RoPE output q, the attention output o,
    h after attention, the MLP activation and h after each layer, one decode step."""
    cfg, w, m = tiny
    P = 12
    prompt = synth.gen_prompts(cfg, 1, P + 1)
    cache = oracle.KVCache(cfg, 1, P + 1)
    oracle.prefill(m, prompt[:, :P], cache)
    z, trace = oracle.decode_step(m, cache, prompt[:, P], [P], keep=True)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + 1)
    dec = lib.Decoder(dm)
    dec.prefill(prompt[:, :P])
    dec.decode_step(prompt[:, P], [P])
    for l in range(cfg.n_layers):
        r = trace[l]
        _close(dec.read_activation(2, l)[0], r["q"][0].reshape(-1), what=f"q layer {l}")
        _close(dec.read_activation(3, l)[0], r["o"][0].reshape(-1), what=f"o layer {l}")
        _close(dec.read_activation(1, l)[0], r["h_mid"][0], what=f"h_mid layer {l}")
        _close(dec.read_activation(4, l)[0], r["a"][0], what=f"a layer {l}")
        _close(dec.read_activation(0, l + 1)[0], r["h_out"][0], what=f"h layer {l}")
    # the cache holds the rotated key of the new position, rounded like the oracle's
    k_gpu = dm.k_cache[0][0, :, P].cpu().numpy().view(np.uint16)
    k_ref = cache.k[0][0, :, P]
    got = oracle.upcast(k_gpu, cfg.dtype)
    _close(got, k_ref, what="new key in the cache")
    dec.close()


@pytest.mark.parametrize("B", [2, 4])
def test_tiny_batched(lib, tiny, B):
    cfg, w, m = tiny
    P, n_new = 10, 8
    prompt = synth.gen_prompts(cfg, B, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    dm = lib.DeviceModel(cfg, w, max_batch=4, max_ctx=P + n_new)
    dec = lib.Decoder(dm)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


def test_tiny_ragged_positions(lib, tiny):
    """Sequences of a batch at different positions in the same step."""
    cfg, w, m = tiny
    lag = 5
    seqs = synth.gen_prompts(cfg, 2, 20)
    dm = lib.DeviceModel(cfg, w, max_batch=2, max_ctx=32)
    dec = lib.Decoder(dm)
    cache = oracle.KVCache(cfg, 2, 32)
    logits = torch.zeros((2, cfg.vocab), dtype=torch.float32, device=dm.device)
    for t in range(lag):                    # sequence 0 alone (batch slot 0)
        dec.decode_step([seqs[0, t]], [t])
    cache0 = oracle.KVCache(cfg, 1, 32)
    for t in range(lag):
        oracle.decode_step(m, cache0, [seqs[0, t]], [t])
    for l in range(cfg.n_layers):
        cache.k[l][0] = cache0.k[l][0]
        cache.v[l][0] = cache0.v[l][0]
    for t in range(8):                      # both sequences, positions t + lag and t
        pos = [t + lag, t]
        tok = [seqs[0, t + lag], seqs[1, t]]
        dec.decode_step(tok, pos, logits=logits)
        zr = oracle.decode_step(m, cache, tok, pos)
        zg = logits.cpu().numpy()
        for b in range(2):
            assert np.abs(zg[b] - zr[b]).max() <= 1e-2 * np.abs(zr[b]).max()
    dec.close()


def test_tiny_deterministic(lib, tiny):
    """Same inputs, same bits: no atomics in any floating-point reduction."""
    cfg, w, m = tiny
    prompt = synth.gen_prompts(cfg, 1, 12)
    outs = []
    for _ in range(2):
        dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=16)
        dec = lib.Decoder(dm)
        logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device=dm.device)
        dec.prefill(prompt, logits=logits)
        outs.append(logits.cpu().numpy().copy())
        dec.close()
    np.testing.assert_array_equal(outs[0], outs[1])


def test_chained_decode_matches_stepwise(lib, tiny):
    """mk_decode_steps (device-fed tokens, no host round trip) == greedy step by step."""
    cfg, w, m = tiny
    P, n = 8, 12
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, _ = oracle_run(cfg, w, prompt, n + 1, model=m)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + n + 1)
    dec = lib.Decoder(dm)
    first = dec.prefill(prompt)
    out = torch.zeros((n, 1), dtype=torch.int32, device=dm.device)
    dec.decode_steps(first, [P], n, out)
    dec.synchronize()
    got = out.cpu().numpy()[:, 0]
    dec.close()
    assert first[0] == toks[0, P]
    np.testing.assert_array_equal(got, toks[0, P + 1: P + 1 + n])


@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
@pytest.mark.parametrize("B", [1, 2, 4])
def test_multi_step_launch_matches_single_step_launches(lib, tiny, sync, B):
    """n greedy steps in ONE persistent launch (the kernel walks its queue once per step,
    each step waiting for the tokens the step before published) give the same tokens and
    the same last-step activations, bit for bit, as n launches of one step each."""
    cfg, w, m = tiny
    P, n = 6, 9
    prompt = synth.gen_prompts(cfg, B, P)
    runs = []
    for one_launch in (True, False):
        dm = lib.DeviceModel(cfg, w, max_batch=B, max_ctx=P + n + 1)
        dec = lib.Decoder(dm, sync_mode=sync)
        first = dec.prefill(prompt)
        out = torch.zeros((n, B), dtype=torch.int32, device=dm.device)
        if one_launch:
            dec.decode_steps(first, [P] * B, n, out)
        else:
            for k in range(n):
                dec.decode_steps(first if k == 0 else None, [P + k] * B, 1, out[k:k + 1])
        dec.synchronize()
        h = dec.read_activation(0, cfg.n_layers)   # the final residual stream of the last step
        runs.append((first, out.cpu().numpy().copy(), h))
        dec.close()
    assert list(runs[0][0]) == list(runs[1][0])
    np.testing.assert_array_equal(runs[0][1], runs[1][1])
    np.testing.assert_array_equal(runs[0][2], runs[1][2])
    # and the chain is the oracle's greedy chain for sequence 0
    toks, _ = oracle_run(cfg, w, prompt[:1], n + 1, model=m)
    np.testing.assert_array_equal(runs[0][1][:, 0], toks[0, P + 1: P + 1 + n])


@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_host_token_steps_match_device_chain(lib, tiny, sync):
    """mk_decode_step without logits (tokens come back through the mapped host mailbox, no
    copy or stream sync) returns the same greedy chain as device-fed steps, and a step with
    logits (the synchronous path) in the middle of it changes nothing."""
    cfg, w, m = tiny
    P, n = 5, 10
    prompt = synth.gen_prompts(cfg, 2, P)
    dm = lib.DeviceModel(cfg, w, max_batch=2, max_ctx=P + n + 1)
    dec = lib.Decoder(dm, sync_mode=sync)
    first = dec.prefill(prompt)
    out = torch.zeros((n, 2), dtype=torch.int32, device=dm.device)
    dec.decode_steps(first, [P] * 2, n, out)
    dec.synchronize()
    want = out.cpu().numpy()
    dec.close()
    dm2 = lib.DeviceModel(cfg, w, max_batch=2, max_ctx=P + n + 1)
    dec2 = lib.Decoder(dm2, sync_mode=sync)
    tok = dec2.prefill(prompt)
    got = []
    logits = torch.zeros((2, cfg.vocab), dtype=torch.float32, device=dm2.device)
    for k in range(n):
        tok = dec2.decode_step(tok, [P + k] * 2, logits=logits if k == 4 else None)
        got.append(list(tok))
    dec2.close()
    np.testing.assert_array_equal(np.array(got), want)


def test_fault_injection_times_out_and_recovers(lib, tiny):
    """A dropped counter signal (injected on the host, validator skipped) makes a device
    wait run out: the step returns MK_ERR_TIMEOUT within the limit, the context refuses
    work until mk_reset, and the GPU stays usable."""
    from persistent_sm_decode_megakernel_gb300 import MK_ERR_STATE, MK_ERR_TIMEOUT
    cfg, w, m = tiny
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=8)
    dec = lib.Decoder(dm, timeout_s=0.2, fault_drop_signal=7)
    st, _ = dec.decode_step_status([1], [0])
    assert st == MK_ERR_TIMEOUT
    st, _ = dec.decode_step_status([1], [0])
    assert st == MK_ERR_STATE
    dec.reset()
    dec.close()
    # the device still runs a correct step afterwards
    dec = lib.Decoder(dm)
    logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device=dm.device)
    dec.decode_step([3], [0], logits=logits)
    cache = oracle.KVCache(cfg, 1, 8)
    zr = oracle.decode_step(m, cache, [3], [0])
    assert np.abs(logits.cpu().numpy() - zr).max() <= 1e-2 * np.abs(zr).max()
    dec.close()


def test_small_page_pool_and_splits(lib, tiny):
    """Geometry variants: 8 KB pages, 2-page pool, 3 KV splits, 5 CTAs -- the ring wraps
    constantly and many instructions share a CTA."""
    cfg, w, m = tiny
    P, n_new = 9, 5
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + n_new)
    dec = lib.Decoder(dm, page_bytes=8192, n_pages=2, kv_splits=3, max_ctas=5)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


def test_half_billion_teacher_forced(lib):
    cfg = synth.CONFIGS["0.5b"]
    w = synth.gen_weights(cfg)
    P, n_new = cfg.prompt_len, 6
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + n_new)
    dec = lib.Decoder(dm)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


def test_2b_fp16_full_prompt_teacher_forced(lib):
    """The benchmarked workload's model and launch configuration: 2B fp16, 512-token
    prompt through mk_prefill, then teacher-forced decode steps."""
    cfg = synth.CONFIGS["2b"]
    w = synth.gen_weights(cfg)
    P, n_new = cfg.prompt_len, 4
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + n_new)
    dec = lib.Decoder(dm)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


@pytest.mark.parametrize("page_bytes", [0, 8192])
@pytest.mark.parametrize("merge", [1, 2, 3], ids=["merge-step", "merge-in-oproj", "merge-last-arriver"])
def test_tiny_long_context_many_splits(lib, tiny, page_bytes, merge):
    """A 600-position context: the step uses several KV splits (one page of positions
    each, up to the schedule's count), merged in a separate step (the ATTN_REDUCE op with
    sentinels, the last-arriving split with counters), inside the O-proj staging, or by the
    last-arriving split under either synchronisation."""
    cfg, w, m = tiny
    P, n_new = 600, 4
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    for sync in (0, 1):
        dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + n_new)
        dec = lib.Decoder(dm, sync_mode=sync, page_bytes=page_bytes, attn_merge=merge)
        z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
        dec.close()
        assert_parity(z, tg, zref, toks, P)


@pytest.mark.parametrize("B", [2, 5, 11])
@pytest.mark.parametrize("merge", [1, 2, 3], ids=["merge-step", "merge-in-oproj", "merge-last-arriver"])
@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_tiny_batched_merge_modes(lib, tiny, merge, sync, B):
    """Batches 2 (CUDA-core GEMV), 5 and 11 (tensor-core GEMV with one and two tiles of 8
    sequences, three and five of them empty; O-proj input in fragment form from the merge)
    under every split-merge placement."""
    cfg, w, m = tiny
    P, n_new = cfg.prompt_len, 6
    prompt = synth.gen_prompts(cfg, B, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    dm = lib.DeviceModel(cfg, w, max_batch=B, max_ctx=P + n_new)
    dec = lib.Decoder(dm, sync_mode=sync, attn_merge=merge)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


@pytest.mark.parametrize("kv_splits", [2, 3])
@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_tiny_g4_long_context_chunked(lib, sync, kv_splits):
    """Four query heads per kv head (the 8b model's group) at a 600-position context with
    few, long splits: each split's block holds more than two passes of positions, so the
    grouped attention instance takes its four-pass chunks (and, with two splits, a second
    block and single-pass tail)."""
    cfg = synth.CONFIGS["tiny-g4"]
    w = synth.gen_weights(cfg)
    m = oracle.Model(cfg, w)
    P, n_new = cfg.prompt_len, cfg.decode_len
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + n_new)
    dec = lib.Decoder(dm, sync_mode=sync, kv_splits=kv_splits)
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
@pytest.mark.parametrize("B", [1, 4])
def test_attention_pool_matches_static_units(lib, tiny, sync, B):
    """Dynamic work queue of the attention units (§8.8: each CTA's loader claims units of
    the layer's pool as its ring frees): a unit computes the same thing on whichever CTA
    claims it and the split merge keeps its fixed order, so the logits equal the static
    placement's bit for bit -- at a 600-position context (many splits per sequence and
    head), at batch 1 and 4 -- and match the oracle."""
    cfg, w, m = tiny
    P, n = 600, 3
    seqs = synth.gen_prompts(cfg, B, P + n)
    zs = []
    for pool in (0, 1):
        dm = lib.DeviceModel(cfg, w, max_batch=B, max_ctx=P + n + 1)
        dec = lib.Decoder(dm, sync_mode=sync, attn_pool=pool)
        dec.prefill(seqs[:, :P])
        logits = torch.zeros((B, cfg.vocab), dtype=torch.float32, device=dm.device)
        z = []
        for t in range(n):
            dec.decode_step(seqs[:, P + t], [P + t] * B, logits=logits)
            z.append(logits.cpu().numpy().copy())
        dec.close()
        zs.append(np.stack(z))
    np.testing.assert_array_equal(zs[0], zs[1])
    cache = oracle.KVCache(cfg, B, P + n)
    oracle.prefill(m, seqs[:, :P], cache)
    for t in range(n):
        zr = oracle.decode_step(m, cache, seqs[:, P + t], [P + t] * B)
        for b in range(B):
            assert np.abs(zs[1][t, b] - zr[b]).max() <= 1e-2 * np.abs(zr[b]).max()


@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_attention_pool_multi_step_launch(lib, tiny, sync):
    """Several greedy steps in one launch with the attention pool: the loader's claims of a
    later step count against that step's epoch while the compute warps finish the one
    before; the tokens equal those of one launch per step."""
    cfg, w, m = tiny
    P, n, B = 40, 7, 2
    prompt = synth.gen_prompts(cfg, B, P)
    runs = []
    for one_launch in (True, False):
        dm = lib.DeviceModel(cfg, w, max_batch=B, max_ctx=P + n + 1)
        dec = lib.Decoder(dm, sync_mode=sync, attn_pool=1)
        first = dec.prefill(prompt)
        out = torch.zeros((n, B), dtype=torch.int32, device=dm.device)
        if one_launch:
            dec.decode_steps(first, [P] * B, n, out)
        else:
            for k in range(n):
                dec.decode_steps(first if k == 0 else None, [P + k] * B, 1, out[k:k + 1])
        dec.synchronize()
        runs.append(out.cpu().numpy().copy())
        dec.close()
    np.testing.assert_array_equal(runs[0], runs[1])

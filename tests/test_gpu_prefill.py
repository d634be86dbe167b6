"""mk_prefill in prompt chunks against the fp64 oracle's batched causal prefill.

A chunk is one launch of the persistent kernel over up to 16 rows -- consecutive positions
of each prompt -- on the tensor-core GEMV; every row attends to the cached positions below
its chunk and to the chunk's rows up to its own ("7 · AMD et le monokernel", §7.1: the
prefill runs in the same persistent kernel as the decode steps).  Checked: the last
position's logits (1e-2 of the oracle's largest |logit|), the returned greedy token where
the oracle's top-2 margin exceeds that tolerance, and every cached key and value the
prefill wrote: each within one storage ulp of the oracle's (an entry whose fp32 value
falls on the other side of a rounding boundary from the fp64 value moves by one ulp) plus
1e-3 of the largest magnitude (near zero the ulp is tiny and the arithmetic's own error
shows: the tensor-core GEMV carries its inputs as hi/lo 16-bit halves, ~16 significant
bits).  Ragged cases:
a prompt that is not a multiple of the chunk, and three sequences (five positions of each
per chunk).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import LOGIT_RTOL

pytestmark = pytest.mark.gpu
ULP_REL = {"bf16": 2.0 ** -7, "f16": 2.0 ** -10}   # one storage ulp, relative, at most


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from persistent_sm_decode_megakernel_gb300 import model
    return model


def _check(lib, name, B, P, sync, layers=None, max_batch=None):
    cfg = synth.CONFIGS[name]
    w = synth.gen_weights(cfg)
    prompt = synth.gen_prompts(cfg, B, P)
    m = oracle.Model(cfg, w)
    cache = oracle.KVCache(cfg, B, P)
    zref = oracle.prefill(m, prompt, cache)[:, -1]                  # [B, V]
    dm = lib.DeviceModel(cfg, w, max_batch=max_batch or B, max_ctx=P + 1)
    dec = lib.Decoder(dm, sync_mode=sync)
    logits = torch.zeros((B, cfg.vocab), dtype=torch.float32, device=dm.device)
    tok = dec.prefill(prompt, logits=logits)
    z = logits.cpu().numpy()
    dec.close()
    for b in range(B):
        scale = np.abs(zref[b]).max()
        err = np.abs(z[b] - zref[b]).max()
        assert err <= LOGIT_RTOL * scale, f"seq {b}: max |dlogit| {err:.3e} > {LOGIT_RTOL * scale:.3e}"
        if oracle.top2_margin(zref[b]) > LOGIT_RTOL * scale:
            assert tok[b] == int(np.argmax(zref[b])), f"seq {b}: token {tok[b]} != {int(np.argmax(zref[b]))}"
    for l in (layers if layers is not None else range(cfg.n_layers)):
        for got_t, want in ((dm.k_cache[l], cache.k[l]), (dm.v_cache[l], cache.v[l])):
            got = oracle.upcast(got_t[:B, :, :P].cpu().numpy().view(np.uint16), cfg.dtype)
            want = want[:, :, :P]
            err = np.abs(got - want)
            bound = ULP_REL[cfg.dtype] * np.abs(want) + 1e-3 * np.abs(want).max()
            assert np.all(err <= bound), f"layer {l}: cache err {err.max():.3e}, worst over bound {(err - bound).max():.3e}"


@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_tiny_prefill_600_chunks(lib, sync):
    """600 positions of one prompt: 37 chunks of 16 rows and a ragged chunk of 8."""
    _check(lib, "tiny", 1, 600, sync)


@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_tiny_prefill_three_sequences(lib, sync):
    """Three prompts of 37 positions: chunks of 5 positions of each (15 rows), then 2."""
    _check(lib, "tiny", 3, 37, sync)


def test_tiny_g4_prefill(lib):
    """Four query heads per kv head, on a batch-1 context (the chunk geometry differs from
    the decode geometry)."""
    _check(lib, "tiny-g4", 1, 300, 1, max_batch=1)


def test_2b_prefill_512(lib):
    """The benchmarked model's 512-token prompt: 32 chunks of 16 rows."""
    _check(lib, "2b", 1, 512, 1, layers=(0, 11, 23), max_batch=1)


def test_prefill_then_decode_chain(lib):
    """Decode steps fed by the device after a chunked prefill continue the oracle's greedy
    chain (the chunk's token is the sequence's last position, not the chunk's first row)."""
    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_weights(cfg)
    m = oracle.Model(cfg, w)
    P, n = 21, 6
    prompt = synth.gen_prompts(cfg, 2, P)
    toks, _ = oracle.greedy_generate(m, prompt, n + 1)
    dm = lib.DeviceModel(cfg, w, max_batch=2, max_ctx=P + n + 2)
    dec = lib.Decoder(dm, sync_mode=1)
    first = dec.prefill(prompt)
    out = torch.zeros((n, 2), dtype=torch.int32, device=dm.device)
    dec.decode_steps(None, [P] * 2, n, out)
    dec.synchronize()
    got = out.cpu().numpy()
    dec.close()
    np.testing.assert_array_equal(first, toks[:, P])
    np.testing.assert_array_equal(got.T, toks[:, P + 1: P + 1 + n])


def test_tiny_prefill_32k_equals_stepwise_decode(lib):
    """A 32768-token prompt (2048 chunks, attention over up to 32k cached positions per
    row): prefill in chunks and the same prompt fed one position per decode step leave the
    same cache (sampled positions, each entry within one storage ulp plus 1e-3 of the
    largest magnitude) and give the same last-position logits (1e-2 of the largest) --
    prefill equals incremental decode, a property that holds at any length, where the
    fp64 oracle's causal prefill would need 8 GB score matrices per head."""
    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_weights(cfg)
    P = 32768
    prompt = synth.gen_prompts(cfg, 1, P)
    out = []
    for chunked in (True, False):
        dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=P + 1)
        dec = lib.Decoder(dm, sync_mode=1)
        logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device=dm.device)
        if chunked:
            dec.prefill(prompt, logits=logits)
        else:
            for t in range(P):
                dec.decode_step(prompt[:, t], [t], logits=logits if t == P - 1 else None)
        dec.close()
        idx = torch.as_tensor(np.r_[np.arange(0, P, 997), np.arange(P - 16, P)], device=dm.device)
        caches = [np.stack([oracle.upcast(c[0][:, idx].cpu().numpy().view(np.uint16), cfg.dtype)
                            for c in (dm.k_cache[l], dm.v_cache[l])]) for l in range(cfg.n_layers)]
        out.append((logits.cpu().numpy()[0], caches))
        del dm
    (za, ca), (zb, cb) = out
    assert np.abs(za - zb).max() <= LOGIT_RTOL * np.abs(zb).max()
    for l in range(cfg.n_layers):
        err = np.abs(ca[l] - cb[l])
        bound = ULP_REL[cfg.dtype] * np.abs(cb[l]) + 1e-3 * np.abs(cb[l]).max()
        assert np.all(err <= bound), f"layer {l}: cache err {err.max():.3e}"

"""The tensor-core split-KV attention ("8 · Écrire son megakernel", §8.2 ATTENTION; the
flash-decoding split of «7 · AMD et le monokernel», §7.1) against the oracle and against the
CUDA-core attention of the same context.

A unit of at least half a page of cached positions (64 at head_dim 128, 128 at 64) runs
q K^T and P V on mma.sync with its K / V pages landed by tensor-map boxes; the last box of a
unit ends at its last cached position, so the contexts below pick unit lengths that hit the
half-page threshold, a first box that starts before position 0 (zero rows), a box that
starts inside the previous split, several boxes with a ragged tail, and prompt chunks whose
rows carry up to 16 new keys."""
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


# head_dim 128 with one, two and four query heads per kv head (the 2b and 8b attention
# shapes) on the tiny decoder's other sizes
HD128 = {
    1: synth.with_overrides(synth.CONFIGS["tiny"], name="tiny-hd128-g1", n_heads=2, n_kv_heads=2, head_dim=128),
    2: synth.with_overrides(synth.CONFIGS["tiny"], name="tiny-hd128-g2", n_heads=4, n_kv_heads=2, head_dim=128),
    4: synth.with_overrides(synth.CONFIGS["tiny"], name="tiny-hd128-g4", n_heads=8, n_kv_heads=2, head_dim=128),
}


def _run(lib, cfg, w, prompt, toks, n_new, **opts):
    B = prompt.shape[0]
    dm = lib.DeviceModel(cfg, w, max_batch=B, max_ctx=prompt.shape[1] + n_new)
    dec = lib.Decoder(dm, **opts)
    want = 2 if B >= 3 else (1 if opts.get("attn_tensor_cores", 0) == 1 else 0)
    assert dec.info()["kernel_variant"] == want
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    return z, tg


@pytest.mark.parametrize("P,kv_splits", [(64, 1), (100, 1), (200, 2), (300, 1), (600, 3)],
                         ids=["half-page", "box-before-0", "box-in-prev-split", "ragged-blocks", "three-splits"])
@pytest.mark.parametrize("G", [1, 2, 4])
@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_hd128_tensor_core_attention(lib, sync, G, P, kv_splits):
    """head_dim 128 (page = 128 positions): the tensor-core units match the oracle and the
    CUDA-core attention of the same schedule."""
    cfg = HD128[G]
    w = synth.gen_weights(cfg)
    m = oracle.Model(cfg, w)
    n_new = 3
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    z1, t1 = _run(lib, cfg, w, prompt, toks, n_new, sync_mode=sync, kv_splits=kv_splits, attn_tensor_cores=1)
    assert_parity(z1, t1, zref, toks, P)
    z0, _ = _run(lib, cfg, w, prompt, toks, n_new, sync_mode=sync, kv_splits=kv_splits, attn_tensor_cores=-1)
    # the two attentions differ only in rounding: q and P as hi/lo 16-bit halves on the
    # tensor cores against fp32 products on the CUDA cores
    scale = np.abs(zref).max()
    assert np.abs(z1 - z0).max() <= 1e-3 * scale


@pytest.mark.parametrize("B", [1, 3, 6])
@pytest.mark.parametrize("sync", [0, 1], ids=["counter", "sentinel"])
def test_hd64_batched_tensor_core_attention(lib, sync, B):
    """head_dim 64 (page = 256 positions: two passes of 128 rows per page) at a 600-position
    context, one split per sequence and head: batches 1 (CUDA-core GEMV) and 3 / 6 (the
    tensor-core instance; cache rows of several sequences through one tensor map)."""
    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_weights(cfg)
    m = oracle.Model(cfg, w)
    P, n_new = 600, 3
    prompt = synth.gen_prompts(cfg, B, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    z, tg = _run(lib, cfg, w, prompt, toks, n_new, sync_mode=sync, kv_splits=1, attn_tensor_cores=1)
    assert_parity(z, tg, zref, toks, P)


def test_hd128_long_prompt_chunks(lib):
    """A 520-position prompt through prompt chunks of 16 rows on the tensor-core instance
    (each row's unit carries up to 16 new keys in its new-row page), then decode: matches
    the oracle, and the CUDA-core attention to rounding."""
    cfg = HD128[2]
    w = synth.gen_weights(cfg)
    m = oracle.Model(cfg, w)
    B, P, n_new = 3, 520, 3
    prompt = synth.gen_prompts(cfg, B, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    z1, t1 = _run(lib, cfg, w, prompt, toks, n_new, sync_mode=0)
    assert_parity(z1, t1, zref, toks, P)
    z0, _ = _run(lib, cfg, w, prompt, toks, n_new, sync_mode=0, attn_tensor_cores=-1)
    assert np.abs(z1 - z0).max() <= 1e-3 * np.abs(zref).max()


def test_long_capacity_batch1_context_takes_the_attention_variant(lib):
    """A batch-1 context of KV capacity >= 8192 runs the kernel variant with the
    tensor-core attention by default, and its decode matches the oracle."""
    cfg = HD128[2]
    w = synth.gen_weights(cfg)
    m = oracle.Model(cfg, w)
    P, n_new = 200, 3
    prompt = synth.gen_prompts(cfg, 1, P)
    toks, zref = oracle_run(cfg, w, prompt, n_new, model=m)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=8192)
    dec = lib.Decoder(dm, sync_mode=1, kv_splits=2)
    assert dec.info()["kernel_variant"] == 1
    z, tg = gpu_teacher_forced(dec, prompt, toks, n_new, cfg.vocab)
    dec.close()
    assert_parity(z, tg, zref, toks, P)


@pytest.mark.parametrize("B", [1, 4])
def test_multi_step_launch_with_tensor_core_attention(lib, B):
    """Several greedy steps in ONE launch (the multi-step instances of the attention-only
    and the tensor-core variant: the loader waits for the previous step's tokens before a
    unit's K / V boxes, which then include the rows that step appended) give the same tokens
    and last-step activations, bit for bit, as one launch per step."""
    import torch
    cfg = HD128[2]
    w = synth.gen_weights(cfg)
    P, n = 130, 6
    prompt = synth.gen_prompts(cfg, B, P)
    runs = []
    for one_launch in (True, False):
        dm = lib.DeviceModel(cfg, w, max_batch=B, max_ctx=P + n + 1)
        dec = lib.Decoder(dm, sync_mode=1, kv_splits=1, attn_tensor_cores=1)
        assert dec.info()["kernel_variant"] == (1 if B == 1 else 2)
        first = dec.prefill(prompt)
        out = torch.zeros((n, B), dtype=torch.int32, device=dm.device)
        if one_launch:
            dec.decode_steps(first, [P] * B, n, out)
        else:
            for k in range(n):
                dec.decode_steps(first if k == 0 else None, [P + k] * B, 1, out[k:k + 1])
        dec.synchronize()
        h = dec.read_activation(0, cfg.n_layers)
        runs.append((first, out.cpu().numpy().copy(), h))
        dec.close()
    assert list(runs[0][0]) == list(runs[1][0])
    np.testing.assert_array_equal(runs[0][1], runs[1][1])
    np.testing.assert_array_equal(runs[0][2], runs[1][2])


def test_attn_tensor_cores_option_range(lib):
    """attn_tensor_cores is -1, 0 or 1; anything else is refused at creation."""
    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_weights(cfg)
    dm = lib.DeviceModel(cfg, w, max_batch=1, max_ctx=64)
    from persistent_sm_decode_megakernel_gb300 import MkError
    with pytest.raises(MkError):
        lib.Decoder(dm, attn_tensor_cores=2)

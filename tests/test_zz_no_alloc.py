"""mk_decode_step_noalloc against mk_decode_step, on the GPU, through the C ABI.

The allocation-free entry point serves callers that cannot call cudaMalloc (code inside
an allocator, or under a host framework that owns every device allocation): it keeps
its working buffers in a fixed device array compiled into the library.  It runs the same
kernel instance (counter sync) over the same schedule as a context, so its logits must
equal the context entry point's bit for bit, with the same tokens and the same key and
value rows written to the cache -- on calls in a row, where each call finds the previous
call's leftovers in the shared array (including a schedule of another batch size) and
must clear what needs clearing.  The file sorts last so that a run stopping at the first
failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

P32 = ctypes.POINTER(ctypes.c_int32)


def _noalloc(mk, dm, toks, pos, logits, stream):
    desc = dm.desc()
    wts, kv, keep = dm.abi_structs()
    tok = np.ascontiguousarray(toks, dtype=np.int32)
    ps = np.ascontiguousarray(pos, dtype=np.int32)
    out = np.zeros(len(tok), dtype=np.int32)
    st = mk.mk_decode_step_noalloc(ctypes.byref(desc), ctypes.byref(wts), ctypes.byref(kv), tok.ctypes.data_as(P32),
                                   ps.ctypes.data_as(P32), len(tok), out.ctypes.data_as(P32),
                                   ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert st == mk.MK_OK, mk.mk_last_error()
    return out


def _same_rows(dm_a, dm_b, cfg, pos):
    """The key and value rows each sequence's step wrote, in every layer, are identical."""
    for l in range(cfg.n_layers):
        for b, p in enumerate(pos):
            for ca, cb in ((dm_a.k_cache[l], dm_b.k_cache[l]), (dm_a.v_cache[l], dm_b.v_cache[l])):
                np.testing.assert_array_equal(ca[b, :, p].cpu().numpy(), cb[b, :, p].cpu().numpy())


def test_noalloc_matches_context_entry_point_twice():
    import __graft_entry__
    __graft_entry__.build()
    import persistent_sm_decode_megakernel_gb300 as mk
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel

    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_weights(cfg)
    toks = synth.gen_prompts(cfg, 1, 2)[0]
    ref_dm = DeviceModel(cfg, w, max_batch=1, max_ctx=8)
    na_dm = DeviceModel(cfg, w, max_batch=1, max_ctx=8)
    dec = Decoder(ref_dm)
    stream = torch.cuda.current_stream()
    z_ref = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda:0")
    z_na = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda:0")
    for t in range(2):                                  # two calls in a row
        out_ref = dec.decode_step([int(toks[t])], [t], logits=z_ref)
        out = _noalloc(mk, na_dm, [toks[t]], [t], z_na, stream)
        np.testing.assert_array_equal(z_na.cpu().numpy(), z_ref.cpu().numpy())
        assert out[0] == out_ref[0]
        _same_rows(na_dm, ref_dm, cfg, [t])
    dec.close()


def test_noalloc_batches_in_a_row_match_context():
    """max_batch 8: a batch-1 call, then a batch-4 call at ragged positions (the tensor-core
    GEMV path and a wider activation arena in the same array), then batch 1 twice (the
    schedule is rebuilt, then reused); each against the context entry point."""
    import persistent_sm_decode_megakernel_gb300 as mk
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel

    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_weights(cfg)
    seqs = synth.gen_prompts(cfg, 4, 4)
    ref_dm = DeviceModel(cfg, w, max_batch=8, max_ctx=16)
    na_dm = DeviceModel(cfg, w, max_batch=8, max_ctx=16)
    dec = Decoder(ref_dm)
    stream = torch.cuda.current_stream()
    calls = [([seqs[0, 0]], [0]),
             ([seqs[0, 1], seqs[1, 0], seqs[2, 0], seqs[3, 0]], [1, 0, 0, 0]),
             ([seqs[0, 2]], [2]),
             ([seqs[0, 3]], [3])]
    for toks, pos in calls:
        B = len(toks)
        z_ref = torch.zeros((B, cfg.vocab), dtype=torch.float32, device="cuda:0")
        z_na = torch.zeros((B, cfg.vocab), dtype=torch.float32, device="cuda:0")
        out_ref = dec.decode_step([int(t) for t in toks], pos, logits=z_ref)
        out = _noalloc(mk, na_dm, toks, pos, z_na, stream)
        np.testing.assert_array_equal(z_na.cpu().numpy(), z_ref.cpu().numpy())
        np.testing.assert_array_equal(out, np.asarray(out_ref))
        _same_rows(na_dm, ref_dm, cfg, pos)
    dec.close()


def test_noalloc_long_context_tensor_core_attention_matches_context():
    """max_batch 4 at ~3000 cached positions (synthetic keys and values, the same in both
    caches): every split-KV unit holds more than half a page of positions, so both entry
    points run the tensor-core attention with its K / V tensor maps -- the allocation-free
    one keeps them in its array -- and the logits, tokens and written rows agree bit for bit,
    at ragged positions."""
    import persistent_sm_decode_megakernel_gb300 as mk
    from persistent_sm_decode_megakernel_gb300.model import Decoder, DeviceModel

    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_weights(cfg)
    T, B = 3000, 4
    dms = [DeviceModel(cfg, w, max_batch=B, max_ctx=T + 8) for _ in range(2)]
    for dm in dms:
        g = torch.Generator(device=dm.device)
        g.manual_seed(5)
        for l in range(cfg.n_layers):
            for cache in (dm.k_cache[l], dm.v_cache[l]):
                x = torch.randn((B, cfg.n_kv_heads, T, cfg.head_dim), generator=g, device=dm.device)
                cache[:, :, :T] = (x * 0.9).to(torch.bfloat16).view(torch.int16)
    ref_dm, na_dm = dms
    dec = Decoder(ref_dm)
    assert dec.info()["kernel_variant"] == 2
    stream = torch.cuda.current_stream()
    toks = synth.gen_prompts(cfg, 1, B)[0]
    pos = [T, T - 700, T - 1300, T - 1]
    z_ref = torch.zeros((B, cfg.vocab), dtype=torch.float32, device="cuda:0")
    z_na = torch.zeros((B, cfg.vocab), dtype=torch.float32, device="cuda:0")
    out_ref = dec.decode_step([int(t) for t in toks], pos, logits=z_ref)
    out = _noalloc(mk, na_dm, toks, pos, z_na, stream)
    np.testing.assert_array_equal(z_na.cpu().numpy(), z_ref.cpu().numpy())
    np.testing.assert_array_equal(out, np.asarray(out_ref))
    _same_rows(na_dm, ref_dm, cfg, pos)
    dec.close()


def test_noalloc_refuses_models_beyond_its_scratch():
    """A descriptor whose schedule alone outgrows the array (the tiny model's tensors
    repeated over 400 layers: ~19 MB of instructions) is refused before anything runs."""
    import persistent_sm_decode_megakernel_gb300 as mk
    from persistent_sm_decode_megakernel_gb300 import mk_kv, mk_weights
    from persistent_sm_decode_megakernel_gb300.model import _LAYER_TENSORS, DeviceModel

    cfg = synth.CONFIGS["tiny"]
    dm = DeviceModel(cfg, synth.gen_weights(cfg), max_batch=1, max_ctx=8)
    L = 400
    desc = dm.desc()
    desc.n_layers = L
    arr = ctypes.c_void_p * L
    tabs = {n: arr(*[dm.layers[l % 2][n].data_ptr() for l in range(L)]) for n in _LAYER_TENSORS}
    wts = mk_weights(dm.embed.data_ptr(), dm.final_norm.data_ptr(), dm.lm_head.data_ptr(),
                     *[ctypes.cast(tabs[n], ctypes.POINTER(ctypes.c_void_p)) for n in _LAYER_TENSORS])
    kt = arr(*[dm.k_cache[l % 2].data_ptr() for l in range(L)])
    vt = arr(*[dm.v_cache[l % 2].data_ptr() for l in range(L)])
    kv = mk_kv(ctypes.cast(kt, ctypes.POINTER(ctypes.c_void_p)), ctypes.cast(vt, ctypes.POINTER(ctypes.c_void_p)))
    tok = np.array([1], dtype=np.int32)
    pos = np.array([0], dtype=np.int32)
    out = np.zeros(1, dtype=np.int32)
    st = mk.mk_decode_step_noalloc(ctypes.byref(desc), ctypes.byref(wts), ctypes.byref(kv), tok.ctypes.data_as(P32),
                                   pos.ctypes.data_as(P32), 1, out.ctypes.data_as(P32), None, None)
    assert st == mk.MK_ERR_INVALID
    assert b"scratch" in mk.mk_last_error()

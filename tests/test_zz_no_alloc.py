"""mk_decode_step_noalloc against mk_decode_step, on the GPU, through the C ABI.

The allocation-free entry point serves callers that cannot call cudaMalloc (code inside
an allocator, or under a host framework that owns every device allocation): it keeps
its working buffers in a fixed device array compiled into the library.  Here it must
give the same logits (within the tolerance of the other parity tests) and the same
tokens as the context-based entry point, on two calls in a row -- the second call finds
the first call's leftovers in the shared array and must clear what needs clearing.
The file sorts last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


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
    desc = na_dm.desc()
    wts, kv, keep = na_dm.abi_structs()
    z_ref = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda:0")
    z_na = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda:0")
    for t in range(2):                                  # two calls in a row
        out_ref = dec.decode_step([int(toks[t])], [t], logits=z_ref)
        tok = np.array([toks[t]], dtype=np.int32)
        pos = np.array([t], dtype=np.int32)
        out = np.zeros(1, dtype=np.int32)
        P = ctypes.POINTER(ctypes.c_int32)
        st = mk.mk_decode_step_noalloc(ctypes.byref(desc), ctypes.byref(wts), ctypes.byref(kv),
                                       tok.ctypes.data_as(P), pos.ctypes.data_as(P), 1, out.ctypes.data_as(P),
                                       ctypes.c_void_p(z_na.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert st == mk.MK_OK, mk.mk_last_error()
        a, b = z_na.cpu().numpy(), z_ref.cpu().numpy()
        assert np.abs(a - b).max() <= 1e-2 * np.abs(b).max()
        assert out[0] == out_ref[0]
        # the cache position this step wrote matches too
        np.testing.assert_array_equal(na_dm.k_cache[0][0, :, t].cpu().numpy(), ref_dm.k_cache[0][0, :, t].cpu().numpy())
    dec.close()


def test_noalloc_refuses_models_beyond_its_scratch():
    import persistent_sm_decode_megakernel_gb300 as mk
    from persistent_sm_decode_megakernel_gb300.model import DeviceModel

    # a tiny model with a context so long that its RoPE rows alone exceed the array
    cfg = synth.CONFIGS["tiny"]
    dm = DeviceModel(cfg, synth.gen_weights(cfg), max_batch=1, max_ctx=80000)
    desc = dm.desc()
    wts, kv, keep = dm.abi_structs()
    P = ctypes.POINTER(ctypes.c_int32)
    tok = np.array([1], dtype=np.int32)
    pos = np.array([79999], dtype=np.int32)
    out = np.zeros(1, dtype=np.int32)
    st = mk.mk_decode_step_noalloc(ctypes.byref(desc), ctypes.byref(wts), ctypes.byref(kv), tok.ctypes.data_as(P),
                                   pos.ctypes.data_as(P), 1, out.ctypes.data_as(P), None, None)
    assert st == mk.MK_ERR_INVALID
    assert b"scratch" in mk.mk_last_error()

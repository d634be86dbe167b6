"""CPU-only checks of the C-ABI library: it builds, loads without a GPU, exports every
function include/mk.h declares, and its host-side schedule builder and static
validator ("8 · Écrire son megakernel", §8.7, static verification) accept every
workload shape, reject injected faults, and refuse bad descriptors."""
import ctypes

import pytest

import synth


@pytest.fixture(scope="module")
def mk():
    import __graft_entry__
    __graft_entry__.build()
    import persistent_sm_decode_megakernel_gb300 as m
    return m


def _desc(mk, cfg, max_batch=1, max_ctx=4096):
    return mk.mk_model_desc(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                            cfg.vocab, mk.MK_F16 if cfg.dtype == "f16" else mk.MK_BF16, cfg.rms_eps, cfg.rope_theta,
                            max_batch, max_ctx)


def _plan(mk, desc, n_ctas, **opt):
    o = mk.mk_options()
    for k, v in opt.items():
        setattr(o, k, v)
    info = mk.mk_info_t()
    st = mk.mk_plan(ctypes.byref(desc), ctypes.byref(o), n_ctas, ctypes.byref(info))
    return st, info


def test_library_exports_every_declared_symbol(mk):
    names = mk.declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(mk.lib, n), f"{n} declared in include/mk.h but not exported"
    for required in ("mk_create", "mk_prefill", "mk_decode_step", "mk_destroy"):
        assert required in names


def test_status_strings(mk):
    assert mk.mk_status_string(mk.MK_ERR_TIMEOUT) == b"MK_ERR_TIMEOUT"
    assert mk.mk_status_string(mk.MK_OK) == b"MK_OK"


@pytest.mark.parametrize("name", ["tiny", "0.5b", "2b", "8b"])
@pytest.mark.parametrize("n_ctas", [152, 148, 132, 7])
def test_plan_validates_every_workload(mk, name, n_ctas):
    cfg = synth.CONFIGS[name]
    st, info = _plan(mk, _desc(mk, cfg), n_ctas)
    assert st == mk.MK_OK, mk.mk_last_error()
    assert info.weight_bytes_per_step == cfg.streamed_weight_bytes()
    assert info.n_pages >= 2 and info.smem_bytes <= 232448
    assert info.kv_splits >= 1


def test_plan_batches_and_sizes(mk):
    cfg = synth.CONFIGS["2b"]
    for B in (1, 2, 4):
        st, info = _plan(mk, _desc(mk, cfg, max_batch=B), 152)
        assert st == mk.MK_OK, mk.mk_last_error()
    # one wave of split-KV units: B * Hkv * S is a multiple of the CTA count
    st, info = _plan(mk, _desc(mk, cfg), 152)
    assert (cfg.n_kv_heads * info.kv_splits) % 152 == 0


def test_plan_multilaunch_counts_launches(mk):
    cfg = synth.CONFIGS["2b"]
    L = cfg.n_layers
    # the KV-split merge: inside the O-proj staging (attn_merge 2) or in the last-arriving
    # split (counter sync) -- five launches per layer either way -- or a separate reduce
    # launch per layer (sentinel sync); auto (0) keeps the separate step at the 2b size
    for execm in (mk.MK_EXEC_MULTILAUNCH, mk.MK_EXEC_GRAPH):
        for sync, merge, per_layer in ((0, 0, 5), (1, 0, 6), (0, 2, 5), (1, 2, 5), (0, 1, 5), (1, 1, 6)):
            st, info = _plan(mk, _desc(mk, cfg), 152, exec_mode=execm, sync_mode=sync, attn_merge=merge)
            assert st == mk.MK_OK, mk.mk_last_error()
            assert info.launches_per_step == per_layer * L + 2, (sync, merge)


def test_plan_merge_choice_and_bad_option(mk):
    cfg = synth.CONFIGS["2b"]
    for merge in (0, 1, 2, 3):
        for b in (1, 2, 4):
            for sync in (0, 1):
                st, _ = _plan(mk, _desc(mk, cfg, max_batch=b), 152, attn_merge=merge, sync_mode=sync)
                assert st == mk.MK_OK, (merge, b, sync, mk.mk_last_error())
    st, _ = _plan(mk, _desc(mk, cfg), 152, attn_merge=4)
    assert st == mk.MK_ERR_INVALID


@pytest.mark.parametrize("sync", [0, 1])
def test_plan_validates_both_sync_schedules(mk, sync):
    for name in ("tiny", "2b"):
        st, _ = _plan(mk, _desc(mk, synth.CONFIGS[name], max_batch=2), 152, sync_mode=sync)
        assert st == mk.MK_OK, mk.mk_last_error()


def test_validator_rejects_dropped_signal(mk):
    # fault injection on the host: with one counter signal removed the waiters can never
    # complete; the validator must name the mismatch instead of letting it deadlock
    cfg = synth.CONFIGS["tiny"]
    for k in (1, 5, 40):
        st, _ = _plan(mk, _desc(mk, cfg), 16, fault_drop_signal=k)
        assert st == mk.MK_ERR_INVALID
        msg = mk.mk_last_error().decode()
        assert "validator" in msg and ("signals" in msg or "deadlock" in msg)


@pytest.mark.parametrize("field,value", [("n_heads", 5), ("head_dim", 96), ("max_batch", 17), ("dtype", 7),
                                         ("vocab", 0), ("d_model", 100)])
def test_bad_descriptors_rejected(mk, field, value):
    d = _desc(mk, synth.CONFIGS["tiny"])
    setattr(d, field, value)
    st, _ = _plan(mk, d, 16)
    assert st == mk.MK_ERR_INVALID


def test_bad_page_size_rejected(mk):
    d = _desc(mk, synth.CONFIGS["2b"])
    for pb in (3000, 1 << 16, 4096):       # not a power of two / too big / < 64 * head_dim
        st, _ = _plan(mk, d, 152, page_bytes=pb)
        assert st == mk.MK_ERR_INVALID


def test_create_rejects_null_and_misaligned_pointers(mk):
    # argument checks run before any CUDA call, so they work without a GPU
    cfg = synth.CONFIGS["tiny"]
    d = _desc(mk, cfg)
    h = ctypes.c_void_p()
    o = mk.mk_options()
    assert mk.mk_create(ctypes.byref(d), None, None, ctypes.byref(o), None, ctypes.byref(h)) == mk.MK_ERR_INVALID
    L = cfg.n_layers
    arr = (ctypes.c_void_p * L)(*([0x1001] * L))   # misaligned
    P = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    w = mk.mk_weights(0x1000, 0x2000, 0x3000, P, P, P, P, P, P, P, P, P)
    kv = mk.mk_kv(P, P)
    st = mk.mk_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(kv), ctypes.byref(o), None, ctypes.byref(h))
    assert st == mk.MK_ERR_INVALID and b"aligned" in mk.mk_last_error()


@pytest.mark.parametrize("name,max_batch", [("tiny", 1), ("tiny", 4), ("2b", 1), ("2b", 16), ("8b", 2)])
@pytest.mark.parametrize("sync", [0, 1])
def test_plan_with_attention_pool_validates(mk, name, max_batch, sync):
    """Dynamic attention (one claim loop per CTA and layer, the units in per-layer pools):
    the validator runs each pool whole on the first CTA that reaches it and checks
    coverage, signal counts and ordering as for static units; the instruction count
    is the static plan's minus the units plus the claim loops."""
    cfg = synth.CONFIGS[name]
    d = _desc(mk, cfg, max_batch=max_batch)
    st0, static = _plan(mk, d, 152, sync_mode=sync)
    st1, pooled = _plan(mk, d, 152, sync_mode=sync, attn_pool=1)
    assert st0 == mk.MK_OK and st1 == mk.MK_OK, mk.mk_last_error()
    assert pooled.n_instructions == static.n_instructions + 152 * cfg.n_layers
    assert pooled.n_counters == static.n_counters + cfg.n_layers   # one claim counter per layer


def test_attention_pool_option_range(mk):
    cfg = synth.CONFIGS["tiny"]
    st, _ = _plan(mk, _desc(mk, cfg), 152, attn_pool=1, exec_mode=1)   # multi-launch: static units
    assert st == mk.MK_OK


@pytest.mark.parametrize("max_batch,max_ctx,attn,page_bytes,variant", [
    (1, 4096, 0, 0, 0), (1, 8192, 0, 0, 1), (2, 32800, 0, 0, 1), (3, 64, 0, 0, 2), (16, 64, 0, 0, 2),
    (1, 64, 1, 0, 1), (1, 32800, -1, 0, 0), (8, 64, -1, 0, 2), (1, 32800, 0, 16384, 0)])
def test_kernel_variant_choice(mk, max_batch, max_ctx, attn, page_bytes, variant):
    """The step kernel variant a context runs: with the tensor-core GEMV and attention from
    max_batch 3 on; with the tensor-core attention alone for batch-1..2 contexts of KV
    capacity >= 8192 (or when asked for); without tensor-core code otherwise, or when the
    attention is kept on CUDA cores, or with pages smaller than the 32 KB box."""
    cfg = synth.CONFIGS["2b"]
    st, info = _plan(mk, _desc(mk, cfg, max_batch, max_ctx), 152, attn_tensor_cores=attn, page_bytes=page_bytes)
    assert st == mk.MK_OK, mk.mk_last_error()
    assert info.kernel_variant == variant


def test_attn_tensor_cores_option_range(mk):
    for bad in (-2, 2):
        st, _ = _plan(mk, _desc(mk, synth.CONFIGS["tiny"]), 152, attn_tensor_cores=bad)
        assert st == mk.MK_ERR_INVALID

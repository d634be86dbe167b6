"""Model-level pins of the fp64 oracle: causality, prefill == incremental decode,
batch independence, and agreement with an independent formulation built from
PyTorch library routines (F.rms_norm, F.scaled_dot_product_attention with GQA and a
causal mask, F.silu, F.linear, complex rotation for RoPE) in float64 on the CPU."""
import json
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.CONFIGS["tiny"]
    return cfg, O.Model(cfg, synth.gen_weights(cfg))


def _small_gqa_cfg():
    # 3 layers, G = 3 query heads per kv head, odd sizes: exercises the grouping
    return synth.with_overrides(synth.CONFIGS["tiny"], name="small3", n_layers=3, d_model=96,
                                n_heads=6, n_kv_heads=2, head_dim=16, ffn_dim=160, vocab=97, seed=11)


def test_causality_appending_tokens_keeps_earlier_logits(tiny):
    cfg, m = tiny
    p = synth.gen_prompts(cfg, 1, 12)
    c1 = O.KVCache(cfg, 1, 12)
    z_short = O.prefill(m, p[:, :7], O.KVCache(cfg, 1, 7))
    z_long = O.prefill(m, p, c1)
    # a missing or transposed causal mask changes these by O(1); BLAS blocking may
    # change the last bits, so compare to 1e-12 of the logit scale
    np.testing.assert_allclose(z_long[:, :7], z_short, rtol=0, atol=1e-12 * np.abs(z_short).max())


def test_prefill_equals_incremental_decode(tiny):
    cfg, m = tiny
    P = 10
    p = synth.gen_prompts(cfg, 2, P)
    cache_a = O.KVCache(cfg, 2, P)
    za = O.prefill(m, p, cache_a)
    cache_b = O.KVCache(cfg, 2, P)
    zb = np.stack([O.decode_step(m, cache_b, p[:, t], [t, t]) for t in range(P)], axis=1)
    np.testing.assert_allclose(zb, za, rtol=1e-10, atol=1e-12 * np.abs(za).max())
    for l in range(cfg.n_layers):
        np.testing.assert_array_equal(cache_a.k[l], cache_b.k[l])
        np.testing.assert_array_equal(cache_a.v[l], cache_b.v[l])


def test_batch_rows_are_independent(tiny):
    cfg, m = tiny
    p = synth.gen_prompts(cfg, 3, 6)
    z3 = O.prefill(m, p, O.KVCache(cfg, 3, 6))
    z1 = O.prefill(m, p[1:2], O.KVCache(cfg, 1, 6))
    np.testing.assert_allclose(z3[1:2], z1, rtol=1e-12, atol=1e-13)


def _torch_reference_prefill(cfg, weights, tokens):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    dt = torch.float64

    def W(name, l=-1):
        src = weights[name] if l < 0 else weights["layers"][l][name]
        t = torch.from_numpy(np.ascontiguousarray(src).view(np.int16).copy())
        t = t.view(torch.float16 if cfg.dtype == "f16" else torch.bfloat16)
        return t.to(dt)

    B, P = tokens.shape
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    tok = torch.from_numpy(tokens.astype(np.int64))
    h = F.embedding(tok, W("embed"))
    pos = torch.arange(P, dtype=dt)
    freq = cfg.rope_theta ** (-torch.arange(hd // 2, dtype=dt) * 2.0 / hd)
    rot = torch.polar(torch.ones(P, hd // 2, dtype=dt), pos[:, None] * freq[None])   # [P, hd/2]

    def rope(x):                                    # x [B, H, P, hd]
        z = torch.complex(x[..., : hd // 2], x[..., hd // 2:]) * rot
        return torch.cat([z.real, z.imag], dim=-1)

    def to_cache(x):
        return x.to(torch.float16 if cfg.dtype == "f16" else torch.bfloat16).to(dt)

    for l in range(cfg.n_layers):
        x = F.rms_norm(h, (cfg.d_model,), W("attn_norm", l), eps=cfg.rms_eps)
        q = rope(F.linear(x, W("wq", l)).view(B, P, Hq, hd).transpose(1, 2))
        k = to_cache(rope(F.linear(x, W("wk", l)).view(B, P, Hkv, hd).transpose(1, 2)))
        v = to_cache(F.linear(x, W("wv", l)).view(B, P, Hkv, hd).transpose(1, 2))
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
        h = h + F.linear(o.transpose(1, 2).reshape(B, P, Hq * hd), W("wo", l))
        x2 = F.rms_norm(h, (cfg.d_model,), W("mlp_norm", l), eps=cfg.rms_eps)
        h = h + F.linear(F.silu(F.linear(x2, W("w_gate", l))) * F.linear(x2, W("w_up", l)), W("w_down", l))
    z = F.linear(F.rms_norm(h, (cfg.d_model,), W("final_norm"), eps=cfg.rms_eps), W("lm_head"))
    return z.numpy()


@pytest.mark.parametrize("which", ["tiny", "small3", "small3-f16"])
def test_oracle_matches_torch_library_formulation(which):
    if which == "tiny":
        cfg = synth.CONFIGS["tiny"]
    else:
        cfg = _small_gqa_cfg()
        if which.endswith("f16"):
            cfg = synth.with_overrides(cfg, dtype="f16", seed=12)
    weights = synth.gen_weights(cfg)
    m = O.Model(cfg, weights)
    p = synth.gen_prompts(cfg, 2, 9)
    za = O.prefill(m, p, O.KVCache(cfg, 2, 9))
    zt = _torch_reference_prefill(cfg, weights, p)
    # both sides are fp64 with the same cache rounding; they agree to ~1e-15 here, and
    # 1e-10 leaves room for BLAS summation order only
    np.testing.assert_allclose(za, zt, rtol=0, atol=1e-10 * np.abs(zt).max())


def test_greedy_generate_consistent_with_decode(tiny):
    cfg, m = tiny
    p = synth.gen_prompts(cfg, 1, 5)
    toks, logits = O.greedy_generate(m, p, 4)
    assert toks.shape == (1, 9) and logits.shape == (1, 9, cfg.vocab)
    np.testing.assert_array_equal(toks[:, :5], p)
    for t in range(4, 8):
        assert toks[0, t + 1] == np.argmax(logits[0, t])


def test_golden_tiny_greedy(tiny):
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    cfg, m = tiny
    with open(os.path.join(GOLDEN, "tiny_greedy.json")) as f:
        g = json.load(f)
    p = synth.gen_prompts(cfg, 1, g["prompt_len"])
    assert p[0].tolist() == g["prompt"]
    toks, logits = O.greedy_generate(m, p, g["n_new"])
    assert toks[0].tolist() == g["tokens"]
    np.testing.assert_allclose(logits[0, :, :8], np.array(g["logits_head"]), rtol=1e-12, atol=1e-14)

"""Seeded synthetic inputs shared by the CUDA path's harness and the CPU oracle.

This module holds no arithmetic of the decoder: only the model shapes of the five
workloads, and seeded generators for weights, prompts and (for long-context tests)
KV-cache contents.  Both sides receive the *same bytes* from here:
  * weights and KV entries are returned as uint16 bit patterns of the storage dtype
    (IEEE fp16 or bfloat16), so that the GPU uploads exactly what the oracle upcasts;
  * prompts are int32 token ids.

Generation recipe (stated once, used everywhere):
  * every tensor has a fixed index in the order
      embed, per layer [attn_norm, wq, wk, wv, wo, mlp_norm, w_gate, w_up, w_down],
      final_norm, lm_head
    and is drawn from numpy PCG64 streams seeded by SeedSequence([seed, index, block]),
    one stream per block of BLOCK consecutive elements (row-major), so blocks can be
    drawn in parallel threads and a reader can regenerate any tensor on its own;
  * projections, embedding and LM head: N(0, 0.02); norm gains: 1 + N(0, 0.1);
    draws are float32 and rounded to the storage dtype with round-to-nearest-even;
  * prompt of sequence b: uniform integers in [0, vocab) from default_rng(1000 + 100*cfg + b);
  * synthetic KV entries (long-context decode tests): N(0, KV_SIGMA) rounded to the
    cache dtype, SeedSequence([seed, 7777, layer, b, k_or_v]).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

BLOCK = 1 << 22          # elements per independent RNG stream
KV_SIGMA = 0.9           # std of synthetic k/v entries (matches W x-hat with unit-RMS x-hat)

F16 = "f16"
BF16 = "bf16"


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    dtype: str                  # storage dtype of weights and KV cache
    seed: int
    cfg_index: int              # 1-based workload number (prompt seeds)
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    batch: int = 1
    prompt_len: int = 16
    decode_len: int = 32
    batches: tuple = field(default=())

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def n_params(self) -> int:
        d, L = self.d_model, self.n_layers
        per_layer = 2 * d + d * (self.q_dim + 2 * self.kv_dim) + self.q_dim * d + 3 * d * self.ffn_dim
        return L * per_layer + 2 * self.vocab * d + d

    def streamed_weight_bytes(self) -> int:
        """Bytes of weights one decode step must read (all but the embedding table)."""
        d, L = self.d_model, self.n_layers
        per_layer = 2 * d + d * (self.q_dim + 2 * self.kv_dim) + self.q_dim * d + 3 * d * self.ffn_dim
        return 2 * (L * per_layer + self.vocab * d + d)

    def kv_bytes_per_position(self) -> int:
        return self.n_layers * 2 * self.kv_dim * 2


CONFIGS = {
    "tiny": ModelConfig("tiny", 2, 256, 4, 2, 64, 768, 1024, BF16, seed=0, cfg_index=1,
                        batch=1, prompt_len=16, decode_len=32),
    "0.5b": ModelConfig("0.5b", 24, 1024, 16, 8, 64, 2816, 32000, BF16, seed=2, cfg_index=2,
                        batch=1, prompt_len=128, decode_len=256),
    "2b": ModelConfig("2b", 24, 2048, 16, 8, 128, 8192, 128256, F16, seed=3, cfg_index=3,
                      batch=1, prompt_len=512, decode_len=1024),
    "8b": ModelConfig("8b", 32, 4096, 32, 8, 128, 14336, 128256, BF16, seed=4, cfg_index=4,
                      batch=1, prompt_len=8192, decode_len=512),
    # a tiny decoder with four query heads per kv head (the 8b model's GQA group) for the
    # grouped attention instance at long contexts in test time
    "tiny-g4": ModelConfig("tiny-g4", 2, 256, 8, 2, 64, 768, 1024, BF16, seed=6, cfg_index=6,
                           batch=1, prompt_len=600, decode_len=4),
    # the 2B fp16 model under a batch / 32k-context sweep: same weights as "2b"
    "2b-32k": ModelConfig("2b-32k", 24, 2048, 16, 8, 128, 8192, 128256, F16, seed=3, cfg_index=5,
                          batch=1, prompt_len=32768, decode_len=128, batches=(1, 2, 4, 8, 16)),
}


def tensor_names(cfg: ModelConfig):
    """(name, layer) in generation order; layer is -1 for model-level tensors."""
    out = [("embed", -1)]
    for l in range(cfg.n_layers):
        for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"):
            out.append((n, l))
    out += [("final_norm", -1), ("lm_head", -1)]
    return out


def tensor_shape(cfg: ModelConfig, name: str):
    d, F = cfg.d_model, cfg.ffn_dim
    return {
        "embed": (cfg.vocab, d), "lm_head": (cfg.vocab, d),
        "attn_norm": (d,), "mlp_norm": (d,), "final_norm": (d,),
        "wq": (cfg.q_dim, d), "wk": (cfg.kv_dim, d), "wv": (cfg.kv_dim, d),
        "wo": (d, cfg.q_dim),
        "w_gate": (F, d), "w_up": (F, d), "w_down": (d, F),
    }[name]


def tensor_index(cfg: ModelConfig, name: str, layer: int) -> int:
    if name == "embed":
        return 0
    if name == "final_norm":
        return 1 + 9 * cfg.n_layers
    if name == "lm_head":
        return 2 + 9 * cfg.n_layers
    order = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")
    return 1 + 9 * layer + order.index(name)


# ---------------------------------------------------------------- rounding to storage bits
def f32_to_storage_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> uint16 bit pattern of fp16 / bf16, round-to-nearest-even (finite inputs)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = x.view(np.uint32).astype(np.uint64)
        r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return r.astype(np.uint16)
    raise ValueError(dtype)


def storage_bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


# ---------------------------------------------------------------- generators
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def _normal_blocks(key: tuple, n: int, mean: float, std: float, dtype: str) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)

    def fill(bi):
        lo = bi * BLOCK
        hi = min(n, lo + BLOCK)
        rng = np.random.default_rng(np.random.SeedSequence(list(key) + [bi]))
        v = rng.standard_normal(hi - lo, dtype=np.float32)
        v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)
        out[lo:hi] = f32_to_storage_bits(v, dtype)

    nb = (n + BLOCK - 1) // BLOCK
    if nb == 1:
        fill(0)
    else:
        list(_pool().map(fill, range(nb)))
    return out


def gen_tensor(cfg: ModelConfig, name: str, layer: int = -1) -> np.ndarray:
    """Storage bits (uint16) of one weight tensor, shaped like the tensor."""
    shape = tensor_shape(cfg, name)
    n = int(np.prod(shape))
    idx = tensor_index(cfg, name, layer)
    if name.endswith("norm"):
        bits = _normal_blocks((cfg.seed, idx), n, 1.0, 0.1, cfg.dtype)
    else:
        bits = _normal_blocks((cfg.seed, idx), n, 0.0, 0.02, cfg.dtype)
    return bits.reshape(shape)


def gen_weights(cfg: ModelConfig) -> dict:
    """All tensors: {'embed': bits, 'final_norm': bits, 'lm_head': bits, 'layers': [dict, ...]}."""
    w = {"layers": [dict() for _ in range(cfg.n_layers)]}
    for name, layer in tensor_names(cfg):
        t = gen_tensor(cfg, name, layer)
        if layer < 0:
            w[name] = t
        else:
            w["layers"][layer][name] = t
    return w


def gen_prompt(cfg: ModelConfig, b: int, length: int) -> np.ndarray:
    rng = np.random.default_rng(1000 + 100 * cfg.cfg_index + b)
    return rng.integers(0, cfg.vocab, size=length, dtype=np.int64).astype(np.int32)


def gen_prompts(cfg: ModelConfig, batch: int, length: int) -> np.ndarray:
    return np.stack([gen_prompt(cfg, b, length) for b in range(batch)])


def gen_kv(cfg: ModelConfig, layer: int, b: int, which: int, length: int) -> np.ndarray:
    """Synthetic cache entries [n_kv_heads, length, head_dim] (storage bits) of sequence b.

    which = 0 for keys, 1 for values.  Used where the prompt's own prefill would be too
    slow for the fp64 oracle; the state then stands for an already-filled cache.
    """
    n = cfg.n_kv_heads * length * cfg.head_dim
    bits = _normal_blocks((cfg.seed, 7777, layer, b, which, length), n, 0.0, KV_SIGMA, cfg.dtype)
    return bits.reshape(cfg.n_kv_heads, length, cfg.head_dim)


def with_overrides(cfg: ModelConfig, **kw) -> ModelConfig:
    return replace(cfg, **kw)

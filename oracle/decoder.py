"""fp64 reference decoder (TEST INFRASTRUCTURE ONLY -- see the package header).

Every quantity is float64.  Weights arrive as the exact storage bits (fp16 or bf16)
the GPU receives and are upcast exactly.  Cached keys and values are rounded to the
storage dtype (round-to-nearest-even from the exact fp64 value) before they are used,
because the GPU reads them back from a cache of that dtype; nothing else is rounded.

Readings taken where the pages are silent (the pages group the ops but never define
the layer; the workload is "Llama-style"):
  * RMSNorm(h; g)_i = g_i * h_i / sqrt(mean_j h_j^2 + eps)
  * rotary embedding, "rotate-half" pairing of dims (i, i + hd/2), i < hd/2, with
    frequency theta^(-2i/hd) and angle pos * frequency; positions are 0-based
  * query head i reads kv head floor(i / (Hq/Hkv)) (contiguous groups)
  * attention scale 1/sqrt(hd); no bias, no soft-cap, no window
  * silu(u) = u / (1 + exp(-u)); MLP = W_down (silu(W_gate x) * (W_up x))
  * final RMSNorm with its own gain before the untied LM head
  * greedy token = argmax of the logits, lowest index among equal maxima
"""
from __future__ import annotations

import numpy as np

F16 = "f16"
BF16 = "bf16"


# ---------------------------------------------------------------- storage dtype
def upcast(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact value of fp16 / bf16 storage bits as float64."""
    bits = np.ascontiguousarray(bits).view(np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float64)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round exact fp64 values to the nearest fp16 / bf16 value (ties to even), as fp64.

    fp16: numpy's double->half conversion rounds the double directly (one rounding).
    bf16: written out from the format: 8 significant bits, exponent range of fp32.
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == F16:
        return x.astype(np.float16).astype(np.float64)
    if dtype == BF16:
        out = np.zeros_like(x)
        nz = x != 0
        _, e = np.frexp(x[nz])                    # x = m * 2^e, 0.5 <= |m| < 1
        e = np.maximum(e, -125)                   # below the normal range the grid is fixed
        step = np.ldexp(1.0, e - 8)               # spacing of 8-significant-bit numbers
        out[nz] = np.rint(x[nz] / step) * step    # np.rint: round half to even
        return out
    raise ValueError(dtype)


# ---------------------------------------------------------------- the seven ops' pieces
def rms_norm(h: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis (reading above)."""
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return g * h / np.sqrt(ms + eps)


def rope_cos_sin(pos: int, head_dim: int, theta: float):
    i = np.arange(head_dim // 2, dtype=np.float64)
    freq = theta ** (-2.0 * i / head_dim)
    ang = float(pos) * freq
    return np.cos(ang), np.sin(ang)


def apply_rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of x[..., hd] at position pos."""
    hd = x.shape[-1]
    c, s = rope_cos_sin(pos, hd, theta)
    x1 = x[..., : hd // 2]
    x2 = x[..., hd // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(s: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def kv_head_of(i: int, n_heads: int, n_kv_heads: int) -> int:
    return i // (n_heads // n_kv_heads)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """One new token attending to all cached positions (ATTENTION + ATTN_REDUCE, §8.2).

    q [Hq, hd]; k, v [Hkv, T, hd] hold positions 0..T-1 (the new one included).
    Returns o [Hq, hd] = sum_t softmax_t(q_i . k_t / sqrt(hd)) v_t per query head.
    """
    n_heads, hd = q.shape
    n_kv = k.shape[0]
    o = np.empty_like(q)
    for i in range(n_heads):
        j = kv_head_of(i, n_heads, n_kv)
        p = softmax(k[j] @ q[i] / np.sqrt(hd))
        o[i] = p @ v[j]
    return o


def silu(u: np.ndarray) -> np.ndarray:
    return u / (1.0 + np.exp(-u))


def argmax_lowest(z: np.ndarray) -> np.ndarray:
    """Greedy token: index of the largest logit, lowest index among ties (last axis)."""
    return np.argmax(z, axis=-1)          # numpy returns the first occurrence


# ---------------------------------------------------------------- split-KV partials
def split_partials(q: np.ndarray, k: np.ndarray, v: np.ndarray, bounds):
    """Flash-decoding partial results of one query head over position ranges (§8.2,
    ATTENTION).  For each range [t0, t1): m = max score, l = sum exp(s - m),
    o = sum exp(s - m) v (unnormalised).  Empty ranges give (-inf, 0, 0)."""
    hd = q.shape[-1]
    out = []
    for t0, t1 in bounds:
        if t1 <= t0:
            out.append((-np.inf, 0.0, np.zeros(hd)))
            continue
        s = k[t0:t1] @ q / np.sqrt(hd)
        m = np.max(s)
        e = np.exp(s - m)
        out.append((m, float(np.sum(e)), e @ v[t0:t1]))
    return out


def merge_partials(parts) -> np.ndarray:
    """Log-sum-exp merge of split partials into the normalised output (§8.2, ATTN_REDUCE)."""
    M = max(p[0] for p in parts)
    num = sum(np.exp(m - M) * o for m, _, o in parts if m != -np.inf)
    den = sum(np.exp(m - M) * l for m, l, _ in parts if m != -np.inf)
    return num / den


# ---------------------------------------------------------------- model
class Model:
    """fp64 view of the synthetic model.  `weights` follows synth.gen_weights' layout
    (uint16 storage bits); matrices are nn.Linear-style [out, in]."""

    def __init__(self, cfg, weights):
        self.cfg = cfg
        dt = cfg.dtype
        self.dtype = dt
        self._bits = weights
        self._cache = {}
        self.eps = float(cfg.rms_eps)
        self.theta = float(cfg.rope_theta)

    def w(self, name: str, layer: int = -1) -> np.ndarray:
        key = (name, layer)
        if key not in self._cache:
            src = self._bits[name] if layer < 0 else self._bits["layers"][layer][name]
            self._cache[key] = upcast(src, self.dtype)
        return self._cache[key]

    def embed_rows(self, tokens) -> np.ndarray:
        E = self._bits["embed"]
        return upcast(E[np.asarray(tokens)], self.dtype)


class KVCache:
    """Per layer k, v [B, Hkv, capacity, hd] as fp64 values of the storage dtype."""

    def __init__(self, cfg, batch: int, capacity: int):
        shape = (batch, cfg.n_kv_heads, capacity, cfg.head_dim)
        self.k = [np.zeros(shape) for _ in range(cfg.n_layers)]
        self.v = [np.zeros(shape) for _ in range(cfg.n_layers)]


def layer_step(m: Model, l: int, h: np.ndarray, cache: KVCache, pos) -> dict:
    """One decoder layer for B new tokens at positions pos[b] (the §8.2 ops in order).
    Returns the intermediate vectors (used by per-op parity checks)."""
    cfg = m.cfg
    B = h.shape[0]
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    # RMSNORM_QKV_ROPE
    x = rms_norm(h, m.w("attn_norm", l), m.eps)
    q = (x @ m.w("wq", l).T).reshape(B, Hq, hd)
    k = (x @ m.w("wk", l).T).reshape(B, Hkv, hd)
    v = (x @ m.w("wv", l).T).reshape(B, Hkv, hd)
    o = np.empty((B, Hq, hd))
    for b in range(B):
        t = int(pos[b])
        q[b] = apply_rope(q[b], t, m.theta)
        k[b] = apply_rope(k[b], t, m.theta)
        cache.k[l][b, :, t] = round_to_storage(k[b], m.dtype)
        cache.v[l][b, :, t] = round_to_storage(v[b], m.dtype)
        # ATTENTION + ATTN_REDUCE over positions 0..t
        o[b] = attention(q[b], cache.k[l][b, :, : t + 1], cache.v[l][b, :, : t + 1])
    # O_PROJ with the residual add
    h_mid = h + o.reshape(B, Hq * hd) @ m.w("wo", l).T
    # MLP_UP_GATE
    x2 = rms_norm(h_mid, m.w("mlp_norm", l), m.eps)
    a = silu(x2 @ m.w("w_gate", l).T) * (x2 @ m.w("w_up", l).T)
    # MLP_DOWN with the residual add
    h_out = h_mid + a @ m.w("w_down", l).T
    return {"x": x, "q": q, "k": k, "v": v, "o": o, "h_mid": h_mid, "a": a, "h_out": h_out}


def decode_step(m: Model, cache: KVCache, tokens, pos, keep=False):
    """One decode step for B sequences: token tokens[b] sits at position pos[b] and the
    cache already holds positions 0..pos[b]-1.  Returns logits [B, V] (and the per-layer
    intermediates when keep=True)."""
    h = m.embed_rows(tokens)
    trace = []
    for l in range(m.cfg.n_layers):
        r = layer_step(m, l, h, cache, pos)
        h = r["h_out"]
        if keep:
            trace.append(r)
    # LM_HEAD
    z = rms_norm(h, m.w("final_norm"), m.eps) @ m.w("lm_head").T
    return (z, trace) if keep else z


def prefill(m: Model, tokens: np.ndarray, cache: KVCache):
    """All prompt positions at once with a causal mask (batched form of decode_step).
    tokens [B, P]; writes cache positions 0..P-1; returns logits [B, P, V]."""
    cfg = m.cfg
    B, P = tokens.shape
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    G = Hq // Hkv
    h = m.embed_rows(tokens)                                   # [B, P, d]
    causal = np.tril(np.ones((P, P), dtype=bool))
    c_tab = np.stack([rope_cos_sin(t, hd, m.theta)[0] for t in range(P)])   # [P, hd/2]
    s_tab = np.stack([rope_cos_sin(t, hd, m.theta)[1] for t in range(P)])

    def rope_all(x):                                           # x [B, P, H, hd]
        x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
        c = c_tab[None, :, None, :]
        s = s_tab[None, :, None, :]
        return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)

    for l in range(cfg.n_layers):
        x = rms_norm(h, m.w("attn_norm", l), m.eps)
        q = rope_all((x @ m.w("wq", l).T).reshape(B, P, Hq, hd))
        k = round_to_storage(rope_all((x @ m.w("wk", l).T).reshape(B, P, Hkv, hd)), m.dtype)
        v = round_to_storage((x @ m.w("wv", l).T).reshape(B, P, Hkv, hd), m.dtype)
        cache.k[l][:, :, :P] = k.transpose(0, 2, 1, 3)
        cache.v[l][:, :, :P] = v.transpose(0, 2, 1, 3)
        o = np.empty((B, P, Hq, hd))
        for b in range(B):
            for i in range(Hq):
                j = i // G
                s = (q[b, :, i] @ k[b, :, j].T) / np.sqrt(hd)       # [P, P]
                s = np.where(causal, s, -np.inf)
                o[b, :, i] = softmax(s) @ v[b, :, j]
        h = h + o.reshape(B, P, Hq * hd) @ m.w("wo", l).T
        x2 = rms_norm(h, m.w("mlp_norm", l), m.eps)
        h = h + (silu(x2 @ m.w("w_gate", l).T) * (x2 @ m.w("w_up", l).T)) @ m.w("w_down", l).T
    return rms_norm(h, m.w("final_norm"), m.eps) @ m.w("lm_head").T


def greedy_generate(m: Model, prompt: np.ndarray, n_new: int, capacity=None):
    """Prompt [B, P] through decode steps (one position at a time), then n_new greedy
    tokens.  Returns (tokens [B, P + n_new], logits [B, P + n_new, V]) where logits[:, t]
    is the step that consumed tokens[:, t]."""
    B, P = prompt.shape
    cap = capacity or (P + n_new)
    cache = KVCache(m.cfg, B, cap)
    toks = np.zeros((B, P + n_new), dtype=np.int64)
    toks[:, :P] = prompt
    logits = []
    for t in range(P + n_new):
        z = decode_step(m, cache, toks[:, t], [t] * B)
        logits.append(z)
        if P <= t + 1 < P + n_new:
            toks[:, t + 1] = argmax_lowest(z)
    return toks, np.stack(logits, axis=1)


def top2_margin(z: np.ndarray) -> np.ndarray:
    """Gap between the largest and second-largest logit (last axis)."""
    s = np.sort(z, axis=-1)
    return s[..., -1] - s[..., -2]

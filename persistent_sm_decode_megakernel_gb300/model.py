"""Device-side model holder and a decoder handle over the C ABI.

PyTorch is used for device memory and streams only: weights and KV caches are torch
tensors on the GPU whose raw addresses go into mk_weights / mk_kv; all arithmetic of
the decode step runs in libmk.so.
"""
import ctypes

import numpy as np
import torch

from . import (MK_BF16, MK_F16, MK_OK, MK_ERR_NAN, check, mk_create, mk_decode_step, mk_decode_steps,
               mk_destroy, mk_get_trace, mk_info, mk_info_t, mk_kv, mk_model_desc, mk_options, mk_prefill,
               mk_read_activation, mk_reset, mk_synchronize, mk_trace_rec, mk_weights, P_i32)

_LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


def _to_device(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 storage bits -> int16 device tensor holding the same bytes."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device, non_blocking=False)


class DeviceModel:
    """Weights (storage bits) resident in HBM plus a KV cache of max_ctx positions."""

    def __init__(self, cfg, weights, max_batch, max_ctx, device="cuda:0"):
        self.cfg = cfg
        self.device = torch.device(device)
        self.max_batch = max_batch
        self.max_ctx = max_ctx
        self.embed = _to_device(weights["embed"], self.device)
        self.final_norm = _to_device(weights["final_norm"], self.device)
        self.lm_head = _to_device(weights["lm_head"], self.device)
        self.layers = [{n: _to_device(weights["layers"][l][n], self.device) for n in _LAYER_TENSORS}
                       for l in range(cfg.n_layers)]
        shape = (max_batch, cfg.n_kv_heads, max_ctx, cfg.head_dim)
        self.k_cache = [torch.zeros(shape, dtype=torch.int16, device=self.device) for _ in range(cfg.n_layers)]
        self.v_cache = [torch.zeros(shape, dtype=torch.int16, device=self.device) for _ in range(cfg.n_layers)]

    def desc(self):
        c = self.cfg
        return mk_model_desc(c.n_layers, c.d_model, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.vocab,
                             MK_F16 if c.dtype == "f16" else MK_BF16, c.rms_eps, c.rope_theta,
                             self.max_batch, self.max_ctx)

    def abi_structs(self):
        L = self.cfg.n_layers
        arr = ctypes.c_void_p * L
        tabs = {n: arr(*[self.layers[l][n].data_ptr() for l in range(L)]) for n in _LAYER_TENSORS}
        w = mk_weights(self.embed.data_ptr(), self.final_norm.data_ptr(), self.lm_head.data_ptr(),
                       *[ctypes.cast(tabs[n], ctypes.POINTER(ctypes.c_void_p)) for n in _LAYER_TENSORS])
        kt = arr(*[t.data_ptr() for t in self.k_cache])
        vt = arr(*[t.data_ptr() for t in self.v_cache])
        kv = mk_kv(ctypes.cast(kt, ctypes.POINTER(ctypes.c_void_p)), ctypes.cast(vt, ctypes.POINTER(ctypes.c_void_p)))
        return w, kv, (tabs, kt, vt)   # keep the host tables alive while mk_create reads them

    def set_kv(self, layer, b, k_bits, v_bits):
        """Fill positions 0..T-1 of sequence b's cache in one layer from storage bits
        [n_kv_heads, T, head_dim] (uint16)."""
        T = k_bits.shape[1]
        self.k_cache[layer][b, :, :T] = _to_device(k_bits, self.device)
        self.v_cache[layer][b, :, :T] = _to_device(v_bits, self.device)

    def weight_bytes(self):
        n = self.lm_head.numel() + self.final_norm.numel()
        for lt in self.layers:
            n += sum(t.numel() for t in lt.values())
        return 2 * n


def _i32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(P_i32)


class Decoder:
    """A context over a DeviceModel (mk_create ... mk_destroy)."""

    def __init__(self, dm: DeviceModel, sync_mode=0, exec_mode=0, trace=0, timeout_s=2.0, page_bytes=0,
                 n_pages=0, kv_splits=0, max_ctas=0, fault_drop_signal=0, backoff_max_ns=0,
                 split_min_positions=0, attn_merge=0, inflight_pages=0, attn_pool=0, attn_tensor_cores=0,
                 stream=None):
        self.dm = dm
        self.stream = stream if stream is not None else torch.cuda.current_stream(dm.device)
        self.opts = mk_options(sync_mode, exec_mode, page_bytes, n_pages, kv_splits, trace, timeout_s,
                               backoff_max_ns, max_ctas, fault_drop_signal, split_min_positions,
                               attn_merge, inflight_pages, attn_pool, attn_tensor_cores)
        d = dm.desc()
        w, kv, _keep = dm.abi_structs()
        h = ctypes.c_void_p()
        check(mk_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(kv), ctypes.byref(self.opts),
                        ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h)), "mk_create")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self):
        i = mk_info_t()
        check(mk_info(self.h, ctypes.byref(i)), "mk_info")
        return {k: getattr(i, k) for k, _ in mk_info_t._fields_}

    def prefill(self, tokens, logits=None, allow_nan=False):
        tokens = np.asarray(tokens, dtype=np.int32)
        B, P = tokens.shape
        t, tp = _i32(tokens)
        out, op = _i32(np.zeros(B))
        st = mk_prefill(self.h, tp, B, P, op, ctypes.c_void_p(logits.data_ptr() if logits is not None else 0))
        if not (allow_nan and st == MK_ERR_NAN):
            check(st, "mk_prefill")
        return out.copy()

    def decode_step(self, in_tok, pos, logits=None):
        B = len(in_tok)
        t, tp = _i32(in_tok)
        p, pp = _i32(pos)
        out, op = _i32(np.zeros(B))
        st = mk_decode_step(self.h, tp, pp, B, op, ctypes.c_void_p(logits.data_ptr() if logits is not None else 0))
        check(st, "mk_decode_step")
        return out.copy()

    def decode_step_status(self, in_tok, pos, logits=None):
        B = len(in_tok)
        t, tp = _i32(in_tok)
        p, pp = _i32(pos)
        out, op = _i32(np.zeros(B))
        st = mk_decode_step(self.h, tp, pp, B, op, ctypes.c_void_p(logits.data_ptr() if logits is not None else 0))
        return st, out.copy()

    def decode_steps(self, in_tok, pos0, n_steps, out_dev=None):
        """in_tok None continues from the token the previous step chose on the device."""
        B = len(pos0)
        if in_tok is None:
            tp = None
        else:
            t, tp = _i32(in_tok)
        p, pp = _i32(pos0)
        ptr = ctypes.c_void_p(out_dev.data_ptr() if out_dev is not None else 0)
        check(mk_decode_steps(self.h, tp, pp, B, n_steps, ptr), "mk_decode_steps")

    def synchronize(self):
        check(mk_synchronize(self.h), "mk_synchronize")

    def reset(self):
        check(mk_reset(self.h), "mk_reset")

    def read_activation(self, which, layer):
        c = self.dm.cfg
        width = {0: c.d_model, 1: c.d_model, 2: c.q_dim, 3: c.q_dim, 4: c.ffn_dim}[which]
        out = np.zeros((self.dm.max_batch, width), dtype=np.float32)
        check(mk_read_activation(self.h, which, layer, out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                 out.nbytes), "mk_read_activation")
        return out

    def trace(self, max_records=1 << 20):
        buf = (mk_trace_rec * max_records)()
        n = ctypes.c_int()
        check(mk_get_trace(self.h, buf, max_records, ctypes.byref(n)), "mk_get_trace")
        return [(r.cta, r.pc, r.op, r.layer, r.t_fetch, r.t_ready, r.t_end, *list(r.t_mark))
                for r in buf[: n.value]]

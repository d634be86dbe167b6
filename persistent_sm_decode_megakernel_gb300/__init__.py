"""Python binding of the persistent decode megakernel's C ABI (include/mk.h).

Argument marshalling only: every step of the decode path runs in the CUDA kernels of
libmk.so.  There is no CPU fallback -- importing this package fails loudly when the
library has not been built (`python -c "import __graft_entry__ as g; g.build()"`).
The functions keep the C names (mk_create, mk_prefill, mk_decode_step, ...) and return
the C status codes; `check(status)` raises MkError with mk_last_error()'s text.
"""
import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmk.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "mk.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with __graft_entry__.build(); the decode path has no CPU fallback")
lib = ctypes.CDLL(LIB_PATH)

MK_OK, MK_ERR_INVALID, MK_ERR_OCCUPANCY, MK_ERR_CUDA, MK_ERR_TIMEOUT, MK_ERR_STATE, MK_ERR_NAN = range(7)
MK_F16, MK_BF16 = 0, 1
MK_SYNC_COUNTER, MK_SYNC_SENTINEL = 0, 1
MK_EXEC_PERSISTENT, MK_EXEC_MULTILAUNCH, MK_EXEC_GRAPH = 0, 1, 2

c_int, c_float, c_double, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_void_p
P_void = ctypes.POINTER(ctypes.c_void_p)
P_i32 = ctypes.POINTER(ctypes.c_int32)
P_f32 = ctypes.POINTER(ctypes.c_float)


class mk_model_desc(ctypes.Structure):
    _fields_ = [("n_layers", c_int), ("d_model", c_int), ("n_heads", c_int), ("n_kv_heads", c_int),
                ("head_dim", c_int), ("ffn_dim", c_int), ("vocab", c_int), ("dtype", c_int),
                ("rms_eps", c_float), ("rope_theta", c_float), ("max_batch", c_int), ("max_ctx", c_int)]


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("final_norm", c_void_p), ("lm_head", c_void_p)] + [
        (n, P_void) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")]


class mk_kv(ctypes.Structure):
    _fields_ = [("k_cache", P_void), ("v_cache", P_void)]


class mk_options(ctypes.Structure):
    _fields_ = [("sync_mode", c_int), ("exec_mode", c_int), ("page_bytes", c_int), ("n_pages", c_int),
                ("kv_splits", c_int), ("trace", c_int), ("wait_timeout_s", c_double),
                ("backoff_max_ns", c_int), ("max_ctas", c_int), ("fault_drop_signal", c_int),
                ("split_min_positions", c_int),
                ("attn_merge", c_int), ("inflight_pages", c_int), ("attn_pool", c_int),
                ("attn_tensor_cores", c_int)]


class mk_info_t(ctypes.Structure):
    _fields_ = [("n_sm", c_int), ("blocks_per_sm", c_int), ("n_ctas", c_int), ("threads_per_cta", c_int),
                ("smem_bytes", c_int), ("page_bytes", c_int), ("n_pages", c_int), ("kv_splits", c_int),
                ("n_instructions", c_int), ("n_counters", c_int), ("launches_per_step", c_int),
                ("weight_bytes_per_step", ctypes.c_longlong), ("kernel_variant", c_int)]


class mk_trace_rec(ctypes.Structure):
    _fields_ = [("cta", ctypes.c_int32), ("pc", ctypes.c_int32), ("op", ctypes.c_int32), ("layer", ctypes.c_int32),
                ("t_fetch", ctypes.c_uint64), ("t_ready", ctypes.c_uint64), ("t_mark", ctypes.c_uint64 * 6),
                ("t_end", ctypes.c_uint64)]


def _fn(name, argtypes, restype=c_int):
    f = getattr(lib, name)
    f.argtypes = argtypes
    f.restype = restype
    return f


mk_create = _fn("mk_create", [ctypes.POINTER(mk_model_desc), ctypes.POINTER(mk_weights), ctypes.POINTER(mk_kv),
                              ctypes.POINTER(mk_options), c_void_p, ctypes.POINTER(c_void_p)])
mk_prefill = _fn("mk_prefill", [c_void_p, P_i32, c_int, c_int, P_i32, c_void_p])
mk_decode_step = _fn("mk_decode_step", [c_void_p, P_i32, P_i32, c_int, P_i32, c_void_p])
mk_decode_steps = _fn("mk_decode_steps", [c_void_p, P_i32, P_i32, c_int, c_int, c_void_p])
mk_synchronize = _fn("mk_synchronize", [c_void_p])
mk_reset = _fn("mk_reset", [c_void_p])
mk_destroy = _fn("mk_destroy", [c_void_p])
mk_info = _fn("mk_info", [c_void_p, ctypes.POINTER(mk_info_t)])
mk_get_trace = _fn("mk_get_trace", [c_void_p, ctypes.POINTER(mk_trace_rec), c_int, ctypes.POINTER(c_int)])
mk_read_activation = _fn("mk_read_activation", [c_void_p, c_int, c_int, P_f32, ctypes.c_size_t])
mk_plan = _fn("mk_plan", [ctypes.POINTER(mk_model_desc), ctypes.POINTER(mk_options), c_int,
                          ctypes.POINTER(mk_info_t)])
mk_selftest = _fn("mk_selftest", [c_int, ctypes.POINTER(ctypes.c_int64), c_int])
mk_barrier_bench = _fn("mk_barrier_bench", [c_int, c_int, ctypes.POINTER(c_double)])
mk_die_map = _fn("mk_die_map", [c_int, c_int, ctypes.POINTER(c_int), ctypes.POINTER(ctypes.c_float),
                                ctypes.POINTER(c_int)])
mk_two_groups = _fn("mk_two_groups", [ctypes.POINTER(ctypes.c_float), c_int, ctypes.POINTER(c_int),
                                      ctypes.POINTER(ctypes.c_float)])
mk_line_latency = _fn("mk_line_latency", [ctypes.c_longlong, ctypes.POINTER(ctypes.c_int64), c_int, c_int, c_int, c_int,
                                          ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)])
mk_stream_bench = _fn("mk_stream_bench", [c_int, c_int, c_int, c_int, ctypes.c_longlong, ctypes.POINTER(c_double)])
mk_decode_step_noalloc = _fn("mk_decode_step_noalloc", [ctypes.POINTER(mk_model_desc), ctypes.POINTER(mk_weights),
                                                        ctypes.POINTER(mk_kv), P_i32, P_i32, c_int, P_i32, c_void_p,
                                                        c_void_p])
mk_last_error = _fn("mk_last_error", [], ctypes.c_char_p)
mk_status_string = _fn("mk_status_string", [c_int], ctypes.c_char_p)


class MkError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        msg = mk_last_error().decode(errors="replace")
        super().__init__(f"{where}: {mk_status_string(status).decode()} ({status}): {msg}")


def check(status, where=""):
    if status != MK_OK:
        raise MkError(status, where)
    return status


def declared_functions():
    """Names of the functions include/mk.h declares (for the export check)."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:mk_status|const char \*)\s*(mk_\w+)\s*\(", text, re.M)))

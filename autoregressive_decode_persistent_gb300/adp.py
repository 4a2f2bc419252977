"""ctypes binding of the engine's C ABI (include/adp.h), with the same names.

Argument marshalling only: every step of the decode path runs in the CUDA kernels of
libadp.so. There is no fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libadp.so")
# The test build (libadp_test.so) also exports the test-only hooks; it is loaded instead of the
# release library when the environment sets ADP_TEST_HOOKS=1 (the test suite does).
TEST_LIB_PATH = os.path.join(_HERE, "libadp_test.so")
TEST_HOOKS = ("adp_debug_set_epoch_base", "adp_debug_set_wait_limit", "adp_debug_skip_publication")


def default_library_path() -> str:
    return TEST_LIB_PATH if os.environ.get("ADP_TEST_HOOKS") == "1" else LIB_PATH

ADP_F16, ADP_BF16, ADP_E4M3, ADP_F32, ADP_NVFP4 = 0, 1, 2, 3, 4
DTYPES = {"f16": ADP_F16, "bf16": ADP_BF16, "e4m3": ADP_E4M3, "f32": ADP_F32, "nvfp4": ADP_NVFP4}

ADP_OK = 0
ADP_ERR_INVALID_ARG = -1
ADP_ERR_UNSUPPORTED_CONFIG = -2
ADP_ERR_CONTEXT_OVERFLOW = -3
ADP_ERR_CUDA = -4
ADP_ERR_NOT_CORESIDENT = -5
ADP_ERR_BARRIER_TIMEOUT = -6
ADP_ERR_PIPELINE_TIMEOUT = -7
ADP_ERR_UNIMPLEMENTED = -8


class AdpError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = status_string(code)
        if code == ADP_ERR_CUDA:
            msg += ": " + last_error()
        super().__init__(f"{where}: {msg} ({code})")


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim",
                                               "d_ff", "vocab", "max_ctx")] + \
               [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)] + \
               [(n, ctypes.c_int32) for n in ("tied_embeddings", "weight_dtype", "kv_dtype", "n_experts",
                                               "top_k", "d_expert", "router_dtype", "expert_dtype",
                                               "embed_dtype")]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up",
                                                "w_down", "router", "e_gate", "e_up", "e_down", "e_gate_scale",
                                                "e_up_scale", "e_down_scale", "wq_scale", "wk_scale", "wv_scale",
                                                "wo_scale", "w_gate_scale", "w_up_scale", "w_down_scale",
                                                "wq_bscale", "wk_bscale", "wv_bscale", "wo_bscale",
                                                "w_gate_bscale", "w_up_bscale", "w_down_bscale")]


class Weights(ctypes.Structure):
    _fields_ = [("tok_emb", ctypes.c_void_p), ("lm_head", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeights))]


class Sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("u", ctypes.c_float)]


class PhasePlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("kind", "layer", "n_units", "unit_rows", "slots", "K", "KC",
                                               "n_chunks", "upr", "dtype", "src_phase", "res_phase",
                                               "sel_phase", "replicated")] + \
               [("region", ctypes.c_uint64), ("expert_stride", ctypes.c_uint64)]


class BatchLayout(ctypes.Structure):
    _fields_ = [("ring_slots", ctypes.c_int32), ("attention_slots", ctypes.c_int32), ("xbuf_floats", ctypes.c_int32),
                ("down_segment", ctypes.c_int32), ("control_bytes", ctypes.c_uint64), ("smem_bytes", ctypes.c_uint64)]


_lib = None

# (name, restype, argtypes)
_SIGS = [
    ("adp_create_model", ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(Weights), ctypes.c_void_p,
                                        ctypes.POINTER(ctypes.c_void_p)]),
    ("adp_destroy_model", None, [ctypes.c_void_p]),
    ("adp_kv_create", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    ("adp_kv_destroy", None, [ctypes.c_void_p]),
    ("adp_kv_reset", ctypes.c_int, [ctypes.c_void_p]),
    ("adp_kv_truncate", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("adp_kv_len", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    ("adp_kv_load", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]),
    ("adp_kv_read", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]),
    ("adp_decode_step", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(Sampling),
                                       ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]),
    ("adp_decode_step_noalloc", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                               ctypes.POINTER(Sampling), ctypes.POINTER(ctypes.c_int32),
                                               ctypes.c_void_p]),
    ("adp_prefill", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                   ctypes.POINTER(Sampling), ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]),
    ("adp_prefill_tc", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                      ctypes.POINTER(Sampling), ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]),
    ("adp_generate_async", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]),
    ("adp_sync", ctypes.c_int, [ctypes.c_void_p]),
    ("adp_decode_batch", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.POINTER(Sampling), ctypes.c_void_p, ctypes.c_void_p]),
    ("adp_generate_batch_async", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    ("adp_max_batch", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    ("adp_debug_tc_gemm_time", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.POINTER(ctypes.c_float)]),
    ("adp_debug_tc_gemm", ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    ("adp_reset", ctypes.c_int, [ctypes.c_void_p]),
    ("adp_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("adp_last_error", ctypes.c_char_p, []),
    ("adp_num_ctas", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    ("adp_image_bytes", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64)]),
    ("adp_plan", ctypes.c_int, [ctypes.POINTER(Config), ctypes.c_int32, ctypes.POINTER(PhasePlan), ctypes.c_int32,
                                ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_uint64)]),
    ("adp_batch_plan", ctypes.c_int, [ctypes.POINTER(Config), ctypes.c_int32, ctypes.c_int32,
                                      ctypes.POINTER(BatchLayout), ctypes.POINTER(ctypes.c_int32)]),
    ("adp_launches_per_step", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    ("adp_debug_kernel_mode", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    ("adp_debug_force_experts", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    ("adp_debug_read_experts", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    ("adp_debug_trace_residual", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    ("adp_debug_timeline", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    ("adp_debug_timeline_shape", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                                                ctypes.POINTER(ctypes.c_int32)]),
    ("adp_debug_barriers", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    ("adp_debug_set_l2_lookahead", ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32]),
    ("adp_debug_set_prefetch_flags", ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32]),
    ("adp_debug_set_l2_pacing", ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32]),
    ("adp_measure_read_bandwidth", ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int32, ctypes.c_void_p,
                                                  ctypes.POINTER(ctypes.c_double)]),
    ("adp_debug_set_ring_slots", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("adp_debug_ring_slots", ctypes.c_int, [ctypes.c_void_p]),
    ("adp_debug_set_epoch_base", ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32]),
    ("adp_debug_set_wait_limit", ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint64]),
    ("adp_debug_skip_publication", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]),
]


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libadp.so (build it first with autoregressive_decode_persistent_gb300.build.build())."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or default_library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: the CUDA engine must be built (no CPU fallback exists)")
    L = ctypes.CDLL(p)
    for name, res, args in _SIGS:
        if name in TEST_HOOKS and not hasattr(L, name):
            continue  # the release build: calling the hook raises below
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = L
    return L


def _hook(name: str):
    L = load_library()
    if not hasattr(L, name):
        raise RuntimeError(f"{name} is a test-only hook: load the test build (ADP_TEST_HOOKS=1, libadp_test.so)")
    return getattr(L, name)


def _check(rc: int, where: str):
    if rc != ADP_OK:
        raise AdpError(rc, where)


def status_string(code: int) -> str:
    return load_library().adp_status_string(code).decode()


def last_error() -> str:
    return load_library().adp_last_error().decode()


def _ptr(x) -> int | None:
    """Device or host address of a torch tensor / numpy array / int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


# ---------------------------------------------------------------- the C ABI, one to one

def adp_create_model(cfg: Config, weights: Weights, stream: int = 0):
    h = ctypes.c_void_p()
    _check(load_library().adp_create_model(ctypes.byref(cfg), ctypes.byref(weights), stream or None,
                                           ctypes.byref(h)), "adp_create_model")
    return h


def adp_destroy_model(model):
    load_library().adp_destroy_model(model)


def adp_kv_create(model):
    h = ctypes.c_void_p()
    _check(load_library().adp_kv_create(model, ctypes.byref(h)), "adp_kv_create")
    return h


def adp_kv_destroy(kv):
    load_library().adp_kv_destroy(kv)


def adp_kv_reset(kv):
    _check(load_library().adp_kv_reset(kv), "adp_kv_reset")


def adp_kv_truncate(kv, length: int):
    _check(load_library().adp_kv_truncate(kv, int(length)), "adp_kv_truncate")


def adp_kv_len(kv) -> int:
    n = ctypes.c_int32()
    _check(load_library().adp_kv_len(kv, ctypes.byref(n)), "adp_kv_len")
    return n.value


def adp_kv_load(kv, host_k: np.ndarray, host_v: np.ndarray, length: int):
    _check(load_library().adp_kv_load(kv, _ptr(np.ascontiguousarray(host_k)), _ptr(np.ascontiguousarray(host_v)),
                                      length), "adp_kv_load")


def adp_kv_read(kv, host_k: np.ndarray, host_v: np.ndarray, length: int):
    assert host_k.flags["C_CONTIGUOUS"] and host_v.flags["C_CONTIGUOUS"]
    _check(load_library().adp_kv_read(kv, _ptr(host_k), _ptr(host_v), length), "adp_kv_read")


def _sampling(temperature: float, u: float):
    return ctypes.byref(Sampling(float(temperature), float(u))) if temperature > 0 else None


def adp_decode_step(model, kv, token: int, temperature: float = 0.0, u: float = 0.0, dev_logits=None) -> int:
    nxt = ctypes.c_int32()
    _check(load_library().adp_decode_step(model, kv, int(token), _sampling(temperature, u), ctypes.byref(nxt),
                                          _ptr(dev_logits)), "adp_decode_step")
    return nxt.value


def adp_decode_step_noalloc(model, kv, token: int, temperature: float = 0.0, u: float = 0.0,
                            dev_logits=None) -> int:
    nxt = ctypes.c_int32()
    _check(load_library().adp_decode_step_noalloc(model, kv, int(token), _sampling(temperature, u),
                                                  ctypes.byref(nxt), _ptr(dev_logits)), "adp_decode_step_noalloc")
    return nxt.value


def adp_prefill(model, kv, tokens, temperature: float = 0.0, u: float = 0.0, dev_logits=None) -> int:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    nxt = ctypes.c_int32()
    _check(load_library().adp_prefill(model, kv, _ptr(t), len(t), _sampling(temperature, u), ctypes.byref(nxt),
                                      _ptr(dev_logits)), "adp_prefill")
    return nxt.value


def adp_prefill_tc(model, kv, tokens, temperature: float = 0.0, u: float = 0.0, dev_logits=None) -> int:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    nxt = ctypes.c_int32()
    _check(load_library().adp_prefill_tc(model, kv, _ptr(t), len(t), _sampling(temperature, u), ctypes.byref(nxt),
                                         _ptr(dev_logits)), "adp_prefill_tc")
    return nxt.value


def adp_generate_async(model, kv, token: int, n: int, temperature: float, dev_u, dev_tokens_out):
    _check(load_library().adp_generate_async(model, kv, int(token), int(n), float(temperature), _ptr(dev_u),
                                             _ptr(dev_tokens_out)), "adp_generate_async")


def adp_sync(model):
    _check(load_library().adp_sync(model), "adp_sync")


def _kv_table(kvs):
    """HOST array of adp_kv handles (kept alive by the caller for the duration of the call)."""
    return (ctypes.c_void_p * len(kvs))(*[k.value if isinstance(k, ctypes.c_void_p) else k for k in kvs])


def adp_decode_batch(model, kvs, tokens, temperatures=None, us=None, dev_logits=None) -> list[int]:
    """One batched step: kvs[r] takes tokens[r]; returns the chosen tokens (HOST list)."""
    nb = len(kvs)
    table = _kv_table(kvs)
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    assert len(tok) == nb
    samp = None
    if temperatures is not None:
        arr = (Sampling * nb)(*[Sampling(float(temperatures[r]), float(us[r] if us is not None else 0.0))
                                for r in range(nb)])
        samp = ctypes.cast(arr, ctypes.POINTER(Sampling))
    out = np.zeros(nb, dtype=np.int32)
    _check(load_library().adp_decode_batch(model, table, nb, _ptr(tok), samp, _ptr(out), _ptr(dev_logits)),
           "adp_decode_batch")
    return [int(t) for t in out]


def adp_generate_batch_async(model, kvs, tokens, n: int, temperatures=None, dev_u=None, dev_tokens_out=None):
    nb = len(kvs)
    table = _kv_table(kvs)
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    assert len(tok) == nb
    temps = None if temperatures is None else np.ascontiguousarray(temperatures, dtype=np.float32)
    _check(load_library().adp_generate_batch_async(model, table, nb, _ptr(tok), int(n), _ptr(temps), _ptr(dev_u),
                                                   _ptr(dev_tokens_out)), "adp_generate_batch_async")


def adp_debug_tc_gemm(bf16: bool, A, W, C):
    """C = A W^T on the tensor cores (A [M, K], W [N, K] 16-bit, C [M, N] fp32; device tensors)."""
    M, K = A.shape
    N = W.shape[0]
    _check(load_library().adp_debug_tc_gemm(int(bf16), M, N, K, _ptr(A), _ptr(W), _ptr(C)), "adp_debug_tc_gemm")


def adp_debug_tc_gemm_time(model, which: int, M: int, reps: int) -> float:
    ms = ctypes.c_float()
    _check(load_library().adp_debug_tc_gemm_time(model, int(which), int(M), int(reps), ctypes.byref(ms)),
           "adp_debug_tc_gemm_time")
    return ms.value


def adp_max_batch(model) -> int:
    nb = ctypes.c_int32()
    _check(load_library().adp_max_batch(model, ctypes.byref(nb)), "adp_max_batch")
    return nb.value


def adp_reset(model):
    _check(load_library().adp_reset(model), "adp_reset")


def adp_num_ctas(model) -> int:
    n = ctypes.c_int32()
    _check(load_library().adp_num_ctas(model, ctypes.byref(n)), "adp_num_ctas")
    return n.value


def adp_image_bytes(model) -> int:
    n = ctypes.c_uint64()
    _check(load_library().adp_image_bytes(model, ctypes.byref(n)), "adp_image_bytes")
    return n.value


def adp_plan(config: Config, n_sms: int) -> tuple[list[dict], int]:
    """The phase plan and weight-image size of a config on a GPU with n_sms SMs (host only)."""
    L = load_library()
    n, img = ctypes.c_int32(), ctypes.c_uint64()
    _check(L.adp_plan(ctypes.byref(config), n_sms, None, 0, ctypes.byref(n), ctypes.byref(img)), "adp_plan")
    out = (PhasePlan * n.value)()
    _check(L.adp_plan(ctypes.byref(config), n_sms, out, n.value, ctypes.byref(n), ctypes.byref(img)), "adp_plan")
    return [{f: getattr(p, f) for f, _ in PhasePlan._fields_} for p in out], img.value


def adp_batch_plan(config: Config, n_sms: int, smem_optin: int) -> tuple[list[dict], int]:
    """The batched kernel's layout for 1..4 requests and the largest batch that fits (host only)."""
    out = (BatchLayout * 4)()
    mb = ctypes.c_int32()
    _check(load_library().adp_batch_plan(ctypes.byref(config), n_sms, smem_optin, out, ctypes.byref(mb)),
           "adp_batch_plan")
    return [{f: getattr(o, f) for f, _ in BatchLayout._fields_} for o in out], mb.value


def adp_launches_per_step(model) -> int:
    n = ctypes.c_int32()
    _check(load_library().adp_launches_per_step(model, ctypes.byref(n)), "adp_launches_per_step")
    return n.value


def adp_debug_kernel_mode(model, mode: int):
    _check(load_library().adp_debug_kernel_mode(model, mode), "adp_debug_kernel_mode")


def adp_debug_force_experts(model, host_idx):
    arr = None if host_idx is None else np.ascontiguousarray(host_idx, dtype=np.int32)
    _check(load_library().adp_debug_force_experts(model, _ptr(arr)), "adp_debug_force_experts")


def adp_debug_read_experts(model, n_layers: int, top_k: int) -> np.ndarray:
    out = np.zeros((n_layers, top_k), dtype=np.int32)
    _check(load_library().adp_debug_read_experts(model, _ptr(out)), "adp_debug_read_experts")
    return out


def adp_debug_trace_residual(model, dev_buf):
    _check(load_library().adp_debug_trace_residual(model, _ptr(dev_buf)), "adp_debug_trace_residual")


def adp_debug_timeline(model, dev_buf):
    _check(load_library().adp_debug_timeline(model, _ptr(dev_buf)), "adp_debug_timeline")


def adp_debug_timeline_shape(model):
    c, p = ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().adp_debug_timeline_shape(model, ctypes.byref(c), ctypes.byref(p)),
           "adp_debug_timeline_shape")
    return c.value, p.value


def adp_debug_barriers(model, on: bool):
    _check(load_library().adp_debug_barriers(model, 1 if on else 0), "adp_debug_barriers")


def adp_debug_set_l2_lookahead(model, nbytes: int):
    _check(load_library().adp_debug_set_l2_lookahead(model, int(nbytes)), "adp_debug_set_l2_lookahead")


def adp_measure_read_bandwidth(dev_buf, nbytes: int, reps: int, stream: int = 0) -> float:
    """GB/s of 16-byte reads over a device buffer (see include/adp.h)."""
    g = ctypes.c_double()
    _check(load_library().adp_measure_read_bandwidth(_ptr(dev_buf), int(nbytes), int(reps), stream or None,
                                                      ctypes.byref(g)), "adp_measure_read_bandwidth")
    return g.value


def adp_debug_set_l2_pacing(model, bytes_per_us: int, burst_bytes: int):
    _check(load_library().adp_debug_set_l2_pacing(model, int(bytes_per_us), int(burst_bytes)),
           "adp_debug_set_l2_pacing")


def adp_debug_set_prefetch_flags(model, flags: int):
    _check(load_library().adp_debug_set_prefetch_flags(model, int(flags)), "adp_debug_set_prefetch_flags")


def adp_debug_set_ring_slots(model, slots: int):
    _check(load_library().adp_debug_set_ring_slots(model, int(slots)), "adp_debug_set_ring_slots")


def adp_debug_ring_slots(model) -> int:
    return int(load_library().adp_debug_ring_slots(model))


def adp_debug_set_epoch_base(model, base: int):
    _check(_hook("adp_debug_set_epoch_base")(model, int(base)), "adp_debug_set_epoch_base")


def adp_debug_set_wait_limit(model, ns: int):
    _check(_hook("adp_debug_set_wait_limit")(model, int(ns)), "adp_debug_set_wait_limit")


def adp_debug_skip_publication(model, cta: int, phase: int):
    _check(_hook("adp_debug_skip_publication")(model, int(cta), int(phase)), "adp_debug_skip_publication")

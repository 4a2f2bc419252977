"""ctypes wrapper of oracle.c (test infrastructure only; shares no code with the engine).

The C file computes one decode step of the decoder on the CPU in fp32, in two modes:
PLAIN (the textbook step) and EXACT (the same step under the engine's stated
arithmetic contract, for bit-level comparison). See the header of oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

PLAIN, EXACT = 0, 1
_DT = {"f16": 0, "bf16": 1, "e4m3": 2, "f32": 3, "nvfp4": 4}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_c(src: str, out: str) -> str:
    """Compile an oracle source file into a shared library with the oracle's flags."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-ffp-contract=off",
                           "-Wall", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build_lib(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    return compile_c(src, _LIB_PATH)


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim",
                                               "d_ff", "vocab", "max_ctx")] + \
               [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)] + \
               [(n, ctypes.c_int32) for n in ("tied_embeddings", "weight_dtype", "kv_dtype", "n_experts",
                                               "top_k", "d_expert", "router_dtype", "expert_dtype",
                                               "embed_dtype")]


class Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate",
                                                "w_up", "w_down", "router", "e_gate", "e_up", "e_down",
                                                "e_gate_scale", "e_up_scale", "e_down_scale",
                                                "wq_scale", "wk_scale", "wv_scale", "wo_scale",
                                                "w_gate_scale", "w_up_scale", "w_down_scale",
                                                "wq_bscale", "wk_bscale", "wv_bscale", "wo_bscale",
                                                "w_gate_bscale", "w_up_bscale", "w_down_bscale")]


class Weights(ctypes.Structure):
    _fields_ = [("tok_emb", ctypes.c_void_p), ("lm_head", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(Layer))]


def load(path: str):
    """oracle.c's functions from a compiled copy at `path`, with their signatures set."""
    L = ctypes.CDLL(path)
    vp, f32, i32 = ctypes.c_void_p, ctypes.c_float, ctypes.c_int32
    L.orc_init.argtypes = []
    L.orc_step.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, vp, i32, i32, i32, f32, f32,
                           vp, vp, vp, vp, vp, vp]
    L.orc_step.restype = ctypes.c_int
    L.orc_exp_c.argtypes = [f32]
    L.orc_exp_c.restype = f32
    L.orc_dot_exact.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int]
    L.orc_dot_exact.restype = f32
    L.orc_dot_plain.argtypes = [vp, vp, ctypes.c_int]
    L.orc_dot_plain.restype = f32
    L.orc_rmsnorm.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, f32, ctypes.c_int, vp]
    L.orc_rope_row.argtypes = [f32, ctypes.c_int, ctypes.c_int, vp, vp]
    L.orc_rope.argtypes = [vp, ctypes.c_int, ctypes.c_int, f32, ctypes.c_int]
    L.orc_attention_head.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, f32,
                                     ctypes.c_int, vp]
    L.orc_route.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp]
    L.orc_argmax.argtypes = [vp, ctypes.c_int]
    L.orc_argmax.restype = i32
    L.orc_sample.argtypes = [vp, ctypes.c_int, f32, f32, ctypes.c_int]
    L.orc_sample.restype = i32
    L.orc_round_f16.argtypes = [f32]
    L.orc_round_f16.restype = ctypes.c_uint16
    L.orc_round_bf16.argtypes = [f32]
    L.orc_round_bf16.restype = ctypes.c_uint16
    L.orc_e4m3_table.argtypes = []
    L.orc_e4m3_table.restype = ctypes.POINTER(ctypes.c_float)
    L.orc_gemv.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, ctypes.c_int]
    L.orc_gemv.restype = ctypes.c_int
    L.orc_dot_nvfp4.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int]
    L.orc_dot_nvfp4.restype = f32
    L.orc_e2m1_table.argtypes = []
    L.orc_e2m1_table.restype = ctypes.POINTER(ctypes.c_float)
    L.orc_init()
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build_lib()
            _lib = load(_LIB_PATH)
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a):
    return None if a is None else np.ascontiguousarray(a)


class OracleModel:
    """Host model + host KV cache; `step` runs one decode step in the chosen mode."""

    def __init__(self, cfg: dict, W: dict, library=None):
        """library: the compiled oracle to call (default: oracle.c as built by build_lib)."""
        self.cfg = cfg
        self._lib = library
        self.W = W
        c = cfg
        self.c = Config(c["n_layers"], c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"],
                        c.get("d_ff", 0), c["vocab"], c["max_ctx"], c["rms_eps"], c["rope_theta"],
                        1 if c["tied_embeddings"] else 0, _DT[c["weight_dtype"]], _DT[c["kv_dtype"]],
                        c["n_experts"], c["top_k"], c["d_expert"], _DT[c["router_dtype"]], _DT[c["expert_dtype"]],
                        _DT[c.get("embed_dtype") or c["weight_dtype"]])
        self._keep = []
        layers = (Layer * c["n_layers"])()
        for i, Lw in enumerate(W["layers"]):
            f = {}
            for k in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down", "router",
                      "e_gate", "e_up", "e_down", "e_gate_scale", "e_up_scale", "e_down_scale",
                      "wq_scale", "wk_scale", "wv_scale", "wo_scale", "w_gate_scale", "w_up_scale",
                      "w_down_scale", "wq_bscale", "wk_bscale", "wv_bscale", "wo_bscale", "w_gate_bscale",
                      "w_up_bscale", "w_down_bscale"):
                a = _c(Lw.get(k))
                self._keep.append(a)
                f[k] = _p(a)
            layers[i] = Layer(**f)
        self._layers = layers
        te, lm, fn = _c(W["tok_emb"]), _c(W.get("lm_head")), _c(W["final_norm"])
        self._keep += [te, lm, fn]
        self.w = Weights(_p(te), _p(lm), _p(fn), layers)
        shp = (c["n_layers"], c["n_kv_heads"], c["max_ctx"], c["head_dim"])
        self.kc = np.zeros(shp, dtype=np.uint16)
        self.vc = np.zeros(shp, dtype=np.uint16)
        self.len = 0

    def reset(self):
        self.kc[:] = 0
        self.vc[:] = 0
        self.len = 0

    def load_kv_prefix(self, k: np.ndarray, v: np.ndarray):
        n = k.shape[2]
        self.kc[:, :, :n, :] = k
        self.vc[:, :, :n, :] = v
        self.len = n

    def step(self, token: int, mode: int = PLAIN, temperature: float = 0.0, u: float = 0.0, force=None,
             trace: bool = False, pos: int | None = None):
        c = self.cfg
        pos = self.len if pos is None else pos
        logits = np.empty((c["vocab"],), dtype=np.float32)
        nxt = np.zeros((1,), dtype=np.int32)
        k = max(c["top_k"], 1)
        sel = np.zeros((c["n_layers"], k), dtype=np.int32)
        gate = np.zeros((c["n_layers"], k), dtype=np.float32)
        tr = np.zeros((c["n_layers"] + 1, c["d_model"]), dtype=np.float32) if trace else None
        fz = None if force is None else np.ascontiguousarray(force, dtype=np.int32)
        rc = (self._lib or lib()).orc_step(ctypes.byref(self.c), ctypes.byref(self.w), _p(self.kc), _p(self.vc), pos, int(token),
                            mode, float(temperature), float(u), _p(fz), _p(logits), _p(nxt), _p(sel), _p(gate),
                            _p(tr))
        if rc != 0:
            raise RuntimeError(f"orc_step failed: {rc}")
        self.len = pos + 1
        out = {"logits": logits, "next": int(nxt[0])}
        if c["n_experts"]:
            out["experts"], out["gates"] = sel, gate
        if trace:
            out["trace"] = tr
        return out

    def prefill(self, tokens, mode: int = PLAIN, **kw):
        out = None
        for t in tokens:
            out = self.step(int(t), mode, **kw)
        return out

"""Seeded synthetic inputs shared by the CUDA engine's tests/bench and the CPU oracle.

Holds no arithmetic of the decode step: it draws weights (std 0.02 normals
rounded to the storage dtype, RMSNorm gains 1.0, row-scaled e4m3 experts),
prompt ids, sampling uniforms and synthetic KV prefixes, and describes the
workload shapes. Both sides then read the same bytes.

The workloads are the five decoder configurations of the single-request decode
study in "Real-time LLM inference on standard GPUs: 3,000 tokens/s per request"
(Kog AI; summarised at hakusoku.com, section "GPU推論の速度制限要因：メモリ帯域幅",
and aether-echoes.com, section "モデルは 2B・HumanEval 50%": a 2.3B FP16
decoder, 25 layers, context 4096, batch 1), with trained weights replaced by
seeded random ones of the same shapes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import CONFIGS, get_config, shrink  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Seeds (fixed per workload): weights = 1000 + index, prompt = 2000 + index,
# sampling stream = 3000, synthetic KV prefix = 4000 + index.
SEED_WEIGHTS = 1000
SEED_PROMPT = 2000
SEED_SAMPLING = 3000
SEED_KV = 4000

WEIGHT_STD = 0.02


def build_lib(force: bool = False) -> str:
    """Compile gen.c into libsynth.so beside it (gcc, OpenMP)."""
    src = os.path.join(_HERE, "gen.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
                           "-ffp-contract=off", "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build_lib()
            L = ctypes.CDLL(_LIB_PATH)
            u64, f32, sz = ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
            vp = ctypes.c_void_p
            L.synth_normal_f32.argtypes = [u64, u64, f32, vp, sz]
            L.synth_normal_f16.argtypes = [u64, u64, f32, vp, sz]
            L.synth_normal_bf16.argtypes = [u64, u64, f32, vp, sz]
            L.synth_normal_e4m3_rows.argtypes = [u64, u64, f32, sz, sz, vp, vp]
            L.synth_f32_to_f16.argtypes = [vp, vp, sz]
            L.synth_f32_to_bf16.argtypes = [vp, vp, sz]
            L.synth_f32_to_e4m3.argtypes = [vp, vp, sz]
            L.synth_tokens.argtypes = [u64, u64, ctypes.c_uint32, vp, sz]
            L.synth_uniforms.argtypes = [u64, u64, vp, sz]
            L.synth_key.argtypes = [u64, u64]
            L.synth_key.restype = u64
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- primitives

def normal_f32(seed: int, tensor_id: int, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().synth_normal_f32(seed, tensor_id, std, _ptr(out), out.size)
    return out


def normal_stored(seed: int, tensor_id: int, shape, dtype: str, std: float = WEIGHT_STD) -> np.ndarray:
    """std-normal draws x std, rounded RNE to 'f16' or 'bf16'. Returned as raw uint16 bits."""
    out = np.empty(shape, dtype=np.uint16)
    if dtype == "f16":
        lib().synth_normal_f16(seed, tensor_id, std, _ptr(out), out.size)
    elif dtype == "bf16":
        lib().synth_normal_bf16(seed, tensor_id, std, _ptr(out), out.size)
    else:
        raise ValueError(dtype)
    return out


def normal_e4m3_rows(seed: int, tensor_id: int, rows: int, cols: int, std: float = WEIGHT_STD):
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty((rows,), dtype=np.float32)
    lib().synth_normal_e4m3_rows(seed, tensor_id, std, rows, cols, _ptr(q), _ptr(s))
    return q, s


# Magnitudes of the 4-bit E2M1 codes 0..7 (code = 2 * exponent field + fraction bit) and the
# midpoints between neighbours, for round-to-nearest-even quantisation.
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)
_E2M1_MID = (_E2M1_MAG[:-1] + _E2M1_MAG[1:]) / 2


def normal_nvfp4_rows(seed: int, tensor_id: int, rows: int, cols: int, std: float = WEIGHT_STD):
    """NVFP4 quantisation of seeded N(0, std) fp32 draws (an input recipe, not engine arithmetic):
    per row s = max|w| / (6 * 448) (fp32); per 16-element block the scale b = e4m3_RNE(max|w_block|
    / (6 s)); elements q = e2m1_RNE(w / (s * b)), saturating at 6, ties to the even code.
    Returns (codes [rows, cols/2] uint8, element 2i in the low nibble; block scales [rows, cols/16]
    uint8 e4m3; row scales [rows] float32)."""
    assert cols % 16 == 0
    w = normal_f32(seed, tensor_id, (rows, cols), std)
    amax = np.abs(w).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(6.0 * 448.0), np.float32(1.0)).astype(np.float32)
    blk = np.abs(w.reshape(rows, cols // 16, 16)).max(axis=2)
    b_codes = f32_to_stored((blk / (np.float32(6.0) * s[:, None])).astype(np.float32), "e4m3")
    b = _e4m3_values(b_codes)
    denom = (s[:, None] * b).astype(np.float32)
    denom16 = np.repeat(denom, 16, axis=1)
    a = np.where(denom16 > 0, np.abs(w) / np.where(denom16 > 0, denom16, 1), 0).astype(np.float32)
    k = np.searchsorted(_E2M1_MID, a, side="left")
    tie = (k < 7) & (a == _E2M1_MID[np.minimum(k, 6)])
    k = np.where(tie & (k % 2 == 1), k + 1, k)
    k = np.minimum(k, 7)
    code = (k | np.where((w < 0) & (k > 0), 8, 0)).astype(np.uint8)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, b_codes.astype(np.uint8), s


def _e4m3_values(q: np.ndarray) -> np.ndarray:
    """fp32 values of e4m3 codes (finite codes only: the quantiser never stores NaN)."""
    q = q.astype(np.int64)
    e, m = (q >> 3) & 15, q & 7
    v = np.where(e == 0, m * 2.0 ** -9, (8 + m) * 2.0 ** (e - 10.0))
    return np.where(q & 0x80, -v, v).astype(np.float32)


def f32_to_stored(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "e4m3":
        out = np.empty(x.shape, dtype=np.uint8)
        lib().synth_f32_to_e4m3(_ptr(x), _ptr(out), x.size)
        return out
    out = np.empty(x.shape, dtype=np.uint16)
    if dtype == "f16":
        lib().synth_f32_to_f16(_ptr(x), _ptr(out), x.size)
    elif dtype == "bf16":
        lib().synth_f32_to_bf16(_ptr(x), _ptr(out), x.size)
    else:
        raise ValueError(dtype)
    return out


def ones_stored(n: int, dtype: str) -> np.ndarray:
    """RMSNorm gains: exactly 1.0 in the storage dtype."""
    return np.full((n,), 0x3C00 if dtype == "f16" else 0x3F80, dtype=np.uint16)


def tokens(seed: int, stream_id: int, n: int, vocab: int) -> np.ndarray:
    out = np.empty((n,), dtype=np.int32)
    lib().synth_tokens(seed, stream_id, vocab, _ptr(out), n)
    return out


def uniforms(seed: int, first: int, n: int) -> np.ndarray:
    out = np.empty((n,), dtype=np.float32)
    lib().synth_uniforms(seed, first, _ptr(out), n)
    return out


# ---------------------------------------------------------------- tensor ids

def _tid_layer(layer: int, kind: int) -> int:
    return 1000 + layer * 64 + kind


def _tid_expert(layer: int, expert: int, kind: int) -> int:
    return 1_000_000 + (layer * 1024 + expert) * 4 + kind


TID_EMB, TID_LM = 1, 2
K_WQ, K_WK, K_WV, K_WO, K_WG, K_WU, K_WD, K_ROUTER = range(8)
E_GATE, E_UP, E_DOWN = range(3)


# ---------------------------------------------------------------- model weights

def model_weights(cfg: dict, seed: int | None = None) -> dict:
    """Host copies of every stored tensor of a model, as numpy arrays of raw bits.

    Layout (row-major [out, in]):
      tok_emb [V, d]; lm_head [V, d] (None when tied); final_norm [d]   (embed dtype)
      layers[l]: attn_norm [d], ffn_norm [d] (embed dtype), wq [hq*hd, d], wk/wv [hkv*hd, d],
        wo [d, hq*hd]; dense: w_gate/w_up [ff, d], w_down [d, ff] (weight dtype; with e4m3
        weights each matrix M also has M_scale [rows] f32, applied after the dot)
        MoE:   router [E, d]; e_gate/e_up [E, f, d] e4m3; e_down [E, d, f] e4m3;
               e_gate_scale/e_up_scale [E, f] f32; e_down_scale [E, d] f32
    """
    c = cfg
    if seed is None:
        seed = SEED_WEIGHTS + c["index"]
    wdt = c["weight_dtype"]
    edt = c.get("embed_dtype") or wdt
    d, hq, hkv, hd = c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"]
    V = c["vocab"]
    W = {"tok_emb": normal_stored(seed, TID_EMB, (V, d), edt)}
    W["lm_head"] = None if c["tied_embeddings"] else normal_stored(seed, TID_LM, (V, d), edt)
    W["final_norm"] = ones_stored(d, edt)

    def mat(L, name, tid, rows, cols):
        """A layer matrix in the weight dtype; e4m3 ones come with per-row scales `<name>_scale`,
        nvfp4 ones with row scales and e4m3 block scales `<name>_bscale` (codes packed)."""
        if wdt == "e4m3":
            L[name], L[name + "_scale"] = normal_e4m3_rows(seed, tid, rows, cols)
        elif wdt == "nvfp4":
            L[name], L[name + "_bscale"], L[name + "_scale"] = normal_nvfp4_rows(seed, tid, rows, cols)
        else:
            L[name] = normal_stored(seed, tid, (rows, cols), wdt)

    layers = []
    for l in range(c["n_layers"]):
        L = {"attn_norm": ones_stored(d, edt), "ffn_norm": ones_stored(d, edt)}
        mat(L, "wq", _tid_layer(l, K_WQ), hq * hd, d)
        mat(L, "wk", _tid_layer(l, K_WK), hkv * hd, d)
        mat(L, "wv", _tid_layer(l, K_WV), hkv * hd, d)
        mat(L, "wo", _tid_layer(l, K_WO), d, hq * hd)
        if c["n_experts"] == 0:
            ff = c["d_ff"]
            mat(L, "w_gate", _tid_layer(l, K_WG), ff, d)
            mat(L, "w_up", _tid_layer(l, K_WU), ff, d)
            mat(L, "w_down", _tid_layer(l, K_WD), d, ff)
        else:
            E, f = c["n_experts"], c["d_expert"]
            L["router"] = normal_stored(seed, _tid_layer(l, K_ROUTER), (E, d), c["router_dtype"])
            eg = np.empty((E, f, d), np.uint8); eu = np.empty((E, f, d), np.uint8); ed = np.empty((E, d, f), np.uint8)
            sg = np.empty((E, f), np.float32); su = np.empty((E, f), np.float32); sd = np.empty((E, d), np.float32)
            for e in range(E):
                eg[e], sg[e] = normal_e4m3_rows(seed, _tid_expert(l, e, E_GATE), f, d)
                eu[e], su[e] = normal_e4m3_rows(seed, _tid_expert(l, e, E_UP), f, d)
                ed[e], sd[e] = normal_e4m3_rows(seed, _tid_expert(l, e, E_DOWN), d, f)
            L.update(e_gate=eg, e_up=eu, e_down=ed, e_gate_scale=sg, e_up_scale=su, e_down_scale=sd)
        layers.append(L)
    W["layers"] = layers
    return W


def prompt(cfg: dict, n: int | None = None, seed: int | None = None) -> np.ndarray:
    if seed is None:
        seed = SEED_PROMPT + cfg["index"]
    return tokens(seed, 7, cfg["prompt_len"] if n is None else n, cfg["vocab"])


def sampling_uniforms(n: int, first: int = 0, seed: int = SEED_SAMPLING) -> np.ndarray:
    return uniforms(seed, first, n)


def batch_prompts(cfg: dict, lengths) -> list[np.ndarray]:
    """Prompts of independent requests decoded as one batch: request r draws its tokens from the
    prompt stream of seed SEED_PROMPT + config index + 100 * r (request 0 has the usual prompt)."""
    return [prompt(cfg, int(n), seed=SEED_PROMPT + cfg["index"] + 100 * r) for r, n in enumerate(lengths)]


def batch_uniforms(n: int, r: int) -> np.ndarray:
    """Sampling uniforms of request r of a batch: the sampling stream of seed SEED_SAMPLING + r."""
    return uniforms(SEED_SAMPLING + r, 0, n)


def kv_prefix(cfg: dict, length: int, seed: int | None = None):
    """Synthetic KV-cache contents for positions [0, length): N(0, 1) in the KV storage dtype,
    shaped [L, hkv, length, hd] (raw bits). N(0,1) matches the scale of K/V rows that a
    std-0.02 projection produces from a unit-RMS input when d_model ~ 2500."""
    if seed is None:
        seed = SEED_KV + cfg["index"]
    shp = (cfg["n_layers"], cfg["n_kv_heads"], length, cfg["head_dim"])
    k = normal_stored(seed, 11, shp, cfg["kv_dtype"], std=1.0)
    v = normal_stored(seed, 12, shp, cfg["kv_dtype"], std=1.0)
    return k, v

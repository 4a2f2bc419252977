"""Brute-force float64 decoder (test infrastructure only).

Recomputes the whole prefix for every position with no KV cache: one causal
forward pass over the token sequence gives the logits at every position. It is
the independent check of oracle.c: written with NumPy matrix products in float64,
it shares no code with the C oracle or with the CUDA engine. K and V are rounded
to the KV storage dtype before attention reads them, as the step defines (the
cache stores them in full, uncompressed, at that dtype: aether-echoes.com,
"標準 GPU で LLM 推論 3000 tokens/s/req", section "どう出したか").
"""
from __future__ import annotations

import numpy as np


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Raw stored bits -> float64."""
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "e4m3":
        return e4m3_decode(a)
    raise ValueError(dtype)


def e4m3_decode(q: np.ndarray) -> np.ndarray:
    """OCP E4M3 ("fn"): sign, 4 exponent bits (bias 7), 3 fraction bits, subnormals,
    exponent 15 with fraction 7 is NaN, no infinities."""
    q = q.astype(np.int64)
    s = np.where(q & 0x80, -1.0, 1.0)
    e = (q >> 3) & 15
    m = q & 7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


def e2m1_decode(q: np.ndarray) -> np.ndarray:
    """4-bit E2M1 codes (NVFP4 elements): sign bit 3, exponent bits 2..1 (bias 1), one fraction
    bit; exponent 0 is subnormal."""
    q = q.astype(np.int64)
    s = np.where(q & 8, -1.0, 1.0)
    e = (q >> 1) & 3
    m = q & 1
    val = np.where(e == 0, 0.5 * m, (1.0 + m / 2.0) * 2.0 ** (e - 1.0))
    return s * val


def nvfp4_dequant(codes: np.ndarray, bscale: np.ndarray, rscale: np.ndarray) -> np.ndarray:
    """NVFP4 matrix -> float64: packed e2m1 codes [rows, K/2] (element 2i in the low nibble), e4m3
    block scales [rows, K/16], fp32 row scales [rows]: w = rowscale * blockscale * element."""
    rows = codes.shape[0]
    c = codes.astype(np.int64)
    q = np.empty((rows, codes.shape[1] * 2), dtype=np.int64)
    q[:, 0::2] = c & 15
    q[:, 1::2] = c >> 4
    blk = np.repeat(e4m3_decode(bscale), 16, axis=1)
    return rscale.astype(np.float64)[:, None] * blk * e2m1_decode(q)


def store_round(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> value after rounding to the KV storage dtype, back in float64."""
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        f = x.astype(np.float32)
        u = f.view(np.uint32).astype(np.uint64)
        r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
        return r.astype(np.uint32).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope(y: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """y [n, heads, hd]; rotate-half pairs (i, i + hd/2) by pos * theta^(-2i/hd)."""
    hd = y.shape[-1]
    i = np.arange(hd // 2, dtype=np.float64)
    ang = pos[:, None].astype(np.float64) * theta ** (-(2.0 * i) / hd)
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = y[..., : hd // 2], y[..., hd // 2:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def forward(cfg: dict, W: dict, tokens, force=None):
    """Logits [n, V] (float64) at every position of `tokens`, plus per-position routing.

    force: optional [n, n_layers, top_k] expert ids to use instead of this model's own choice
    (gates are then the softmax probabilities of those experts renormalised over them)."""
    c = cfg
    wdt, kvdt = c["weight_dtype"], c["kv_dtype"]
    edt = c.get("embed_dtype") or wdt  # embedding, LM head, norm gains

    def mat(Lw, name):
        """A layer matrix as float64; e4m3 rows times their per-row scale; nvfp4 dequantised."""
        if wdt == "nvfp4":
            return nvfp4_dequant(Lw[name], Lw[name + "_bscale"], Lw[name + "_scale"])
        m = widen(Lw[name], wdt)
        return m * Lw[name + "_scale"].astype(np.float64)[:, None] if wdt == "e4m3" else m

    d, hq, hkv, hd = c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"]
    tokens = np.asarray(tokens, dtype=np.int64)
    n = len(tokens)
    pos = np.arange(n)
    emb = widen(W["tok_emb"], edt)
    x = emb[tokens].copy()
    eps = c["rms_eps"]
    causal = np.tril(np.ones((n, n), dtype=bool))
    group = np.array([(h * hkv) // hq for h in range(hq)])
    routes = []
    for l, Lw in enumerate(W["layers"]):
        xn = rmsnorm(x, widen(Lw["attn_norm"], edt), eps)
        q = (xn @ mat(Lw, "wq").T).reshape(n, hq, hd)
        k = (xn @ mat(Lw, "wk").T).reshape(n, hkv, hd)
        v = (xn @ mat(Lw, "wv").T).reshape(n, hkv, hd)
        q = rope(q, pos, c["rope_theta"])
        k = store_round(rope(k, pos, c["rope_theta"]), kvdt)
        v = store_round(v, kvdt)
        att = np.empty((n, hq, hd))
        for h in range(hq):
            s = (q[:, h, :] @ k[:, group[h], :].T) / np.sqrt(hd)
            s = np.where(causal, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            att[:, h, :] = p @ v[:, group[h], :]
        x = x + att.reshape(n, hq * hd) @ mat(Lw, "wo").T
        xn = rmsnorm(x, widen(Lw["ffn_norm"], edt), eps)
        if not c["n_experts"]:
            g = xn @ mat(Lw, "w_gate").T
            u = xn @ mat(Lw, "w_up").T
            x = x + (silu(g) * u) @ mat(Lw, "w_down").T
        else:
            E, K = c["n_experts"], c["top_k"]
            r = xn @ widen(Lw["router"], c["router_dtype"]).T
            P = np.exp(r - r.max(axis=1, keepdims=True))
            P = P / P.sum(axis=1, keepdims=True)
            out = np.zeros_like(x)
            sel_l = np.zeros((n, K), dtype=np.int64)
            for t in range(n):
                sel = np.argsort(-P[t], kind="stable")[:K]
                if force is not None:
                    sel = np.asarray(force[t][l], dtype=np.int64)
                sel_l[t] = sel
                gates = P[t, sel] / P[t, sel].sum()
                for gk, e in zip(gates, sel):
                    Qg = widen(Lw["e_gate"][e], "e4m3") * Lw["e_gate_scale"][e][:, None]
                    Qu = widen(Lw["e_up"][e], "e4m3") * Lw["e_up_scale"][e][:, None]
                    Qd = widen(Lw["e_down"][e], "e4m3") * Lw["e_down_scale"][e][:, None]
                    h_e = silu(Qg @ xn[t]) * (Qu @ xn[t])
                    out[t] += gk * (Qd @ h_e)
            x = x + out
            routes.append(sel_l)
    xn = rmsnorm(x, widen(W["final_norm"], edt), eps)
    head = W["tok_emb"] if c["tied_embeddings"] else W["lm_head"]
    logits = xn @ widen(head, edt).T
    return logits, (np.stack(routes, axis=1) if routes else None)

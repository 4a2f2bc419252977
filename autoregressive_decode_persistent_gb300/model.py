"""Convenience wrapper: upload host weights with PyTorch (device memory only), fill the C
structs, and hold the engine handles. Every computation runs in libadp.so's kernels."""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import adp

_TORCH_RAW = {np.dtype(np.uint16): torch.int16, np.dtype(np.uint8): torch.uint8,
              np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32}


def to_device(a: np.ndarray | None, device) -> torch.Tensor | None:
    """Raw bytes of a host array -> a device tensor holding the same bytes."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.to(device, non_blocking=False)


def make_config(cfg: dict) -> adp.Config:
    D = adp.DTYPES
    return adp.Config(cfg["n_layers"], cfg["d_model"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                      cfg.get("d_ff", 0), cfg["vocab"], cfg["max_ctx"], cfg["rms_eps"], cfg["rope_theta"],
                      1 if cfg["tied_embeddings"] else 0, D[cfg["weight_dtype"]], D[cfg["kv_dtype"]],
                      cfg["n_experts"], cfg["top_k"], cfg["d_expert"], D[cfg["router_dtype"]],
                      D[cfg["expert_dtype"]], D[cfg.get("embed_dtype") or cfg["weight_dtype"]])


class DecodeModel:
    """A model on one GPU plus its KV caches (see include/adp.h for the semantics)."""

    _MATRICES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "router", "e_gate", "e_up", "e_down",
                 "wq_bscale", "wk_bscale", "wv_bscale", "wo_bscale", "w_gate_bscale", "w_up_bscale",
                 "w_down_bscale")

    def __init__(self, cfg: dict, host_weights: dict, device: str = "cuda:0", stream: torch.cuda.Stream | None = None,
                 keep_matrices: bool = False):
        self.cfg = cfg
        self.device = torch.device(device)
        torch.cuda.set_device(self.device)
        self.stream = stream
        W = host_weights
        self._dev = {}
        keep = []
        matrices = []

        def up(a, matrix=False):
            t = to_device(a, self.device)
            if t is not None:
                (matrices if matrix else keep).append(t)
            return None if t is None else t.data_ptr()

        layers = (adp.LayerWeights * cfg["n_layers"])()
        for i, Lw in enumerate(W["layers"]):
            f = {k: up(Lw.get(k), k in self._MATRICES)
                 for k in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down", "router",
                           "e_gate", "e_up", "e_down", "e_gate_scale", "e_up_scale", "e_down_scale", "wq_scale",
                           "wk_scale", "wv_scale", "wo_scale", "w_gate_scale", "w_up_scale", "w_down_scale",
                           "wq_bscale", "wk_bscale", "wv_bscale", "wo_bscale", "w_gate_bscale", "w_up_bscale",
                           "w_down_bscale")}
            layers[i] = adp.LayerWeights(**f)
        self._layers = layers
        self.weights = adp.Weights(up(W["tok_emb"]), up(W.get("lm_head"), True), up(W["final_norm"]), layers)
        self._keep = keep
        self.config = make_config(cfg)
        torch.cuda.synchronize(self.device)
        sh = stream.cuda_stream if stream is not None else 0
        self.handle = adp.adp_create_model(self.config, self.weights, sh)
        # The engine copied every matrix into its own tile-ordered image at creation and reads
        # only the embedding, norm gains and scales in place afterwards.
        if keep_matrices:
            self._keep += matrices
        del matrices
        torch.cuda.synchronize(self.device)
        torch.cuda.empty_cache()

    def close(self):
        if getattr(self, "handle", None):
            adp.adp_destroy_model(self.handle)
            self.handle = None
        self._keep = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- KV
    def new_kv(self):
        return KVCache(self)

    # -- introspection
    @property
    def num_ctas(self) -> int:
        return adp.adp_num_ctas(self.handle)

    @property
    def image_bytes(self) -> int:
        return adp.adp_image_bytes(self.handle)

    def set_kernel_mode(self, mode: int):
        adp.adp_debug_kernel_mode(self.handle, mode)

    @property
    def launches_per_step(self) -> int:
        return adp.adp_launches_per_step(self.handle)

    # -- small batches: independent requests (one KVCache each) stepped together
    @property
    def max_batch(self) -> int:
        return adp.adp_max_batch(self.handle)

    def step_batch(self, kvs, tokens, temperatures=None, us=None, logits: torch.Tensor | None = None) -> list[int]:
        return adp.adp_decode_batch(self.handle, [k.handle for k in kvs], tokens, temperatures, us, logits)

    def generate_batch_async(self, kvs, tokens, n: int, out: torch.Tensor, temperatures=None,
                             uniforms: torch.Tensor | None = None):
        adp.adp_generate_batch_async(self.handle, [k.handle for k in kvs], tokens, n, temperatures, uniforms, out)


class KVCache:
    def __init__(self, model: DecodeModel):
        self.model = model
        self.handle = adp.adp_kv_create(model.handle)

    def close(self):
        if getattr(self, "handle", None):
            adp.adp_kv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __len__(self):
        return adp.adp_kv_len(self.handle)

    def reset(self):
        adp.adp_kv_reset(self.handle)

    def truncate(self, length: int):
        adp.adp_kv_truncate(self.handle, length)

    def load(self, k: np.ndarray, v: np.ndarray):
        adp.adp_kv_load(self.handle, k, v, k.shape[2])

    def read(self, length: int | None = None):
        c = self.model.cfg
        n = len(self) if length is None else length
        shp = (c["n_layers"], c["n_kv_heads"], n, c["head_dim"])
        k = np.empty(shp, dtype=np.uint16)
        v = np.empty(shp, dtype=np.uint16)
        adp.adp_kv_read(self.handle, k, v, n)
        return k, v

    def step(self, token: int, temperature: float = 0.0, u: float = 0.0, logits: torch.Tensor | None = None) -> int:
        return adp.adp_decode_step(self.model.handle, self.handle, token, temperature, u, logits)

    def prefill(self, tokens, temperature: float = 0.0, u: float = 0.0, logits: torch.Tensor | None = None) -> int:
        return adp.adp_prefill(self.model.handle, self.handle, tokens, temperature, u, logits)

    def prefill_tc(self, tokens, temperature: float = 0.0, u: float = 0.0, logits: torch.Tensor | None = None) -> int:
        return adp.adp_prefill_tc(self.model.handle, self.handle, tokens, temperature, u, logits)

    def generate_async(self, token: int, n: int, out: torch.Tensor, temperature: float = 0.0,
                       uniforms: torch.Tensor | None = None):
        adp.adp_generate_async(self.model.handle, self.handle, token, n, temperature, uniforms, out)

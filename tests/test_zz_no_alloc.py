"""adp_decode_step_noalloc (the decode step with its scratch in the library's static array) against
adp_decode_step (the model's own scratch), both called through the C ABI on identical KV caches.

The entry point exists for callers that must not allocate device memory while they decode (a
process whose memory pool already holds the device's free memory, or a serving loop that cannot
take the synchronisation an allocation may cause).  Both calls run the same kernel on the same
inputs with deterministic reductions, so the logits must be bit-identical (compared as uint32),
as must the next token and the KV rows.  The file sorts last so that it also runs after every
other GPU test; it passes alone in a fresh process too (the model's creation then does the
per-device set-up, and the first no-alloc call still allocates nothing)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    assert torch.cuda.is_available(), "a CUDA GPU is required"
    from autoregressive_decode_persistent_gb300 import adp, build
    build.build()
    return adp


def _pair(cfg, prompt_len):
    """A model and two KV caches holding the same prompt (written by the model's own path)."""
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    model = DecodeModel(cfg, synth.model_weights(cfg))
    prompt = synth.prompt(cfg, prompt_len)
    kv_ref, kv_na = model.new_kv(), model.new_kv()
    t = kv_ref.prefill(prompt)
    assert kv_na.prefill(prompt) == t
    return model, kv_ref, kv_na, t


def _same_bits(a, b):
    return np.array_equal(a.cpu().numpy().view(np.uint32), b.cpu().numpy().view(np.uint32))


def _both(adp, model, kv_ref, kv_na, token, temperature=0.0, u=0.0):
    import torch
    lg_ref = torch.empty(model.cfg["vocab"], device=model.device)
    lg_na = torch.empty(model.cfg["vocab"], device=model.device)
    t_na = adp.adp_decode_step_noalloc(model.handle, kv_na.handle, token, temperature, u, lg_na)
    t_ref = adp.adp_decode_step(model.handle, kv_ref.handle, token, temperature, u, lg_ref)
    assert t_na == t_ref
    assert _same_bits(lg_na, lg_ref)
    return t_ref


def _free_bytes():
    import torch
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def test_two_calls_in_a_row_match_decode_step(lib):
    import torch
    cfg = synth.get_config("tiny")
    model, kv_ref, kv_na, t = _pair(cfg, 12)
    for call in range(2):  # the first no-alloc call after the model's creation, then the next one
        lg_ref = torch.empty(cfg["vocab"], device=model.device)
        lg_na = torch.empty(cfg["vocab"], device=model.device)
        free_before = _free_bytes()
        t_na = lib.adp_decode_step_noalloc(model.handle, kv_na.handle, t, 0.0, 0.0, lg_na)
        free_after = _free_bytes()
        assert free_after == free_before, (call, free_before, free_after)  # no device memory allocated
        t_ref = lib.adp_decode_step(model.handle, kv_ref.handle, t, 0.0, 0.0, lg_ref)
        assert t_na == t_ref
        assert _same_bits(lg_na, lg_ref), call
        t = t_ref
    assert len(kv_na) == len(kv_ref) == 14
    k1, v1 = kv_ref.read()
    k2, v2 = kv_na.read()
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    # without a logits pointer the logits go to the static array; the token still matches
    assert lib.adp_decode_step_noalloc(model.handle, kv_na.handle, t, 0.0, 0.0, None) == \
        lib.adp_decode_step(model.handle, kv_ref.handle, t, 0.0, 0.0, None)
    model.close()


def test_sampling_and_alternating_models(lib):
    """Temperature sampling, and models with different scratch layouts and kernel kinds (16-bit
    dense, e4m3 dense) taking turns."""
    a = _pair(synth.get_config("tiny"), 8)
    b = _pair(synth.shrink(synth.get_config("dense-2.3b-fp16")), 8)
    e = _pair(synth.shrink(synth.get_config("dense-2.3b-e4m3")), 8)
    ta, tb, te = a[3], b[3], e[3]
    for i in range(3):
        ta = _both(lib, *a[:3], ta, 0.7, 0.25 + 0.2 * i)
        tb = _both(lib, *b[:3], tb)
        te = _both(lib, *e[:3], te)
    for m in (a, b, e):
        m[0].close()


def test_device_error_is_returned_and_not_sticky(lib):
    """A dependency wait that runs out (one CTA withholds its outputs of the Wo phase, every wait is
    limited to 1 ms) is returned as ADP_ERR_BARRIER_TIMEOUT; the array is zeroed and the model is
    not left in an error state, so the next no-alloc step, without adp_reset, matches
    adp_decode_step bit for bit."""
    cfg = synth.get_config("tiny")
    model, kv_ref, kv_na, t = _pair(cfg, 10)
    lib.adp_debug_set_wait_limit(model.handle, 1_000_000)
    lib.adp_debug_skip_publication(model.handle, 3, 2)  # CTA 3, the Wo phase of layer 0
    with pytest.raises(lib.AdpError) as e:
        lib.adp_decode_step_noalloc(model.handle, kv_na.handle, t, 0.0, 0.0, None)
    assert e.value.code == lib.ADP_ERR_BARRIER_TIMEOUT
    assert len(kv_na) == 10
    lib.adp_debug_set_wait_limit(model.handle, 200_000_000)
    for _ in range(2):
        t = _both(lib, model, kv_ref, kv_na, t)
    k1, v1 = kv_ref.read()
    k2, v2 = kv_na.read()
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    model.close()


def test_scratch_beyond_the_static_array_is_rejected(lib):
    import torch
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    cfg = synth.shrink(synth.get_config("tiny"), n_heads=32, n_kv_heads=4, max_ctx=40960)
    model = DecodeModel(cfg, synth.model_weights(cfg))
    kv = model.new_kv()
    with pytest.raises(lib.AdpError) as e:
        lib.adp_decode_step_noalloc(model.handle, kv.handle, 1, 0.0, 0.0, None)
    assert e.value.code == lib.ADP_ERR_UNSUPPORTED_CONFIG
    assert "static array" in lib.load_library().adp_last_error().decode()
    assert len(kv) == 0
    torch.cuda.synchronize()
    model.close()

"""Tensor-core prefill: the tcgen05 GEMM against float64 numpy on the same 16-bit operands."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    assert torch.cuda.is_available(), "a CUDA GPU is required"
    from autoregressive_decode_persistent_gb300 import adp, build
    build.build()
    return adp


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 100), (5, 17, 8), (384, 1024, 2560), (130, 512, 704),
                                   (2000, 4864, 100)])
@pytest.mark.parametrize("bf16", [False, True])
def test_tc_gemm_matches_float64(lib, M, N, K, bf16):
    """fp32 accumulation of exact 16-bit products: every entry within 2^-20 of the row's sum of
    |a_k w_k| (fp32 rounding of K partial sums) of the float64 product.  The GEMM takes 128-row
    tiles where 256-row ones would leave a nearly empty last wave: on a 152-SM GB300 the small
    shapes run with 128-row tiles and 2000 x 4864 (one full wave of 256-row tiles) with 256."""
    import torch
    dt = torch.bfloat16 if bf16 else torch.float16
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    a = torch.randn(M, K, generator=g).to(dt)
    w = torch.randn(N, K, generator=g).to(dt)
    ref = a.double() @ w.double().T
    bound = (a.double().abs() @ w.double().abs().T) * 2.0 ** -20 + 1e-30
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.adp_debug_tc_gemm(bf16, a.cuda(), w.cuda(), c)
    err = (c.cpu().double() - ref).abs()
    assert torch.isfinite(c).all()
    assert (err <= bound).all(), float((err / bound).max())


def _kv_within_tolerance(got, ref, vocab):
    """KV rows written by the tensor-core path (an approximation: 16-bit GEMM operands) against a
    reference: the logits' tolerances applied to the cache.  Per layer, and per 128 positions,
    relative L2 <= 5e-3.  Max-abs: 2e-2 is stated for one step's `vocab` logits; over a layer's n
    elements the bound keeps the same per-element tail probability (the extreme of n samples grows
    like sqrt(2 ln n)): 2e-2 * sqrt(ln n / ln vocab), and never below 2e-2."""
    n = ref[0].size
    bound = 2e-2 * max(1.0, float(np.sqrt(np.log(n) / np.log(vocab))))
    for layer in range(ref.shape[0]):
        g = got[layer].astype(np.float64)
        r = ref[layer].astype(np.float64)
        d = g - r
        assert np.max(np.abs(d)) <= bound, (layer, float(np.max(np.abs(d))), bound)
        assert np.linalg.norm(d) / max(np.linalg.norm(r), 1e-30) <= 5e-3, layer
        for p0 in range(0, r.shape[1], 128):  # [kv head][position][head_dim]
            dd, rr = d[:, p0:p0 + 128], r[:, p0:p0 + 128]
            assert np.linalg.norm(dd) / max(np.linalg.norm(rr), 1e-30) <= 5e-3, (layer, p0)


def _as_float(bits, cfg):
    import torch
    t = torch.from_numpy(bits.astype(np.int16).view(np.int16))
    dt = torch.bfloat16 if cfg["kv_dtype"] == "bf16" else torch.float16
    return t.view(dt).float().numpy()


def _prefill_case(cfg, prompt_len, prefix_len=0, n_decode=3):
    """adp_prefill_tc of a prompt (after an optional synthetic KV prefix) against the oracle's plain
    mode: the last prompt token's logits, every new KV row, and a few decode steps after it."""
    import torch
    import synth
    from oracle import PLAIN, OracleModel
    from gpu_common import assert_logits_within_tolerance
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    W = synth.model_weights(cfg)
    prompt = synth.prompt(cfg, prompt_len)
    om = OracleModel(cfg, W)
    kvp = synth.kv_prefix(cfg, prefix_len) if prefix_len else None
    if kvp is not None:
        om.load_kv_prefix(*kvp)
    out = None
    for t in prompt:
        out = om.step(int(t), PLAIN)
    model = DecodeModel(cfg, W)
    kv = model.new_kv()
    if kvp is not None:
        kv.load(*kvp)
    lg = torch.empty(cfg["vocab"], device=model.device)
    nxt = kv.prefill_tc(prompt, logits=lg)
    assert len(kv) == prefix_len + prompt_len
    assert_logits_within_tolerance(lg.cpu().numpy()[None], out["logits"][None].astype(np.float64))
    n = prefix_len + prompt_len
    k, v = kv.read()
    _kv_within_tolerance(_as_float(k[:, :, prefix_len:n], cfg), _as_float(om.kc[:, :, prefix_len:n], cfg), cfg["vocab"])
    _kv_within_tolerance(_as_float(v[:, :, prefix_len:n], cfg), _as_float(om.vc[:, :, prefix_len:n], cfg), cfg["vocab"])
    # decode continues from the tensor-core cache (teacher-forced on the oracle's tokens)
    t = out["next"]
    for _ in range(n_decode):
        ref = om.step(int(t), PLAIN)
        kv.step(int(t), logits=lg)
        assert_logits_within_tolerance(lg.cpu().numpy()[None], ref["logits"][None].astype(np.float64))
        t = ref["next"]
    model.close()
    return nxt


def test_prefill_tc_tiny(lib):
    import synth
    _prefill_case(synth.get_config("tiny"), 40)


def test_prefill_tc_ragged_and_after_prefix(lib):
    """head_dim 128, widths that are not multiples of the GEMM tiles (d 384, ffn 1000), 132
    tensor-core tokens (two 128-row tiles, the second ragged) after a 21-row cache prefix."""
    import synth
    cfg = synth.shrink(synth.get_config("tiny"), head_dim=128, n_heads=4, n_kv_heads=2, d_model=384, d_ff=1000)
    _prefill_case(cfg, 133, prefix_len=21)


@pytest.mark.parametrize("name", ["dense-2.3b-fp16", "dense-2.3b-e4m3", "dense-2.3b-nvfp4"])
def test_prefill_tc_full_size(lib, name):
    """The 2.3B model at full size (fp16, and e4m3 or NVFP4 layer matrices dequantised for the GEMMs): a
    448-row synthetic cache prefix, then a 64-token prompt through the tensor-core path and three
    decode steps."""
    import synth
    _prefill_case(synth.get_config(name), 64, prefix_len=448)


@pytest.mark.parametrize("name", ["dense-2.3b-fp16", "dense-8b-bf16", "dense-2.3b-e4m3", "dense-2.3b-nvfp4"])
def test_prefill_tc_shrunk_workloads(lib, name):
    import synth
    _prefill_case(synth.shrink(synth.get_config(name)), 70)


def test_prefill_tc_single_token_is_a_decode_step(lib):
    import torch
    import synth
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    cfg = synth.get_config("tiny")
    model = DecodeModel(cfg, synth.model_weights(cfg))
    a, b = model.new_kv(), model.new_kv()
    la = torch.empty(cfg["vocab"], device=model.device)
    lb = torch.empty(cfg["vocab"], device=model.device)
    assert a.prefill_tc([17], logits=la) == b.step(17, logits=lb)
    assert torch.equal(la, lb)
    model.close()


def test_prefill_tc_rejects_unsupported_models(lib):
    import synth
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    for name in ("moe-32x1408-top4-e4m3",):
        cfg = synth.shrink(synth.get_config(name))
        model = DecodeModel(cfg, synth.model_weights(cfg))
        kv = model.new_kv()
        with pytest.raises(lib.AdpError) as e:
            kv.prefill_tc([1, 2, 3])
        assert e.value.code == lib.ADP_ERR_UNSUPPORTED_CONFIG
        assert len(kv) == 0
        model.close()


def test_prefill_tc_full_prompt_matches_the_decode_path(lib):
    """The long-context workload's whole 3,584-token prompt at full size (28 query tiles per head, up
    to 28 key blocks on the longest rows, the masked diagonal blocks, the last tile ragged): the
    tensor-core prefill's KV rows and first-token logits against the decode-kernel prefill of the
    same prompt (the bit-exact path, itself checked against the oracle), within the logits'
    tolerances; then the decode steps after either prefix agree."""
    import torch
    import synth
    from gpu_common import assert_logits_within_tolerance
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    cfg = synth.get_config("dense-2.3b-fp16-long-t0.7")
    prompt = synth.prompt(cfg)
    P = len(prompt)
    model = DecodeModel(cfg, synth.model_weights(cfg))
    a, b = model.new_kv(), model.new_kv()
    la = torch.empty(cfg["vocab"], device=model.device)
    lb = torch.empty(cfg["vocab"], device=model.device)
    ta = a.prefill_tc(prompt, logits=la)
    tb = b.prefill(prompt, logits=lb)
    ref = lb.cpu().numpy().astype(np.float64)
    assert_logits_within_tolerance(la.cpu().numpy()[None], ref[None])
    top2 = np.sort(ref)[-2:]
    if top2[1] - top2[0] > 1e-2:
        assert ta == tb
    ka, va = a.read()
    kb, vb = b.read()
    _kv_within_tolerance(_as_float(ka[:, :, :P], cfg), _as_float(kb[:, :, :P], cfg), cfg["vocab"])
    _kv_within_tolerance(_as_float(va[:, :, :P], cfg), _as_float(vb[:, :, :P], cfg), cfg["vocab"])
    t = tb
    for _ in range(2):
        a.step(int(t), logits=la)
        t = b.step(int(t), logits=lb)
        assert_logits_within_tolerance(la.cpu().numpy()[None], lb.cpu().numpy()[None].astype(np.float64))
    model.close()

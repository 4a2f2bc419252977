/*
 * adp.h — C ABI of a batch-1 persistent decode engine for one GB300 (sm_103a).
 *
 * The engine runs one autoregressive decode step of a decoder-only transformer
 * (dense SwiGLU or top-k MoE with e4m3 experts) as ONE persistent CUDA kernel per
 * step, its phases ordered by epoch-tagged exchange words instead of a kernel per
 * operation; a second persistent kernel decodes small batches of independent requests
 * (adp_decode_batch).
 *
 * Pages this interface follows (cited by title and section):
 *  [H] "標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒" (hakusoku.com
 *      summary of Kog AI, "Real-time LLM inference on standard GPUs: 3,000 tokens/s per request"):
 *      §"単一リクエストLLMデコード速度の重要性" (single-request decode speed is the metric),
 *      §"GPU推論の速度制限要因：メモリ帯域幅" (batch-1 decode is matrix-vector work that streams
 *        every active weight and the KV cache: tokens/s <= bandwidth / (beta*weights + KV)),
 *      §"標準推論スタックのボトルネックとKogの工夫" (per-kernel launch/cleanup overhead; one
 *        GPU-resident program runs the whole decode path),
 *      §"Kog Inference Engineの特徴とイノベーション" (the program covers MatMul, attention,
 *        normalization, routing and sampling, and controls sync, prefetch and order).
 *  [A] "標準 GPU で LLM 推論 3000 tokens/s/req — 数字の前提を運用者目線で読む" (aether-echoes.com),
 *      §"どう出したか": no quantization, speculative decoding, pruning or KV compression.
 *  [S] "「ソフトウェア・ファースト」戦略でGPUの限界を突破" (studioglobal.ai),
 *      §"独自の3層共同設計アプローチ" item 1 (monokernel: the whole decode as one persistent kernel).
 *
 * Conventions for every call:
 *  - Return value: ADP_OK (0) or a negative ADP_ERR_* code; no call aborts or throws.
 *  - Device errors (a barrier or pipeline wait that ran out) are sticky: every later
 *    decode call on the model returns the same code until adp_reset.
 *  - Calls on one model are not thread-safe; all GPU work goes on the model's stream.
 *  - "device pointer" = cudaMalloc'd (or equivalent) memory of the current device;
 *    "host pointer" = ordinary (pageable or pinned) host memory.
 */
#ifndef ADP_H_
#define ADP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

/* Storage types of weights and of the KV cache.  ADP_NVFP4: 4-bit E2M1 codes, two per byte (the
 * even element in the low nibble), with one e4m3 scale per 16 consecutive elements of a row. */
typedef enum { ADP_F16 = 0, ADP_BF16 = 1, ADP_E4M3 = 2, ADP_F32 = 3, ADP_NVFP4 = 4 } adp_dtype;

enum {
  ADP_OK = 0,
  ADP_ERR_INVALID_ARG = -1,        /* null pointer, bad token id, n < 0 ... */
  ADP_ERR_UNSUPPORTED_CONFIG = -2, /* shape or dtype combination the kernel does not implement */
  ADP_ERR_CONTEXT_OVERFLOW = -3,   /* position >= max_ctx */
  ADP_ERR_CUDA = -4,               /* a CUDA runtime call failed (message: adp_last_error) */
  ADP_ERR_NOT_CORESIDENT = -5,     /* the persistent grid cannot be co-resident on this GPU */
  ADP_ERR_BARRIER_TIMEOUT = -6,    /* a wait for another CTA's output ran out (sticky until adp_reset) */
  ADP_ERR_PIPELINE_TIMEOUT = -7,   /* a weight-pipeline wait ran out (sticky until adp_reset) */
  ADP_ERR_UNIMPLEMENTED = -8
};

/* Model shape and types.  Row-major [out, in] weights, no biases, pre-norm decoder:
 * x += Wo . attn(rope(Wq xn), rope(Wk xn), Wv xn);  x += FFN(rmsnorm(x));  logits = W_lm rmsnorm(x).
 * RMSNorm with eps inside the root, rotate-half RoPE (pairs i, i + head_dim/2) with
 * inv_freq_i = rope_theta^(-2i/head_dim), grouped-query attention where query head h reads
 * KV head floor(h * n_kv_heads / n_heads).  n_experts == 0 selects the dense SwiGLU FFN
 * (d_ff wide); otherwise a softmax top_k router over n_experts SwiGLU experts of width d_expert,
 * gates renormalised over the chosen experts ([H] §"Kog Inference Engineの特徴とイノベーション":
 * routing is one of the stages; Hacker News author reply: FP8 MoE models at batch 1). */
typedef struct {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, d_ff, vocab, max_ctx;
  float rms_eps, rope_theta;
  int32_t tied_embeddings;          /* 1: logits use tok_emb as the LM head */
  int32_t weight_dtype, kv_dtype;   /* adp_dtype: ADP_F16 or ADP_BF16 for both; weight_dtype may be
                                       ADP_E4M3 or ADP_NVFP4 for a dense model (see embed_dtype and
                                       the scales; NVFP4 needs d_model, d_ff and n_heads*head_dim
                                       to be multiples of 128) */
  int32_t n_experts, top_k, d_expert;
  int32_t router_dtype, expert_dtype; /* router: ADP_F16/ADP_BF16; experts: ADP_E4M3 */
  int32_t embed_dtype;              /* with weight_dtype ADP_E4M3/NVFP4: type of tok_emb, lm_head and the
                                       norm gains (ADP_F16 or ADP_BF16); otherwise ignored */
} adp_config;

/* Per-layer weights: DEVICE pointers, contiguous row-major, borrowed (never written; the
 * engine copies the matrices into its own streaming layout at creation, but tok_emb, the
 * norm gains and the expert scales are read in place, so all must outlive the model). */
typedef struct {
  const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm;   /* [d], [hq*hd, d], [hkv*hd, d] x2, [d, hq*hd], [d] */
  const void *w_gate, *w_up, *w_down;                     /* dense: [ff, d], [ff, d], [d, ff]; else NULL */
  const void *router;                                     /* MoE: [E, d]; else NULL */
  const void *e_gate, *e_up, *e_down;                     /* MoE: [E, f, d], [E, f, d], [E, d, f] e4m3 */
  const float *e_gate_scale, *e_up_scale, *e_down_scale;  /* MoE: [E, f], [E, f], [E, d] fp32, applied
                                                             to each output channel after its dot product */
  /* weight_dtype ADP_E4M3 (dense): one fp32 scale per output row of wq, wk, wv, wo, w_gate, w_up,
   * w_down ([hq*hd], [hkv*hd] x2, [d], [ff] x2, [d]), applied after that row's dot product (read
   * in place); else NULL.  The pages project fp8 weights as the next step for large models
   * ([H] translated comment thread, author reply: "FP8" MoE). */
  const float *wq_scale, *wk_scale, *wv_scale, *wo_scale, *w_gate_scale, *w_up_scale, *w_down_scale;
  /* weight_dtype ADP_NVFP4 (dense): the seven matrices above hold [rows, K/2] bytes of E2M1 codes
   * and these their e4m3 block scales, [rows, K/16] bytes (one per 16 consecutive elements of a
   * row); an element is row scale x block scale x code, the row scale (above) applied after the
   * dot product.  Per 8-element vector of a row the element products are summed by fused
   * multiply-adds from zero, and that sum times its block scale is fused-multiply-added into the
   * vector's lane partial.  Copied into the image at creation; else NULL.  The pages project
   * 4-bit weights for larger models ([H] translated comment thread, author reply: mixed FP4/FP8). */
  const uint8_t *wq_bscale, *wk_bscale, *wv_bscale, *wo_bscale, *w_gate_bscale, *w_up_bscale, *w_down_bscale;
} adp_layer_weights;

typedef struct {
  const void *tok_emb;     /* [vocab, d] device */
  const void *lm_head;     /* [vocab, d] device, or NULL when tied */
  const void *final_norm;  /* [d] device */
  const adp_layer_weights *layers; /* HOST array of n_layers entries */
} adp_weights;

/* Sampling of the next token ([H] §"Kog Inference Engineの特徴とイノベーション": sampling is
 * a stage of the GPU program).  temperature == 0: greedy argmax, lowest index on ties.
 * temperature > 0: inverse-CDF draw from softmax(logits / temperature) with the caller's
 * uniform u in [0, 1) (the engine draws no random numbers itself). */
typedef struct {
  float temperature;
  float u;
} adp_sampling;

typedef struct adp_model adp_model;
typedef struct adp_kv adp_kv;

/* Create a model on the current CUDA device.
 *  cfg, w     host structs as above (w->layers host array; tensors device pointers)
 *  stream     cudaStream_t (as void*) the model launches on; NULL = the legacy default stream
 *  out        receives the model handle
 * Validates the shapes (head_dim even and <= 256; d_model, widths and vocab multiples of 8;
 * the persistent grid co-resident: one CTA per SM), plans the per-SM weight streams, copies
 * the matrices into the engine's own tile-ordered image (device memory owned by the model),
 * and allocates scratch.  Synchronises the stream before returning.
 * Errors: ADP_ERR_INVALID_ARG, ADP_ERR_UNSUPPORTED_CONFIG, ADP_ERR_NOT_CORESIDENT, ADP_ERR_CUDA. */
int adp_create_model(const adp_config* cfg, const adp_weights* w, void* stream, adp_model** out);
void adp_destroy_model(adp_model* m);

/* KV cache of one sequence ([H] §"GPU推論の速度制限要因：メモリ帯域幅": the KV cache is the
 * other stream each token reads; [A] §"どう出したか": kept uncompressed).  Engine-owned device
 * memory, layout [n_layers][n_kv_heads][max_ctx][head_dim] of cfg.kv_dtype for K and for V;
 * K rows hold post-RoPE keys.  A cache belongs to the model it was created from.  The model may
 * be destroyed before its caches: they then accept only adp_kv_destroy (every other call on them
 * returns ADP_ERR_INVALID_ARG). */
int adp_kv_create(adp_model* m, adp_kv** out);
void adp_kv_destroy(adp_kv* kv);
int adp_kv_reset(adp_kv* kv);                        /* length := 0 */
/* Rewind to the first len positions (0 <= len <= current length); later rows are overwritten
 * by the next steps.  Host-side only.  ADP_ERR_INVALID_ARG if len is out of range. */
int adp_kv_truncate(adp_kv* kv, int32_t len);
int adp_kv_len(const adp_kv* kv, int32_t* len);      /* number of cached positions */
/* Copy positions [0, len) in from / out to HOST arrays k, v of shape [n_layers][n_kv_heads][len][head_dim]
 * (storage bits of kv_dtype).  Load sets the length to len.  This is the whole decode state, so
 * it also serves as checkpoint save/restore.  Synchronous.  ADP_ERR_CONTEXT_OVERFLOW if len > max_ctx. */
int adp_kv_load(adp_kv* kv, const void* host_k, const void* host_v, int32_t len);
int adp_kv_read(const adp_kv* kv, void* host_k, void* host_v, int32_t len);

/* One decode step ([H] §"単一リクエストLLMデコード速度の重要性"): token `token` at position
 * p = current length; writes its K/V rows to the cache, returns the next token.
 *  sampling     host struct, NULL = greedy
 *  next_token   host pointer, receives the sampled/greedy next token
 *  dev_logits   optional DEVICE pointer [vocab] fp32 that receives the step's logits
 * One cooperative kernel launch (dependent phases wait on epoch-tagged outputs), a 4-byte token
 * and the 16-byte step state in, the token and status word out; synchronises the stream.
 * Errors: ADP_ERR_CONTEXT_OVERFLOW (p >= max_ctx; nothing launched), ADP_ERR_INVALID_ARG,
 * ADP_ERR_BARRIER_TIMEOUT / ADP_ERR_PIPELINE_TIMEOUT (sticky), ADP_ERR_CUDA. */
int adp_decode_step(adp_model* m, adp_kv* kv, int32_t token, const adp_sampling* sampling,
                    int32_t* next_token, float* dev_logits);

/* adp_decode_step without device allocation.  The persistent-decode method itself has no
 * counterpart to this call: it changes only where the step keeps its scratch (the activation
 * exchange words and their epoch base, the attention partials and counters, the sampling and
 * argmax words, the grid-barrier counter, the error word, the step state and, when dev_logits is
 * NULL, the logits).  These live in one static 8 MiB (8,388,608-byte) device array compiled into
 * the library instead of in the model's own buffers, and the call makes no cudaMalloc/cudaFree or
 * other allocating call.  It is meant for callers that may not allocate device memory while they
 * decode: a process whose memory manager has already reserved the device's free memory for its
 * own pool (a further allocation would fail or make the pool give memory back), or a serving loop
 * that cannot take the device-wide synchronisation that cudaMalloc and cudaFree may cause.
 * Arguments, results and the kernel are those of adp_decode_step (always the single persistent
 * launch), with the same output; the model's own scratch is left untouched.
 *  - Set-up happens in adp_create_model, not here: with the model's device current it looks up the
 *    array's device address once per device (cudaGetSymbolAddress, which may make the CUDA runtime
 *    load the library module holding the array, and so place the 8 MiB array in device memory).
 *    So the first no-alloc call on a device allocates nothing either.
 *  - The model's device must be the current device; otherwise ADP_ERR_INVALID_ARG (with a message in
 *    adp_last_error()) is returned before anything runs.
 *  - A model whose step needs more than 8 MiB of scratch (dominated by 8 * n_heads *
 *    ceil(max_ctx / 32) * head_dim bytes of attention partials plus 4 * vocab bytes of logits) is
 *    rejected with ADP_ERR_UNSUPPORTED_CONFIG before anything runs; adp_last_error() gives both sizes.
 *  - Every call shares the array.  All of it must be zero before a model's first step in it: it
 *    is at load, a completed step leaves it ready for the next one, and the call zeroes it first
 *    when the previous call was for a model with another scratch layout or failed.  Calls that
 *    overlap in time (from two threads, or on two streams) race on the array: serialise them.
 *  - A device-side error (ADP_ERR_BARRIER_TIMEOUT / ADP_ERR_PIPELINE_TIMEOUT) is returned and the
 *    array is zeroed; unlike adp_decode_step it does not leave the model in an error state. */
int adp_decode_step_noalloc(adp_model* m, adp_kv* kv, int32_t token, const adp_sampling* sampling,
                            int32_t* next_token, float* dev_logits);

/* Prefill: n successive decode steps over HOST tokens[0..n) (positions len..len+n-1) through the
 * same kernel, so prompt-written and decode-written KV rows follow one arithmetic; returns the
 * next token after the last one (and its logits if dev_logits).  One host->device copy of the
 * tokens, n launches, one synchronisation. */
int adp_prefill(adp_model* m, adp_kv* kv, const int32_t* host_tokens, int32_t n, const adp_sampling* sampling,
                int32_t* next_token, float* dev_logits);

/* Generation without host round trips: n decode steps starting from `token`, each step feeding
 * the token the previous one chose.  In the persistent kernel mode the n steps run inside ONE
 * cooperative launch: the step's last CTA publishes the chosen token as an epoch-tagged word and
 * every CTA takes it from there before the next step's embedding gather, while the weight stream
 * runs on across the step boundary (the ablation modes launch each step separately).
 * dev_u: optional DEVICE array of n uniforms (used when temperature > 0).  dev_tokens_out: DEVICE
 * array [n] that receives the chosen tokens.  Returns after enqueueing (does not synchronise);
 * adp_sync reports device errors.  adp_prefill likewise runs its n steps in one launch. */
int adp_generate_async(adp_model* m, adp_kv* kv, int32_t token, int32_t n, float temperature, const float* dev_u,
                       int32_t* dev_tokens_out);
int adp_sync(adp_model* m);                          /* synchronise the stream; report sticky errors */

/* Tensor-core prefill: the prompt's first n-1 tokens go through every layer as dense GEMMs on the
 * tcgen05 tensor cores ([P, d] x [d, n] contractions, fp32 accumulation in TMEM, activations
 * rounded to the weights' 16-bit type before each GEMM; RoPE with the K/V cache write and SwiGLU
 * in the GEMMs' epilogues), causal attention as flash-style tcgen05 MMAs (online softmax in fp32)
 * and RMSNorm kernels between them; their K/V rows go into the cache.  The last token
 * then runs as one adp_decode_step, whose logits and next token are returned.  The pages time
 * time-to-first-token ("標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒",
 * §"単一リクエストLLMデコード速度の重要性") but fix no prefill algorithm; this path is not the
 * decode step's arithmetic contract, so its KV rows and logits agree with the oracle within the
 * tolerances, not bit for bit (adp_prefill is the bit-exact path).
 * Arguments, errors and synchronisation as adp_prefill.  Dense models with head_dim 64 or 128 only
 * (else ADP_ERR_UNSUPPORTED_CONFIG); e4m3 and NVFP4 layer matrices are dequantised with their
 * row (and block) scales into the embedding's 16-bit type for the GEMMs.  The first call builds a second copy of the
 * layer matrices in the tensor cores' tile layout (16-bit, device memory owned by the model);
 * scratch grows with the longest prompt seen. */
int adp_prefill_tc(adp_model* m, adp_kv* kv, const int32_t* host_tokens, int32_t n, const adp_sampling* sampling,
                   int32_t* next_token, float* dev_logits);

/* Small-batch decode: nb independent requests of one model advance one token each in ONE
 * persistent launch that streams the weights once for all of them.  The pages' authors plan
 * small batches and warn that they trade against per-request speed ([H], the translated comment
 * thread, the author reply on batching); the pages fix no batched algorithm.  Per request the arithmetic is adp_decode_step's contract unchanged, so request
 * r's next token, logits and KV row are bit-identical to decoding it alone.
 *  kvs:        HOST array [nb] of distinct caches of this model, each at its own length (the
 *              request's position); each gains one row.
 *  tokens:     HOST array [nb], each in [0, vocab).
 *  sampling:   HOST array [nb] (temperature and uniform per request), or NULL for greedy.
 *  next_tokens: HOST array [nb] that receives the chosen tokens.
 *  dev_logits: optional DEVICE float array [nb][vocab].
 * nb must be in [1, adp_max_batch]: the batched kernel keeps every request's GEMV input vector
 * (fp32) in shared memory beside a weight ring of at least two slots (the down projection's
 * input in segments of whole K-chunks when nb whole vectors do not fit; see adp_batch_plan), and
 * merges head h of request r on CTA G-1-(r*n_heads+h).  Dense models with 16-bit, e4m3 or NVFP4
 * layer matrices (experts differ per request: MoE models get ADP_ERR_UNSUPPORTED_CONFIG).
 * Synchronises; errors as adp_decode_step (a device error is sticky and no cache grows). */
int adp_decode_batch(adp_model* m, adp_kv* const* kvs, int32_t nb, const int32_t* tokens,
                     const adp_sampling* sampling, int32_t* next_tokens, float* dev_logits);
/* n batched steps in one launch, each request feeding itself the token it chose.
 * temperatures: HOST array [nb] or NULL (greedy); dev_u: DEVICE array [n][nb] of uniforms,
 * required when some temperature is > 0; dev_tokens_out: DEVICE array [n][nb].  Returns after
 * enqueueing; adp_sync reports device errors. */
int adp_generate_batch_async(adp_model* m, adp_kv* const* kvs, int32_t nb, const int32_t* tokens, int32_t n,
                             const float* temperatures, const float* dev_u, int32_t* dev_tokens_out);
/* Largest nb this model can batch (0 when the model cannot batch at all).  The first call sets
 * up the batch buffers (device memory for 4 requests' exchange words and logits). */
int adp_max_batch(adp_model* m, int32_t* nb);

int adp_reset(adp_model* m);                         /* clear a sticky device error and sync counters */
const char* adp_status_string(int status);
const char* adp_last_error(void);                    /* text of the last ADP_ERR_CUDA in this thread */

/* Introspection used by tests and the benchmark. */
/* One phase of a decode step's plan (host-side description, see adp_plan). */
typedef struct {
  int32_t kind;       /* 0 QKV, 1 attention, 2 Wo, 3 FFN gate|up, 4 FFN down, 5 router, 6 expert gate|up,
                         7 expert down, 8 LM head, 9 sampling */
  int32_t layer;      /* n_layers for the LM head and sampling */
  int32_t n_units;    /* units of the phase, split evenly over the persistent CTAs (0: no weights) */
  int32_t unit_rows;  /* weight rows per unit (per expert slot) */
  int32_t slots;      /* expert slots per tile (1 for dense phases) */
  int32_t K;          /* reduction length */
  int32_t KC;         /* K-chunk width (a multiple of 256; the last chunk may be shorter) */
  int32_t n_chunks;   /* ceil(K / KC) */
  int32_t upr;        /* units per round of a CTA (a tile is min(upr, units left) x one K-chunk) */
  int32_t dtype;      /* adp_dtype of the phase's weights, -1 without weights */
  int32_t src_phase;  /* phase whose output vector this phase reads (-1: the embedding row) */
  int32_t res_phase;  /* phase that wrote the residual rows this phase adds to (-1: none) */
  int32_t sel_phase;  /* router phase whose logits choose this phase's experts (-1: none) */
  int32_t replicated; /* 1: every CTA streams the phase's one region and computes all its units
                       * (the router: each CTA chooses its experts without a hop); 0: units split
                       * evenly over the CTAs */
  uint64_t region;        /* byte offset of the phase's region in the weight image */
  uint64_t expert_stride; /* bytes of the region (per expert), a multiple of 256 */
} adp_phase_plan;

/* The plan of a decode step for cfg on a GPU with n_sms SMs (one persistent CTA each), computed on
 * the host without any CUDA call: the phases in step order and the size of the tile-ordered
 * weight image, exactly as adp_create_model lays them out on such a GPU.  CTA c of G owns units
 * [floor(c n / G), floor((c + 1) n / G)) of a phase of n units, stored from byte region +
 * floor(c n / G) x unit bytes as its rounds x K-chunks of tiles.  Writes min(cap, *n_phases) entries
 * of out (caller-owned HOST memory); *n_phases gets the full count and *image_bytes the image size.
 * Errors: ADP_ERR_INVALID_ARG (null pointers, n_sms < 1) and the config errors of adp_create_model. */
int adp_plan(const adp_config* cfg, int32_t n_sms, adp_phase_plan* out, int32_t cap, int32_t* n_phases,
             uint64_t* image_bytes);

/* The batched kernel's shared-memory layout for one batch size (see adp_batch_plan). */
typedef struct {
  int32_t ring_slots;      /* 32 KB weight slots of the ring (0: this batch size does not fit) */
  int32_t attention_slots; /* attention items a CTA stages at once */
  int32_t xbuf_floats;     /* floats of the input-vector / staging area (nb input vectors at least) */
  int32_t down_segment;    /* elements of each request's down-projection input staged at once: d_ff
                              (whole), or a whole number of that phase's K-chunks (segments, when nb
                              whole inputs do not fit beside a ring of two slots) */
  uint64_t control_bytes;  /* the control block (phase table, per-request state) */
  uint64_t smem_bytes;     /* dynamic shared memory of a launch: ring + staging area + control block */
} adp_batch_layout;

/* The batched kernel's layout for 1..4 requests of cfg on a GPU with n_sms SMs and smem_optin bytes
 * of opt-in shared memory per block, computed on the host without any CUDA call, exactly as the
 * first batched call lays it out (adp_decode_batch; GB300: 232,448 bytes).  out: caller-owned HOST
 * array of 4 entries, entry nb - 1 for nb requests; *max_batch gets the largest batch that fits
 * (0: none; MoE models are not batched).  Errors: ADP_ERR_INVALID_ARG (null pointers, n_sms < 1,
 * smem_optin < 1) and the config errors of adp_create_model. */
int adp_batch_plan(const adp_config* cfg, int32_t n_sms, int32_t smem_optin, adp_batch_layout* out,
                   int32_t* max_batch);

int adp_num_ctas(const adp_model* m, int32_t* ctas);            /* persistent grid size (SMs) */
int adp_image_bytes(const adp_model* m, uint64_t* bytes);       /* bytes of the tile-ordered weight image */
int adp_launches_per_step(const adp_model* m, int32_t* n);      /* kernel launches of one decode step */

/* Measurement helper (not part of the decode step): the read bandwidth this GPU delivers on a
 * caller-given DEVICE buffer of `bytes` bytes (16-byte aligned; use one larger than L2 so that the
 * reads come from HBM): `reps` launches of a grid-stride kernel of 16-byte loads on the stream
 * (NULL = the default stream), after one untimed launch, timed with CUDA events; *gb_per_s gets
 * bytes * reps / time.  The buffer is only read (its first word would be written only if the xor of
 * all its words equalled one fixed constant).  Allocates nothing; synchronises the stream.
 * Errors: ADP_ERR_INVALID_ARG, ADP_ERR_CUDA.  Bandwidth is the bound of batch-1 decode
 * ([H] §"GPU推論の速度制限要因：メモリ帯域幅"). */
int adp_measure_read_bandwidth(const void* dev_buf, uint64_t bytes, int32_t reps, void* cuda_stream,
                               double* gb_per_s);

/* Debug and ablation hooks ([H] §"標準推論スタックのボトルネックとKogの工夫": the launch
 * overhead the persistent kernel removes is measured by running the same device code as one
 * launch per phase).
 *  mode 0: persistent (one cooperative launch per step, grid barriers)
 *  mode 1: multi-kernel (one launch per phase, same device functions, same arithmetic)
 *  mode 2: multi-kernel, captured once into a CUDA graph and replayed per step */
int adp_debug_kernel_mode(adp_model* m, int mode);
/* Force MoE expert choices: HOST array [n_layers][top_k] of expert ids (NULL = router decides).
 * Gates are the router's probabilities of the forced experts, renormalised over them. */
int adp_debug_force_experts(adp_model* m, const int32_t* host_idx);
/* The router's own choices of the last step: HOST array [n_layers][top_k]. */
int adp_debug_read_experts(const adp_model* m, int32_t* host_idx);
/* Record the residual entering each layer (and the final one) of every step into a DEVICE
 * buffer [n_layers + 1][d_model] fp32 (NULL = off). */
int adp_debug_trace_residual(adp_model* m, float* dev_buf);
/* Per-phase timeline of every CTA: DEVICE buffer [ctas][phases][16] of %globaltimer stamps (ns):
 * 0 phase entry, 1 after the prologue, 2 after the phase body, 3 after the grid barrier (consumer
 * warp 0), 4 first and 5 last weight tile issued (producer warp), 7 ns the producer spent with
 * the ring full; weighted phases: 8 first tile ready and 9 last K-chunk done (consumer warp 0);
 * attention: 4 first item's data staged, 6 its block computed, 5 its partial published, 7 all
 * items done, 10 a merged head's partials seen, 12 its weights formed, 13 its outputs summed,
 * 11 published.  In builds with -DADP_CYCLE_STAMPS entries 12..15 of weighted phases hold SM
 * cycles of consumer warp 0 (waiting for tiles, computing, whole round loop, epilogues) and of
 * the first attention item (scores, weights, weighted sum, publication).  Unused entries keep
 * what the buffer held.  NULL = off.  Sizes from adp_debug_timeline_shape. */
int adp_debug_timeline(adp_model* m, uint64_t* dev_buf);
int adp_debug_timeline_shape(const adp_model* m, int32_t* ctas, int32_t* phases);
/* 1: also take a grid barrier after every phase (debugging the epoch-tagged exchange). */
int adp_debug_barriers(adp_model* m, int on);
/* Bytes of each SM's weight stream the producer warp keeps prefetched into L2 beyond its TMA
 * loads (default 0 = off).  A tuning knob: it lets HBM keep streaming while the compute
 * warps wait at barriers. */
int adp_debug_set_l2_lookahead(adp_model* m, uint32_t bytes);
/* How the step prefetches into L2 (bits; default 0): 1 = each layer's attention K/V blocks one
 * layer early (during the previous layer's QKV phase), 2 = those K/V prefetches with the L2
 * evict-last priority, 4 = the weight lookahead with the evict-last priority.  Other bits:
 * ADP_ERR_INVALID_ARG.  A tuning knob; results do not depend on it. */
int adp_debug_set_prefetch_flags(adp_model* m, uint32_t flags);
/* Pace the weight lookahead (adp_debug_set_l2_lookahead) with a token bucket per CTA: at most
 * bytes_per_us bytes of prefetch per microsecond, at most burst_bytes (>= 32768) at once;
 * bytes_per_us = 0 (the default) issues the lookahead unpaced.  A tuning knob; results do not
 * depend on it. */
int adp_debug_set_l2_pacing(adp_model* m, uint32_t bytes_per_us, uint32_t burst_bytes);
/* Depth of the per-CTA weight ring in 32 KB slots: the model takes the deepest ring (at most 6)
 * that fits beside its other shared-memory buffers; this lowers it (3 <= slots <= that depth,
 * else ADP_ERR_INVALID_ARG), for measurements.  adp_debug_ring_slots reads the current depth. */
int adp_debug_set_ring_slots(adp_model* m, int32_t slots);
int adp_debug_ring_slots(const adp_model* m);
#ifdef ADP_TEST_HOOKS
/* The three hooks below exist only in the test build of the library (libadp_test.so, compiled with
 * -DADP_TEST_HOOKS); the release build (libadp.so) does not export them.
 *
 * Test hook: clear the exchange buffers and start the model's 32-bit epoch counter at `base`
 * (the engine clears and restarts it by itself before a step would run past 2^32). */
int adp_debug_set_epoch_base(adp_model* m, uint32_t base);
/* Wait limit of every in-kernel spin (grid barrier, weight pipeline), nanoseconds (default 2e8). */
int adp_debug_set_wait_limit(adp_model* m, uint64_t ns);
/* Test hook: in the next step, CTA `cta` withholds the outputs of phase number `phase` (-1 = off),
 * so that every phase waiting for them runs out of time and the step returns
 * ADP_ERR_BARRIER_TIMEOUT (a dependency wait ran out) instead of hanging. */
int adp_debug_skip_publication(adp_model* m, int32_t cta, int32_t phase);
#endif /* ADP_TEST_HOOKS */
/* The prefill path's tensor-core GEMM alone (test hook): C[M, N] = A[M, K] W[N, K]^T in fp32, with
 * A and W DEVICE row-major 16-bit matrices (f16, or bf16 when bf16 = 1) and C a DEVICE fp32 [M, N]
 * array.  Tiles the operands into temporary device buffers, runs, synchronises the device. */
int adp_debug_tc_gemm(int32_t bf16, int32_t M, int32_t N, int32_t K, const void* A, const void* W, float* C);
/* Benchmark hook of the tensor-core prefill: times `reps` back-to-back launches of one of the
 * model's prefill GEMMs (which: 0 QKV (with a plain fp32 store epilogue here), 1 Wo, 2 gate|up
 * (with its SwiGLU epilogue), 3 down; layer 0's weights) on M tokens of a constant operand, with
 * CUDA events on the model's stream; *ms_per_launch receives the mean. */
int adp_debug_tc_gemm_time(adp_model* m, int32_t which, int32_t M, int32_t reps, float* ms_per_launch);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#ifdef __cplusplus
}
#endif
#endif /* ADP_H_ */

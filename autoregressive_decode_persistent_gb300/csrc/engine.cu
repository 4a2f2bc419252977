// Host engine behind the C ABI of include/adp.h: configuration checks, the per-SM weight
// stream plan, the tile-ordered weight image, scratch, KV caches and the decode-step launches.
//
// Pages followed: "標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒" (hakusoku.com),
// sections "単一リクエストLLMデコード速度の重要性" (batch-1, one request), "標準推論スタックのボトルネック
// とKogの工夫" (one GPU-resident launch per step instead of ~10 kernels per layer) and
// "Kog Inference Engineの特徴とイノベーション" (the engine orders sync and prefetch itself).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/adp.h"
#include "launch.h"
#include "plan.h"
#include "scratch.h"

using namespace adp;

namespace {

thread_local std::string g_last_error;

int cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return ADP_ERR_CUDA;
}

#define CK(call)                                   \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

// Bytes per element of a weight type (0 for NVFP4, whose image bytes come from wbytes()).
int elem_bytes(int dt) { return dt == ADP_NVFP4 ? 0 : dt == ADP_E4M3 ? 1 : (dt == ADP_F32 ? 4 : 2); }

// Layer matrices quantised with fp32 row scales (e4m3, NVFP4): the embedding, the LM head and
// the norm gains then keep the 16-bit embed_dtype.
static bool quantised(int wdt) { return wdt == ADP_E4M3 || wdt == ADP_NVFP4; }
static int head_dtype(const adp_config& c) { return quantised(c.weight_dtype) ? c.embed_dtype : c.weight_dtype; }

}  // namespace

struct adp_kv {
  adp_model* m = nullptr;
  uint16_t* k = nullptr;
  uint16_t* v = nullptr;
  int32_t len = 0;
  size_t bytes = 0;  // of each of k and v
};

struct adp_model {
  adp_config cfg{};
  int device = 0;
  cudaStream_t stream = nullptr;
  int G = 0;
  int xbuf_floats = 0;
  size_t smem = 0;
  int max_nslots = 0;
  std::vector<PhaseDesc> phases;
  PhaseDesc* d_phases = nullptr;
  uint8_t* image = nullptr;
  uint64_t image_bytes = 0;
  Params p{};            // fields that do not change between steps
  std::vector<void*> allocs;
  StepState* h_state = nullptr;  // pinned
  cudaEvent_t state_copied = nullptr;  // the last host->device copy of h_state has executed
  int32_t* h_out = nullptr;      // pinned: out_token, err
  int32_t* d_tokseq = nullptr;
  int32_t tokseq_cap = 0;
  int32_t* d_force = nullptr;
  bool force_on = false;
  float* d_logits_scratch = nullptr;
  std::vector<adp_kv*> kvs;  // live caches of this model (orphaned when the model goes first)
  int mode = 0;
  // multi-kernel graph cache
  cudaGraphExec_t graph = nullptr;
  const void* graph_key_kv = nullptr;
  const void* graph_key_logits = nullptr;
  bool graph_key_sample = false;
  int sticky = ADP_OK;
  uint64_t epochs_used = 0;  // epochs handed out since the exchange buffers were last cleared
  size_t ll_bytes[11] = {0};  // sizes of the epoch-tagged exchange buffers
  std::vector<const void*> h_attn_norm, h_ffn_norm;  // per-layer gains (device pointers)
  std::vector<const float*> h_wscale[7];             // e4m3 dense: per-layer row scales of q, k, v, o, gate, up, down
  // Tensor-core prefill (set up at the first adp_prefill_tc): the layer matrices again, as GEMM
  // operand tiles, and scratch for up to tc_cap prompt tokens.
  struct TcState {
    int init_rc = 1;
    std::vector<const uint8_t*> wqkv, wo, wgu, wdown;
    std::vector<const float*> sqkv, swo, sgu, sdown;  // column scales of quantised layer matrices
    int cap = 0;
    int32_t* tokens = nullptr;
    float* x = nullptr;
    uint8_t* A = nullptr;
    uint8_t* A2 = nullptr;
    uint8_t* Qt = nullptr;  // query tiles of the attention kernel
    uint8_t* Kt = nullptr;  // key / transposed value tiles of every cache position (the attention's)
    uint8_t* Vt = nullptr;
    float* C = nullptr;     // fp32 QKV output (the timing hook's plain-store QKV GEMM only)
  } tc;
  // Batched decode (set up at the first batched call): per-request buffers for kMaxBatch
  // requests, the per-request step state and KV cache tables, and the shared-memory layout of
  // each batch size.
  struct BatchHost {
    StepState st[kMaxBatch];
    uint16_t* kcb[kMaxBatch];
    uint16_t* vcb[kMaxBatch];
  };
  struct Batch {
    int init_rc = 1;  // 1: not set up yet; else the set-up's status
    int max_nb = 0;
    size_t smem[kMaxBatch + 1] = {};
    int nslots[kMaxBatch + 1] = {}, xbuf_floats[kMaxBatch + 1] = {}, att_slots[kMaxBatch + 1] = {};
    int down_seg[kMaxBatch + 1] = {};  // elements of the down input staged at once per request
    Params p{};                    // the batch buffers (per-request copies back to back)
    BatchHost* h = nullptr;        // pinned staging of the step state and cache tables
    BatchHost* d = nullptr;
    cudaEvent_t copied = nullptr;  // the last copy out of h has executed
    int32_t* h_out = nullptr;      // pinned: out_token per request, then err
    float* d_logits = nullptr;     // [kMaxBatch][V] logits when the caller passes none
    size_t ll_bytes[11] = {0};
  } bt;

  template <class T>
  int alloc(T** ptr, size_t count) {
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, std::max<size_t>(count * sizeof(T), 16));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    allocs.push_back(q);
    *ptr = static_cast<T*>(q);
    return ADP_OK;
  }
};

// ---------------------------------------------------------------- validation and planning

// The shape and type checks of a config (no weights).
static int validate_config(const adp_config* c) {
  if (!c) return ADP_ERR_INVALID_ARG;
  if (c->n_layers < 1 || c->d_model < 8 || c->n_heads < 1 || c->n_kv_heads < 1 || c->vocab < 8 || c->max_ctx < 1)
    return ADP_ERR_INVALID_ARG;
  if (c->n_kv_heads > c->n_heads) return ADP_ERR_UNSUPPORTED_CONFIG;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return ADP_ERR_UNSUPPORTED_CONFIG;
  if (c->d_model % 8 || c->vocab % 8 || (c->n_heads * c->head_dim) % 8) return ADP_ERR_UNSUPPORTED_CONFIG;
  if (c->d_model > 7680 || c->vocab > 1024 * 256) return ADP_ERR_UNSUPPORTED_CONFIG;
  // fp8 or NVFP4 layer matrices with per-row scales (dense only)
  const bool q8 = quantised(c->weight_dtype), q4 = c->weight_dtype == ADP_NVFP4;
  if (c->weight_dtype != ADP_F16 && c->weight_dtype != ADP_BF16 && !(q8 && c->n_experts == 0))
    return ADP_ERR_UNSUPPORTED_CONFIG;
  if (q8 && c->embed_dtype != ADP_F16 && c->embed_dtype != ADP_BF16) return ADP_ERR_UNSUPPORTED_CONFIG;
  if (q8 && (c->d_model % 16 || c->d_ff % 16 || (c->n_heads * c->head_dim) % 16)) return ADP_ERR_UNSUPPORTED_CONFIG;
  // NVFP4 tiles stay 16-byte multiples when every reduction length is a multiple of 128
  if (q4 && (c->d_model % 128 || c->d_ff % 128 || (c->n_heads * c->head_dim) % 128))
    return ADP_ERR_UNSUPPORTED_CONFIG;
  if (c->kv_dtype != ADP_F16 && c->kv_dtype != ADP_BF16) return ADP_ERR_UNSUPPORTED_CONFIG;
  if (c->n_experts == 0) {
    if (c->d_ff < 8 || c->d_ff % 8) return ADP_ERR_UNSUPPORTED_CONFIG;
  } else {
    if (c->expert_dtype != ADP_E4M3) return ADP_ERR_UNSUPPORTED_CONFIG;
    if (c->router_dtype != ADP_F16 && c->router_dtype != ADP_BF16) return ADP_ERR_UNSUPPORTED_CONFIG;
    if (c->n_experts > 1024 || c->top_k < 1 || c->top_k > c->n_experts) return ADP_ERR_UNSUPPORTED_CONFIG;
    if (c->top_k != 1 && c->top_k != 2 && c->top_k != 4 && c->top_k != 8) return ADP_ERR_UNSUPPORTED_CONFIG;
    if (c->d_expert < 16 || c->d_expert % 16 || c->d_model % 16) return ADP_ERR_UNSUPPORTED_CONFIG;
  }
  return ADP_OK;
}

static int validate(const adp_config* c, const adp_weights* w) {
  if (!c || !w || !w->layers || !w->tok_emb || !w->final_norm) return ADP_ERR_INVALID_ARG;
  const int rc = validate_config(c);
  if (rc) return rc;
  const bool q8 = quantised(c->weight_dtype), q4 = c->weight_dtype == ADP_NVFP4;
  if (!c->tied_embeddings && !w->lm_head) return ADP_ERR_INVALID_ARG;
  for (int l = 0; l < c->n_layers; ++l) {
    const adp_layer_weights& L = w->layers[l];
    if (!L.attn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.ffn_norm) return ADP_ERR_INVALID_ARG;
    if (c->n_experts == 0 && (!L.w_gate || !L.w_up || !L.w_down)) return ADP_ERR_INVALID_ARG;
    if (q8 && (!L.wq_scale || !L.wk_scale || !L.wv_scale || !L.wo_scale || !L.w_gate_scale || !L.w_up_scale ||
               !L.w_down_scale))
      return ADP_ERR_INVALID_ARG;
    if (q4 && (!L.wq_bscale || !L.wk_bscale || !L.wv_bscale || !L.wo_bscale || !L.w_gate_bscale ||
               !L.w_up_bscale || !L.w_down_bscale))
      return ADP_ERR_INVALID_ARG;
    if (c->n_experts && (!L.router || !L.e_gate || !L.e_up || !L.e_down || !L.e_gate_scale || !L.e_up_scale ||
                         !L.e_down_scale))
      return ADP_ERR_INVALID_ARG;
  }
  return ADP_OK;
}

// Append a phase; weighted phases get a region of the image and a K-chunk width such that one
// round of units fits one ring slot.
static void add_phase(adp_model* m, int kind, int layer, int n_units, int unit_rows, int slots, int K, int eb,
                      int wdt, bool weights, int experts, bool replicated = false) {
  PhaseDesc P{};
  P.kind = kind;
  P.layer = layer;
  P.index = (int32_t)m->phases.size();
  P.has_weights = weights ? 1 : 0;
  P.replicated = replicated ? 1 : 0;
  if (weights) {
    P.n_units = n_units;
    P.unit_rows = unit_rows;
    P.slots = slots;
    P.K = K;
    P.eb = eb;
    P.wdt = wdt;
    // balanced rounds of at most kConsumerWarps units over the largest per-CTA share
    const int maxu = replicated ? std::max(1, n_units) : std::max(1, (n_units + m->G - 1) / m->G);
    const int nrounds = (maxu + kConsumerWarps - 1) / kConsumerWarps;
    int upr = (maxu + nrounds - 1) / nrounds;
    while (upr > 1 && wbytes(P, (uint64_t)upr * unit_rows * slots * kChunkAlign) > (uint64_t)kSlotBytes) --upr;
    P.upr = upr;
    // the widest K-chunk (a multiple of kChunkAlign) whose round of tiles fits one slot
    int KC = (int)(kSlotBytes / wbytes(P, (uint64_t)upr * unit_rows * slots * kChunkAlign)) * kChunkAlign;
    const int Kr = (K + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
    KC = std::min(KC, Kr);
    P.KC = KC;
    P.n_chunks = (K + KC - 1) / KC;
    const uint64_t region = wbytes(P, (uint64_t)n_units * unit_rows * K);
    P.region = m->image_bytes;
    P.expert_stride = (region + 255) / 256 * 256;
    m->image_bytes += P.expert_stride * (uint64_t)experts;
  }
  m->phases.push_back(P);
}

static void plan(adp_model* m) {
  const adp_config& c = m->cfg;
  const int d = c.d_model, hq = c.n_heads, hkv = c.n_kv_heads, hd = c.head_dim;
  const int eb = elem_bytes(c.weight_dtype);
  // Which phase produced each input: the residual x, the attention output, the FFN activations
  // and the router logits are read by epoch, so every phase names its producers.
  int x_ph = -1;  // latest writer of the residual (-1 before layer 0: the embedding row)
  auto last = [&]() { return (int)m->phases.size() - 1; };
  auto link = [&](int src, int res, int sel) {
    PhaseDesc& P = m->phases.back();
    P.src_ph = src;
    P.res_ph = res;
    P.sel_ph = sel;
  };
  for (int l = 0; l < c.n_layers; ++l) {
    add_phase(m, PK_QKV, l, (hq + 2 * hkv) * hd / 2, 2, 1, d, eb, c.weight_dtype, true, 1);
    link(x_ph, -1, -1);
    const int qkv = last();
    if (l == 0) x_ph = qkv;  // the QKV phase of layer 0 publishes x = embedding row
    add_phase(m, PK_ATTN, l, 0, 0, 0, 0, 0, 0, false, 0);
    link(qkv, -1, -1);
    const int att = last();
    add_phase(m, PK_WO, l, d / 2, 2, 1, hq * hd, eb, c.weight_dtype, true, 1);
    link(att, x_ph, -1);
    x_ph = last();
    if (c.n_experts == 0) {
      add_phase(m, PK_GU, l, c.d_ff, 2, 1, d, eb, c.weight_dtype, true, 1);
      link(x_ph, -1, -1);
      const int gu = last();
      add_phase(m, PK_DOWN, l, d / 2, 2, 1, c.d_ff, eb, c.weight_dtype, true, 1);
      link(gu, x_ph, -1);
      x_ph = last();
    } else {
      // every CTA computes all router logits itself (its experts are then chosen without a hop), in
      // units of 4 rows when the expert count allows (one round of at most 8 units for 32 experts)
      const int rrows = c.n_experts % 4 == 0 ? 4 : 1;
      add_phase(m, PK_ROUTER, l, c.n_experts / rrows, rrows, 1, d, elem_bytes(c.router_dtype), c.router_dtype, true, 1,
                true);
      link(x_ph, -1, -1);
      const int router = last();
      add_phase(m, PK_EGU, l, c.d_expert, 2, c.top_k, d, 1, ADP_E4M3, true, c.n_experts);
      link(x_ph, -1, router);
      const int egu = last();
      add_phase(m, PK_EDOWN, l, d, 1, c.top_k, c.d_expert, 1, ADP_E4M3, true, c.n_experts);
      link(egu, x_ph, router);
      x_ph = last();
    }
  }
  const int edt = head_dtype(c);  // the LM head's type
  add_phase(m, PK_LM, c.n_layers, c.vocab / 4, 4, 1, d, elem_bytes(edt), edt, true, 1);
  link(x_ph, -1, -1);
  add_phase(m, PK_SAMPLE, c.n_layers, 0, 0, 0, 0, 0, 0, false, 0);
  link(-1, -1, -1);
}

// Zero the epoch base and every epoch-tagged exchange buffer (epoch 0 is never awaited).
static int clear_exchange(adp_model* m) {
  const Params& p = m->p;
  void* bufs[11] = {p.x, p.q, p.attn, p.h, p.rlog, p.knew, p.vnew, p.part_m, p.part_l, p.part_o, p.tok_word};
  for (int i = 0; i < 11; ++i) CK(cudaMemsetAsync(bufs[i], 0, m->ll_bytes[i], m->stream));
  if (m->bt.init_rc == ADP_OK) {
    const Params& b = m->bt.p;
    void* bb[11] = {b.x, b.q, b.attn, b.h, nullptr, b.knew, b.vnew, b.part_m, b.part_l, b.part_o, b.tok_word};
    for (int i = 0; i < 11; ++i)
      if (bb[i]) CK(cudaMemsetAsync(bb[i], 0, m->bt.ll_bytes[i], m->stream));
  }
  CK(cudaMemsetAsync(p.epoch, 0, 4, m->stream));
  m->epochs_used = 0;
  return ADP_OK;
}

// Epochs are 32-bit and every step takes n_phases of them.  Before the steps about to be
// enqueued would run past 2^32, start over: zero the exchange buffers and the epoch base
// (stream-ordered, between launches), so that tags never wrap around.
static int reserve_epochs(adp_model* m, int n_steps) {
  const uint64_t need = (uint64_t)m->phases.size() * ((uint64_t)n_steps + 1);
  if (m->epochs_used + need >= (1ull << 32)) {
    const int rc = clear_exchange(m);
    if (rc) return rc;
  }
  m->epochs_used += (uint64_t)m->phases.size() * (uint64_t)n_steps;
  return ADP_OK;
}

// ---------------------------------------------------------------- model creation

// Most query heads sharing one KV head (query head h reads KV head floor(h hkv / hq)).
static int kv_group_max(const adp_config& c) {
  int gmax = 0;
  for (int g = 0; g < c.n_kv_heads; ++g) {
    const int h0 = (g * c.n_heads + c.n_kv_heads - 1) / c.n_kv_heads;
    const int h1 = ((g + 1) * c.n_heads + c.n_kv_heads - 1) / c.n_kv_heads;
    gmax = std::max(gmax, h1 - h0);
  }
  return gmax;
}

static int create(adp_model* m, const adp_config* cfg, const adp_weights* w) {
  const adp_config& c = *cfg;
  CK(cudaGetDevice(&m->device));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, m->device));
  if (!prop.cooperativeLaunch) return ADP_ERR_NOT_CORESIDENT;
  m->G = prop.multiProcessorCount;  // one persistent CTA per SM
  {
    const int rc = noalloc_prepare_device(m->device);  // the static scratch of adp_decode_step_noalloc
    if (rc) return rc;
  }
  plan(m);
  for (const PhaseDesc& P : m->phases)  // per-CTA shares are computed in 32-bit arithmetic
    if ((uint64_t)P.n_units * (uint64_t)m->G >= (1ull << 32)) return ADP_ERR_UNSUPPORTED_CONFIG;
  const int d = c.d_model, hq = c.n_heads, hkv = c.n_kv_heads, hd = c.head_dim, L = c.n_layers;
  const int ffw = c.n_experts ? c.top_k * c.d_expert : c.d_ff;
  // xbuf holds a phase's input vector, the attention warps' K/V staging areas, or the merge's
  // per-block weights: sized for the largest use that fits beside the ring.
  const int nbmax_ = (c.max_ctx + kAttnBlock - 1) / kAttnBlock;
  const size_t ctl_sz = (ctl_bytes((int)m->phases.size()) + 127) & ~(size_t)127;
  const size_t optin = (size_t)prop.sharedMemPerBlockOptin;
  const int gmax = kv_group_max(c);  // most query heads sharing one KV head
  if (gmax < 1 || gmax > kMaxGroup) return ADP_ERR_UNSUPPORTED_CONFIG;
  if (hq > m->G) return ADP_ERR_UNSUPPORTED_CONFIG;  // CTA G-1-h merges query head h
  // K (rows padded by 16 bytes), V, the group's queries, the weights e_j
  const size_t item = (size_t)kAttnBlock * (hd + 8) * 2 + (size_t)kAttnBlock * hd * 2 + (size_t)kMaxGroup * hd * 4 +
                      (size_t)kMaxGroup * kAttnBlock * 4;
  // GEMV input vectors are stored in shared memory padded to multiples of 256 floats (per expert
  // slot for the expert down projection)
  auto pad256 = [](int n) { return (size_t)((n + 255) / 256 * 256); };
  const size_t vec_floats = std::max({pad256(d), pad256(hq * hd),
                                      c.n_experts ? (size_t)c.top_k * pad256(c.d_expert) : pad256(c.d_ff)});
  const size_t vec_bytes = std::max(vec_floats * 4, ((size_t)2 * 8 * nbmax_ + 8) * 4);
  // The deepest weight ring (kMaxSlots down to 3 slots) that leaves room for the input vector and
  // one attention item; the attention slots then take the room that is left (at most one query
  // head per consumer warp).
  int nslots = 0, att_slots = 0;
  size_t xbytes = 0;
  for (int ns = kMaxSlots; ns >= 3 && !nslots; --ns) {
    if ((size_t)ns * kSlotBytes + ctl_sz > optin) continue;
    const size_t room = optin - (size_t)ns * kSlotBytes - ctl_sz;
    if (room < vec_bytes || room < item) continue;
    nslots = ns;
    att_slots = (int)std::min<size_t>(std::min(kAttnSlots, kConsumerWarps / gmax), room / item);
    xbytes = std::max(vec_bytes, (size_t)att_slots * item);
  }
  if (!nslots) return ADP_ERR_UNSUPPORTED_CONFIG;
  xbytes = (xbytes + 127) & ~(size_t)127;
  // the attention merge stages at least one block's outputs (8-byte words) after the block maxima and sums
  if ((long long)(xbytes / 4) - ((2 * nbmax_ + 2 + 3) & ~3) < 2 * hd) return ADP_ERR_UNSUPPORTED_CONFIG;
  m->xbuf_floats = (int)(xbytes / 4);
  m->p.xbuf_floats = m->xbuf_floats;
  m->smem = (size_t)nslots * kSlotBytes + xbytes + ctl_bytes((int)m->phases.size());
  if (m->smem > optin) return ADP_ERR_UNSUPPORTED_CONFIG;
  m->p.nslots = nslots;
  m->max_nslots = nslots;
  m->p.att_slots = att_slots;
  m->p.att_gmax = gmax;
  m->p.att_slot_bytes = (int)item;
  int bps = 0;
  {
    const int kind = c.n_experts > 0                 ? KK_MOE
                     : c.weight_dtype == ADP_E4M3  ? KK_DENSE8
                     : c.weight_dtype == ADP_NVFP4 ? KK_DENSE4
                                                   : KK_DENSE;
    CK(decode_prepare(m->smem, kind, c.head_dim, c.kv_dtype, kind == KK_DENSE ? c.weight_dtype : head_dtype(c),
                      &bps));
  }
  if (bps < 1) return ADP_ERR_NOT_CORESIDENT;

  // weight image
  int rc;
  if ((rc = m->alloc(&m->image, m->image_bytes))) return rc;
  if ((rc = m->alloc(&m->d_phases, m->phases.size()))) return rc;
  CK(cudaMemcpyAsync(m->d_phases, m->phases.data(), m->phases.size() * sizeof(PhaseDesc), cudaMemcpyHostToDevice,
                     m->stream));
  const int eb = elem_bytes(c.weight_dtype);
  for (const PhaseDesc& P : m->phases) {
    if (!P.has_weights) continue;
    RepackSrc S{};
    S.hd = hd;
    S.hq = hq;
    S.hkv = hkv;
    int experts = 1;
    if (P.kind == PK_LM) {
      S.a = (const uint8_t*)(c.tied_embeddings ? w->tok_emb : w->lm_head);
    } else {
      const adp_layer_weights& Lw = w->layers[P.layer];
      switch (P.kind) {
        case PK_QKV:
          S.a = (const uint8_t*)Lw.wq; S.b = (const uint8_t*)Lw.wk; S.c = (const uint8_t*)Lw.wv;
          S.sa = Lw.wq_bscale; S.sb = Lw.wk_bscale; S.sc = Lw.wv_bscale;
          break;
        case PK_WO: S.a = (const uint8_t*)Lw.wo; S.sa = Lw.wo_bscale; break;
        case PK_GU:
          S.a = (const uint8_t*)Lw.w_gate; S.b = (const uint8_t*)Lw.w_up;
          S.sa = Lw.w_gate_bscale; S.sb = Lw.w_up_bscale;
          break;
        case PK_DOWN: S.a = (const uint8_t*)Lw.w_down; S.sa = Lw.w_down_bscale; break;
        case PK_ROUTER: S.a = (const uint8_t*)Lw.router; break;
        case PK_EGU:
          S.a = (const uint8_t*)Lw.e_gate; S.b = (const uint8_t*)Lw.e_up;
          S.expert_src_stride = (uint64_t)c.d_expert * d;
          experts = c.n_experts;
          break;
        case PK_EDOWN:
          S.a = (const uint8_t*)Lw.e_down;
          S.expert_src_stride = (uint64_t)d * c.d_expert;
          experts = c.n_experts;
          break;
        default: break;
      }
    }
    CK(repack_launch(m->image, P, S, P.replicated ? 1 : m->G, experts, m->stream));
  }
  (void)eb;

  // per-layer pointer tables
  std::vector<const void*> an(L), fn(L);
  std::vector<const float*> sg(L), su(L), sd(L);
  std::vector<const float*> ws[7];  // e4m3 layer-matrix scales: q, k, v, o, gate, up, down
  for (auto& v : ws) v.resize(L);
  for (int l = 0; l < L; ++l) {
    const adp_layer_weights& Lw = w->layers[l];
    an[l] = Lw.attn_norm;
    fn[l] = Lw.ffn_norm;
    m->h_attn_norm.push_back(Lw.attn_norm);
    m->h_ffn_norm.push_back(Lw.ffn_norm);
    sg[l] = Lw.e_gate_scale;
    su[l] = Lw.e_up_scale;
    sd[l] = Lw.e_down_scale;
    const float* s7[7] = {Lw.wq_scale, Lw.wk_scale, Lw.wv_scale, Lw.wo_scale, Lw.w_gate_scale, Lw.w_up_scale,
                          Lw.w_down_scale};
    for (int i = 0; i < 7; ++i) {
      ws[i][l] = quantised(c.weight_dtype) ? s7[i] : nullptr;
      m->h_wscale[i].push_back(ws[i][l]);
    }
  }
  for (int i = 0; i < 7; ++i) {
    const float** t = nullptr;
    if ((rc = m->alloc(&t, L))) return rc;
    CK(cudaMemcpyAsync(t, ws[i].data(), L * sizeof(void*), cudaMemcpyHostToDevice, m->stream));
    m->p.wscale[i] = t;
  }
  const void** d_an; const void** d_fn; const float** d_sg; const float** d_su; const float** d_sd;
  if ((rc = m->alloc(&d_an, L)) || (rc = m->alloc(&d_fn, L)) || (rc = m->alloc(&d_sg, L)) ||
      (rc = m->alloc(&d_su, L)) || (rc = m->alloc(&d_sd, L)))
    return rc;
  CK(cudaMemcpyAsync(d_an, an.data(), L * sizeof(void*), cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(d_fn, fn.data(), L * sizeof(void*), cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(d_sg, sg.data(), L * sizeof(void*), cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(d_su, su.data(), L * sizeof(void*), cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(d_sd, sd.data(), L * sizeof(void*), cudaMemcpyHostToDevice, m->stream));

  // RoPE tables [max_ctx][hd/2]: inv_freq_i = theta^(-2i/hd), angle = p * inv_freq_i (double),
  // cos and sin rounded to fp32 (the reading the step's arithmetic contract fixes).
  const int half = hd / 2;
  std::vector<float> cs((size_t)c.max_ctx * half), sn((size_t)c.max_ctx * half);
  for (int i = 0; i < half; ++i) {
    const double ex = (double)(2 * i) / (double)hd;
    const double inv = std::pow((double)c.rope_theta, -ex);
    for (int p = 0; p < c.max_ctx; ++p) {
      const double ang = (double)p * inv;
      cs[(size_t)p * half + i] = (float)std::cos(ang);
      sn[(size_t)p * half + i] = (float)std::sin(ang);
    }
  }
  float *d_cos, *d_sin;
  if ((rc = m->alloc(&d_cos, cs.size())) || (rc = m->alloc(&d_sin, sn.size()))) return rc;
  CK(cudaMemcpyAsync(d_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(d_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice, m->stream));

  // scratch
  Params& p = m->p;
  const int nbmax = (c.max_ctx + kAttnBlock - 1) / kAttnBlock;
  const int nblk = (c.vocab + kVocabBlock - 1) / kVocabBlock;
  const int topk = std::max(c.top_k, 1);
  if ((rc = m->alloc(&p.x, d)) || (rc = m->alloc(&p.q, hq * hd)) || (rc = m->alloc(&p.attn, hq * hd)) ||
      (rc = m->alloc(&p.h, ffw)) || (rc = m->alloc(&p.rlog, std::max(c.n_experts, 1))) ||
      (rc = m->alloc(&p.knew, hkv * hd)) || (rc = m->alloc(&p.vnew, hkv * hd)) || (rc = m->alloc(&p.epoch, 1)) ||
      (rc = m->alloc(&p.tok_word, 1)) ||
      (rc = m->alloc(&p.part_m, (size_t)hq * nbmax)) || (rc = m->alloc(&p.part_l, (size_t)hq * nbmax)) ||
      (rc = m->alloc(&p.part_o, (size_t)hq * nbmax * hd)) ||
      (rc = m->alloc(&p.sblock, nblk)) || (rc = m->alloc(&p.sample_ctr, 1)) || (rc = m->alloc(&p.argkey, 1)) ||
      (rc = m->alloc(&p.lm_ctr, 1)) || (rc = m->alloc(&p.bar_ctr, 1)) || (rc = m->alloc(&p.err, 1)) ||
      (rc = m->alloc(&p.sel_out, (size_t)L * topk)) || (rc = m->alloc(&p.state, 1)) ||
      (rc = m->alloc(&m->d_force, (size_t)L * topk)) || (rc = m->alloc(&m->d_logits_scratch, c.vocab)))
    return rc;
  m->ll_bytes[0] = (size_t)d * 8;
  m->ll_bytes[1] = (size_t)hq * hd * 8;
  m->ll_bytes[2] = (size_t)hq * hd * 8;
  m->ll_bytes[3] = (size_t)ffw * 8;
  m->ll_bytes[4] = (size_t)std::max(c.n_experts, 1) * 8;
  m->ll_bytes[5] = (size_t)hkv * hd * 8;
  m->ll_bytes[6] = (size_t)hkv * hd * 8;
  m->ll_bytes[7] = (size_t)hq * nbmax * 8;
  m->ll_bytes[8] = (size_t)hq * nbmax * 8;
  m->ll_bytes[9] = (size_t)hq * nbmax * hd * 8;
  m->ll_bytes[10] = 8;
  if ((rc = clear_exchange(m))) return rc;
  CK(cudaMemsetAsync(p.sample_ctr, 0, 4, m->stream));
  CK(cudaMemsetAsync(p.argkey, 0, 8, m->stream));
  CK(cudaMemsetAsync(p.lm_ctr, 0, 4, m->stream));
  CK(cudaMemsetAsync(p.bar_ctr, 0, 8, m->stream));
  CK(cudaMemsetAsync(p.err, 0, 4, m->stream));
  CK(cudaMemsetAsync(p.sel_out, 0, (size_t)L * topk * 4, m->stream));
  CK(cudaMemsetAsync(p.state, 0, sizeof(StepState), m->stream));
  CK(cudaMallocHost(&m->h_state, sizeof(StepState)));
  CK(cudaEventCreateWithFlags(&m->state_copied, cudaEventDisableTiming));
  CK(cudaEventRecord(m->state_copied, m->stream));
  CK(cudaMallocHost(&m->h_out, 2 * sizeof(int32_t)));

  p.image = m->image;
  p.tok_emb = w->tok_emb;
  p.attn_norm = d_an;
  p.ffn_norm = d_fn;
  p.final_norm = w->final_norm;
  p.e_gate_scale = d_sg;
  p.e_up_scale = d_su;
  p.e_down_scale = d_sd;
  p.phases = m->d_phases;
  p.n_phases = (int)m->phases.size();
  p.L = L; p.d = d; p.hq = hq; p.hkv = hkv; p.hd = hd; p.ff = c.d_ff; p.V = c.vocab; p.max_ctx = c.max_ctx;
  p.E = c.n_experts; p.topk = c.n_experts ? c.top_k : 0; p.fexp = c.d_expert;
  p.wdt = c.weight_dtype; p.kvdt = c.kv_dtype; p.rdt = c.router_dtype;
  p.edt = head_dtype(c);
  p.eps = c.rms_eps;
  p.attn_scale = (float)(1.0 / std::sqrt((double)hd));
  p.nbmax = nbmax;
  // on long contexts each query head is merged by up to four CTAs (head_dim slices), as many as
  // the grid has CTAs for; the merge time grows with the block count, the split's fixed cost does
  // not (measured break-even near 50 blocks on the 2.3B model)
  p.merge_split = hq * 4 <= m->G && hd % 4 == 0 ? 4 : hq * 2 <= m->G && hd % 2 == 0 ? 2 : 1;
  p.merge_split_blocks = 64;
  p.rope_cos = d_cos;
  p.rope_sin = d_sin;
  p.wait_ns = 200000000ull;
  p.l2_lookahead = 0;
  p.pf_flags = 0;
  p.l2_rate = 0;
  p.l2_burst = 0;
  p.n_steps = 1;
  p.skip_cta = -1;
  p.skip_phase = -1;
  CK(cudaStreamSynchronize(m->stream));
  CK(cudaGetLastError());
  return ADP_OK;
}

extern "C" int adp_create_model(const adp_config* cfg, const adp_weights* w, void* stream, adp_model** out) {
  if (!out) return ADP_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate(cfg, w);
  if (rc) return rc;
  adp_model* m = new adp_model();
  m->cfg = *cfg;
  m->stream = (cudaStream_t)stream;
  rc = create(m, cfg, w);
  if (rc) {
    adp_destroy_model(m);
    return rc;
  }
  *out = m;
  return ADP_OK;
}

extern "C" void adp_destroy_model(adp_model* m) {
  if (!m) return;
  if (m->stream) cudaStreamSynchronize(m->stream);
  else cudaDeviceSynchronize();
  if (m->graph) cudaGraphExecDestroy(m->graph);
  if (m->state_copied) cudaEventDestroy(m->state_copied);
  for (void* q : m->allocs) cudaFree(q);
  if (m->h_state) cudaFreeHost(m->h_state);
  if (m->h_out) cudaFreeHost(m->h_out);
  if (m->bt.copied) cudaEventDestroy(m->bt.copied);
  if (m->bt.h) cudaFreeHost(m->bt.h);
  if (m->bt.h_out) cudaFreeHost(m->bt.h_out);
  for (adp_kv* kv : m->kvs) kv->m = nullptr;  // still valid for adp_kv_destroy, for nothing else
  delete m;
}

// ---------------------------------------------------------------- KV caches

extern "C" int adp_kv_create(adp_model* m, adp_kv** out) {
  if (!m || !out) return ADP_ERR_INVALID_ARG;
  *out = nullptr;
  const adp_config& c = m->cfg;
  adp_kv* kv = new adp_kv();
  kv->m = m;
  kv->bytes = (size_t)c.n_layers * c.n_kv_heads * c.max_ctx * c.head_dim * 2;
  cudaError_t e = cudaMalloc(&kv->k, kv->bytes);
  if (e == cudaSuccess) e = cudaMalloc(&kv->v, kv->bytes);
  if (e == cudaSuccess) e = cudaMemsetAsync(kv->k, 0, kv->bytes, m->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(kv->v, 0, kv->bytes, m->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
  if (e != cudaSuccess) {
    adp_kv_destroy(kv);
    return cuda_fail(e, "adp_kv_create");
  }
  m->kvs.push_back(kv);
  *out = kv;
  return ADP_OK;
}

extern "C" void adp_kv_destroy(adp_kv* kv) {
  if (!kv) return;
  if (kv->m) {
    if (kv->m->stream) cudaStreamSynchronize(kv->m->stream);
    auto& v = kv->m->kvs;
    v.erase(std::remove(v.begin(), v.end(), kv), v.end());
  }
  if (kv->k) cudaFree(kv->k);
  if (kv->v) cudaFree(kv->v);
  delete kv;
}

extern "C" int adp_kv_reset(adp_kv* kv) {
  if (!kv || !kv->m) return ADP_ERR_INVALID_ARG;
  kv->len = 0;
  return ADP_OK;
}

extern "C" int adp_kv_truncate(adp_kv* kv, int32_t len) {
  if (!kv || !kv->m || len < 0 || len > kv->len) return ADP_ERR_INVALID_ARG;
  kv->len = len;
  return ADP_OK;
}

extern "C" int adp_kv_len(const adp_kv* kv, int32_t* len) {
  if (!kv || !len) return ADP_ERR_INVALID_ARG;
  *len = kv->len;
  return ADP_OK;
}

static int kv_copy(const adp_kv* kv, void* host_k, void* host_v, int32_t len, bool load) {
  const adp_config& c = kv->m->cfg;
  const size_t row = (size_t)c.head_dim * 2;
  for (int l = 0; l < c.n_layers; ++l)
    for (int g = 0; g < c.n_kv_heads; ++g) {
      const size_t dev_off = (((size_t)l * c.n_kv_heads + g) * c.max_ctx) * row;
      const size_t host_off = (((size_t)l * c.n_kv_heads + g) * (size_t)len) * row;
      if (load) {
        CK(cudaMemcpyAsync((uint8_t*)kv->k + dev_off, (const uint8_t*)host_k + host_off, len * row,
                           cudaMemcpyHostToDevice, kv->m->stream));
        CK(cudaMemcpyAsync((uint8_t*)kv->v + dev_off, (const uint8_t*)host_v + host_off, len * row,
                           cudaMemcpyHostToDevice, kv->m->stream));
      } else {
        CK(cudaMemcpyAsync((uint8_t*)host_k + host_off, (const uint8_t*)kv->k + dev_off, len * row,
                           cudaMemcpyDeviceToHost, kv->m->stream));
        CK(cudaMemcpyAsync((uint8_t*)host_v + host_off, (const uint8_t*)kv->v + dev_off, len * row,
                           cudaMemcpyDeviceToHost, kv->m->stream));
      }
    }
  CK(cudaStreamSynchronize(kv->m->stream));
  return ADP_OK;
}

extern "C" int adp_kv_load(adp_kv* kv, const void* host_k, const void* host_v, int32_t len) {
  if (!kv || !kv->m || len < 0 || (len > 0 && (!host_k || !host_v))) return ADP_ERR_INVALID_ARG;
  if (len > kv->m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  int rc = kv_copy(kv, const_cast<void*>(host_k), const_cast<void*>(host_v), len, true);
  if (rc == ADP_OK) kv->len = len;
  return rc;
}

extern "C" int adp_kv_read(const adp_kv* kv, void* host_k, void* host_v, int32_t len) {
  if (!kv || !kv->m || len < 0 || (len > 0 && (!host_k || !host_v))) return ADP_ERR_INVALID_ARG;
  if (len > kv->m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  return kv_copy(kv, host_k, host_v, len, false);
}

// ---------------------------------------------------------------- decode

// Copy the step state to the device; the pinned staging buffer is reused only after the
// previous copy out of it has executed.
static int put_state(adp_model* m, int32_t pos, int32_t token, float T, float u) {
  CK(cudaEventSynchronize(m->state_copied));
  m->h_state->pos = pos;
  m->h_state->token = token;
  m->h_state->temperature = T;
  m->h_state->u = u;
  m->h_state->seq_index = 0;
  m->h_state->out_token = -1;
  CK(cudaMemcpyAsync(m->p.state, m->h_state, sizeof(StepState), cudaMemcpyHostToDevice, m->stream));
  CK(cudaEventRecord(m->state_copied, m->stream));
  return ADP_OK;
}

static int map_device_error(int32_t e) {
  if (e == DE_BARRIER_TIMEOUT) return ADP_ERR_BARRIER_TIMEOUT;
  if (e == DE_PIPELINE_TIMEOUT) return ADP_ERR_PIPELINE_TIMEOUT;
  return e ? ADP_ERR_CUDA : ADP_OK;
}

static Params step_params(adp_model* m, adp_kv* kv, float* logits, const int32_t* tok_seq, const float* u_seq,
                          int32_t* out_seq) {
  Params p = m->p;
  p.kc = kv->k;
  p.vc = kv->v;
  p.logits = logits ? logits : m->d_logits_scratch;
  p.tok_seq = tok_seq;
  p.u_seq = u_seq;
  p.out_seq = out_seq;
  p.force_sel = m->force_on ? m->d_force : nullptr;
  return p;
}

static int enqueue_step(adp_model* m, const Params& p, bool sampling);

// Enqueue n decode steps: in the persistent mode one launch that runs them back to back (each
// step takes the token the previous one chose, or the next of p.tok_seq); in the ablation modes
// the launches of one step, n times.
static int enqueue_steps(adp_model* m, const Params& p, bool sampling, int n) {
  const int rs = reserve_epochs(m, n);
  if (rs) return rs;
  if (m->mode == 0) {
    Params q = p;
    q.n_steps = n;
    return enqueue_step(m, q, sampling);
  }
  for (int i = 0; i < n; ++i) {
    const int rc = enqueue_step(m, p, sampling);
    if (rc) return rc;
  }
  return ADP_OK;
}

// Enqueue the launches of one decode step in the model's kernel mode.
static int enqueue_step(adp_model* m, const Params& p, bool sampling) {
  const int nph = (int)m->phases.size();
  const int last = sampling ? nph : nph - 1;  // the sampling phase runs only at temperature > 0
  if (m->mode == 0) {
    CK(decode_launch(p, 0, last, true, m->G, m->smem, m->xbuf_floats, m->stream));
    return ADP_OK;
  }
  if (m->mode == 2) {
    const bool hit = m->graph && m->graph_key_kv == (const void*)p.kc && m->graph_key_logits == (const void*)p.logits &&
                     m->graph_key_sample == sampling && !p.tok_seq && !p.u_seq && !p.out_seq;
    if (!hit && !p.tok_seq && !p.u_seq && !p.out_seq) {
      if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
      cudaStream_t cap;
      CK(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking));
      cudaGraph_t g;
      CK(cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal));
      for (int ph = 0; ph < last; ++ph) {
        cudaError_t e = decode_launch(p, ph, ph + 1, false, m->G, m->smem, m->xbuf_floats, cap);
        if (e != cudaSuccess) { cudaStreamEndCapture(cap, &g); cudaStreamDestroy(cap); return cuda_fail(e, "capture"); }
      }
      CK(cudaStreamEndCapture(cap, &g));
      CK(cudaGraphInstantiate(&m->graph, g, 0));
      cudaGraphDestroy(g);
      cudaStreamDestroy(cap);
      m->graph_key_kv = p.kc;
      m->graph_key_logits = p.logits;
      m->graph_key_sample = sampling;
    }
    if (m->graph && !p.tok_seq && !p.u_seq && !p.out_seq) {
      CK(cudaGraphLaunch(m->graph, m->stream));
      return ADP_OK;
    }
  }
  for (int ph = 0; ph < last; ++ph) CK(decode_launch(p, ph, ph + 1, false, m->G, m->smem, m->xbuf_floats, m->stream));
  return ADP_OK;
}

static int finish(adp_model* m) {
  CK(cudaMemcpyAsync(&m->h_out[0], &m->p.state->out_token, 4, cudaMemcpyDeviceToHost, m->stream));
  CK(cudaMemcpyAsync(&m->h_out[1], m->p.err, 4, cudaMemcpyDeviceToHost, m->stream));
  CK(cudaStreamSynchronize(m->stream));
  const int rc = map_device_error(m->h_out[1]);
  if (rc) m->sticky = rc;
  return rc;
}

extern "C" int adp_decode_step(adp_model* m, adp_kv* kv, int32_t token, const adp_sampling* sampling,
                               int32_t* next_token, float* dev_logits) {
  if (!m || !kv || !next_token || kv->m != m) return ADP_ERR_INVALID_ARG;
  if (m->sticky) return m->sticky;
  if (token < 0 || token >= m->cfg.vocab) return ADP_ERR_INVALID_ARG;
  if (kv->len >= m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  const float T = sampling ? sampling->temperature : 0.0f;
  int rs = put_state(m, kv->len, token, T, sampling ? sampling->u : 0.0f);
  if (rs) return rs;
  Params p = step_params(m, kv, dev_logits, nullptr, nullptr, nullptr);
  int rc = enqueue_steps(m, p, T > 0.0f, 1);
  m->p.skip_cta = m->p.skip_phase = -1;
  if (rc) return rc;
  rc = finish(m);
  if (rc) return rc;
  *next_token = m->h_out[0];
  kv->len += 1;
  return ADP_OK;
}

extern "C" int adp_prefill(adp_model* m, adp_kv* kv, const int32_t* host_tokens, int32_t n,
                           const adp_sampling* sampling, int32_t* next_token, float* dev_logits) {
  if (!m || !kv || !next_token || kv->m != m || n < 1 || !host_tokens) return ADP_ERR_INVALID_ARG;
  if (m->sticky) return m->sticky;
  if (kv->len + n > m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  for (int i = 0; i < n; ++i)
    if (host_tokens[i] < 0 || host_tokens[i] >= m->cfg.vocab) return ADP_ERR_INVALID_ARG;
  if (n > m->tokseq_cap) {
    int32_t* q = nullptr;
    int rc = m->alloc(&q, (size_t)n);
    if (rc) return rc;
    m->d_tokseq = q;
    m->tokseq_cap = n;
  }
  CK(cudaMemcpyAsync(m->d_tokseq, host_tokens, (size_t)n * 4, cudaMemcpyHostToDevice, m->stream));
  const float T = sampling ? sampling->temperature : 0.0f;
  int rs = put_state(m, kv->len, 0, T, sampling ? sampling->u : 0.0f);
  if (rs) return rs;
  {
    // every step writes its logits to the same place: the last step's remain
    Params p = step_params(m, kv, dev_logits, m->d_tokseq, nullptr, nullptr);
    int rc = enqueue_steps(m, p, T > 0.0f, n);
    if (rc) return rc;
  }
  m->p.skip_cta = m->p.skip_phase = -1;
  int rc = finish(m);
  if (rc) return rc;
  *next_token = m->h_out[0];
  kv->len += n;
  return ADP_OK;
}

extern "C" int adp_generate_async(adp_model* m, adp_kv* kv, int32_t token, int32_t n, float temperature,
                                  const float* dev_u, int32_t* dev_tokens_out) {
  if (!m || !kv || kv->m != m || n < 0 || !dev_tokens_out) return ADP_ERR_INVALID_ARG;
  if (m->sticky) return m->sticky;
  if (token < 0 || token >= m->cfg.vocab) return ADP_ERR_INVALID_ARG;
  if (temperature > 0.0f && !dev_u) return ADP_ERR_INVALID_ARG;
  if (kv->len + n > m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  if (n == 0) return ADP_OK;
  int rs = put_state(m, kv->len, token, temperature, 0.0f);
  if (rs) return rs;
  Params p = step_params(m, kv, nullptr, nullptr, temperature > 0.0f ? dev_u : nullptr, dev_tokens_out);
  int rc = enqueue_steps(m, p, temperature > 0.0f, n);
  if (rc) return rc;
  kv->len += n;
  return ADP_OK;
}

// ---------------------------------------------------------------- small-batch decode

// The batched kernel's shared-memory layout of one batch size (nslots 0: the size does not fit).
struct BatchLayout {
  size_t smem = 0, ctl = 0;
  int nslots = 0, att_slots = 0, xbuf_floats = 0, down_seg = 0;
};

// The layout of every batch size 1..kMaxBatch on a GPU of G SMs with `optin` bytes of shared memory
// per block (host only): nb input vectors of the widest GEMV input beside a ring of at least two
// slots; when nb whole down-projection inputs do not fit, they are staged in segments of whole
// K-chunks (the fewest that fit).  Returns the largest batch that fits (0: none; MoE models, whose
// experts differ per request, are not batched).
static int plan_batches(const adp_config& c, const std::vector<PhaseDesc>& phases, int G, size_t optin,
                        BatchLayout (&out)[kMaxBatch + 1]) {
  for (auto& o : out) o = BatchLayout{};
  if (c.n_experts != 0) return 0;
  const int d = c.d_model, hq = c.n_heads, hd = c.head_dim;
  const int nph = (int)phases.size();
  const size_t ctl_sz = (ctl_bytes(nph) + 16 + batch_ctl_bytes() + 127) & ~(size_t)127;
  const int nbmax = (c.max_ctx + kAttnBlock - 1) / kAttnBlock;
  const size_t item = (size_t)kAttnBlock * (hd + 8) * 2 + (size_t)kAttnBlock * hd * 2 + (size_t)kMaxGroup * hd * 4 +
                      (size_t)kMaxGroup * kAttnBlock * 4;
  auto pad256 = [](int n) { return (size_t)((n + 255) / 256 * 256); };
  const size_t merge_bytes = ((size_t)2 * 8 * nbmax + 8) * 4;
  const int gmax = kv_group_max(c);
  // the down projection's K-chunk: a staged segment of its input is a whole number of chunks
  int down_kc = c.d_ff;
  for (const PhaseDesc& P : phases)
    if (P.kind == PK_DOWN) {
      down_kc = P.KC;
      break;
    }
  const int down_chunks = (c.d_ff + down_kc - 1) / down_kc;
  int max_nb = 0;
  for (int nb = 1; nb <= kMaxBatch; ++nb) {
    if (nb * hq > G) break;  // CTA G-1-(r*hq+h) merges head h of request r
    // the fewest segments of the down input that leave a ring of at least 2 slots: a refetch in the
    // middle of the down GEMV cost more than a deeper ring saved (2.3B, 2 requests: 1,106 tok/s whole
    // against 915 in two segments with 4 slots), so segments only make a batch possible at all
    int ns = 0, att = 0, seg = 0;
    size_t xbytes = 0;
    for (int S = 1; S <= down_chunks; ++S) {
      const int sg = S == 1 ? c.d_ff : ((down_chunks + S - 1) / S) * down_kc;
      if (S > 1 && sg >= c.d_ff) continue;
      const size_t vec_floats = std::max({pad256(d), pad256(hq * hd), pad256(std::min(sg, c.d_ff))});
      const size_t vec_bytes = std::max((size_t)nb * vec_floats * 4, merge_bytes);
      int ks = 0, ka = 0;
      size_t kx = 0;
      for (int k = kMaxSlots; k >= 2 && !ks; --k) {
        if ((size_t)k * kSlotBytes + ctl_sz > optin) continue;
        const size_t room = optin - (size_t)k * kSlotBytes - ctl_sz;
        if (room < vec_bytes || room < item) continue;
        ks = k;
        ka = (int)std::min<size_t>(std::min(kAttnSlots, kConsumerWarps / gmax), room / item);
        kx = std::max(vec_bytes, (size_t)ka * item);
      }
      if (ks) {
        ns = ks;
        att = ka;
        xbytes = kx;
        seg = std::min(sg, c.d_ff);
        break;
      }
    }
    if (!ns) break;
    xbytes = (xbytes + 127) & ~(size_t)127;
    BatchLayout& o = out[nb];
    o.nslots = ns;
    o.att_slots = att;
    o.xbuf_floats = (int)(xbytes / 4);
    o.down_seg = seg;
    o.ctl = ctl_sz;
    o.smem = (size_t)ns * kSlotBytes + xbytes + ctl_sz;
    max_nb = nb;
  }
  return max_nb;
}

// Set up batched decode once per model: the shared-memory layout of every batch size that fits
// (plan_batches), the per-request exchange buffers and the step-state staging.  Dense models only.
static int batch_init(adp_model* m) {
  adp_model::Batch& B = m->bt;
  if (B.init_rc != 1) return B.init_rc;
  const adp_config& c = m->cfg;
  B.init_rc = ADP_ERR_UNSUPPORTED_CONFIG;
  if (c.n_experts != 0) return B.init_rc;  // experts differ per request
  const int d = c.d_model, hq = c.n_heads, hkv = c.n_kv_heads, hd = c.head_dim;
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, m->device));
  const int nbmax = (c.max_ctx + kAttnBlock - 1) / kAttnBlock;
  BatchLayout lay[kMaxBatch + 1];
  B.max_nb = plan_batches(c, m->phases, m->G, (size_t)prop.sharedMemPerBlockOptin, lay);
  size_t smem_max = 0;
  for (int nb = 1; nb <= B.max_nb; ++nb) {
    B.nslots[nb] = lay[nb].nslots;
    B.att_slots[nb] = lay[nb].att_slots;
    B.xbuf_floats[nb] = lay[nb].xbuf_floats;
    B.down_seg[nb] = lay[nb].down_seg;
    B.smem[nb] = lay[nb].smem;
    smem_max = std::max(smem_max, B.smem[nb]);
  }
  if (B.max_nb == 0) return B.init_rc;
  int bps = 0;
  CK(decode_batch_prepare(smem_max, &bps));
  if (bps < 1) return B.init_rc = ADP_ERR_NOT_CORESIDENT;
  // per-request copies of the exchange buffers, for kMaxBatch requests
  Params& p = B.p;
  p = m->p;
  const size_t R = kMaxBatch;
  const int nblk = (c.vocab + kVocabBlock - 1) / kVocabBlock;
  int rc;
  if ((rc = m->alloc(&p.x, R * d)) || (rc = m->alloc(&p.q, R * hq * hd)) || (rc = m->alloc(&p.attn, R * hq * hd)) ||
      (rc = m->alloc(&p.h, R * c.d_ff)) || (rc = m->alloc(&p.knew, R * hkv * hd)) ||
      (rc = m->alloc(&p.vnew, R * hkv * hd)) || (rc = m->alloc(&p.tok_word, R)) ||
      (rc = m->alloc(&p.part_m, R * hq * nbmax)) || (rc = m->alloc(&p.part_l, R * hq * nbmax)) ||
      (rc = m->alloc(&p.part_o, R * hq * nbmax * hd)) || (rc = m->alloc(&p.sblock, R * nblk)) ||
      (rc = m->alloc(&p.sample_ctr, R)) || (rc = m->alloc(&p.argkey, R)) || (rc = m->alloc(&B.d, 1)) ||
      (rc = m->alloc(&B.d_logits, R * c.vocab)))
    return B.init_rc = rc;
  p.rlog = nullptr;
  const size_t sizes[11] = {R * d * 8, R * hq * hd * 8, R * hq * hd * 8, R * c.d_ff * 8, 0, R * hkv * hd * 8,
                            R * hkv * hd * 8, R * hq * nbmax * 8, R * hq * nbmax * 8, R * hq * nbmax * hd * 8, R * 8};
  for (int i = 0; i < 11; ++i) B.ll_bytes[i] = sizes[i];
  void* bb[11] = {p.x, p.q, p.attn, p.h, nullptr, p.knew, p.vnew, p.part_m, p.part_l, p.part_o, p.tok_word};
  for (int i = 0; i < 11; ++i)
    if (bb[i]) CK(cudaMemsetAsync(bb[i], 0, sizes[i], m->stream));
  CK(cudaMemsetAsync(p.sample_ctr, 0, 4 * R, m->stream));
  CK(cudaMemsetAsync(p.argkey, 0, 8 * R, m->stream));
  CK(cudaMemsetAsync(B.d, 0, sizeof(adp_model::BatchHost), m->stream));
  CK(cudaMallocHost(&B.h, sizeof(adp_model::BatchHost)));
  std::memset(B.h, 0, sizeof(adp_model::BatchHost));
  CK(cudaMallocHost(&B.h_out, (kMaxBatch + 1) * sizeof(int32_t)));
  CK(cudaEventCreateWithFlags(&B.copied, cudaEventDisableTiming));
  CK(cudaEventRecord(B.copied, m->stream));
  uint8_t* dbase = reinterpret_cast<uint8_t*>(B.d);  // device addresses of the staged fields
  p.state = reinterpret_cast<StepState*>(dbase + offsetof(adp_model::BatchHost, st));
  p.kcb = reinterpret_cast<uint16_t* const*>(dbase + offsetof(adp_model::BatchHost, kcb));
  p.vcb = reinterpret_cast<uint16_t* const*>(dbase + offsetof(adp_model::BatchHost, vcb));
  p.force_sel = nullptr;
  p.trace = nullptr;
  CK(cudaStreamSynchronize(m->stream));
  return B.init_rc = ADP_OK;
}

// Checks shared by the batched entry points; on success the batch is set up.
static int batch_check(adp_model* m, adp_kv* const* kvs, int32_t nb, const int32_t* tokens, int32_t n_steps) {
  if (!m || !kvs || !tokens || nb < 1 || n_steps < 0) return ADP_ERR_INVALID_ARG;
  if (m->sticky) return m->sticky;
  for (int r = 0; r < nb; ++r) {
    if (!kvs[r] || kvs[r]->m != m) return ADP_ERR_INVALID_ARG;
    for (int s = 0; s < r; ++s)
      if (kvs[s] == kvs[r]) return ADP_ERR_INVALID_ARG;  // one cache cannot take two tokens per step
    if (tokens[r] < 0 || tokens[r] >= m->cfg.vocab) return ADP_ERR_INVALID_ARG;
  }
  const int rc = batch_init(m);
  if (rc) return rc;
  if (nb > m->bt.max_nb) return ADP_ERR_UNSUPPORTED_CONFIG;
  for (int r = 0; r < nb; ++r)
    if (kvs[r]->len + std::max(n_steps, 1) > m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  return ADP_OK;
}

// Stage the step state and KV cache tables of the batch and enqueue n steps in one launch.
static int batch_enqueue(adp_model* m, adp_kv* const* kvs, int32_t nb, const int32_t* tokens, const float* temps,
                         const float* us, int32_t n, const float* dev_u, int32_t* dev_out, float* dev_logits) {
  adp_model::Batch& B = m->bt;
  CK(cudaEventSynchronize(B.copied));
  bool sampling = false;
  for (int r = 0; r < nb; ++r) {
    StepState& st = B.h->st[r];
    st.pos = kvs[r]->len;
    st.token = tokens[r];
    st.temperature = temps ? temps[r] : 0.0f;
    st.u = us ? us[r] : 0.0f;
    st.seq_index = 0;
    st.out_token = -1;
    B.h->kcb[r] = kvs[r]->k;
    B.h->vcb[r] = kvs[r]->v;
    sampling = sampling || st.temperature > 0.0f;
  }
  CK(cudaMemcpyAsync(B.d, B.h, sizeof(adp_model::BatchHost), cudaMemcpyHostToDevice, m->stream));
  CK(cudaEventRecord(B.copied, m->stream));
  const int rs = reserve_epochs(m, n);
  if (rs) return rs;
  Params q = B.p;
  q.nb = nb;
  q.n_steps = n;
  q.nslots = B.nslots[nb];
  q.att_slots = B.att_slots[nb];
  q.xbuf_floats = B.xbuf_floats[nb];
  q.logits = dev_logits ? dev_logits : B.d_logits;
  q.tok_seq = nullptr;
  q.u_seq = dev_u;
  q.out_seq = dev_out;
  q.timeline = m->p.timeline;
  q.wait_ns = m->p.wait_ns;
  q.debug_barriers = m->p.debug_barriers;
  q.skip_cta = q.skip_phase = -1;
  const int nph = (int)m->phases.size();
  CK(decode_batch_launch(q, 0, sampling ? nph : nph - 1, m->G, B.smem[nb], B.xbuf_floats[nb], B.down_seg[nb],
                         m->stream));
  return ADP_OK;
}

extern "C" int adp_debug_tc_gemm(int32_t bf16, int32_t M, int32_t N, int32_t K, const void* A, const void* W,
                                 float* C) {
  if (M < 1 || N < 1 || K < 1 || !A || !W || !C || (bf16 != 0 && bf16 != 1)) return ADP_ERR_INVALID_ARG;
  uint8_t *at = nullptr, *wt = nullptr;
  int32_t* err = nullptr;
  int32_t herr = 0;
  cudaError_t e = cudaMalloc(&at, tc_tiled_bytes(M, K, 256));  // rows padded to the GEMM's 256-row blocks
  if (e == cudaSuccess) e = cudaMalloc(&wt, tc_tiled_bytes(N, K, 256));
  if (e == cudaSuccess) e = cudaMalloc(&err, 4);
  if (e == cudaSuccess) e = cudaMemset(err, 0, 4);
  if (e == cudaSuccess) e = tc_tile((const uint16_t*)A, M, K, K, at, 128, 0);
  if (e == cudaSuccess) e = tc_tile((const uint16_t*)W, N, K, K, wt, 256, 0);
  if (e == cudaSuccess) e = tc_gemm(bf16, TC_STORE, at, wt, C, N, M, N, K, err, 1000000000ull, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  cudaFree(at);
  cudaFree(wt);
  cudaFree(err);
  if (e != cudaSuccess) return cuda_fail(e, "adp_debug_tc_gemm");
  return herr ? ADP_ERR_PIPELINE_TIMEOUT : ADP_OK;
}

extern "C" int adp_max_batch(adp_model* m, int32_t* nb) {
  if (!m || !nb) return ADP_ERR_INVALID_ARG;
  const int rc = batch_init(m);
  *nb = rc == ADP_OK ? m->bt.max_nb : 0;
  return rc == ADP_ERR_UNSUPPORTED_CONFIG ? ADP_OK : rc;
}

extern "C" int adp_decode_batch(adp_model* m, adp_kv* const* kvs, int32_t nb, const int32_t* tokens,
                                const adp_sampling* sampling, int32_t* next_tokens, float* dev_logits) {
  if (!next_tokens) return ADP_ERR_INVALID_ARG;
  int rc = batch_check(m, kvs, nb, tokens, 1);
  if (rc) return rc;
  float temps[kMaxBatch], us[kMaxBatch];
  for (int r = 0; r < nb; ++r) {
    temps[r] = sampling ? sampling[r].temperature : 0.0f;
    us[r] = sampling ? sampling[r].u : 0.0f;
  }
  rc = batch_enqueue(m, kvs, nb, tokens, temps, us, 1, nullptr, nullptr, dev_logits);
  if (rc) return rc;
  adp_model::Batch& B = m->bt;
  for (int r = 0; r < nb; ++r)
    CK(cudaMemcpyAsync(&B.h_out[r], &B.p.state[r].out_token, 4, cudaMemcpyDeviceToHost, m->stream));
  CK(cudaMemcpyAsync(&B.h_out[kMaxBatch], m->p.err, 4, cudaMemcpyDeviceToHost, m->stream));
  CK(cudaStreamSynchronize(m->stream));
  rc = map_device_error(B.h_out[kMaxBatch]);
  if (rc) {
    m->sticky = rc;
    return rc;
  }
  for (int r = 0; r < nb; ++r) {
    next_tokens[r] = B.h_out[r];
    kvs[r]->len += 1;
  }
  return ADP_OK;
}

extern "C" int adp_generate_batch_async(adp_model* m, adp_kv* const* kvs, int32_t nb, const int32_t* tokens,
                                        int32_t n, const float* temperatures, const float* dev_u,
                                        int32_t* dev_tokens_out) {
  if (!dev_tokens_out) return ADP_ERR_INVALID_ARG;
  int rc = batch_check(m, kvs, nb, tokens, n);
  if (rc) return rc;
  bool sampling = false;
  for (int r = 0; r < nb && temperatures; ++r) sampling = sampling || temperatures[r] > 0.0f;
  if (sampling && !dev_u) return ADP_ERR_INVALID_ARG;
  for (int r = 0; r < nb; ++r)
    if (kvs[r]->len + n > m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  if (n == 0) return ADP_OK;
  rc = batch_enqueue(m, kvs, nb, tokens, temperatures, nullptr, n, sampling ? dev_u : nullptr, dev_tokens_out,
                     nullptr);
  if (rc) return rc;
  for (int r = 0; r < nb; ++r) kvs[r]->len += n;
  return ADP_OK;
}

// ---------------------------------------------------------------- tensor-core prefill

// The 16-bit type of the tensor-core prefill's GEMM operands: the weights' own, or for e4m3
// layer matrices the embedding's (the matrices are dequantised into it).
static int tc_operand_bf16(const adp_config& c) {
  return head_dtype(c) == ADP_BF16 ? 1 : 0;
}

// Set up the tensor-core prefill once per model: every layer matrix again as GEMM operand tiles
// (rebuilt from the decode image), for dense models (16-bit, e4m3 or NVFP4 layer matrices) with head_dim
// 64 or 128.
static int tc_init(adp_model* m) {
  adp_model::TcState& T = m->tc;
  if (T.init_rc != 1) return T.init_rc;
  const adp_config& c = m->cfg;
  T.init_rc = ADP_ERR_UNSUPPORTED_CONFIG;
  if (c.n_experts != 0) return T.init_rc;
  if (c.head_dim != 64 && c.head_dim != 128) return T.init_rc;
  const int d = c.d_model, hq = c.n_heads, hkv = c.n_kv_heads, hd = c.head_dim;
  for (const PhaseDesc& P : m->phases) {
    int rows = 0;
    std::vector<const uint8_t*>* dst = nullptr;
    std::vector<const float*>* sdst = nullptr;
    const float* sc3[3] = {nullptr, nullptr, nullptr};  // row scales of e4m3 / NVFP4 matrices
    auto scale = [&](int i) { return m->h_wscale[i].empty() ? nullptr : m->h_wscale[i][P.layer]; };
    switch (P.kind) {
      case PK_QKV:
        rows = (hq + 2 * hkv) * hd;
        dst = &T.wqkv;
        sdst = &T.sqkv;
        sc3[0] = scale(0);
        sc3[1] = scale(1);
        sc3[2] = scale(2);
        break;
      case PK_WO: rows = d; dst = &T.wo; sdst = &T.swo; sc3[0] = scale(3); break;
      case PK_GU: rows = 2 * c.d_ff; dst = &T.wgu; sdst = &T.sgu; sc3[0] = scale(4); sc3[1] = scale(5); break;
      case PK_DOWN: rows = d; dst = &T.wdown; sdst = &T.sdown; sc3[0] = scale(6); break;
      default: continue;
    }
    uint8_t* buf = nullptr;
    const size_t bytes = tc_tiled_bytes(rows, P.K, 256);
    int rc = m->alloc(&buf, bytes);
    if (rc) return T.init_rc = rc;
    CK(cudaMemsetAsync(buf, 0, bytes, m->stream));
    CK(tc_unpack(m->image, P, m->G, hd, hq, hkv, c.d_ff, buf, tc_operand_bf16(c), m->stream));
    dst->push_back(buf);
    if (sc3[0]) {  // quantised: the row scales become the GEMM's column scales
      float* cs = nullptr;
      if ((rc = m->alloc(&cs, (size_t)rows))) return T.init_rc = rc;
      CK(tc_colscale(P, rows, hd, hq, hkv, c.d_ff, sc3[0], sc3[1], sc3[2], cs, m->stream));
      sdst->push_back(cs);
    }
  }
  // 128 positions x head_dim 16-bit values per block, for every KV head: K tiles and V^T tiles
  const size_t kv_bytes = (size_t)hkv * ((c.max_ctx + 127) / 128) * 128 * hd * 2;
  if (!T.sqkv.empty() && (T.sqkv.size() != T.wqkv.size() || T.swo.size() != T.wo.size() ||
                          T.sgu.size() != T.wgu.size() || T.sdown.size() != T.wdown.size()))
    return T.init_rc = ADP_ERR_INVALID_ARG;  // every layer matrix quantised, or none
  int rc = m->alloc(&T.Kt, kv_bytes);
  if (!rc) rc = m->alloc(&T.Vt, kv_bytes);
  if (rc) return T.init_rc = rc;
  CK(cudaMemsetAsync(T.Kt, 0, kv_bytes, m->stream));
  CK(cudaMemsetAsync(T.Vt, 0, kv_bytes, m->stream));
  CK(cudaStreamSynchronize(m->stream));
  return T.init_rc = ADP_OK;
}

// Scratch of the tensor-core prefill for P tokens (grown on demand; the old buffers are freed).
static int tc_reserve(adp_model* m, int P) {
  adp_model::TcState& T = m->tc;
  if (P <= T.cap) return ADP_OK;
  CK(cudaStreamSynchronize(m->stream));
  for (void* q : {(void*)T.tokens, (void*)T.x, (void*)T.A, (void*)T.A2, (void*)T.Qt, (void*)T.C}) {
    if (!q) continue;
    m->allocs.erase(std::remove(m->allocs.begin(), m->allocs.end(), q), m->allocs.end());
    cudaFree(q);
  }
  T.tokens = nullptr;
  T.x = nullptr;
  T.A = nullptr;
  T.A2 = nullptr;
  T.Qt = nullptr;
  T.C = nullptr;
  T.cap = 0;
  const adp_config& c = m->cfg;
  const int kmax = std::max(c.d_model, c.n_heads * c.head_dim);
  const size_t nmax = (size_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  int rc;
  if ((rc = m->alloc(&T.tokens, (size_t)P)) || (rc = m->alloc(&T.x, (size_t)P * c.d_model)) ||
      (rc = m->alloc(&T.A, tc_tiled_bytes(P, kmax, 256))) || (rc = m->alloc(&T.A2, tc_tiled_bytes(P, c.d_ff, 256))) ||
      (rc = m->alloc(&T.Qt, (size_t)c.n_heads * tc_tiled_bytes(P, c.head_dim, 128))) ||
      (rc = m->alloc(&T.C, (size_t)P * nmax)))
    return rc;
  CK(cudaMemsetAsync(T.Qt, 0, (size_t)c.n_heads * tc_tiled_bytes(P, c.head_dim, 128), m->stream));
  // the A tiles' padding (rows beyond P up to the GEMM's 256-row blocks, columns beyond a GEMM's
  // K) must read as zero
  CK(cudaMemsetAsync(T.A, 0, tc_tiled_bytes(P, kmax, 256), m->stream));
  CK(cudaMemsetAsync(T.A2, 0, tc_tiled_bytes(P, c.d_ff, 256), m->stream));
  T.cap = P;
  return ADP_OK;
}

extern "C" int adp_debug_tc_gemm_time(adp_model* m, int32_t which, int32_t M, int32_t reps, float* ms_per_launch) {
  if (!m || !ms_per_launch || which < 0 || which > 3 || M < 1 || reps < 1) return ADP_ERR_INVALID_ARG;
  int rc = tc_init(m);
  if (rc) return rc;
  if ((rc = tc_reserve(m, M))) return rc;
  const adp_config& c = m->cfg;
  const int qkv_n = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  const int N[4] = {qkv_n, c.d_model, 2 * c.d_ff, c.d_model};
  const int K[4] = {c.d_model, c.n_heads * c.head_dim, c.d_model, c.d_ff};
  const uint8_t* Wt[4] = {m->tc.wqkv[0], m->tc.wo[0], m->tc.wgu[0], m->tc.wdown[0]};
  const bool q = !m->tc.sqkv.empty();
  const float* Cs[4] = {q ? m->tc.sqkv[0] : nullptr, q ? m->tc.swo[0] : nullptr, q ? m->tc.sgu[0] : nullptr,
                        q ? m->tc.sdown[0] : nullptr};
  // each GEMM as the prefill runs it: QKV stores into C, Wo and down add into the residual x,
  // gate|up writes SwiGLU into the down GEMM's A tiles; down reads those tiles
  const int kmax = std::max(c.d_model, c.n_heads * c.head_dim);
  const int mode[4] = {TC_STORE, TC_ADD, TC_SWIGLU, TC_ADD};
  const uint8_t* Ain[4] = {m->tc.A, m->tc.A, m->tc.A, m->tc.A2};
  float* out[4] = {m->tc.C, m->tc.x, reinterpret_cast<float*>(m->tc.A2), m->tc.x};
  const int ldo[4] = {qkv_n, c.d_model, (c.d_ff + 63) / 64, c.d_model};
  // operands A: every element 0x3C3C (about 1.06 in f16, 0.0115 in bf16); the residual zero
  CK(cudaMemsetAsync(m->tc.A, 0x3C, tc_tiled_bytes(M, kmax, 256), m->stream));
  CK(cudaMemsetAsync(m->tc.A2, 0x3C, tc_tiled_bytes(M, c.d_ff, 256), m->stream));
  CK(cudaMemsetAsync(m->tc.x, 0, (size_t)M * c.d_model * 4, m->stream));
  const int bf16 = tc_operand_bf16(c);
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  const int w = which;
  CK(tc_gemm(bf16, mode[w], Ain[w], Wt[w], out[w], ldo[w], M, N[w], K[w], m->p.err, 1000000000ull, m->stream,
             nullptr, Cs[w]));
  CK(cudaEventRecord(e0, m->stream));
  for (int i = 0; i < reps; ++i)
    CK(tc_gemm(bf16, mode[w], Ain[w], Wt[w], out[w], ldo[w], M, N[w], K[w], m->p.err, 1000000000ull, m->stream,
               nullptr, Cs[w]));
  CK(cudaEventRecord(e1, m->stream));
  CK(cudaEventSynchronize(e1));
  float ms = 0.0f;
  CK(cudaEventElapsedTime(&ms, e0, e1));
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  // padding reads as zero again
  CK(cudaMemsetAsync(m->tc.A, 0, tc_tiled_bytes(M, kmax, 256), m->stream));
  CK(cudaMemsetAsync(m->tc.A2, 0, tc_tiled_bytes(M, c.d_ff, 256), m->stream));
  CK(cudaStreamSynchronize(m->stream));
  *ms_per_launch = ms / (float)reps;
  return ADP_OK;
}

extern "C" int adp_prefill_tc(adp_model* m, adp_kv* kv, const int32_t* host_tokens, int32_t n,
                              const adp_sampling* sampling, int32_t* next_token, float* dev_logits) {
  if (!m || !kv || !next_token || kv->m != m || n < 1 || !host_tokens) return ADP_ERR_INVALID_ARG;
  if (m->sticky) return m->sticky;
  if (kv->len + n > m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  for (int i = 0; i < n; ++i)
    if (host_tokens[i] < 0 || host_tokens[i] >= m->cfg.vocab) return ADP_ERR_INVALID_ARG;
  int rc = tc_init(m);
  if (rc) return rc;
  const int P = n - 1;  // the last prompt token goes through the decode kernel
  if (P > 0) {
    if ((rc = tc_reserve(m, P))) return rc;
    const adp_config& c = m->cfg;
    CK(cudaMemcpyAsync(m->tc.tokens, host_tokens, (size_t)P * 4, cudaMemcpyHostToDevice, m->stream));
    TcPrefill a{};
    a.P = P;
    a.pos0 = kv->len;
    a.n_layers = c.n_layers;
    a.d = c.d_model;
    a.hq = c.n_heads;
    a.hkv = c.n_kv_heads;
    a.hd = c.head_dim;
    a.ff = c.d_ff;
    a.max_ctx = c.max_ctx;
    a.bf16 = tc_operand_bf16(c);
    a.kvdt = c.kv_dtype;
    a.eps = c.rms_eps;
    a.scale = m->p.attn_scale;
    a.tokens = m->tc.tokens;
    a.tok_emb = m->p.tok_emb;
    a.attn_norm = m->h_attn_norm.data();
    a.ffn_norm = m->h_ffn_norm.data();
    a.wqkv = m->tc.wqkv.data();
    a.wo = m->tc.wo.data();
    a.wgu = m->tc.wgu.data();
    a.wdown = m->tc.wdown.data();
    a.sqkv = m->tc.sqkv.empty() ? nullptr : m->tc.sqkv.data();
    a.swo = m->tc.swo.empty() ? nullptr : m->tc.swo.data();
    a.sgu = m->tc.sgu.empty() ? nullptr : m->tc.sgu.data();
    a.sdown = m->tc.sdown.empty() ? nullptr : m->tc.sdown.data();
    a.kc = kv->k;
    a.vc = kv->v;
    a.rope_cos = m->p.rope_cos;
    a.rope_sin = m->p.rope_sin;
    a.x = m->tc.x;
    a.A = m->tc.A;
    a.A2 = m->tc.A2;
    a.Qt = m->tc.Qt;
    a.Kt = m->tc.Kt;
    a.Vt = m->tc.Vt;
    a.n_kb = (c.max_ctx + 127) / 128;
    a.err = m->p.err;
    a.wait_ns = std::max<uint64_t>(m->p.wait_ns, 1000000000ull);
    CK(tc_prefill(a, m->stream));
    kv->len += P;
  }
  // the last token: one decode step (synchronises and reports any device error, the GEMMs' too)
  return adp_decode_step(m, kv, host_tokens[n - 1], sampling, next_token, dev_logits);
}

extern "C" int adp_sync(adp_model* m) {
  if (!m) return ADP_ERR_INVALID_ARG;
  if (m->sticky) return m->sticky;
  return finish(m);
}

extern "C" int adp_reset(adp_model* m) {
  if (!m) return ADP_ERR_INVALID_ARG;
  cudaStreamSynchronize(m->stream);
  const Params& p = m->p;
  CK(cudaMemsetAsync(p.sample_ctr, 0, 4, m->stream));
  CK(cudaMemsetAsync(p.argkey, 0, 8, m->stream));
  CK(cudaMemsetAsync(p.lm_ctr, 0, 4, m->stream));
  CK(cudaMemsetAsync(p.bar_ctr, 0, 8, m->stream));
  CK(cudaMemsetAsync(p.err, 0, 4, m->stream));
  if (m->bt.init_rc == ADP_OK) {
    CK(cudaMemsetAsync(m->bt.p.sample_ctr, 0, 4 * kMaxBatch, m->stream));
    CK(cudaMemsetAsync(m->bt.p.argkey, 0, 8 * kMaxBatch, m->stream));
  }
  int rc = clear_exchange(m);
  if (rc) return rc;
  CK(cudaStreamSynchronize(m->stream));
  m->sticky = ADP_OK;
  m->p.skip_cta = m->p.skip_phase = -1;
  return ADP_OK;
}

extern "C" const char* adp_status_string(int status) {
  switch (status) {
    case ADP_OK: return "ok";
    case ADP_ERR_INVALID_ARG: return "invalid argument";
    case ADP_ERR_UNSUPPORTED_CONFIG: return "unsupported configuration";
    case ADP_ERR_CONTEXT_OVERFLOW: return "position beyond max_ctx";
    case ADP_ERR_CUDA: return "CUDA runtime error";
    case ADP_ERR_NOT_CORESIDENT: return "persistent grid cannot be co-resident";
    case ADP_ERR_BARRIER_TIMEOUT: return "grid barrier wait ran out (sticky until adp_reset)";
    case ADP_ERR_PIPELINE_TIMEOUT: return "weight pipeline wait ran out (sticky until adp_reset)";
    case ADP_ERR_UNIMPLEMENTED: return "unimplemented";
    default: return "unknown status";
  }
}

extern "C" const char* adp_last_error(void) { return g_last_error.c_str(); }

// ---------------------------------------------------------------- step in caller-given scratch

void adp::set_last_error(const char* msg) { g_last_error = msg; }

int adp::model_device(const adp_model* m) { return m ? m->device : -1; }

int adp::scratch_layout(const adp_model* m, ScratchLayout* out) {
  if (!m || !out) return ADP_ERR_INVALID_ARG;
  const adp_config& c = m->cfg;
  const size_t d = c.d_model, hq = c.n_heads, hkv = c.n_kv_heads, hd = c.head_dim, L = c.n_layers;
  const size_t ffw = c.n_experts ? (size_t)c.top_k * c.d_expert : (size_t)c.d_ff;
  const size_t nbmax = ((size_t)c.max_ctx + kAttnBlock - 1) / kAttnBlock;
  const size_t nblk = ((size_t)c.vocab + kVocabBlock - 1) / kVocabBlock;
  const size_t topk = c.n_experts ? (size_t)c.top_k : 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = (off + std::max<size_t>(bytes, 16) + 255) & ~(size_t)255;
    return at;
  };
  ScratchLayout& l = *out;
  l.x = take(d * 8);
  l.q = take(hq * hd * 8);
  l.attn = take(hq * hd * 8);
  l.h = take(ffw * 8);
  l.rlog = take((size_t)std::max(c.n_experts, 1) * 8);
  l.knew = take(hkv * hd * 8);
  l.vnew = take(hkv * hd * 8);
  l.epoch = take(4);
  l.tok_word = take(8);
  l.part_m = take(hq * nbmax * 8);
  l.part_l = take(hq * nbmax * 8);
  l.part_o = take(hq * nbmax * hd * 8);
  l.sblock = take(nblk * 4);
  l.sample_ctr = take(4);
  l.argkey = take(8);
  l.lm_ctr = take(4);
  l.bar_ctr = take(8);
  l.err = take(4);
  l.sel_out = take(L * topk * 4);
  l.state = take(sizeof(StepState));
  l.logits = take((size_t)c.vocab * 4);
  l.total = off;
  l.n_phases = m->phases.size();
  return ADP_OK;
}

int adp::decode_step_in_scratch(adp_model* m, adp_kv* kv, int32_t token, const adp_sampling* sampling,
                                int32_t* next_token, float* dev_logits, uint8_t* base, const ScratchLayout& lay,
                                size_t zero_bytes, size_t clear_bytes) {
  if (!m || !kv || !next_token || kv->m != m || !base) return ADP_ERR_INVALID_ARG;
  if (m->sticky) return m->sticky;
  if (token < 0 || token >= m->cfg.vocab) return ADP_ERR_INVALID_ARG;
  if (kv->len >= m->cfg.max_ctx) return ADP_ERR_CONTEXT_OVERFLOW;
  if (zero_bytes) CK(cudaMemsetAsync(base, 0, zero_bytes, m->stream));
  const float T = sampling ? sampling->temperature : 0.0f;
  StepState* d_state = reinterpret_cast<StepState*>(base + lay.state);
  CK(cudaEventSynchronize(m->state_copied));
  m->h_state->pos = kv->len;
  m->h_state->token = token;
  m->h_state->temperature = T;
  m->h_state->u = sampling ? sampling->u : 0.0f;
  m->h_state->seq_index = 0;
  m->h_state->out_token = -1;
  CK(cudaMemcpyAsync(d_state, m->h_state, sizeof(StepState), cudaMemcpyHostToDevice, m->stream));
  CK(cudaEventRecord(m->state_copied, m->stream));
  Params p = step_params(m, kv, dev_logits, nullptr, nullptr, nullptr);
  auto at = [&](size_t o) { return base + o; };
  p.x = reinterpret_cast<unsigned long long*>(at(lay.x));
  p.q = reinterpret_cast<unsigned long long*>(at(lay.q));
  p.attn = reinterpret_cast<unsigned long long*>(at(lay.attn));
  p.h = reinterpret_cast<unsigned long long*>(at(lay.h));
  p.rlog = reinterpret_cast<unsigned long long*>(at(lay.rlog));
  p.knew = reinterpret_cast<unsigned long long*>(at(lay.knew));
  p.vnew = reinterpret_cast<unsigned long long*>(at(lay.vnew));
  p.epoch = reinterpret_cast<uint32_t*>(at(lay.epoch));
  p.tok_word = reinterpret_cast<unsigned long long*>(at(lay.tok_word));
  p.n_steps = 1;
  p.part_m = reinterpret_cast<unsigned long long*>(at(lay.part_m));
  p.part_l = reinterpret_cast<unsigned long long*>(at(lay.part_l));
  p.part_o = reinterpret_cast<unsigned long long*>(at(lay.part_o));
  p.sblock = reinterpret_cast<float*>(at(lay.sblock));
  p.sample_ctr = reinterpret_cast<uint32_t*>(at(lay.sample_ctr));
  p.argkey = reinterpret_cast<unsigned long long*>(at(lay.argkey));
  p.lm_ctr = reinterpret_cast<uint32_t*>(at(lay.lm_ctr));
  p.bar_ctr = reinterpret_cast<unsigned long long*>(at(lay.bar_ctr));
  p.err = reinterpret_cast<int32_t*>(at(lay.err));
  p.sel_out = reinterpret_cast<int32_t*>(at(lay.sel_out));
  p.state = d_state;
  if (!dev_logits) p.logits = reinterpret_cast<float*>(at(lay.logits));
  const int nph = (int)m->phases.size();
  CK(decode_launch(p, 0, T > 0.0f ? nph : nph - 1, true, m->G, m->smem, m->xbuf_floats, m->stream));
  m->p.skip_cta = m->p.skip_phase = -1;  // the publication test hook covers one step, as in adp_decode_step
  CK(cudaMemcpyAsync(&m->h_out[0], &d_state->out_token, 4, cudaMemcpyDeviceToHost, m->stream));
  CK(cudaMemcpyAsync(&m->h_out[1], p.err, 4, cudaMemcpyDeviceToHost, m->stream));
  CK(cudaStreamSynchronize(m->stream));
  const int rc = map_device_error(m->h_out[1]);
  if (rc) {
    // counters and exchange words may be left mid-step: start the area over from zero
    CK(cudaMemsetAsync(base, 0, clear_bytes, m->stream));
    CK(cudaStreamSynchronize(m->stream));
    return rc;
  }
  *next_token = m->h_out[0];
  kv->len += 1;
  return ADP_OK;
}

extern "C" int adp_num_ctas(const adp_model* m, int32_t* ctas) {
  if (!m || !ctas) return ADP_ERR_INVALID_ARG;
  *ctas = m->G;
  return ADP_OK;
}

extern "C" int adp_image_bytes(const adp_model* m, uint64_t* bytes) {
  if (!m || !bytes) return ADP_ERR_INVALID_ARG;
  *bytes = m->image_bytes;
  return ADP_OK;
}

// The phase plan of a config on a GPU with n_sms SMs, computed on the host alone (no CUDA call):
// the same plan() a model built on such a GPU streams.
extern "C" int adp_plan(const adp_config* cfg, int32_t n_sms, adp_phase_plan* out, int32_t cap, int32_t* n_phases,
                        uint64_t* image_bytes) {
  if (!cfg || n_sms < 1 || cap < 0 || (cap > 0 && !out) || !n_phases || !image_bytes) return ADP_ERR_INVALID_ARG;
  const int rc = validate_config(cfg);
  if (rc) return rc;
  adp_model m;
  m.cfg = *cfg;
  m.G = n_sms;
  plan(&m);
  for (const PhaseDesc& P : m.phases)
    if ((uint64_t)P.n_units * (uint64_t)m.G >= (1ull << 32)) return ADP_ERR_UNSUPPORTED_CONFIG;
  *n_phases = (int32_t)m.phases.size();
  *image_bytes = m.image_bytes;
  for (int i = 0; i < cap && i < (int)m.phases.size(); ++i) {
    const PhaseDesc& P = m.phases[i];
    adp_phase_plan& o = out[i];
    o.kind = P.kind;
    o.layer = P.layer;
    o.n_units = P.n_units;
    o.unit_rows = P.unit_rows;
    o.slots = P.slots;
    o.K = P.K;
    o.KC = P.KC;
    o.n_chunks = P.n_chunks;
    o.upr = P.upr;
    o.dtype = P.has_weights ? P.wdt : -1;
    o.src_phase = P.src_ph;
    o.res_phase = P.res_ph;
    o.sel_phase = P.sel_ph;
    o.replicated = P.replicated;
    o.region = P.region;
    o.expert_stride = P.expert_stride;
  }
  return ADP_OK;
}

extern "C" int adp_batch_plan(const adp_config* cfg, int32_t n_sms, int32_t smem_optin, adp_batch_layout* out,
                              int32_t* max_batch) {
  if (!cfg || n_sms < 1 || smem_optin < 1 || !out || !max_batch) return ADP_ERR_INVALID_ARG;
  const int rc = validate_config(cfg);
  if (rc) return rc;
  adp_model m;
  m.cfg = *cfg;
  m.G = n_sms;
  plan(&m);
  BatchLayout lay[kMaxBatch + 1];
  *max_batch = plan_batches(m.cfg, m.phases, n_sms, (size_t)smem_optin, lay);
  for (int nb = 1; nb <= kMaxBatch; ++nb) {
    adp_batch_layout& o = out[nb - 1];
    o.ring_slots = lay[nb].nslots;
    o.attention_slots = lay[nb].att_slots;
    o.xbuf_floats = lay[nb].xbuf_floats;
    o.down_segment = lay[nb].down_seg;
    o.control_bytes = lay[nb].ctl;
    o.smem_bytes = lay[nb].smem;
  }
  return ADP_OK;
}

extern "C" int adp_launches_per_step(const adp_model* m, int32_t* n) {
  if (!m || !n) return ADP_ERR_INVALID_ARG;
  *n = m->mode == 0 ? 1 : (int32_t)m->phases.size() - 1;
  return ADP_OK;
}

// ---------------------------------------------------------------- debug and ablation hooks

extern "C" int adp_debug_kernel_mode(adp_model* m, int mode) {
  if (!m || mode < 0 || mode > 2) return ADP_ERR_INVALID_ARG;
  m->mode = mode;
  return ADP_OK;
}

extern "C" int adp_debug_force_experts(adp_model* m, const int32_t* host_idx) {
  if (!m) return ADP_ERR_INVALID_ARG;
  if (!m->cfg.n_experts) return host_idx ? ADP_ERR_UNSUPPORTED_CONFIG : ADP_OK;
  if (!host_idx) {
    m->force_on = false;
    return ADP_OK;
  }
  const size_t n = (size_t)m->cfg.n_layers * m->cfg.top_k;
  for (size_t i = 0; i < n; ++i)
    if (host_idx[i] < 0 || host_idx[i] >= m->cfg.n_experts) return ADP_ERR_INVALID_ARG;
  CK(cudaMemcpyAsync(m->d_force, host_idx, n * 4, cudaMemcpyHostToDevice, m->stream));
  CK(cudaStreamSynchronize(m->stream));
  m->force_on = true;
  return ADP_OK;
}

extern "C" int adp_debug_read_experts(const adp_model* m, int32_t* host_idx) {
  if (!m || !host_idx) return ADP_ERR_INVALID_ARG;
  if (!m->cfg.n_experts) return ADP_ERR_UNSUPPORTED_CONFIG;
  CK(cudaMemcpyAsync(host_idx, m->p.sel_out, (size_t)m->cfg.n_layers * m->cfg.top_k * 4, cudaMemcpyDeviceToHost,
                     m->stream));
  CK(cudaStreamSynchronize(m->stream));
  return ADP_OK;
}

extern "C" int adp_debug_trace_residual(adp_model* m, float* dev_buf) {
  if (!m) return ADP_ERR_INVALID_ARG;
  m->p.trace = dev_buf;
  if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
  return ADP_OK;
}

extern "C" int adp_debug_timeline(adp_model* m, uint64_t* dev_buf) {
  if (!m) return ADP_ERR_INVALID_ARG;
  m->p.timeline = reinterpret_cast<unsigned long long*>(dev_buf);
  if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
  return ADP_OK;
}

extern "C" int adp_debug_timeline_shape(const adp_model* m, int32_t* ctas, int32_t* phases) {
  if (!m || !ctas || !phases) return ADP_ERR_INVALID_ARG;
  *ctas = m->G;
  *phases = (int32_t)m->phases.size();
  return ADP_OK;
}

extern "C" int adp_debug_barriers(adp_model* m, int on) {
  if (!m) return ADP_ERR_INVALID_ARG;
  m->p.debug_barriers = on ? 1 : 0;
  if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
  return ADP_OK;
}

extern "C" int adp_debug_set_l2_lookahead(adp_model* m, uint32_t bytes) {
  if (!m) return ADP_ERR_INVALID_ARG;
  m->p.l2_lookahead = bytes;
  if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
  return ADP_OK;
}

extern "C" int adp_debug_set_l2_pacing(adp_model* m, uint32_t bytes_per_us, uint32_t burst_bytes) {
  if (!m || (bytes_per_us && burst_bytes < 32768)) return ADP_ERR_INVALID_ARG;
  m->p.l2_rate = bytes_per_us;
  m->p.l2_burst = burst_bytes;
  if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
  return ADP_OK;
}

extern "C" int adp_debug_set_prefetch_flags(adp_model* m, uint32_t flags) {
  if (!m || (flags & ~(uint32_t)(PF_KV_AHEAD | PF_KV_LAST | PF_W_LAST))) return ADP_ERR_INVALID_ARG;
  m->p.pf_flags = flags;
  if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
  return ADP_OK;
}

extern "C" int adp_debug_set_ring_slots(adp_model* m, int32_t slots) {
  if (!m || slots < 3 || slots > m->max_nslots) return ADP_ERR_INVALID_ARG;
  m->p.nslots = slots;  // the shared-memory size stays the one chosen at creation
  if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
  return ADP_OK;
}

extern "C" int adp_debug_ring_slots(const adp_model* m) { return m ? m->p.nslots : 0; }

// Test-only hooks: compiled into the test build of the library (-DADP_TEST_HOOKS) only, so that a
// release caller cannot make a model withhold outputs, shorten its waits or move its epoch counter.
#ifdef ADP_TEST_HOOKS
extern "C" int adp_debug_set_epoch_base(adp_model* m, uint32_t base) {
  if (!m) return ADP_ERR_INVALID_ARG;
  CK(cudaStreamSynchronize(m->stream));
  int rc = clear_exchange(m);
  if (rc) return rc;
  CK(cudaMemcpyAsync(m->p.epoch, &base, 4, cudaMemcpyHostToDevice, m->stream));
  CK(cudaStreamSynchronize(m->stream));
  m->epochs_used = base;
  return ADP_OK;
}

extern "C" int adp_debug_set_wait_limit(adp_model* m, uint64_t ns) {
  if (!m || ns == 0) return ADP_ERR_INVALID_ARG;
  m->p.wait_ns = ns;
  if (m->graph) { cudaGraphExecDestroy(m->graph); m->graph = nullptr; }
  return ADP_OK;
}

extern "C" int adp_debug_skip_publication(adp_model* m, int32_t cta, int32_t phase) {
  if (!m) return ADP_ERR_INVALID_ARG;
  m->p.skip_cta = cta;
  m->p.skip_phase = phase;
  return ADP_OK;
}
#endif  // ADP_TEST_HOOKS

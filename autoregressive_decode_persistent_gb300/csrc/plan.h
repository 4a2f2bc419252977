// Plan and parameter structures shared by the host engine and the decode kernel.
//
// The decode step is a fixed sequence of phases per layer (QKV, attention, Wo, FFN
// gate|up, FFN down; for MoE: router, expert gate|up, expert down), then the LM head
// and, when sampling, a sampling phase.  Weighted phases split their "units" (one row,
// a RoPE pair, a gate/up pair, a row group) evenly over the persistent CTAs (one per
// SM); each CTA streams its share as tiles of whole units x one K-chunk, laid out
// contiguously in a model-owned weight image in exactly the order the CTA consumes
// them, so one TMA bulk copy moves a tile.
#pragma once
#include <stdint.h>

namespace adp {

constexpr int kConsumerWarps = 15;                  // compute warps per CTA (16 warps in all: <= 128 registers)
constexpr int kThreads = (kConsumerWarps + 1) * 32; // + one producer (TMA) warp
constexpr int kSlotBytes = 32768;                   // one ring slot
constexpr int kMaxSlots = 6;                        // ring depth limit (the model picks what fits)
constexpr int kAttnBlock = 32;                      // positions per attention block (contract)
constexpr int kVocabBlock = 256;                    // vocabulary entries per sampling block (contract)
constexpr int kMaxTopK = 8;
constexpr int kAttnSlots = 8;                       // attention items in flight per CTA (max)
constexpr int kMaxGroup = 8;                        // query heads per KV head (max)
constexpr int kChunkAlign = 256;                    // K-chunks start at multiples of 32 lanes x 8 elements
constexpr int kStamps = 16;                         // timeline stamps per (CTA, phase)
constexpr int kMaxBatch = 4;                        // requests of one batched decode step (max)

enum PhaseKind : int32_t {
  PK_QKV = 0,    // rmsnorm prologue; RoPE pairs of q/k, v; epilogue writes q and the KV rows
  PK_ATTN = 1,   // split-sequence attention + per-head merge (no weights)
  PK_WO = 2,     // x += Wo attn
  PK_GU = 3,     // h = silu(Wg xn) * (Wu xn)
  PK_DOWN = 4,   // x += Wd h
  PK_ROUTER = 5, // r = Wr xn
  PK_EGU = 6,    // per chosen expert: h_s = silu(sg*(Qg xn)) * (su*(Qu xn))
  PK_EDOWN = 7,  // x += sum_s gate_s * sd*(Qd_s h_s)
  PK_LM = 8,     // logits = W_lm rmsnorm(x), running argmax
  PK_SAMPLE = 9  // inverse-CDF sampling over the logits (temperature > 0 only)
};

// DT_NVFP4: 4-bit E2M1 codes (two per byte, the even element in the low nibble) with one e4m3
// scale per 16 consecutive elements of a row.
enum DType : int32_t { DT_F16 = 0, DT_BF16 = 1, DT_E4M3 = 2, DT_F32 = 3, DT_NVFP4 = 4 };

// Kernel instantiations: dense 16-bit weights, top-k experts, dense e4m3 layer matrices, the
// batched kernel (dense 16-bit or e4m3 weights, up to kMaxBatch requests per step), and dense
// NVFP4 layer matrices.
enum KernelKind : int32_t { KK_DENSE = 0, KK_MOE = 1, KK_DENSE8 = 2, KK_BATCH = 3, KK_DENSE4 = 4 };

struct PhaseDesc {
  int32_t kind, layer;
  int32_t n_units;        // units of the whole phase
  int32_t unit_rows;      // weight rows per unit (per expert slot)
  int32_t slots;          // expert slots per tile: 1, or top_k for expert phases
  int32_t K;              // reduction length
  int32_t KC;             // K-chunk width, multiple of kChunkAlign
  int32_t n_chunks;       // ceil(K / KC)
  int32_t upr;            // units per round (<= kConsumerWarps)
  int32_t eb;             // weight element bytes (0 for NVFP4: see wbytes)
  int32_t wdt;            // weight DType
  int32_t has_weights;
  int32_t index;          // position of this phase in the step's phase list
  int32_t src_ph;         // phase whose output vector is this phase's input (-1: the embedding row)
  int32_t res_ph;         // phase that wrote the residual rows this phase updates (-1: none)
  int32_t sel_ph;         // router phase whose logits choose this phase's experts (-1: none)
  int32_t replicated;     // 1: every CTA takes all units (one shared region of the image), 0: an even split
  uint64_t region;        // byte offset of the phase's region in the image (expert 0 for expert phases)
  uint64_t expert_stride; // bytes of one expert's region
};

struct StepState {
  int32_t pos;        // position of the token being decoded
  int32_t token;      // input token (ignored when a token sequence is given)
  float temperature;  // 0: greedy
  float u;            // uniform for sampling (ignored when a uniform sequence is given)
  int32_t seq_index;  // index into token / uniform / output sequences
  int32_t out_token;  // chosen token of the last completed step
  int32_t pad0, pad1;
};

struct Params {
  // weights
  const uint8_t* image;
  const void* tok_emb;
  const void* const* attn_norm;       // [L] device pointers
  const void* const* ffn_norm;        // [L]
  const void* final_norm;
  const float* const* e_gate_scale;   // [L] -> [E][f]
  const float* const* e_up_scale;     // [L] -> [E][f]
  const float* const* e_down_scale;   // [L] -> [E][d]
  const float* const* wscale[7];      // e4m3 dense: [L] -> per-row scales of q, k, v, o, gate, up, down
  const PhaseDesc* phases;
  int32_t n_phases;
  // shapes
  int32_t L, d, hq, hkv, hd, ff, V, max_ctx, E, topk, fexp;
  int32_t wdt, kvdt, rdt;
  int32_t edt;                        // embedding, LM head and norm gains (= wdt unless wdt is e4m3)
  float eps;
  float attn_scale;
  int32_t nbmax;                      // max attention blocks = ceil(max_ctx / 32)
  int32_t att_slots;                  // attention items a CTA works on at once
  int32_t att_gmax;                   // warps per slot (largest number of query heads per KV head)
  int32_t att_slot_bytes;             // shared-memory staging bytes of one slot
  int32_t xbuf_floats;                // floats of the shared input-vector / staging area
  int32_t merge_split;                // CTAs merging each query head, one slice of head_dim each (1, 2, 4),
  int32_t merge_split_blocks;         // from this many attention blocks on (fewer: one CTA per head)
  // KV cache [L][hkv][max_ctx][hd]
  uint16_t* kc;
  uint16_t* vc;
  // RoPE tables [max_ctx][hd/2]
  const float* rope_cos;
  const float* rope_sin;
  // Activations exchanged between CTAs, as 64-bit words {fp32 bits (low), epoch (high)} written
  // with one store each: a reader polls a word until it carries the epoch of the phase that
  // produces it, so no grid barrier separates dependent phases.
  unsigned long long* x;     // [d] residual
  unsigned long long* q;     // [hq*hd] post-RoPE queries
  unsigned long long* knew;  // [hkv*hd] this step's K rows (storage bits)
  unsigned long long* vnew;  // [hkv*hd] this step's V rows (storage bits)
  unsigned long long* attn;  // [hq*hd] attention output
  unsigned long long* h;     // [max(ff, topk*f)] FFN activations
  unsigned long long* rlog;  // [E] router logits
  uint32_t* epoch;           // epoch base of the next step (advanced by the step's last CTA)
  unsigned long long* tok_word;  // the token a step chose, tagged with the next step's epoch base
  unsigned long long* part_m;  // [hq][nbmax] attention block maxima (epoch-tagged)
  unsigned long long* part_l;  // [hq][nbmax] attention block sums (epoch-tagged)
  unsigned long long* part_o;  // [hq][nbmax][hd] attention block outputs (epoch-tagged)
  float* sblock;               // [ceil(V/256)] sampling block sums
  uint32_t* sample_ctr;
  unsigned long long* argkey;  // packed (ordered logit, ~index) maximum
  uint32_t* lm_ctr;
  unsigned long long* bar_ctr; // monotonic grid-barrier counter
  int32_t* err;                // sticky device error word
  int32_t* sel_out;            // [L][topk] router choices
  const int32_t* force_sel;    // [L][topk] forced experts or null
  float* trace;                // [L+1][d] residual trace or null
  StepState* state;
  const int32_t* tok_seq;      // token per step (prefill) or null
  const float* u_seq;          // uniform per step or null
  int32_t* out_seq;            // chosen token per step or null
  float* logits;               // [V] logits output
  unsigned long long* timeline; // [G][n_phases][kStamps] %globaltimer stamps or null
  uint64_t wait_ns;            // limit of every in-kernel wait
  uint32_t l2_lookahead;       // bytes of weight stream prefetched into L2 beyond the TMA loads
  uint32_t pf_flags;           // PF_* bits: how the KV cache and the weight lookahead are prefetched
  uint32_t l2_rate;            // lookahead pacing: bytes per microsecond per CTA (0 = unpaced)
  uint32_t l2_burst;           // lookahead pacing: most bytes issued at once (token-bucket depth)
  int32_t debug_barriers;      // 1: also take a grid barrier after every phase (debugging)
  int32_t n_steps;             // decode steps this launch runs back to back (persistent launch)
  int32_t nslots;              // weight ring depth (slots of kSlotBytes)
  int32_t skip_cta, skip_phase;  // test hook: that CTA does not publish that phase's outputs
  // Batched kernel only: nb requests per step.  Every per-request buffer above (x, q, knew, vnew,
  // attn, h, part_*, logits, argkey, sblock, sample_ctr, tok_word, state) then holds nb copies of
  // its single-request layout back to back, and the token / uniform / output sequences are
  // [step][nb].
  int32_t nb;
  uint16_t* const* kcb;        // [nb] each request's K cache [L][hkv][max_ctx][hd]
  uint16_t* const* vcb;        // [nb] each request's V cache
};

#ifdef __CUDACC__
#define ADP_HD __host__ __device__
#else
#define ADP_HD
#endif

// Image bytes of n consecutive weight elements of one row (n * eb).  NVFP4 rows take n / 2 bytes
// of codes plus n / 16 block-scale bytes (n a multiple of 16): within one tile of R rows x kck
// elements the R x kck / 2 code bytes come first, row after row, then the R x kck / 16 scales.
ADP_HD inline uint64_t wbytes(const PhaseDesc& P, uint64_t n) {
  return P.wdt == DT_NVFP4 ? n / 16 * 9 : n * (uint64_t)P.eb;
}

// Prefetch options (Params::pf_flags).  PF_KV_AHEAD: a layer's attention K/V blocks are brought
// into L2 one layer early (during the previous layer's QKV phase) instead of during its own QKV
// phase; PF_KV_LAST / PF_W_LAST: those K/V prefetches / the weight-stream lookahead carry the L2
// evict-last priority.
enum PrefetchFlags : uint32_t { PF_KV_AHEAD = 1u, PF_KV_LAST = 2u, PF_W_LAST = 4u };

// Device error codes (the host maps them to ADP_ERR_*).
enum DevErr : int32_t { DE_NONE = 0, DE_BARRIER_TIMEOUT = 1, DE_PIPELINE_TIMEOUT = 2 };  // 1: a dependency wait

}  // namespace adp

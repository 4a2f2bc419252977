// One batch-1 decode step as one persistent kernel (or, for the launch-overhead ablation,
// the same device code as one launch per phase).
//
// Pages followed (title, section):
//  "標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒" (hakusoku.com summary of
//   Kog AI's "Real-time LLM inference on standard GPUs: 3,000 tokens/s per request"):
//   - "GPU推論の速度制限要因：メモリ帯域幅": at batch 1 the step is matrix-vector products that
//     stream every active weight (and the KV cache) once, so it is bound by memory bandwidth;
//   - "標準推論スタックのボトルネックとKogの工夫": per-kernel launch and cleanup cost (4.5 µs x 10
//     kernels x 25 layers) is removed by one GPU-resident program for the whole decode path;
//   - "Kog Inference Engineの特徴とイノベーション": that program covers MatMul, attention,
//     normalization, routing and sampling, and controls sync, prefetch and ordering itself.
//  "「ソフトウェア・ファースト」戦略でGPUの限界を突破" (studioglobal.ai), "独自の3層共同設計アプローチ"
//   item 1: the whole decode runs as one persistent kernel with no launches between layers.
//
// GB300 design (not the pages' H200/MI300X code, which is not public):
//  - one CTA per SM (152), 16 consumer warps + 1 producer warp;
//  - the producer streams this CTA's weight tiles, in consumption order, from a model-owned
//    image through a 4 x 32 KB shared-memory ring with TMA bulk copies (cp.async.bulk +
//    mbarrier, L2 evict-first).  Weights never depend on activations, so it runs ahead across
//    phase boundaries and grid barriers: HBM keeps streaming while the consumers wait;
//  - consumers compute GEMV rows with the contract's dot product (lane l takes 8-element
//    vectors l, l+32, ..., fused multiply-adds in order, then a fixed butterfly), RMSNorm in the
//    prologue, RoPE / KV store / SwiGLU / residual / argmax in the epilogue;
//  - attention is split over 32-position blocks and query heads across all warps of the grid;
//    the last block of a head to finish merges the head by log-sum-exp.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace adp {

struct Ctl {
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  uint64_t sel_bar;
  int32_t abort;
  int32_t pad;
  unsigned long long red_k[kConsumerWarps];
  float bcast;
  int32_t flag;
  int32_t sel[kMaxTopK];
  float gate[kMaxTopK];
};

struct Step {
  int32_t pos, token, seq_index;
  float temperature, u;
};

__device__ __forceinline__ void set_error(const Params& p, Ctl* ctl, int32_t code) {
  atomicCAS(p.err, 0, code);
  *(volatile int32_t*)&ctl->abort = 1;
}

__device__ __forceinline__ bool aborted(Ctl* ctl) { return *(volatile int32_t*)&ctl->abort != 0; }

// Per-CTA share of a phase: units [u0, u0 + n).
__device__ __forceinline__ void cta_units(const PhaseDesc& P, uint32_t c, uint32_t G, int32_t& u0, int32_t& n) {
  const long long a = (long long)c * P.n_units / G, b = (long long)(c + 1) * P.n_units / G;
  u0 = (int32_t)a;
  n = (int32_t)(b - a);
}

// ---------------------------------------------------------------- producer (TMA) warp

__device__ void producer(const Params& p, Ctl* ctl, uint8_t* ring, uint32_t c, uint32_t G, int ph0, int ph1) {
  const uint64_t pol = policy_evict_first();
  uint32_t t = 0;
  uint32_t sel_uses = 0;
  int sel_layer = -1;
  bool stop = false;
  for (int ph = ph0; ph < ph1 && !stop; ++ph) {
    const PhaseDesc P = p.phases[ph];
    if (!P.has_weights) continue;
    int32_t u0, n;
    cta_units(P, c, G, u0, n);
    const bool expert = P.kind == PK_EGU || P.kind == PK_EDOWN;
    if (expert && sel_layer != P.layer) {
      // expert weights are known only after routing: wait for this layer's selection
      if (!mbar_wait(&ctl->sel_bar, sel_uses & 1, &ctl->abort, p.wait_ns)) {
        if (!aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
        break;
      }
      ++sel_uses;
      sel_layer = P.layer;
    }
    if (n <= 0) continue;
    const uint64_t unit_bytes = (uint64_t)P.unit_rows * P.K * P.eb;
    const uint8_t* base = p.image + P.region + (uint64_t)u0 * unit_bytes;
    const int rounds = (n + P.upr - 1) / P.upr;
    for (int r = 0; r < rounds && !stop; ++r) {
      const int m = min(P.upr, n - r * P.upr);
      const uint64_t round_off = (uint64_t)r * P.upr * unit_bytes;
      for (int ck = 0; ck < P.n_chunks; ++ck) {
        if (aborted(ctl)) { stop = true; break; }
        const int kck = min(P.KC, P.K - ck * P.KC);
        const uint32_t bytes = (uint32_t)m * P.unit_rows * kck * P.eb;
        const uint64_t off = round_off + (uint64_t)m * P.unit_rows * ck * P.KC * P.eb;
        const uint32_t slot = t % kSlots, use = t / kSlots;
        if (t >= kSlots && !mbar_wait(&ctl->empty[slot], (use - 1) & 1, &ctl->abort, p.wait_ns)) {
          if (!aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
          stop = true;
          break;
        }
        mbar_arrive_expect_tx(&ctl->full[slot], bytes * P.slots);
        uint8_t* dst = ring + (size_t)slot * kSlotBytes;
        for (int s = 0; s < P.slots; ++s) {
          const uint8_t* src = base + off;
          if (expert) src += (uint64_t)(*(volatile int32_t*)&ctl->sel[s]) * P.expert_stride;
          tma_load_1d(dst + (size_t)s * bytes, src, bytes, &ctl->full[slot], pol);
        }
        ++t;
      }
    }
  }
  // No bulk copy may still be writing this CTA's shared memory when it exits.
  int32_t never = 0;
  for (uint32_t i = (t > (uint32_t)kSlots ? t - kSlots : 0); i < t; ++i)
    mbar_wait(&ctl->full[i % kSlots], (i / kSlots) & 1, &never, p.wait_ns);
}

// ---------------------------------------------------------------- consumer helpers

__device__ __forceinline__ void load_x8(const float* xs, float (&x)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(xs);
  const float4 b = *reinterpret_cast<const float4*>(xs + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void ldcg_x8(const float* g, float (&x)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(g));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(g) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// xn = rmsnorm(src) * gain into xbuf (all consumer warps; ends with consumer_sync).
// src is the fp32 residual in global memory, or (layer 0) the token's embedding row.
__device__ void rmsnorm_prologue(const Params& p, Ctl* ctl, float* xbuf, const void* gain, const void* emb_row,
                                 int cw, int lane) {
  const int d = p.d;
  if (cw == 0) {
    float acc = 0.0f;
    for (int v = lane; v < d / 8; v += 32) {
      float x8[8];
      if (emb_row) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x8[e] = load_elem(emb_row, (size_t)v * 8 + e, p.wdt);
      } else {
        ldcg_x8(p.x + v * 8, x8);
      }
      acc = fma8(x8, x8, acc);
    }
    const float ss = warp_fold(acc);
    const float mean = __fdiv_rn(ss, (float)d);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, p.eps)));
    if (lane == 0) ctl->bcast = r;
  }
  consumer_sync();
  const float r = ctl->bcast;
  for (int i = cw * 32 + lane; i < d; i += kConsumerWarps * 32) {
    const float xi = emb_row ? load_elem(emb_row, (size_t)i, p.wdt) : __ldcg(p.x + i);
    xbuf[i] = __fmul_rn(__fmul_rn(xi, r), load_elem(gain, (size_t)i, p.wdt));
  }
  consumer_sync();
}

__device__ void copy_prologue(float* xbuf, const float* src, int n, int cw, int lane) {
  for (int i = cw * 32 + lane; i < n; i += kConsumerWarps * 32) xbuf[i] = __ldcg(src + i);
  consumer_sync();
}

// Router softmax + top-k in one lane (ties to the lower index), gates renormalised over the
// choice; forced experts (test hook) keep the router's probabilities of those experts.
__device__ void select_experts(const Params& p, Ctl* ctl, int layer) {
  const int E = p.E, K = p.topk;
  float M = __ldcg(p.rlog);
  for (int e = 1; e < E; ++e) {
    const float r = __ldcg(p.rlog + e);
    M = r > M ? r : M;
  }
  float Z = 0.0f;
  for (int e = 0; e < E; ++e) Z = __fadd_rn(Z, exp_c(__fsub_rn(__ldcg(p.rlog + e), M)));
  uint32_t used[32] = {0};  // bit set over up to 1024 experts
  float Zs = 0.0f;
  for (int i = 0; i < K; ++i) {
    int best = -1;
    float bp = 0.0f;
    if (p.force_sel) {
      best = p.force_sel[layer * K + i];
      bp = __fdiv_rn(exp_c(__fsub_rn(__ldcg(p.rlog + best), M)), Z);
    } else {
      for (int e = 0; e < E; ++e) {
        if (used[e >> 5] & (1u << (e & 31))) continue;
        const float pe = __fdiv_rn(exp_c(__fsub_rn(__ldcg(p.rlog + e), M)), Z);
        if (best < 0 || pe > bp) { best = e; bp = pe; }
      }
      used[best >> 5] |= 1u << (best & 31);
    }
    ctl->sel[i] = best;
    ctl->gate[i] = bp;  // probability for now
    Zs = __fadd_rn(Zs, bp);
  }
  for (int i = 0; i < K; ++i) ctl->gate[i] = __fdiv_rn(ctl->gate[i], Zs);
}

// ---------------------------------------------------------------- GEMV phases

template <int ROWS, int SLOTS, int WDT, bool XPERSLOT>
__device__ void gemv_phase(const Params& p, Ctl* ctl, uint8_t* ring, float* xbuf, const PhaseDesc& P,
                           const Step& st, uint32_t c, uint32_t G, int cw, int lane, uint32_t& t) {
  int32_t u0, n;
  cta_units(P, c, G, u0, n);
  const int L = P.layer;
  unsigned long long best = 0ull;  // LM: packed running maximum of this warp
  const int rounds = n > 0 ? (n + P.upr - 1) / P.upr : 0;
  for (int r = 0; r < rounds; ++r) {
    const int m = min(P.upr, n - r * P.upr);
    const bool active = cw < m;
    const int unit = u0 + r * P.upr + cw;
    float acc[SLOTS * ROWS];
#pragma unroll
    for (int i = 0; i < SLOTS * ROWS; ++i) acc[i] = 0.0f;
    for (int ck = 0; ck < P.n_chunks; ++ck) {
      const uint32_t slot = t % kSlots, use = t / kSlots;
      bool ok = aborted(ctl) || mbar_wait(&ctl->full[slot], use & 1, &ctl->abort, p.wait_ns);
      if (!ok) {
        if (lane == 0 && !aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
        __syncwarp();
      }
      if (active && !aborted(ctl)) {
        const int kck = min(P.KC, P.K - ck * P.KC);
        const int nvec = kck >> 3;
        const uint32_t slot_bytes = (uint32_t)m * ROWS * kck * P.eb;
        const uint8_t* tile = ring + (size_t)slot * kSlotBytes;
        const int xoff = ck * P.KC;
        for (int v = lane; v < nvec; v += 32) {
          float x8[8];
          if (!XPERSLOT) load_x8(xbuf + xoff + v * 8, x8);
#pragma unroll
          for (int s = 0; s < SLOTS; ++s) {
            if (XPERSLOT) load_x8(xbuf + s * P.K + xoff + v * 8, x8);
#pragma unroll
            for (int j = 0; j < ROWS; ++j) {
              float w8[8];
              load8<WDT>(tile + (size_t)s * slot_bytes + ((size_t)(cw * ROWS + j) * kck + (size_t)v * 8) * P.eb, w8);
              acc[s * ROWS + j] = fma8(w8, x8, acc[s * ROWS + j]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[slot]);
      ++t;
    }
    if (!active || aborted(ctl)) continue;
#pragma unroll
    for (int i = 0; i < SLOTS * ROWS; ++i) acc[i] = warp_fold(acc[i]);
    // ---- epilogues
    if (P.kind == PK_QKV) {
      if (lane == 0) {
        const int half = p.hd / 2;
        const int nq = p.hq * half, nk = p.hkv * half;
        const float a = acc[0], b = acc[1];
        if (unit < nq + nk) {
          const bool isq = unit < nq;
          const int uu = isq ? unit : unit - nq;
          const int head = uu / half, i = uu % half;
          const float cs = __ldg(p.rope_cos + (size_t)st.pos * half + i);
          const float sn = __ldg(p.rope_sin + (size_t)st.pos * half + i);
          const float a2 = fmaf(a, cs, -__fmul_rn(b, sn));
          const float b2 = fmaf(b, cs, __fmul_rn(a, sn));
          if (isq) {
            __stcg(p.q + head * p.hd + i, a2);
            __stcg(p.q + head * p.hd + i + half, b2);
          } else {
            const size_t row = (((size_t)L * p.hkv + head) * p.max_ctx + st.pos) * p.hd;
            p.kc[row + i] = round_kv(a2, p.kvdt);
            p.kc[row + i + half] = round_kv(b2, p.kvdt);
          }
        } else {
          const int uu = unit - nq - nk;
          const int head = uu / half, i = uu % half;
          const size_t row = (((size_t)L * p.hkv + head) * p.max_ctx + st.pos) * p.hd;
          p.vc[row + i] = round_kv(a, p.kvdt);
          p.vc[row + i + half] = round_kv(b, p.kvdt);
        }
      }
    } else if (P.kind == PK_WO || P.kind == PK_DOWN) {
      if (lane < ROWS) {
        const int row = unit * ROWS + lane;
        float y = acc[0];
#pragma unroll
        for (int j = 1; j < ROWS; ++j) if (lane == j) y = acc[j];
        __stcg(p.x + row, __fadd_rn(__ldcg(p.x + row), y));
      }
    } else if (P.kind == PK_GU) {
      if (lane == 0) __stcg(p.h + unit, silu_mul(acc[0], acc[1]));
    } else if (P.kind == PK_ROUTER) {
      if (lane < ROWS) {
        float y = acc[0];
#pragma unroll
        for (int j = 1; j < ROWS; ++j) if (lane == j) y = acc[j];
        __stcg(p.rlog + unit * ROWS + lane, y);
      }
    } else if (P.kind == PK_EGU) {
      if (lane < p.topk) {
        float g = acc[0], uval = acc[1];
#pragma unroll
        for (int s = 1; s < SLOTS; ++s)
          if (lane == s) { g = acc[s * ROWS]; uval = acc[s * ROWS + 1]; }
        const int e = ctl->sel[lane];
        const float sg = __ldg(p.e_gate_scale[L] + (size_t)e * p.fexp + unit);
        const float su = __ldg(p.e_up_scale[L] + (size_t)e * p.fexp + unit);
        __stcg(p.h + lane * p.fexp + unit, silu_mul(__fmul_rn(sg, g), __fmul_rn(su, uval)));
      }
    } else if (P.kind == PK_EDOWN) {
      if (lane == 0) {
        float ax = 0.0f;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
          if (s < p.topk) {
            const int e = ctl->sel[s];
            const float y = __fmul_rn(__ldg(p.e_down_scale[L] + (size_t)e * p.d + unit), acc[s]);
            ax = fmaf(ctl->gate[s], y, ax);
          }
        }
        __stcg(p.x + unit, __fadd_rn(__ldcg(p.x + unit), ax));
      }
    } else if (P.kind == PK_LM) {
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < ROWS; ++j) {
          const int row = unit * ROWS + j;
          __stcg(p.logits + row, acc[j]);
          const unsigned long long k = argmax_key(acc[j], (uint32_t)row);
          best = k > best ? k : best;
        }
      }
    }
  }
  if (P.kind == PK_LM) {
    if (lane == 0) ctl->red_k[cw] = best;
    consumer_sync();
    if (cw == 0 && lane == 0) {
      unsigned long long k = 0ull;
      for (int w = 0; w < kConsumerWarps; ++w) k = ctl->red_k[w] > k ? ctl->red_k[w] : k;
      if (!aborted(ctl)) {
        if (k) atomicMax(p.argkey, k);
        __threadfence();
        const uint32_t old = atomicAdd(p.lm_ctr, 1u);
        ctl->flag = (old == G - 1) ? 1 : 0;
      } else {
        ctl->flag = 0;
      }
    }
    consumer_sync();
  }
}

// ---------------------------------------------------------------- finalisation

__device__ void finalize_token(const Params& p, const Step& st, int32_t token) {
  StepState* s = p.state;
  s->out_token = token;
  if (p.out_seq) p.out_seq[st.seq_index] = token;
  s->token = token;
  s->pos = st.pos + 1;
  s->seq_index = st.seq_index + 1;
  __threadfence();
}

// ---------------------------------------------------------------- attention phase

template <int NV>  // 8-element vectors per head (head_dim / 8)
__device__ void attention_phase(const Params& p, Ctl* ctl, const PhaseDesc& P, const Step& st, uint32_t c,
                                uint32_t G, int cw, int lane) {
  constexpr int HD = NV * 8;
  constexpr int DPL = HD / 32;  // output dims per lane
  const int L = P.layer;
  const int ctx = st.pos + 1;
  const int nb = (ctx + kAttnBlock - 1) / kAttnBlock;
  const int items = p.hq * nb;
  const int stride = (int)G * kConsumerWarps;
  for (int it = cw * (int)G + (int)c; it < items; it += stride) {
    if (aborted(ctl)) break;
    const int h = it % p.hq, b = it / p.hq;
    const int g = (int)(((long long)h * p.hkv) / p.hq);
    const size_t cache0 = ((size_t)L * p.hkv + g) * p.max_ctx * HD;
    const int j0 = b * kAttnBlock;
    const int nvalid = min(kAttnBlock, ctx - j0);
    const float* qh = p.q + h * HD;
    // scores: lane <-> position j0 + lane; contract dot over head_dim
    float s = __int_as_float(0xFF800000);  // -inf
    if (lane < nvalid) {
      float pv[32];
      const uint16_t* krow = p.kc + cache0 + (size_t)(j0 + lane) * HD;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const uint4 kw = __ldcg(reinterpret_cast<const uint4*>(krow) + v);
        const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w};
        float k8[8], q8[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          k8[2 * i] = kv_to_f32((uint16_t)(kk[i] & 0xFFFFu), p.kvdt);
          k8[2 * i + 1] = kv_to_f32((uint16_t)(kk[i] >> 16), p.kvdt);
        }
        ldcg_x8(qh + v * 8, q8);
        pv[v] = fma8(k8, q8, 0.0f);
      }
#pragma unroll
      for (int v = NV; v < 32; ++v) pv[v] = 0.0f;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
        for (int i = 0; i < off; ++i) pv[i] = __fadd_rn(pv[i], pv[i + off]);
      s = __fmul_rn(pv[0], p.attn_scale);
    }
    float mb = s;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, off));
    const float e = lane < nvalid ? exp_c(__fsub_rn(s, mb)) : 0.0f;
    float l = 0.0f;
    float o[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = 0.0f;
    const uint16_t* vblk = p.vc + cache0 + (size_t)j0 * HD + lane * DPL;
    for (int j = 0; j < nvalid; ++j) {
      const float ej = __shfl_sync(0xFFFFFFFFu, e, j);
      l = __fadd_rn(l, ej);
      const uint16_t* vr = vblk + (size_t)j * HD;
      float vv[DPL];
      if constexpr (DPL == 4) {
        const uint2 w = __ldcg(reinterpret_cast<const uint2*>(vr));
        vv[0] = kv_to_f32((uint16_t)(w.x & 0xFFFFu), p.kvdt);
        vv[1] = kv_to_f32((uint16_t)(w.x >> 16), p.kvdt);
        vv[2] = kv_to_f32((uint16_t)(w.y & 0xFFFFu), p.kvdt);
        vv[3] = kv_to_f32((uint16_t)(w.y >> 16), p.kvdt);
      } else {
#pragma unroll
        for (int i = 0; i < DPL; ++i) vv[i] = kv_to_f32(__ldcg(vr + i), p.kvdt);
      }
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[i] = fmaf(ej, vv[i], o[i]);
    }
    const size_t pi = (size_t)h * p.nbmax + b;
    if (lane == 0) {
      __stcg(p.part_m + pi, mb);
      __stcg(p.part_l + pi, l);
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) __stcg(p.part_o + pi * HD + lane * DPL + i, o[i]);
    __threadfence();
    __syncwarp();
    uint32_t last = 0;
    if (lane == 0) last = atomicAdd(p.head_ctr + h, 1u) == (uint32_t)(nb - 1) ? 1u : 0u;
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    // this warp completed head h: merge its nb blocks in ascending order
    __threadfence();
    float M = __int_as_float(0xFF800000);
    for (int bb = lane; bb < nb; bb += 32) M = fmaxf(M, __ldcg(p.part_m + (size_t)h * p.nbmax + bb));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
    float Lsum = 0.0f;
    float O[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) O[i] = 0.0f;
    for (int bb = 0; bb < nb; ++bb) {
      const size_t q = (size_t)h * p.nbmax + bb;
      const float w = exp_c(__fsub_rn(__ldcg(p.part_m + q), M));
      Lsum = fmaf(w, __ldcg(p.part_l + q), Lsum);
#pragma unroll
      for (int i = 0; i < DPL; ++i) O[i] = fmaf(w, __ldcg(p.part_o + q * HD + lane * DPL + i), O[i]);
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) __stcg(p.attn + h * HD + lane * DPL + i, __fdiv_rn(O[i], Lsum));
    if (lane == 0) p.head_ctr[h] = 0u;
  }
}

// ---------------------------------------------------------------- sampling phase

__device__ void sample_phase(const Params& p, Ctl* ctl, const Step& st, uint32_t c, uint32_t G, int cw, int lane) {
  const unsigned long long key = __ldcg(p.argkey);
  const float M = order_float((uint32_t)(key >> 32));
  const float T = st.temperature;
  const int V = p.V;
  const int nblk = (V + kVocabBlock - 1) / kVocabBlock;
  const int stride = (int)G * kConsumerWarps;
  for (int it = cw * (int)G + (int)c; it < nblk; it += stride) {
    if (aborted(ctl)) break;
    const int i0 = it * kVocabBlock;
    const int nn = min(kVocabBlock, V - i0);
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = lane * 8 + e;
      if (k < nn) {
        const float ev = exp_c(__fdiv_rn(__fsub_rn(__ldcg(p.logits + i0 + k), M), T));
        acc = fmaf(ev, 1.0f, acc);
      }
    }
    const float S = warp_fold(acc);
    if (lane == 0) __stcg(p.sblock + it, S);
    __threadfence();
    __syncwarp();
    uint32_t last = 0;
    if (lane == 0) last = atomicAdd(p.sample_ctr, 1u) == (uint32_t)(nblk - 1) ? 1u : 0u;
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    __threadfence();
    // inverse CDF over the block sums, then within the chosen block
    float Z = 0.0f;
    for (int b = 0; b < nblk; ++b) Z = __fadd_rn(Z, __ldcg(p.sblock + b));
    const float tau = __fmul_rn(st.u, Z);
    float P = 0.0f;
    int bstar = -1;
    for (int b = 0; b < nblk; ++b) {
      const float Pn = __fadd_rn(P, __ldcg(p.sblock + b));
      if (Pn > tau) { bstar = b; break; }
      P = Pn;
    }
    bool from_end = false;
    if (bstar < 0) {  // tau rounded up to Z: take the last token with nonzero weight
      from_end = true;
      bstar = 0;
      for (int b = nblk - 1; b >= 0; --b)
        if (__ldcg(p.sblock + b) > 0.0f) { bstar = b; break; }
    }
    const int b0 = bstar * kVocabBlock;
    const int nb2 = min(kVocabBlock, V - b0);
    float ev[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = lane * 8 + e;
      ev[e] = k < nb2 ? exp_c(__fdiv_rn(__fsub_rn(__ldcg(p.logits + b0 + k), M), T)) : 0.0f;
    }
    int32_t token = -1, lastpos = b0;
    float run = P;
    for (int k = 0; k < nb2; ++k) {
      float val = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float t = __shfl_sync(0xFFFFFFFFu, ev[e], k >> 3);
        if ((k & 7) == e) val = t;
      }
      if (val > 0.0f) lastpos = b0 + k;
      if (!from_end && token < 0) {
        run = __fadd_rn(run, val);
        if (run > tau) token = b0 + k;
      }
    }
    if (token < 0) token = lastpos;
    if (lane == 0) {
      finalize_token(p, st, token);
      *p.argkey = 0ull;
      *p.sample_ctr = 0u;
    }
  }
}

// ---------------------------------------------------------------- the kernel

__device__ bool grid_barrier(const Params& p, Ctl* ctl, uint32_t c, uint32_t G, int& bidx) {
  consumer_sync();
  if (threadIdx.x == 0) {
    const bool skip = (int)c == p.skip_cta && bidx == p.skip_barrier;
    const bool was_aborted = aborted(ctl);
    if (!grid_arrive_wait(p.bar_ctr, G, !skip, !was_aborted, p.wait_ns)) set_error(p, ctl, DE_BARRIER_TIMEOUT);
    if (!aborted(ctl) && *(volatile int32_t*)p.err != 0) *(volatile int32_t*)&ctl->abort = 1;
  }
  ++bidx;
  consumer_sync();
  return !aborted(ctl);
}

template <int WDT>
__device__ void run_gemv(const Params& p, Ctl* ctl, uint8_t* ring, float* xbuf, const PhaseDesc& P, const Step& st,
                         uint32_t c, uint32_t G, int cw, int lane, uint32_t& t) {
  switch (P.kind) {
    case PK_QKV:
    case PK_GU:
      gemv_phase<2, 1, WDT, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
      break;
    case PK_WO:
    case PK_DOWN:
      gemv_phase<2, 1, WDT, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
      break;
    case PK_LM:
      gemv_phase<4, 1, WDT, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
      break;
    default:
      break;
  }
}

template <int SLOTS>
__device__ void run_expert(const Params& p, Ctl* ctl, uint8_t* ring, float* xbuf, const PhaseDesc& P, const Step& st,
                           uint32_t c, uint32_t G, int cw, int lane, uint32_t& t) {
  if (P.kind == PK_EGU)
    gemv_phase<2, SLOTS, DT_E4M3, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
  else
    gemv_phase<1, SLOTS, DT_E4M3, true>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
}

__device__ void consumer(const Params& p, Ctl* ctl, uint8_t* ring, float* xbuf, const Step& st, uint32_t c,
                         uint32_t G, int ph0, int ph1, bool use_barrier, int cw, int lane) {
  uint32_t t = 0;
  int bidx = 0;
  int sel_layer = -1;
  for (int ph = ph0; ph < ph1; ++ph) {
    const PhaseDesc P = p.phases[ph];
    const int L = P.layer;
    const bool ab = aborted(ctl);
    // ---- prologue: the GEMV input vector into shared memory
    switch (P.kind) {
      case PK_QKV: {
        const void* emb = L == 0 ? (const uint8_t*)p.tok_emb + (size_t)st.token * p.d * (p.wdt == DT_E4M3 ? 1 : 2)
                                 : nullptr;
        if (L == 0 && !ab) {
          const int a = (int)((long long)c * p.d / G), b = (int)((long long)(c + 1) * p.d / G);
          for (int i = a + cw * 32 + lane; i < b; i += kConsumerWarps * 32)
            __stcg(p.x + i, load_elem(emb, (size_t)i, p.wdt));
        }
        if (p.trace && c == 0 && !ab) {
          for (int i = cw * 32 + lane; i < p.d; i += kConsumerWarps * 32)
            p.trace[(size_t)L * p.d + i] = emb ? load_elem(emb, (size_t)i, p.wdt) : __ldcg(p.x + i);
        }
        rmsnorm_prologue(p, ctl, xbuf, p.attn_norm[L], emb, cw, lane);
        break;
      }
      case PK_WO: copy_prologue(xbuf, p.attn, p.hq * p.hd, cw, lane); break;
      case PK_DOWN: copy_prologue(xbuf, p.h, p.ff, cw, lane); break;
      case PK_EDOWN:
        if (sel_layer != L) {
          if (cw == 0 && lane == 0) {
            select_experts(p, ctl, L);
            mbar_arrive(&ctl->sel_bar);
          }
          sel_layer = L;
        }
        copy_prologue(xbuf, p.h, p.topk * p.fexp, cw, lane);
        break;
      case PK_GU:
      case PK_ROUTER: rmsnorm_prologue(p, ctl, xbuf, p.ffn_norm[L], nullptr, cw, lane); break;
      case PK_EGU: {
        if (cw == 0 && lane == 0) {
          select_experts(p, ctl, L);
          if (c == 0 && !ab) for (int i = 0; i < p.topk; ++i) p.sel_out[L * p.topk + i] = ctl->sel[i];
          mbar_arrive(&ctl->sel_bar);  // release the choice to the producer
        }
        sel_layer = L;
        rmsnorm_prologue(p, ctl, xbuf, p.ffn_norm[L], nullptr, cw, lane);
        break;
      }
      case PK_LM: {
        if (p.trace && c == 0 && !ab)
          for (int i = cw * 32 + lane; i < p.d; i += kConsumerWarps * 32)
            p.trace[(size_t)p.L * p.d + i] = __ldcg(p.x + i);
        rmsnorm_prologue(p, ctl, xbuf, p.final_norm, nullptr, cw, lane);
        break;
      }
      default: break;
    }
    // ---- body
    if (P.kind == PK_ATTN) {
      if (p.hd == 128) attention_phase<16>(p, ctl, P, st, c, G, cw, lane);
      else if (p.hd == 64) attention_phase<8>(p, ctl, P, st, c, G, cw, lane);
      else attention_phase<32>(p, ctl, P, st, c, G, cw, lane);
    } else if (P.kind == PK_SAMPLE) {
      if (st.temperature > 0.0f) sample_phase(p, ctl, st, c, G, cw, lane);
    } else if (P.kind == PK_EGU || P.kind == PK_EDOWN) {
      switch (p.topk) {
        case 1: run_expert<1>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t); break;
        case 2: run_expert<2>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t); break;
        case 4: run_expert<4>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t); break;
        default: run_expert<8>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t); break;
      }
    } else if (P.kind == PK_ROUTER) {
      if (p.rdt == DT_BF16) gemv_phase<1, 1, DT_BF16, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
      else gemv_phase<1, 1, DT_F16, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
    } else {
      if (p.wdt == DT_BF16) run_gemv<DT_BF16>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
      else run_gemv<DT_F16>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t);
    }
    // ---- the LM head's last CTA picks the greedy token
    if (P.kind == PK_LM && ctl->flag && st.temperature <= 0.0f && cw == 0 && lane == 0) {
      __threadfence();
      const unsigned long long key = atomicAdd(p.argkey, 0ull);
      finalize_token(p, st, (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull)));
      *p.argkey = 0ull;
      *p.lm_ctr = 0u;
    } else if (P.kind == PK_LM && ctl->flag && cw == 0 && lane == 0) {
      *p.lm_ctr = 0u;  // sampling: the maximum stays in argkey for the sampling phase
    }
    // ---- grid barrier between dependent phases
    if (use_barrier && ph + 1 < ph1) {
      const bool need = !(P.kind == PK_LM && st.temperature <= 0.0f);
      if (need) grid_barrier(p, ctl, c, G, bidx);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const Params p, int32_t ph0, int32_t ph1, int32_t use_barrier, int32_t xbuf_floats) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* xbuf = reinterpret_cast<float*>(smem + (size_t)kSlots * kSlotBytes);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)kSlots * kSlotBytes + (((size_t)xbuf_floats * 4 + 127) & ~(size_t)127));
  const uint32_t c = blockIdx.x, G = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], kConsumerWarps);
    }
    mbar_init(&ctl->sel_bar, 1);
    ctl->abort = *(volatile int32_t*)p.err != 0 ? 1 : 0;
    ctl->flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (*(volatile int32_t*)&ctl->abort) return;  // sticky device error: nothing runs until reset
  Step st;
  {
    const StepState* s = p.state;
    st.pos = __ldcg(&s->pos);
    st.seq_index = __ldcg(&s->seq_index);
    st.temperature = __ldcg(&s->temperature);
    st.token = p.tok_seq ? __ldcg(p.tok_seq + st.seq_index) : __ldcg(&s->token);
    st.u = p.u_seq ? __ldcg(p.u_seq + st.seq_index) : __ldcg(&s->u);
  }
  if (warp == kConsumerWarps) {
    if (lane == 0) producer(p, ctl, ring, c, G, ph0, ph1);
  } else {
    consumer(p, ctl, ring, xbuf, st, c, G, ph0, ph1, use_barrier != 0, warp, lane);
  }
}

}  // namespace adp

namespace adp {

// Host-side launchers of the decode kernel.
cudaError_t decode_prepare(size_t smem_bytes, int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_kernel, kThreads, smem_bytes);
}

cudaError_t decode_launch(const Params& p, int ph0, int ph1, bool persistent, int grid, size_t smem_bytes,
                          int xbuf_floats, cudaStream_t stream) {
  int32_t a0 = ph0, a1 = ph1, ub = persistent ? 1 : 0, xf = xbuf_floats;
  void* args[] = {(void*)&p, &a0, &a1, &ub, &xf};
  if (persistent)
    return cudaLaunchCooperativeKernel((const void*)decode_kernel, dim3(grid), dim3(kThreads), args, smem_bytes, stream);
  return cudaLaunchKernel((const void*)decode_kernel, dim3(grid), dim3(kThreads), args, smem_bytes, stream);
}

}  // namespace adp

namespace adp {
size_t ctl_bytes() { return sizeof(Ctl); }
}  // namespace adp

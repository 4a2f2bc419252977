// Small-batch decode: nb (<= kMaxBatch) independent requests of one model, each with its own KV
// cache and position, advance one token each per step of one persistent kernel.  The weight
// stream is the single-request kernel's (same tiles, same producer warp); every weight vector a
// consumer lane loads from the ring is multiplied into nb input vectors, so each weight byte
// read from HBM serves nb tokens.
//
// Pages followed (title, section):
//  "標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒": the batch-1 step streams every
//   active weight once per token ("GPU推論の速度制限要因：メモリ帯域幅"); one GPU-resident program
//   runs the whole decode path ("Kog Inference Engineの特徴とイノベーション"); in the translated
//   comment thread the authors answer on batching: small batches are planned, traded against
//   per-request speed.
//
// Per request the arithmetic is the single-request kernel's contract, unchanged: the same
// lane-partial dot products in the same order, RMSNorm, RoPE, attention blocks of 32 positions,
// the block merge, SwiGLU, argmax and inverse-CDF sampling.  So request r's tokens, logits and
// KV rows are bit-identical to decoding it alone.  What differs is only who computes what:
//  - GEMV phases: acc[r][row] for every request in one pass over the tile; the input vectors of
//    all requests sit in shared memory one after the other (nb x K floats, split layout);
//  - attention items are (request, KV group, block) and the merger of (request r, head h) is
//    CTA G-1-(r*hq+h);
//  - the epilogues write request r's outputs from lane r (or lanes r*ROWS+j);
//  - the LM head keeps one running argmax per request; sampling runs per request.
#include "decode_core.cuh"

namespace adp {

// Per-request state of the step, in shared memory (each CTA keeps its own identical copy).
struct Req {
  int32_t pos, token, seq_index;
  float temperature, u;
  int32_t nblk;  // attention blocks of this step: ceil((pos + 1) / 32)
  int32_t pad0, pad1;
};

// Batched kernel's shared-memory block after the phase and share tables.
struct BCtl {
  Req rq[kMaxBatch];
  float rope_cs[kMaxBatch][128], rope_sn[kMaxBatch][128];  // RoPE rows of each request's position
  float xres[kMaxBatch][64];                               // residual rows this CTA updates
  float rnorm[kMaxBatch];                                  // 1 / rms of each request's input
  unsigned long long red_k[kConsumerWarps][kMaxBatch];     // per-warp argmax keys (LM head)
  int32_t any_sample;                                      // some request samples (temperature > 0)
  int32_t down_seg;  // elements of each request's down-projection input staged at once (< ff: segments)
};

__device__ __forceinline__ BCtl* bctl_of(const Ctl* ctl, int n_phases) {
  return reinterpret_cast<BCtl*>(reinterpret_cast<uint8_t*>(share_table(ctl, n_phases)) +
                                 (((size_t)n_phases * sizeof(int2) + 15) & ~(size_t)15));
}

// The element of a register array at a lane-dependent index (every index is a compile-time one).
template <int N>
__device__ __forceinline__ float pick(const float (&a)[N], int i) {
  float y = a[0];
#pragma unroll
  for (int k = 1; k < N; ++k)
    if (i == k) y = a[k];
  return y;
}

// Floats of one request's GEMV input vector in shared memory (split layout, padded to 256).
__device__ __forceinline__ int vec_stride(int n) { return (n + 255) & ~255; }

// Request r's token / step outputs, and its tagged token word for the next step of the launch.
__device__ void finalize_request(const Params& p, const BCtl* bc, int r, uint32_t ebase, int32_t token) {
  const uint32_t next = ebase + (uint32_t)p.n_phases;
  const Req& q = bc->rq[r];
  *p.epoch = next;
  StepState* s = p.state + r;
  s->out_token = token;
  if (p.out_seq) p.out_seq[(size_t)q.seq_index * p.nb + r] = token;
  s->token = token;
  s->pos = q.pos + 1;
  s->seq_index = q.seq_index + 1;
  __threadfence();
  ll_store(p.tok_word + r, ll_pack_bits((uint32_t)token, next));
}

// rmsnorm(x_r) * gain for every request into xbuf (request r at r * vec_stride(d)).  x_r is the
// residual published by phase `x_epoch`, or, for layer 0, the request's embedding row.
__device__ void rmsnorm_batch(const Params& p, Ctl* ctl, BCtl* bc, float* xbuf, const void* gain, bool emb,
                              uint32_t x_epoch, int cw, int lane) {
  const int d = p.d, nb = p.nb, Kp = vec_stride(d);
  const int tid = cw * 32 + lane;
  constexpr int T = kConsumerWarps * 32;
  uint16_t gr[kPrologueRegs];
#pragma unroll
  for (int k = 0; k < kPrologueRegs; ++k) {
    const int i = tid + k * T;
    gr[k] = i < d ? __ldg(reinterpret_cast<const unsigned short*>(gain) + i) : (uint16_t)0;
  }
  if (emb) {
    for (int r = 0; r < nb; ++r) {
      const void* row = (const uint8_t*)p.tok_emb + (size_t)bc->rq[r].token * d * 2;
      for (int i = tid; i < d; i += T) xbuf[r * Kp + xpos(i)] = load_elem(row, (size_t)i, p.edt);
    }
    consumer_sync();
  } else {
    ll_fetch(p, ctl, xbuf, p.x, nb * d, d, Kp, x_epoch, tid);
  }
  if (cw < nb) {
    const float* xr = xbuf + cw * Kp;
    float acc = 0.0f;
    for (int v = lane; v < d / 8; v += 32) {
      float x8[8];
      load_xs8(xr, v, x8);
      acc = fma8(x8, x8, acc);
    }
    const float ss = warp_fold(acc);
    const float mean = __fdiv_rn(ss, (float)d);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, p.eps)));
    if (lane == 0) bc->rnorm[cw] = r;
  }
  consumer_sync();
  for (int r = 0; r < nb; ++r) {
    const float rr = bc->rnorm[r];
    float* xr = xbuf + r * Kp;
#pragma unroll
    for (int k = 0; k < kPrologueRegs; ++k) {
      const int i = tid + k * T;
      if (i < d) {
        const float g = p.edt == DT_BF16 ? bf16_bits_to_f32(gr[k]) : __half2float(__ushort_as_half(gr[k]));
        xr[xpos(i)] = __fmul_rn(__fmul_rn(xr[xpos(i)], rr), g);
      }
    }
  }
  consumer_sync();
}

// The residual rows this CTA's units update, for every request (visible after the next
// consumer_sync).
__device__ void stage_residual_batch(const Params& p, Ctl* ctl, BCtl* bc, const PhaseDesc& P, int rows_per_unit,
                                     uint32_t x_epoch, int tid) {
  int32_t u0, n;
  cta_share(p, ctl, P, u0, n);
  const int rows = n * rows_per_unit;
  if (tid < p.nb * rows) {
    const int r = tid / rows, k = tid % rows;
    const ll_t* src = p.x + (size_t)r * p.d + (size_t)u0 * rows_per_unit + k;
    ll_t w = ll_load(src);
    if (ll_wait(src, x_epoch, w, p, ctl)) bc->xres[r][k] = ll_value(w);
  }
}

// One GEMV phase for nb requests: each weight vector of the tile, loaded once, meets every
// request's input vector.  Per (request, row) the dot product is the contract's: lane l takes
// vectors l, l + 32, ... in order with fused multiply-adds, then the fixed butterfly.
// The down projection's input may be staged in segments of down_seg elements per request (when
// nb whole vectors would leave the ring too few slots): at the chunk where the next segment starts,
// every consumer warp has finished the previous one, and the segment's words (epoch e_src) replace
// it; the chunks, and so the operations of every dot product, keep their order.
// A segment of seg words of the down projection's input for each of the n / seg requests (request
// r's words at src + r ff) once each carries `epoch`, into xbuf in the split layout (request r at
// r segp), as ll_fetch does for whole vectors (eight loads in flight per thread; ends with
// consumer_sync).  Out of line: inlined into the GEMV loop, where every accumulator is live, its
// loads in flight pushed an accumulator array to local memory.
__device__ __noinline__ void fetch_down_segment(const Params& p, Ctl* ctl, float* xbuf, const ll_t* src, int n, int seg,
                                                int segp, uint32_t epoch, int tid) {
  constexpr int B = 8, T = kConsumerWarps * 32;
  auto at = [=](int i) { return src + (size_t)(i / seg) * p.ff + i % seg; };
  for (int base = tid; base < n; base += B * T) {
    ll_t w[B];
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int i = base + k * T;
      w[k] = i < n ? ll_load(at(i)) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int i = base + k * T;
      if (i < n) {
        if (ll_epoch(w[k]) != epoch) {
          if (!ll_wait(at(i), epoch, w[k], p, ctl)) break;
#pragma unroll
          for (int j = k + 1; j < B; ++j) {  // the later words of the batch: reload those still behind
            const int ij = base + j * T;
            if (ij < n && ll_epoch(w[j]) != epoch) w[j] = ll_load(at(ij));
          }
        }
        xbuf[(i / seg) * segp + xpos(i % seg)] = ll_value(w[k]);
      }
    }
  }
  consumer_sync();
}

template <int ROWS, int WDT, bool SEG>
__device__ __forceinline__ void gemv_batch(const Params& p, Ctl* ctl, BCtl* bc, uint8_t* ring, float* xbuf,
                                           const PhaseDesc& Pd, uint32_t c, uint32_t G, int cw, int lane,
                                           uint32_t& t_io, uint32_t ew, uint32_t e_src) {
  constexpr int EB = WDT == DT_E4M3 ? 1 : 2;
  constexpr int NA = kMaxBatch * ROWS;
  constexpr bool kScaled = WDT == DT_E4M3 || WDT == DT_NVFP4;  // per-row scales after the fold
  const int kind = Pd.kind, L = Pd.layer, K = Pd.K, KC = Pd.KC, n_chunks = Pd.n_chunks, upr = Pd.upr;
  const int dseg = SEG ? bc->down_seg : K;
  const bool segd = SEG && ROWS == 2 && kind == PK_DOWN && dseg < K;
  const int Kp = vec_stride(segd ? dseg : K);
  int seg_cur = 0, seg_k0 = 0;  // the staged segment of the down input (segment 0 from the prologue)
  const int nb = p.nb;
  const uint64_t wait_ns = p.wait_ns;
  const uint32_t ns = (uint32_t)p.nslots;
  uint32_t slot = t_io & 0xFFu, par = t_io >> 8;
  int32_t u0, n;
  cta_share(p, ctl, Pd, u0, n);
  unsigned long long best[kMaxBatch];  // LM: running maximum of this warp, per request
#pragma unroll
  for (int r = 0; r < kMaxBatch; ++r) best[r] = 0ull;
  const int rounds = n > 0 ? (n + upr - 1) / upr : 0;
  for (int rd = 0; rd < rounds; ++rd) {
    const int m = min(upr, n - rd * upr);
    const bool active = cw < m;
    const int unit = u0 + rd * upr + cw;
    float acc[NA];
#pragma unroll
    for (int i = 0; i < NA; ++i) acc[i] = 0.0f;
    // e4m3 and NVFP4 layer matrices: this unit's row scales, applied after the fold (as for one
    // request)
    float sc[ROWS];
    if constexpr (kScaled) {
      if (active) {
        int mi, r0, rstep = 1;
        if (kind == PK_QKV) {
          const int half = p.hd / 2, nq = p.hq * half, nk = p.hkv * half;
          const int uu = unit < nq ? unit : unit < nq + nk ? unit - nq : unit - nq - nk;
          mi = unit < nq ? 0 : unit < nq + nk ? 1 : 2;
          r0 = (uu / half) * p.hd + uu % half;
          rstep = half;
        } else if (kind == PK_GU) {
          mi = 4;
          r0 = unit;
          rstep = 0;
        } else {
          mi = kind == PK_WO ? 3 : 6;
          r0 = unit * ROWS;
        }
        const float* tab = p.wscale[mi][L];
#pragma unroll
        for (int j = 0; j < ROWS; ++j)
          sc[j] = (kind == PK_GU) ? __ldg(p.wscale[4 + j][L] + r0) : __ldg(tab + r0 + j * rstep);
      }
    }
    for (int ck = 0; ck < n_chunks; ++ck) {
      if (SEG && ROWS == 2 && segd && (ck * KC) / dseg != seg_cur) {
        consumer_sync();  // no warp reads the previous segment any more
        seg_cur = (ck * KC) / dseg;
        seg_k0 = seg_cur * dseg;
        const int len = min(dseg, K - seg_k0);
        fetch_down_segment(p, ctl, xbuf, p.h + seg_k0, nb * len, len, Kp, e_src, cw * 32 + lane);
      }
      const bool ok = mbar_wait(&ctl->full[slot], par, &ctl->abort, wait_ns);
      if (!ok) {
        if (lane == 0 && !aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
        __syncwarp();
      }
      if (rd == 0 && ck == 0 && cw == 0 && lane == 0) stamp(p, c, Pd.index, 8);
      if (active && ok) {
        const int kck = min(KC, K - ck * KC);
        const int nvec = kck >> 3;
        const int xv = (ck * KC - seg_k0) >> 3;
        if constexpr (WDT == DT_NVFP4) {
          // [m * ROWS rows][kck / 2] code bytes, then [m * ROWS][kck / 16] block scales; per 8-element
          // vector the products summed from zero, times the block scale, into the lane partial (the
          // single-request contract, per request)
          const uint8_t* base = ring + (size_t)slot * kSlotBytes;
          const uint8_t* codes = base + (size_t)cw * ROWS * (kck >> 1);
          const uint8_t* bsc = base + (size_t)m * ROWS * (kck >> 1) + (size_t)cw * ROWS * (kck >> 4);
          for (int v = lane; v < nvec; v += 32) {
            float w[ROWS][8], bs[ROWS];
#pragma unroll
            for (int j = 0; j < ROWS; ++j) {
              load8_e2m1(*reinterpret_cast<const uint32_t*>(codes + (size_t)j * (kck >> 1) + (size_t)v * 4), w[j]);
              bs[j] = e4m3_to_f32(bsc[(size_t)j * (kck >> 4) + (v >> 1)]);
            }
            // each request's input vector read once for all rows of the unit
#pragma unroll
            for (int r = 0; r < kMaxBatch; ++r) {
              if (r < nb) {
                float x8[8];
                load_xs8(xbuf + r * Kp, xv + v, x8);
#pragma unroll
                for (int j = 0; j < ROWS; ++j) acc[r * ROWS + j] = fmaf(bs[j], fma8(w[j], x8, 0.0f), acc[r * ROWS + j]);
              }
            }
          }
        } else {
        const uint8_t* tile = ring + (size_t)slot * kSlotBytes + (size_t)cw * ROWS * kck * EB;
        for (int v = lane; v < nvec; v += 32) {
          float w[ROWS][8];
#pragma unroll
          for (int j = 0; j < ROWS; ++j) load8<WDT>(tile + ((size_t)j * kck + (size_t)v * 8) * EB, w[j]);
#pragma unroll
          for (int r = 0; r < kMaxBatch; ++r) {
            if (r < nb) {
              float x8[8];
              load_xs8(xbuf + r * Kp, xv + v, x8);
#pragma unroll
              for (int j = 0; j < ROWS; ++j) acc[r * ROWS + j] = fma8(w[j], x8, acc[r * ROWS + j]);
            }
          }
        }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[slot]);
      if (++slot == ns) {
        slot = 0;
        par ^= 1u;
      }
    }
    if (rd == rounds - 1 && cw == 0 && lane == 0) stamp(p, c, Pd.index, 9);
    if (!active || aborted(ctl)) continue;
#pragma unroll
    for (int r = 0; r < kMaxBatch; ++r)
      if (r < nb)
#pragma unroll
        for (int j = 0; j < ROWS; ++j) {
          acc[r * ROWS + j] = warp_fold(acc[r * ROWS + j]);
          if constexpr (kScaled) acc[r * ROWS + j] = __fmul_rn(sc[j], acc[r * ROWS + j]);
        }
    // ---- epilogues (every lane holds every folded sum)
    if (kind == PK_QKV) {
      if (lane < nb) {
        const int r = lane;
        const int half = p.hd / 2;
        const int nq = p.hq * half, nk = p.hkv * half;
        const float a = pick(acc, 2 * r), b = pick(acc, 2 * r + 1);
        const int pos = bc->rq[r].pos;
        if (unit < nq + nk) {
          const bool isq = unit < nq;
          const int uu = isq ? unit : unit - nq;
          const int head = uu / half, i = uu % half;
          const float cs = bc->rope_cs[r][i];
          const float sn = bc->rope_sn[r][i];
          const float a2 = fmaf(a, cs, -__fmul_rn(b, sn));
          const float b2 = fmaf(b, cs, __fmul_rn(a, sn));
          if (isq) {
            ll_t* q = p.q + (size_t)r * p.hq * p.hd + head * p.hd;
            ll_store(q + i, ll_pack(a2, ew));
            ll_store(q + i + half, ll_pack(b2, ew));
          } else {
            uint16_t* kc = p.kcb[r];
            const size_t row = (((size_t)L * p.hkv + head) * p.max_ctx + pos) * p.hd;
            const uint16_t ka = round_kv(a2, p.kvdt), kb = round_kv(b2, p.kvdt);
            kc[row + i] = ka;
            kc[row + i + half] = kb;
            ll_t* kn = p.knew + (size_t)r * p.hkv * p.hd + head * p.hd;
            ll_store(kn + i, ll_pack_bits(ka, ew));
            ll_store(kn + i + half, ll_pack_bits(kb, ew));
          }
        } else {
          const int uu = unit - nq - nk;
          const int head = uu / half, i = uu % half;
          uint16_t* vc = p.vcb[r];
          const size_t row = (((size_t)L * p.hkv + head) * p.max_ctx + pos) * p.hd;
          const uint16_t va = round_kv(a, p.kvdt), vb = round_kv(b, p.kvdt);
          vc[row + i] = va;
          vc[row + i + half] = vb;
          ll_t* vn = p.vnew + (size_t)r * p.hkv * p.hd + head * p.hd;
          ll_store(vn + i, ll_pack_bits(va, ew));
          ll_store(vn + i + half, ll_pack_bits(vb, ew));
        }
      }
    } else if (kind == PK_WO || kind == PK_DOWN) {
      if (lane < nb * ROWS) {
        const int r = lane / ROWS, j = lane % ROWS;
        const int row = unit * ROWS + j;
        const float y = pick(acc, lane);
        ll_store(p.x + (size_t)r * p.d + row, ll_pack(__fadd_rn(bc->xres[r][row - u0 * ROWS], y), ew));
      }
    } else if (kind == PK_GU) {
      if (lane < nb) ll_store(p.h + (size_t)lane * p.ff + unit, ll_pack(silu_mul(pick(acc, 2 * lane), pick(acc, 2 * lane + 1)), ew));
    } else if (kind == PK_LM) {
      // (compiled only where the LM head runs: 4-row units of a 16-bit matrix)
      if constexpr (ROWS == 4 && !kScaled) {
        if (lane == 0) {
#pragma unroll
          for (int r = 0; r < kMaxBatch; ++r) {
            if (r < nb) {
#pragma unroll
              for (int j = 0; j < ROWS; ++j) {
                const int row = unit * ROWS + j;
                __stcg(p.logits + (size_t)r * p.V + row, acc[r * ROWS + j]);
                const unsigned long long k = argmax_key(acc[r * ROWS + j], (uint32_t)row);
                best[r] = k > best[r] ? k : best[r];
              }
            }
          }
        }
      }
    }
  }
  if constexpr (ROWS == 4 && !kScaled) {
    if (kind == PK_LM) {
      if (lane == 0)
#pragma unroll
        for (int r = 0; r < kMaxBatch; ++r) bc->red_k[cw][r] = best[r];
      consumer_sync();
      if (cw == 0 && lane == 0) {
        if (!aborted(ctl)) {
          for (int r = 0; r < nb; ++r) {
            unsigned long long k = 0ull;
            for (int w = 0; w < kConsumerWarps; ++w) k = bc->red_k[w][r] > k ? bc->red_k[w][r] : k;
            if (k) atomicMax(p.argkey + r, k);
          }
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
  t_io = slot | (par << 8);
}

// The K/V blocks of this CTA's attention items of layer L for every request, into L2 during the
// layer's QKV phase.
__device__ __forceinline__ void prefetch_attention_kv_batch(const Params& p, const BCtl* bc, int L, uint32_t c,
                                                            uint32_t G) {
  int base = 0;  // item index of the request's first item
  for (int r = 0; r < p.nb; ++r) {
    const int ctx = bc->rq[r].pos + 1;
    const int items = p.hkv * bc->rq[r].nblk;
    const uint16_t* kc = p.kcb[r];
    const uint16_t* vc = p.vcb[r];
    for (int it = ((int)c - base % (int)G + (int)G) % (int)G; it < items; it += (int)G) {
      const int g = it % p.hkv, b = it / p.hkv;
      const int j0 = b * kAttnBlock;
      const uint32_t bytes = (uint32_t)min(kAttnBlock, ctx - j0) * p.hd * 2;
      const size_t cache0 = (((size_t)L * p.hkv + g) * p.max_ctx + j0) * p.hd;
      prefetch_l2(kc + cache0, bytes);
      prefetch_l2(vc + cache0, bytes);
    }
    base += items;
  }
}

// Attention for every request: items (request r, KV group g, block b) over all CTAs, each item
// one warp per query head of the group on the block's 32 cached positions (staged in shared
// memory by TMA); the block partials (m_b, l_b, o_b) are published as tagged words and merged
// per (request, head) by CTA G-1-(r*hq+h) in block order, as in the single-request kernel.
template <int HD, int KVDT>
__device__ __forceinline__ void attention_batch(const Params& p, Ctl* ctl, BCtl* bc, float* xbuf, const PhaseDesc& P,
                                                uint32_t ebase, uint32_t c, uint32_t G, int cw, int lane,
                                                uint32_t& att_uses_io, uint32_t& merge_uses, uint32_t ew) {
  constexpr int NV = HD / 8;
  constexpr int KSTR = HD + 8;
  constexpr int DPL = HD / 32;
  const int L = P.layer;
  const int nbmax = p.nbmax, max_ctx = p.max_ctx, nb = p.nb;
  const int slots = p.att_slots, gmax = p.att_gmax, slot_bytes = p.att_slot_bytes;
  const float scale = p.attn_scale;
  const uint64_t wait_ns = p.wait_ns;
  const uint32_t qe = ebase + 1 + (uint32_t)P.src_ph;
  const int hq = p.hq, hkv = p.hkv;
  uint32_t att_uses = att_uses_io;
  int items = 0;
  for (int r = 0; r < nb; ++r) items += hkv * bc->rq[r].nblk;
  const int tid = cw * 32 + lane;
  const int slot = cw / gmax, hh = cw % gmax;
  if (slot < slots && !aborted(ctl)) {
    uint8_t* stg = reinterpret_cast<uint8_t*>(xbuf) + (size_t)slot * slot_bytes;
    uint16_t* SK = reinterpret_cast<uint16_t*>(stg);
    uint16_t* SV = SK + kAttnBlock * KSTR;
    float* SQ = reinterpret_cast<float*>(SV + kAttnBlock * HD);
    float* SS = SQ + kMaxGroup * HD;
    for (int it = (int)c + (int)G * slot; it < items; it += (int)G * slots) {
      int r = 0, rem = it;
      while (r < nb - 1 && rem >= hkv * bc->rq[r].nblk) {
        rem -= hkv * bc->rq[r].nblk;
        ++r;
      }
      const int ctx = bc->rq[r].pos + 1;
      const int g = rem % hkv, b = rem / hkv;
      int h0, h1;
      group_heads(g, hq, hkv, h0, h1);
      const bool active = hh < h1 - h0;
      const int h = h0 + hh;
      const int j0 = b * kAttnBlock;
      const int nvalid = min(kAttnBlock, ctx - j0);
      const size_t cache0 = (((size_t)L * hkv + g) * max_ctx + j0) * HD;
      const uint32_t bytes = (uint32_t)nvalid * HD * 2;
      const uint16_t* kc = p.kcb[r];
      const uint16_t* vc = p.vcb[r];
      if (hh == 0) {
        if (lane == 0) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          mbar_arrive_expect_tx(&ctl->att_bar[slot], 2 * bytes);
          tma_load_1d(SV, vc + cache0, bytes, &ctl->att_bar[slot], policy_evict_first());
        }
        __syncwarp();
        if (lane < nvalid)
          tma_load_1d(SK + (size_t)lane * KSTR, kc + cache0 + (size_t)lane * HD, HD * 2, &ctl->att_bar[slot],
                      policy_evict_first());
      }
      float* sq = SQ + hh * HD;
      if (active) {
        const ll_t* qs = p.q + ((size_t)r * hq + h) * HD;
        ll_t w[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) w[i] = ll_load(qs + lane + 32 * i);
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          if (ll_epoch(w[i]) != qe) {
            if (!ll_wait(qs + lane + 32 * i, qe, w[i], p, ctl)) break;
#pragma unroll
            for (int j = i + 1; j < DPL; ++j)
              if (ll_epoch(w[j]) != qe) w[j] = ll_load(qs + lane + 32 * j);
          }
          sq[lane + 32 * i] = ll_value(w[i]);
        }
      }
      bool ok = mbar_wait(&ctl->att_bar[slot], att_uses & 1, &ctl->abort, wait_ns);
      ++att_uses;
      if (!ok && lane == 0 && !aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
      if (hh == 0 && j0 + nvalid == ctx) {
        // the block holding this step's position: its K/V row comes from the tagged copies
        const int jr = ctx - 1 - j0;
        const ll_t* kn = p.knew + ((size_t)r * hkv + g) * HD + lane;
        const ll_t* vn = p.vnew + ((size_t)r * hkv + g) * HD + lane;
        ll_t w[2 * DPL];
#pragma unroll
        for (int i = 0; i < 2 * DPL; ++i) w[i] = ll_load(i < DPL ? kn + 32 * i : vn + 32 * (i - DPL));
#pragma unroll
        for (int i = 0; i < 2 * DPL; ++i) {
          if (ll_epoch(w[i]) != qe) {
            if (!ll_wait(i < DPL ? kn + 32 * i : vn + 32 * (i - DPL), qe, w[i], p, ctl)) break;
#pragma unroll
            for (int j = i + 1; j < 2 * DPL; ++j)
              if (ll_epoch(w[j]) != qe) w[j] = ll_load(j < DPL ? kn + 32 * j : vn + 32 * (j - DPL));
          }
          if (i < DPL) SK[(size_t)jr * KSTR + lane + 32 * i] = (uint16_t)w[i];
          else SV[(size_t)jr * HD + lane + 32 * (i - DPL)] = (uint16_t)w[i];
        }
      }
      asm volatile("bar.sync %0, %1;" ::"r"(2 + slot), "r"(gmax * 32) : "memory");
      ok = ok && !aborted(ctl);
      if (active && ok) {
        float sj = __int_as_float(0xFF800000);  // -inf
        if (lane < nvalid) {
          float a[32];
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            float k8[8], q8[8];
            kv8<KVDT>(*reinterpret_cast<const uint4*>(SK + (size_t)lane * KSTR + v * 8), k8);
            load_x8(sq + v * 8, q8);
            a[v] = fma8(k8, q8, 0.0f);
          }
#pragma unroll
          for (int v = NV; v < 32; ++v) a[v] = 0.0f;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
            for (int i = 0; i < off; ++i) a[i] = __fadd_rn(a[i], a[i + off]);
          sj = __fmul_rn(a[0], scale);
        }
        float m = sj;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
        float* se = SS + hh * kAttnBlock;
        se[lane] = lane < nvalid ? exp_c(__fsub_rn(sj, m)) : 0.0f;
        __syncwarp();
        float l = 0.0f, o[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[i] = 0.0f;
        const uint16_t* vcol = SV + lane * DPL;
        for (int jb = 0; jb < nvalid; jb += 8) {
          float vv[8][DPL], ee[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int j = min(jb + k, nvalid - 1);
            kv_dims_smem<KVDT, DPL>(vcol + (size_t)j * HD, vv[k]);
            ee[k] = se[j];
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (jb + k < nvalid) {
              l = __fadd_rn(l, ee[k]);
#pragma unroll
              for (int i = 0; i < DPL; ++i) o[i] = fmaf(ee[k], vv[k][i], o[i]);
            }
          }
        }
        const size_t pb = ((size_t)r * hq + h) * nbmax + b;
        if (lane == 0) {
          ll_store(p.part_m + pb, ll_pack(m, ew));
          ll_store(p.part_l + pb, ll_pack(l, ew));
        }
#pragma unroll
        for (int i = 0; i < DPL; ++i) ll_store(p.part_o + pb * HD + lane * DPL + i, ll_pack(o[i], ew));
      }
      asm volatile("bar.sync %0, %1;" ::"r"(2 + slot), "r"(gmax * 32) : "memory");
    }
  }
  consumer_sync();
  // Merge of (request r, head h) on CTA G-1-(r*hq+h): block weights w_b = exp(m_b - M),
  // L = sum_b w_b l_b and o_d = (sum_b w_b o_bd) / L, both sums in block order.
  const int mi = (int)G - 1 - (int)c;
  if (mi >= 0 && mi < nb * hq && !aborted(ctl)) {
    const int r = mi / hq, h = mi % hq;
    const int nbk = bc->rq[r].nblk;
    const size_t pb0 = ((size_t)r * hq + h) * nbmax;
    float* Wm = xbuf;
    float* Wl = xbuf + nbmax;
    constexpr int T = kConsumerWarps * 32;
    for (int i = tid; i < 2 * nbk; i += T) {
      const ll_t* src = i < nbk ? p.part_m + pb0 + i : p.part_l + pb0 + (i - nbk);
      ll_t x = ll_load(src);
      if (ll_wait(src, ew, x, p, ctl)) (i < nbk ? Wm[i] : Wl[i - nbk]) = ll_value(x);
    }
    consumer_sync();
    ll_t* So = reinterpret_cast<ll_t*>(xbuf + ((2 * nbmax + 2 + 3) & ~3));
    const int batch = (int)(((size_t)p.xbuf_floats - (size_t)((2 * nbmax + 2 + 3) & ~3)) * 4 / ((size_t)HD * 8));
    auto issue = [&](int b0) {
      const int k = min(batch, nbk - b0);
      asm volatile("fence.proxy.async.global;" ::: "memory");
      mbar_arrive_expect_tx(&ctl->merge_bar, (uint32_t)k * HD * 8);
      tma_load_1d(So, p.part_o + (pb0 + b0) * HD, (uint32_t)k * HD * 8, &ctl->merge_bar, policy_evict_first());
    };
    if (tid == 0) issue(0);
    if (cw == 0) {
      float M = __int_as_float(0xFF800000);
      for (int bb = lane; bb < nbk; bb += 32) M = fmaxf(M, Wm[bb]);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
      for (int bb = lane; bb < nbk; bb += 32) Wm[bb] = exp_c(__fsub_rn(Wm[bb], M));
      __syncwarp();
      if (lane == 0) {
        float Ls = 0.0f;
        for (int bb = 0; bb < nbk; ++bb) Ls = fmaf(Wm[bb], Wl[bb], Ls);
        Wl[nbmax] = Ls;
      }
    }
    consumer_sync();
    float O = 0.0f;
    bool ok = true;
    for (int b0 = 0; b0 < nbk; b0 += batch) {
      const int k = min(batch, nbk - b0);
      ok = ok && mbar_wait(&ctl->merge_bar, merge_uses & 1, &ctl->abort, wait_ns);
      ++merge_uses;
      if (!ok && tid == 0 && !aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
      if (ok && tid < HD) {
        for (int t2 = 0; t2 < k && ok; ++t2) {
          ll_t x = So[(size_t)t2 * HD + tid];
          if (ll_epoch(x) != ew) ok = ll_wait(p.part_o + (pb0 + b0 + t2) * HD + tid, ew, x, p, ctl);
          O = fmaf(Wm[b0 + t2], ll_value(x), O);
        }
      }
      if (b0 + k < nbk) {
        consumer_sync();
        if (tid == 0) issue(b0 + k);
      }
    }
    if (ok && tid < HD) ll_store(p.attn + ((size_t)r * hq + h) * HD + tid, ll_pack(__fdiv_rn(O, Wl[nbmax]), ew));
  }
  att_uses_io = att_uses;
}

// Inverse-CDF sampling for the requests with temperature > 0: items (request, vocabulary block
// of 256); the CTA that completes a request's last block picks its token, as in the
// single-request kernel.
__device__ __forceinline__ void sample_batch(const Params& p, Ctl* ctl, BCtl* bc, uint32_t ebase, uint32_t c,
                                             uint32_t G, int cw, int lane) {
  const int V = p.V, nb = p.nb;
  const int nblk = (V + kVocabBlock - 1) / kVocabBlock;
  const int stride = (int)G * kConsumerWarps;
  for (int it = cw * (int)G + (int)c; it < nb * nblk; it += stride) {
    if (aborted(ctl)) break;
    const int r = it / nblk, blk = it % nblk;
    const float T = bc->rq[r].temperature;
    if (!(T > 0.0f)) continue;
    const float* lg = p.logits + (size_t)r * V;
    float* sblock = p.sblock + (size_t)r * nblk;
    const unsigned long long key = __ldcg(p.argkey + r);
    const float M = order_float((uint32_t)(key >> 32));
    const int i0 = blk * kVocabBlock;
    const int nn = min(kVocabBlock, V - i0);
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = lane * 8 + e;
      if (k < nn) acc = fmaf(exp_c(__fdiv_rn(__fsub_rn(__ldcg(lg + i0 + k), M), T)), 1.0f, acc);
    }
    const float Sb = warp_fold(acc);
    if (lane == 0) __stcg(sblock + blk, Sb);
    __threadfence();
    __syncwarp();
    uint32_t last = 0;
    if (lane == 0) last = atomicAdd(p.sample_ctr + r, 1u) == (uint32_t)(nblk - 1) ? 1u : 0u;
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    __threadfence();
    // several warps of a CTA may each complete a request here: the block sums are read from L2,
    // not staged in the CTA's shared memory
    float Z = 0.0f;
    for (int b = 0; b < nblk; ++b) Z = __fadd_rn(Z, __ldcg(sblock + b));
    const float tau = __fmul_rn(bc->rq[r].u, Z);
    float P = 0.0f;
    int bstar = -1;
    for (int b = 0; b < nblk; ++b) {
      const float Pn = __fadd_rn(P, __ldcg(sblock + b));
      if (Pn > tau) {
        bstar = b;
        break;
      }
      P = Pn;
    }
    bool from_end = false;
    if (bstar < 0) {
      from_end = true;
      bstar = 0;
      for (int b = nblk - 1; b >= 0; --b)
        if (__ldcg(sblock + b) > 0.0f) {
          bstar = b;
          break;
        }
    }
    const int b0 = bstar * kVocabBlock;
    const int nb2 = min(kVocabBlock, V - b0);
    float ev[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = lane * 8 + e;
      ev[e] = k < nb2 ? exp_c(__fdiv_rn(__fsub_rn(__ldcg(lg + b0 + k), M), T)) : 0.0f;
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
      p.argkey[r] = 0ull;
      p.sample_ctr[r] = 0u;
      finalize_request(p, bc, r, ebase, token);
    }
  }
}

template <int WDT, bool SEG>
__device__ void run_gemv_batch(const Params& p, Ctl* ctl, BCtl* bc, uint8_t* ring, float* xbuf, const PhaseDesc& P,
                               uint32_t c, uint32_t G, int cw, int lane, uint32_t& t, uint32_t ew, uint32_t e_src) {
  if (P.kind == PK_LM) gemv_batch<4, WDT, false>(p, ctl, bc, ring, xbuf, P, c, G, cw, lane, t, ew, e_src);
  else gemv_batch<2, WDT, SEG>(p, ctl, bc, ring, xbuf, P, c, G, cw, lane, t, ew, e_src);
}

template <bool SEG>
__device__ void consumer_batch(const Params& p, Ctl* ctl, BCtl* bc, uint8_t* ring, float* xbuf, uint32_t ebase,
                               uint32_t c, uint32_t G, int ph0, int ph1, bool use_barrier, int cw, int lane) {
  uint32_t t = 0;
  int bidx = 0;
  uint32_t att_uses = 0, merge_uses = 0;
  const int tid = cw * 32 + lane;
  const int nb = p.nb;
  constexpr int T = kConsumerWarps * 32;
  for (int step = 0; step < p.n_steps; ++step) {
    if (step > 0) {
      // the next step of the launch: each request's position advances by one and its token is
      // the one the last step chose for it (or the next of the given sequence)
      ebase += (uint32_t)p.n_phases;
      if (tid < nb) {
        Req& q = bc->rq[tid];
        q.pos += 1;
        q.seq_index += 1;
        q.nblk = (q.pos + 1 + kAttnBlock - 1) / kAttnBlock;
        if (p.u_seq) q.u = __ldcg(p.u_seq + (size_t)q.seq_index * nb + tid);
        if (p.tok_seq) {
          q.token = __ldcg(p.tok_seq + (size_t)q.seq_index * nb + tid);
        } else {
          ll_t w = ll_load(p.tok_word + tid);
          q.token = ll_wait(p.tok_word + tid, ebase, w, p, ctl) ? (int32_t)(uint32_t)w : 0;
        }
      }
      consumer_sync();
    }
    for (int ph = ph0; ph < ph1; ++ph) {
      if (ph > ph0 || step > 0) consumer_sync();
      const PhaseDesc P = phase_table(ctl)[ph];
      const int L = P.layer;
      const bool ab = aborted(ctl);
      const uint32_t ew = ((int)c == p.skip_cta && ph == p.skip_phase) ? 0u : ebase + 1 + (uint32_t)ph;
      const uint32_t e_src = ebase + 1 + (uint32_t)P.src_ph;
      const uint32_t e_res = ebase + 1 + (uint32_t)P.res_ph;
      int32_t u0, n;
      cta_share(p, ctl, P, u0, n);
      if (cw == 0 && lane == 0) stamp(p, c, ph, 0);
      switch (P.kind) {
        case PK_QKV: {
          if (L == 0 && !ab) {  // each residual starts as its request's embedding row
            const int a = (int)((long long)c * p.d / G), b = (int)((long long)(c + 1) * p.d / G);
            for (int r = 0; r < nb; ++r) {
              const void* row = (const uint8_t*)p.tok_emb + (size_t)bc->rq[r].token * p.d * 2;
              for (int i = a + tid; i < b; i += T) ll_store(p.x + (size_t)r * p.d + i, ll_pack(load_elem(row, (size_t)i, p.edt), ew));
            }
          }
          if (cw == kConsumerWarps - 1 && lane == 0 && !ab) prefetch_attention_kv_batch(p, bc, L, c, G);
          if (n > 0) {
            const int half = p.hd / 2;
            for (int i = tid; i < nb * half; i += T) {
              const int r = i / half, k = i % half;
              const size_t o = (size_t)bc->rq[r].pos * half + k;
              bc->rope_cs[r][k] = __ldg(p.rope_cos + o);
              bc->rope_sn[r][k] = __ldg(p.rope_sin + o);
            }
            rmsnorm_batch(p, ctl, bc, xbuf, p.attn_norm[L], L == 0, e_src, cw, lane);
          }
          break;
        }
        case PK_WO:
          if (n > 0) {
            stage_residual_batch(p, ctl, bc, P, 2, e_res, tid);
            ll_fetch(p, ctl, xbuf, p.attn, nb * p.hq * p.hd, p.hq * p.hd, vec_stride(p.hq * p.hd), e_src, tid);
          }
          break;
        case PK_DOWN:
          if (n > 0) {
            stage_residual_batch(p, ctl, bc, P, 2, e_res, tid);
            // the whole input, or its first segment (the GEMV fetches the others)
            if (SEG && bc->down_seg < p.ff)
              fetch_down_segment(p, ctl, xbuf, p.h, nb * bc->down_seg, bc->down_seg, vec_stride(bc->down_seg), e_src,
                                 tid);
            else
              ll_fetch(p, ctl, xbuf, p.h, nb * p.ff, p.ff, vec_stride(p.ff), e_src, tid);
          }
          break;
        case PK_GU:
          if (n > 0) rmsnorm_batch(p, ctl, bc, xbuf, p.ffn_norm[L], false, e_src, cw, lane);
          break;
        case PK_LM:
          if (n > 0) rmsnorm_batch(p, ctl, bc, xbuf, p.final_norm, false, e_src, cw, lane);
          break;
        default:
          break;
      }
      if (cw == 0 && lane == 0) stamp(p, c, ph, 1);
      if (P.kind == PK_ATTN) {
        if (p.kvdt == DT_BF16) {
          if (p.hd == 128) attention_batch<128, DT_BF16>(p, ctl, bc, xbuf, P, ebase, c, G, cw, lane, att_uses, merge_uses, ew);
          else if (p.hd == 64) attention_batch<64, DT_BF16>(p, ctl, bc, xbuf, P, ebase, c, G, cw, lane, att_uses, merge_uses, ew);
          else attention_batch<256, DT_BF16>(p, ctl, bc, xbuf, P, ebase, c, G, cw, lane, att_uses, merge_uses, ew);
        } else {
          if (p.hd == 128) attention_batch<128, DT_F16>(p, ctl, bc, xbuf, P, ebase, c, G, cw, lane, att_uses, merge_uses, ew);
          else if (p.hd == 64) attention_batch<64, DT_F16>(p, ctl, bc, xbuf, P, ebase, c, G, cw, lane, att_uses, merge_uses, ew);
          else attention_batch<256, DT_F16>(p, ctl, bc, xbuf, P, ebase, c, G, cw, lane, att_uses, merge_uses, ew);
        }
      } else if (P.kind == PK_SAMPLE) {
        if (bc->any_sample) sample_batch(p, ctl, bc, ebase, c, G, cw, lane);
      } else if (p.wdt == DT_E4M3 && P.kind != PK_LM) {
        gemv_batch<2, DT_E4M3, SEG>(p, ctl, bc, ring, xbuf, P, c, G, cw, lane, t, ew, e_src);
      } else if (p.wdt == DT_NVFP4 && P.kind != PK_LM) {
        gemv_batch<2, DT_NVFP4, SEG>(p, ctl, bc, ring, xbuf, P, c, G, cw, lane, t, ew, e_src);
      } else if ((P.kind == PK_LM ? p.edt : p.wdt) == DT_BF16) {
        run_gemv_batch<DT_BF16, SEG>(p, ctl, bc, ring, xbuf, P, c, G, cw, lane, t, ew, e_src);
      } else {
        run_gemv_batch<DT_F16, SEG>(p, ctl, bc, ring, xbuf, P, c, G, cw, lane, t, ew, e_src);
      }
      // ---- the LM head's last CTA picks the greedy requests' tokens
      if (P.kind == PK_LM && ctl->flag && cw == 0 && lane == 0) {
        __threadfence();
        *p.lm_ctr = 0u;
        // each key is cleared before its token is published (finalize_request fences): the next
        // step's LM head starts only after every request's token word has arrived
        for (int r = 0; r < nb; ++r) {
          if (!(bc->rq[r].temperature > 0.0f)) {
            const unsigned long long key = atomicAdd(p.argkey + r, 0ull);
            p.argkey[r] = 0ull;
            finalize_request(p, bc, r, ebase, (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull)));
          }
        }
      }
      if (cw == 0 && lane == 0) stamp(p, c, ph, 2);
      if (use_barrier && ph + 1 < ph1 && ((P.kind == PK_LM && bc->any_sample) || p.debug_barriers))
        grid_barrier(p, ctl, c, G, bidx);
      if (cw == 0 && lane == 0) stamp(p, c, ph, 3);
    }
  }
}

// SEG: the down projection's input staged in segments (down_seg < ff; an instantiation of its own,
// so that batches whose inputs fit whole run none of that code).
template <bool SEG>
__global__ void __launch_bounds__(kThreads, 1)
    decode_batch_kernel(const __grid_constant__ Params p, int32_t ph0, int32_t ph1, int32_t use_barrier,
                        int32_t xbuf_floats, int32_t down_seg) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* xbuf = reinterpret_cast<float*>(smem + (size_t)p.nslots * kSlotBytes);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)p.nslots * kSlotBytes + (((size_t)xbuf_floats * 4 + 127) & ~(size_t)127));
  const uint32_t c = blockIdx.x, G = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BCtl* bc = bctl_of(ctl, p.n_phases);
  cta_setup(p, ctl);
  if (threadIdx.x == 0) bc->down_seg = down_seg;
  if (threadIdx.x < (unsigned)p.nb) {
    const int r = threadIdx.x;
    const StepState* s = p.state + r;
    Req& q = bc->rq[r];
    q.pos = __ldcg(&s->pos);
    q.seq_index = __ldcg(&s->seq_index);
    q.temperature = __ldcg(&s->temperature);
    q.token = p.tok_seq ? __ldcg(p.tok_seq + (size_t)q.seq_index * p.nb + r) : __ldcg(&s->token);
    q.u = p.u_seq ? __ldcg(p.u_seq + (size_t)q.seq_index * p.nb + r) : __ldcg(&s->u);
    q.nblk = (q.pos + 1 + kAttnBlock - 1) / kAttnBlock;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int any = 0;
    for (int r = 0; r < p.nb; ++r) any |= bc->rq[r].temperature > 0.0f ? 1 : 0;
    bc->any_sample = any;
  }
  __syncthreads();
  if (*(volatile int32_t*)&ctl->abort) return;  // sticky device error: nothing runs until reset
  const uint32_t ebase = __ldcg(p.epoch);
  if (warp == kConsumerWarps) {
    if (lane == 0) producer(p, ctl, ring, c, G, ph0, ph1);
  } else {
    consumer_batch<SEG>(p, ctl, bc, ring, xbuf, ebase, c, G, ph0, ph1, use_barrier != 0, warp, lane);
  }
}

}  // namespace adp

namespace adp {

cudaError_t decode_batch_prepare(size_t smem_bytes, int* blocks_per_sm) {
  int bmin = 1 << 30;
  for (const void* k : {(const void*)decode_batch_kernel<false>, (const void*)decode_batch_kernel<true>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return e;
    int b = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, kThreads, smem_bytes)) != cudaSuccess) return e;
    bmin = b < bmin ? b : bmin;
  }
  *blocks_per_sm = bmin;
  return cudaSuccess;
}

cudaError_t decode_batch_launch(const Params& p, int ph0, int ph1, int grid, size_t smem_bytes, int xbuf_floats,
                                int down_seg, cudaStream_t stream) {
  int32_t a0 = ph0, a1 = ph1, ub = 1, xf = xbuf_floats, ds = down_seg;
  void* args[] = {(void*)&p, &a0, &a1, &ub, &xf, &ds};
  const void* k = down_seg < p.ff ? (const void*)decode_batch_kernel<true> : (const void*)decode_batch_kernel<false>;
  return cudaLaunchCooperativeKernel(k, dim3(grid), dim3(kThreads), args, smem_bytes, stream);
}

size_t batch_ctl_bytes() { return sizeof(BCtl); }

}  // namespace adp

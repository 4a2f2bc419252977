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

#include "decode_core.cuh"

namespace adp {


// xn = rmsnorm(x) * gain into xbuf (all consumer warps; ends with consumer_sync).  x is the
// residual as published by phase `x_epoch`, or, for layer 0, the token's embedding row.
__device__ void rmsnorm_prologue(const Params& p, Ctl* ctl, float* xbuf, const void* gain, const void* emb_row,
                                 uint32_t x_epoch, int trace_layer, uint32_t c, int cw, int lane) {
  const int d = p.d;
  const int tid = cw * 32 + lane;
  constexpr int T = kConsumerWarps * 32;
  uint16_t gr[kPrologueRegs];  // gains kept in their 16-bit storage form
#pragma unroll
  for (int k = 0; k < kPrologueRegs; ++k) {
    const int i = tid + k * T;
    gr[k] = i < d ? __ldg(reinterpret_cast<const unsigned short*>(gain) + i) : (uint16_t)0;
  }
  if (emb_row) {
    for (int i = tid; i < d; i += T) xbuf[xpos(i)] = load_elem(emb_row, (size_t)i, p.edt);
    consumer_sync();
  } else {
    ll_fetch(p, ctl, xbuf, p.x, d, d, 0, x_epoch, tid);
  }
  if (p.trace && c == 0 && trace_layer >= 0)
    for (int i = tid; i < d; i += T) p.trace[(size_t)trace_layer * d + i] = xbuf[xpos(i)];
  if (cw == 0) {
    float acc = 0.0f;
    for (int v = lane; v < d / 8; v += 32) {
      float x8[8];
      load_xs8(xbuf, v, x8);
      acc = fma8(x8, x8, acc);
    }
    const float ss = warp_fold(acc);
    const float mean = __fdiv_rn(ss, (float)d);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, p.eps)));
    if (lane == 0) ctl->bcast = r;
  }
  consumer_sync();
  const float r = ctl->bcast;
#pragma unroll
  for (int k = 0; k < kPrologueRegs; ++k) {
    const int i = tid + k * T;
    if (i < d) {
      const float g = p.edt == DT_BF16 ? bf16_bits_to_f32(gr[k]) : __half2float(__ushort_as_half(gr[k]));
      xbuf[xpos(i)] = __fmul_rn(__fmul_rn(xbuf[xpos(i)], r), g);
    }
  }
  consumer_sync();
}

// The residual row this thread stages for the CTA's units (rows_per_unit rows each): fetched
// alongside the phase's input vector, into shared memory, so that the epilogue does not wait for
// a load.
__device__ __forceinline__ SideWord residual_word(const Params& p, Ctl* ctl, const PhaseDesc& P, int rows_per_unit,
                                                  uint32_t x_epoch, int tid) {
  int32_t u0, n;
  cta_share(p, ctl, P, u0, n);
  if (tid >= n * rows_per_unit) return SideWord{nullptr, nullptr, 0};
  return SideWord{p.x + (size_t)u0 * rows_per_unit + tid, &ctl->xres[tid], x_epoch};
}

// Router softmax + top-k (ties to the lower index), gates renormalised over the choice; forced
// experts (test hook) keep the router's probabilities of those experts.  Called by a whole warp,
// lane-parallel: the logits are staged in shared memory in one batch; lane l computes
// e_i = exp(r_i - M) and then P_i = e_i / Z for experts i = l, l + 32, ...; lane 0 forms
// Z = sum_i e_i sequentially in expert order; each of the top_k choices is a warp argmax over
// (P_i, lowest index) of the experts not yet chosen; lane 0 sums the chosen P in slot order and
// divides.  Every value is the same operation on the same operands as a sequential evaluation.
// local: the CTA computed the router logits itself and left them in ctl->stage (the router phase
// ran in this launch); else they are fetched from the published words.
__device__ void select_experts(const Params& p, Ctl* ctl, int layer, uint32_t r_epoch, int lane, bool local) {
  const int E = p.E, K = p.topk;
  float* st = ctl->stage;
  if (!local) {
    for (int e = lane; e < E; e += 32) {
      ll_t w = ll_load(p.rlog + e);
      st[e] = ll_wait(p.rlog + e, r_epoch, w, p, ctl) ? ll_value(w) : 0.0f;
    }
  }
  __syncwarp();
  float M = __int_as_float(0xFF800000);
  for (int e = lane; e < E; e += 32) M = fmaxf(M, st[e]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
  for (int e = lane; e < E; e += 32) st[e] = exp_c(__fsub_rn(st[e], M));
  __syncwarp();
  float Z = 0.0f;
  if (lane == 0) {
    int e = 0;
    for (; e + 8 <= E; e += 8) {  // eight loads in flight, then the sums in expert order
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = st[e + k];
#pragma unroll
      for (int k = 0; k < 8; ++k) Z = __fadd_rn(Z, v[k]);
    }
    for (; e < E; ++e) Z = __fadd_rn(Z, st[e]);
  }
  Z = __shfl_sync(0xFFFFFFFFu, Z, 0);
  for (int e = lane; e < E; e += 32) st[e] = __fdiv_rn(st[e], Z);  // P_e
  __syncwarp();
  float Zs = 0.0f;
  for (int i = 0; i < K; ++i) {
    int best;
    if (p.force_sel) {
      best = p.force_sel[layer * K + i];
    } else {
      unsigned long long key = 0ull;  // chosen experts hold -1 and never win
      for (int e = lane; e < E; e += 32) {
        const unsigned long long k = argmax_key(st[e], (uint32_t)e);
        key = k > key ? k : key;
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, key, off);
        key = o > key ? o : key;
      }
      best = (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
    }
    const float bp = st[best];
    __syncwarp();
    if (lane == 0) {
      ctl->sel[i] = best;
      ctl->gate[i] = bp;  // probability for now
      Zs = __fadd_rn(Zs, bp);
      if (!p.force_sel) st[best] = -1.0f;
    }
    __syncwarp();
  }
  if (lane == 0)
    for (int i = 0; i < K; ++i) ctl->gate[i] = __fdiv_rn(ctl->gate[i], Zs);
  __syncwarp();
}

// ---------------------------------------------------------------- GEMV phases

template <int ROWS, int SLOTS, int WDT, bool XPERSLOT>
__device__ __forceinline__ void gemv_phase(const Params& p, Ctl* ctl, uint8_t* ring, float* xbuf, const PhaseDesc& Pd,
                                        const Step& st, uint32_t c, uint32_t G, int cw, int lane, uint32_t& t_io,
                                        uint32_t ew) {
  // every field the loops use lives in registers (the descriptors are in local memory, and each
  // mbarrier asm statement would otherwise force them to be reloaded)
  constexpr int EB = WDT == DT_E4M3 ? 1 : 2;  // element bytes (NVFP4 tiles are addressed apart)
  const int kind = Pd.kind, L = Pd.layer, K = Pd.K, KC = Pd.KC, n_chunks = Pd.n_chunks, upr = Pd.upr;
  const int Kp = (K + 255) & ~255;  // floats per input vector in the split layout
  const int pos = st.pos;
  const uint64_t wait_ns = p.wait_ns;
  const uint32_t ns = (uint32_t)p.nslots;
  // the consumer's ring cursor: slot of its next tile (low byte) and that slot's use parity
  uint32_t slot = t_io & 0xFFu, par = t_io >> 8;
  int32_t u0, n;
  cta_share(p, ctl, Pd, u0, n);
  unsigned long long best = 0ull;  // LM: packed running maximum of this warp
  long long cyc_wait = 0, cyc_comp = 0, cyc_epi = 0;  // timeline: SM cycles waiting / computing / epilogues
  const int rounds = n > 0 ? (n + upr - 1) / upr : 0;
  const long long cyc_start = cyc_now();
  for (int r = 0; r < rounds; ++r) {
    const int m = min(upr, n - r * upr);
    const bool active = cw < m;
    const int unit = u0 + r * upr + cw;
    float acc[SLOTS * ROWS];
#pragma unroll
    for (int i = 0; i < SLOTS * ROWS; ++i) acc[i] = 0.0f;
    // e4m3 and NVFP4 layer matrices: the per-row scales of this unit, loaded now, applied after
    // the dot
    constexpr bool kScaled = (WDT == DT_E4M3 || WDT == DT_NVFP4) && SLOTS == 1;
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
          rstep = 0;  // gate row `unit` (scale table 4), up row `unit` (table 5)
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
      const long long cy0 = cyc_now();
      // the wait itself gives up when another warp has aborted the step
      const bool ok = mbar_wait(&ctl->full[slot], par, &ctl->abort, wait_ns);
      const long long cy1 = cyc_now();
      cyc_wait += cy1 - cy0;
      if (!ok) {
        if (lane == 0 && !aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
        __syncwarp();
      }
      if (r == 0 && ck == 0 && cw == 0 && lane == 0) stamp(p, c, Pd.index, 8);
      if (active && ok) {
        const int kck = min(KC, K - ck * KC);
        const int nvec = kck >> 3;
        const uint32_t slot_bytes = (uint32_t)m * ROWS * kck * EB;
        const uint8_t* tile = ring + (size_t)slot * kSlotBytes;
        const int xoff = ck * KC;
        if constexpr (WDT == DT_NVFP4) {
          // [m * ROWS rows][kck / 2] code bytes, then [m * ROWS][kck / 16] block scales.  Per
          // 8-element vector: the element products fused-multiply-added from zero, then that sum
          // times its block scale added into the lane partial.
          const uint8_t* codes = tile + (size_t)cw * ROWS * (kck >> 1);
          const uint8_t* bsc = tile + (size_t)m * ROWS * (kck >> 1) + (size_t)cw * ROWS * (kck >> 4);
          auto vec4 = [&](int v, const float (&x8)[8]) {
            if constexpr (ROWS % 2 == 0) {
              // rows j and j + 1 share each instruction: packed fp32 FMAs (two independent IEEE fmas)
#pragma unroll
              for (int j = 0; j < ROWS; j += 2) {
                float wa[8], wb[8];
                load8_e2m1(*reinterpret_cast<const uint32_t*>(codes + (size_t)j * (kck >> 1) + (size_t)v * 4), wa);
                load8_e2m1(*reinterpret_cast<const uint32_t*>(codes + (size_t)(j + 1) * (kck >> 1) + (size_t)v * 4),
                           wb);
                const float2 bs = make_float2(e4m3_to_f32(bsc[(size_t)j * (kck >> 4) + (v >> 1)]),
                                              e4m3_to_f32(bsc[(size_t)(j + 1) * (kck >> 4) + (v >> 1)]));
                const float2 t = fma8x2(wa, wb, x8, make_float2(0.0f, 0.0f));
                const float2 a = __ffma2_rn(bs, t, make_float2(acc[j], acc[j + 1]));
                acc[j] = a.x;
                acc[j + 1] = a.y;
              }
            } else {
#pragma unroll
              for (int j = 0; j < ROWS; ++j) {
                float w8[8];
                load8_e2m1(*reinterpret_cast<const uint32_t*>(codes + (size_t)j * (kck >> 1) + (size_t)v * 4), w8);
                const float bs = e4m3_to_f32(bsc[(size_t)j * (kck >> 4) + (v >> 1)]);
                acc[j] = fmaf(bs, fma8(w8, x8, 0.0f), acc[j]);
              }
            }
          };
          for (int v = lane; v < nvec; v += 32) {
            float x8[8];
            load_xs8(xbuf, (xoff >> 3) + v, x8);
            vec4(v, x8);
          }
        } else {
          for (int v = lane; v < nvec; v += 32) {
            float x8[8];
            if (!XPERSLOT) load_xs8(xbuf, (xoff >> 3) + v, x8);
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
              if (XPERSLOT) load_xs8(xbuf + s * Kp, (xoff >> 3) + v, x8);
              if constexpr (ROWS % 2 == 0) {
                // rows j and j + 1 share each instruction: packed fp32 FMAs (two independent IEEE fmas)
#pragma unroll
                for (int j = 0; j < ROWS; j += 2) {
                  float wa[8], wb[8];
                  load8<WDT>(tile + (size_t)s * slot_bytes + ((size_t)(cw * ROWS + j) * kck + (size_t)v * 8) * EB, wa);
                  load8<WDT>(tile + (size_t)s * slot_bytes + ((size_t)(cw * ROWS + j + 1) * kck + (size_t)v * 8) * EB,
                             wb);
                  const float2 a = fma8x2(wa, wb, x8, make_float2(acc[s * ROWS + j], acc[s * ROWS + j + 1]));
                  acc[s * ROWS + j] = a.x;
                  acc[s * ROWS + j + 1] = a.y;
                }
              } else {
#pragma unroll
                for (int j = 0; j < ROWS; ++j) {
                  float w8[8];
                  load8<WDT>(tile + (size_t)s * slot_bytes + ((size_t)(cw * ROWS + j) * kck + (size_t)v * 8) * EB, w8);
                  acc[s * ROWS + j] = fma8(w8, x8, acc[s * ROWS + j]);
                }
              }
            }
          }
        }
      }
      cyc_comp += cyc_now() - cy1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[slot]);
      if (++slot == ns) {
        slot = 0;
        par ^= 1u;
      }
    }
    if (r == rounds - 1 && cw == 0 && lane == 0) {
      stamp(p, c, Pd.index, 9);
      if (p.timeline) {
        p.timeline[((size_t)c * p.n_phases + Pd.index) * kStamps + 12] = (unsigned long long)cyc_wait;
        p.timeline[((size_t)c * p.n_phases + Pd.index) * kStamps + 13] = (unsigned long long)cyc_comp;
      }
    }
    const long long ce0 = cyc_now();
    if (!active || aborted(ctl)) continue;
#pragma unroll
    for (int i = 0; i < SLOTS * ROWS; ++i) acc[i] = warp_fold(acc[i]);
    if constexpr (kScaled) {
#pragma unroll
      for (int j = 0; j < ROWS; ++j) acc[j] = __fmul_rn(sc[j], acc[j]);
    }
    // ---- epilogues
    if (kind == PK_QKV) {
      if (lane == 0) {
        const int half = p.hd / 2;
        const int nq = p.hq * half, nk = p.hkv * half;
        const float a = acc[0], b = acc[1];
        if (unit < nq + nk) {
          const bool isq = unit < nq;
          const int uu = isq ? unit : unit - nq;
          const int head = uu / half, i = uu % half;
          const float cs = ctl->rope_cs[i];
          const float sn = ctl->rope_sn[i];
          const float a2 = fmaf(a, cs, -__fmul_rn(b, sn));
          const float b2 = fmaf(b, cs, __fmul_rn(a, sn));
          if (isq) {
            ll_store(p.q + head * p.hd + i, ll_pack(a2, ew));
            ll_store(p.q + head * p.hd + i + half, ll_pack(b2, ew));
          } else {
            const size_t row = (((size_t)L * p.hkv + head) * p.max_ctx + pos) * p.hd;
            const uint16_t ka = round_kv(a2, p.kvdt), kb = round_kv(b2, p.kvdt);
            p.kc[row + i] = ka;
            p.kc[row + i + half] = kb;
            ll_store(p.knew + head * p.hd + i, ll_pack_bits(ka, ew));
            ll_store(p.knew + head * p.hd + i + half, ll_pack_bits(kb, ew));
          }
        } else {
          const int uu = unit - nq - nk;
          const int head = uu / half, i = uu % half;
          const size_t row = (((size_t)L * p.hkv + head) * p.max_ctx + pos) * p.hd;
          const uint16_t va = round_kv(a, p.kvdt), vb = round_kv(b, p.kvdt);
          p.vc[row + i] = va;
          p.vc[row + i + half] = vb;
          ll_store(p.vnew + head * p.hd + i, ll_pack_bits(va, ew));
          ll_store(p.vnew + head * p.hd + i + half, ll_pack_bits(vb, ew));
        }
      }
    } else if (kind == PK_WO || kind == PK_DOWN) {
      if (lane < ROWS) {
        const int row = unit * ROWS + lane;
        float y = acc[0];
#pragma unroll
        for (int j = 1; j < ROWS; ++j) if (lane == j) y = acc[j];
        ll_store(p.x + row, ll_pack(__fadd_rn(ctl->xres[row - u0 * ROWS], y), ew));
      }
    } else if (kind == PK_GU) {
      if (lane == 0) ll_store(p.h + unit, ll_pack(silu_mul(acc[0], acc[1]), ew));
    } else if (kind == PK_ROUTER) {
      // every CTA computes every logit (a replicated phase): into shared memory for its own
      // choice of experts; CTA 0 also publishes them, for a launch that starts at the expert phase
      if (lane < ROWS) {
        float y = acc[0];
#pragma unroll
        for (int j = 1; j < ROWS; ++j) if (lane == j) y = acc[j];
        ctl->stage[unit * ROWS + lane] = y;
        if (c == 0) ll_store(p.rlog + unit * ROWS + lane, ll_pack(y, ew));
      }
    } else if (kind == PK_EGU) {
      if (lane < p.topk) {
        float g = acc[0], uval = acc[1];
#pragma unroll
        for (int s = 1; s < SLOTS; ++s)
          if (lane == s) { g = acc[s * ROWS]; uval = acc[s * ROWS + 1]; }
        const int e = ctl->sel[lane];
        const float sg = __ldg(p.e_gate_scale[L] + (size_t)e * p.fexp + unit);
        const float su = __ldg(p.e_up_scale[L] + (size_t)e * p.fexp + unit);
        ll_store(p.h + lane * p.fexp + unit, ll_pack(silu_mul(__fmul_rn(sg, g), __fmul_rn(su, uval)), ew));
      }
    } else if (kind == PK_EDOWN) {
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
        ll_store(p.x + unit, ll_pack(__fadd_rn(ctl->xres[unit - u0], ax), ew));
      }
    } else if (kind == PK_LM) {
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
    cyc_epi += cyc_now() - ce0;
  }
  if (p.timeline && cw == 0 && lane == 0 && rounds > 0) {
    p.timeline[((size_t)c * p.n_phases + Pd.index) * kStamps + 14] = (unsigned long long)(cyc_now() - cyc_start);
    p.timeline[((size_t)c * p.n_phases + Pd.index) * kStamps + 15] = (unsigned long long)cyc_epi;
  }
  if (kind == PK_LM) {
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
  t_io = slot | (par << 8);
}

// ---------------------------------------------------------------- finalisation

// The step's token: into the step state and output sequence for the host, and as an
// epoch-tagged word for the next step of the same launch (which every CTA waits on before it
// gathers the embedding row).  Called after the step's shared counters are reset.
__device__ void finalize_token(const Params& p, const Step& st, int32_t token) {
  const uint32_t next = st.ebase + (uint32_t)p.n_phases;  // the next step's epoch base
  *p.epoch = next;
  StepState* s = p.state;
  s->out_token = token;
  if (p.out_seq) p.out_seq[st.seq_index] = token;
  s->token = token;
  s->pos = st.pos + 1;
  s->seq_index = st.seq_index + 1;
  __threadfence();
  ll_store(p.tok_word, ll_pack_bits((uint32_t)token, next));
}

// ---------------------------------------------------------------- attention phase


// The K/V blocks of this CTA's attention items of layer L (the items the attention phase gives
// it), prefetched into L2 while the layer's QKV phase runs: they do not depend on this step
// except for the newest row, which the attention phase takes from the exchange words anyway.
__device__ __forceinline__ void prefetch_attention_kv(const Params& p, int L, int ctx, uint32_t c, uint32_t G) {
  const uint64_t pol = policy_evict_last();
  const bool last = (p.pf_flags & PF_KV_LAST) != 0;
  const int nb = (ctx + kAttnBlock - 1) / kAttnBlock;
  const int items = p.hkv * nb;
  for (int it = (int)c; it < items; it += (int)G) {
    const int g = it % p.hkv, b = it / p.hkv;
    const int j0 = b * kAttnBlock;
    const uint32_t bytes = (uint32_t)min(kAttnBlock, ctx - j0) * p.hd * 2;  // a multiple of 128
    const size_t cache0 = (((size_t)L * p.hkv + g) * p.max_ctx + j0) * p.hd;
    if (last) {
      prefetch_l2_hint(p.kc + cache0, bytes, pol);
      prefetch_l2_hint(p.vc + cache0, bytes, pol);
    } else {
      prefetch_l2(p.kc + cache0, bytes);
      prefetch_l2(p.vc + cache0, bytes);
    }
  }
}

// Attention over the KV cache, split along the sequence.  Item = (KV group g, block b of 32
// positions).  A CTA runs p.att_slots items at a time; slot s uses warps [s*gmax, (s+1)*gmax)
// (gmax = largest group), one warp per query head of the group, sharing the block's K and V
// rows that the slot's first warp fetches into the slot's staging area with two TMA bulk
// copies.  Each warp produces its head's block partial (m_b, l_b, o_b) of the contract.  The
// CTA that finishes a group's last block merges the group's blocks with all consumer warps.
template <int HD, int KVDT>
__device__ __forceinline__ void attention_phase(const Params& p, Ctl* ctl, float* xbuf, const PhaseDesc& P,
                                             const Step& st, uint32_t c, uint32_t G, int cw, int lane,
                                             uint32_t& att_uses_io, uint32_t ew) {
  constexpr int NV = HD / 8;         // 8-element vectors per K row (partial sums of the contract dot)
  constexpr int KSTR = HD + 8;       // padded K row stride in shared memory (conflict-free row reads)
  constexpr int DPL = HD / 32;       // output dims per lane in the PV pass
  // parameters in registers (see gemv_phase)
  const int L = P.layer;
  const int ctx = st.pos + 1;
  const int nbmax = p.nbmax, max_ctx = p.max_ctx;
  const int slots = p.att_slots, gmax = p.att_gmax, slot_bytes = p.att_slot_bytes;
  const float scale = p.attn_scale;
  const uint64_t wait_ns = p.wait_ns;
  const uint16_t* __restrict__ kc = p.kc;
  const uint16_t* __restrict__ vc = p.vc;
  const ll_t* qg = p.q;
  const ll_t* knew = p.knew;
  const ll_t* vnew = p.vnew;
  const uint32_t qe = st.ebase + 1 + (uint32_t)P.src_ph;  // epoch of this layer's QKV outputs
  ll_t* part_m = p.part_m;
  ll_t* part_l = p.part_l;
  ll_t* part_o = p.part_o;
  ll_t* attn = p.attn;
  uint32_t att_uses = att_uses_io;
  const int nb = (ctx + kAttnBlock - 1) / kAttnBlock;
  const int hq = p.hq, hkv = p.hkv;
  const int items = hkv * nb;
  const int tid = cw * 32 + lane;
  const int slot = cw / gmax, hh = cw % gmax;
  if (slot < slots && !aborted(ctl)) {
    uint8_t* stg = reinterpret_cast<uint8_t*>(xbuf) + (size_t)slot * slot_bytes;
    uint16_t* SK = reinterpret_cast<uint16_t*>(stg);             // [32][KSTR] K rows, padded
    uint16_t* SV = SK + kAttnBlock * KSTR;                       // [32][HD] V rows
    float* SQ = reinterpret_cast<float*>(SV + kAttnBlock * HD);  // [gmax][HD] queries
    float* SS = SQ + kMaxGroup * HD;                             // [gmax][32] weights e_j
    for (int it = (int)c + (int)G * slot; it < items; it += (int)G * slots) {
      const int g = it % hkv, b = it / hkv;
      int h0, h1;
      group_heads(g, hq, hkv, h0, h1);
      const bool active = hh < h1 - h0;
      const int h = h0 + hh;
      const int j0 = b * kAttnBlock;
      const int nvalid = min(kAttnBlock, ctx - j0);
      const size_t cache0 = (((size_t)L * hkv + g) * max_ctx + j0) * HD;
      const uint32_t bytes = (uint32_t)nvalid * HD * 2;
      if (hh == 0) {
        // the newest row was written this step by generic stores of other CTAs
        if (lane == 0) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          mbar_arrive_expect_tx(&ctl->att_bar[slot], 2 * bytes);
          tma_load_1d(SV, vc + cache0, bytes, &ctl->att_bar[slot], policy_evict_first());
        }
        __syncwarp();
        if (lane < nvalid)  // one K row per lane, into the padded layout
          tma_load_1d(SK + (size_t)lane * KSTR, kc + cache0 + (size_t)lane * HD, HD * 2, &ctl->att_bar[slot],
                      policy_evict_first());
      }
      // the block holding this step's position takes its K/V row from the tagged copies (the cache
      // row may not have landed when the bulk copy read it): those words are loaded now, with the
      // query's, so that both round trips overlap
      // Every thread of the slot takes words t, t + 32 * gmax, ... of that row (K then V, 2 * HD
      // words); the first PWE of them are loaded here.
      constexpr int PWE = 2;
      const bool patch = j0 + nvalid == ctx;
      const int tslot = hh * 32 + lane, nthr = gmax * 32;
      const ll_t* kn = knew + (size_t)g * HD;
      const ll_t* vn = vnew + (size_t)g * HD;
      auto pword = [&](int wi) { return wi < HD ? kn + wi : vn + (wi - HD); };
      ll_t pe[PWE];
#pragma unroll
      for (int k = 0; k < PWE; ++k) {
        const int wi = tslot + k * nthr;
        pe[k] = patch && wi < 2 * HD ? ll_load(pword(wi)) : 0ull;
      }
      // this head's query, staged in shared memory (read by every lane in the score pass)
      float* sq = SQ + hh * HD;
      if (active) {
        const ll_t* qs = qg + (size_t)h * HD;
        ll_t w[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) w[i] = ll_load(qs + lane + 32 * i);
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          if (ll_epoch(w[i]) != qe) {
            if (!ll_wait(qs + lane + 32 * i, qe, w[i], p, ctl)) break;
#pragma unroll
            for (int j = i + 1; j < DPL; ++j)  // reload the rest together (see ll_fetch)
              if (ll_epoch(w[j]) != qe) w[j] = ll_load(qs + lane + 32 * j);
          }
          sq[lane + 32 * i] = ll_value(w[i]);
        }
      }
      bool ok = mbar_wait(&ctl->att_bar[slot], att_uses & 1, &ctl->abort, wait_ns);
      ++att_uses;
      if (!ok && lane == 0 && !aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
      if (patch) {
        const int jr = ctx - 1 - j0;
        auto put = [&](int wi, ll_t w) {
          if (wi < HD) SK[(size_t)jr * KSTR + wi] = (uint16_t)w;
          else SV[(size_t)jr * HD + (wi - HD)] = (uint16_t)w;
        };
#pragma unroll
        for (int k = 0; k < PWE; ++k) {
          const int wi = tslot + k * nthr;
          if (wi < 2 * HD && ll_wait(pword(wi), qe, pe[k], p, ctl)) put(wi, pe[k]);
        }
        for (int wi = tslot + PWE * nthr; wi < 2 * HD; wi += nthr) {  // groups of fewer than 4 heads
          ll_t w = ll_load(pword(wi));
          if (ll_wait(pword(wi), qe, w, p, ctl)) put(wi, w);
        }
      }
      asm volatile("bar.sync %0, %1;" ::"r"(2 + slot), "r"(gmax * 32) : "memory");
      ok = ok && !aborted(ctl);
      if (cw == 0 && lane == 0 && it == (int)c) stamp(p, c, P.index, 4);
      if (active && ok) {
        const long long cs0 = cyc_now();
        // score of position j0 + lane: the contract dot over the K row, its 32-slot tree in registers
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
        const long long cs1 = cyc_now();
        // block maximum and weights e_j = exp(s_j - m_b), shared with the warp through SS
        float m = sj;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
        float* se = SS + hh * kAttnBlock;
        se[lane] = lane < nvalid ? exp_c(__fsub_rn(sj, m)) : 0.0f;
        __syncwarp();
        const long long cs2 = cyc_now();
        // l = sequential sum of e_j; o = sequential fma chain over j
        float l = 0.0f, o[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[i] = 0.0f;
        const uint16_t* vcol = SV + lane * DPL;
        if (nvalid == kAttnBlock) {  // a full block: no bounds in the chain
#pragma unroll
          for (int jb = 0; jb < kAttnBlock; jb += 8) {
            float vv[8][DPL], ee[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              kv_dims_smem<KVDT, DPL>(vcol + (size_t)(jb + k) * HD, vv[k]);
              ee[k] = se[jb + k];
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              l = __fadd_rn(l, ee[k]);
#pragma unroll
              for (int i = 0; i < DPL; ++i) o[i] = fmaf(ee[k], vv[k][i], o[i]);
            }
          }
        } else for (int jb = 0; jb < nvalid; jb += 8) {
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
        const long long cs3 = cyc_now();
        if (cw == 0 && lane == 0 && it == (int)c) stamp(p, c, P.index, 6);
        // block partial as epoch-tagged words, [head][block] and [head][block][dim]: the head's
        // merger polls them directly (no counter, no fence on this side)
        // the outputs go first and the maximum and sum after them, so that a merger that has seen
        // the block's maximum and sum usually finds its outputs in place too
#pragma unroll
        for (int i = 0; i < DPL; ++i) ll_store(part_o + ((size_t)h * nbmax + b) * HD + lane * DPL + i, ll_pack(o[i], ew));
        __syncwarp();
        if (lane == 0) {
          ll_store(part_m + (size_t)h * nbmax + b, ll_pack(m, ew));
          ll_store(part_l + (size_t)h * nbmax + b, ll_pack(l, ew));
        }
        if (cw == 0 && lane == 0 && it == (int)c) {
          stamp(p, c, P.index, 5);
          if (p.timeline) {
            unsigned long long* tl = p.timeline + ((size_t)c * p.n_phases + P.index) * kStamps;
            tl[12] = (unsigned long long)(cs1 - cs0);
            tl[13] = (unsigned long long)(cs2 - cs1);
            tl[14] = (unsigned long long)(cs3 - cs2);
            tl[15] = (unsigned long long)(cyc_now() - cs3);
          }
        }
      }
      // the slot's staging area is reused by its next item only after every warp of the slot is done
      asm volatile("bar.sync %0, %1;" ::"r"(2 + slot), "r"(gmax * 32) : "memory");
    }
  }
  consumer_sync();
  if (tid == 0) stamp(p, c, P.index, 7);
  // Merge: S CTAs merge each query head, one slice of HD / S output dimensions each: CTA
  // G-1-(h S + s) takes dimensions [s HD/S, (s+1) HD/S) of head h (after its own items, if any).
  // S = merge_split on long contexts (at least merge_split_blocks blocks), else 1: every slice
  // polls all block maxima and sums, which costs more than the split saves on few blocks.  Thread d < HD / S owns one output dimension; the block maxima and sums are staged in
  // shared memory, the weights w_b = exp(m_b - M) and L = sum_b w_b l_b computed once (every slice
  // computes the same ones), then o_d = (sum_b w_b o_bd) / L, both sums fused-multiply-added in
  // block order.  Every partial is polled by its epoch, so the merge starts as soon as the last one
  // lands.
  const int S = nb >= p.merge_split_blocks ? p.merge_split : 1;
  const int HS = HD / S, hs_log = __ffs(HS) - 1;  // HS: a power of two
  const int mi = (int)G - 1 - (int)c;
  const int h = mi >= 0 ? mi / S : -1, hs = mi >= 0 ? (mi % S) * HS : 0;
  if (h >= 0 && h < hq && !aborted(ctl)) {
    float* Wm = xbuf;           // [nb] block maxima, then weights w_b
    float* Wl = xbuf + nbmax;   // [nb] block sums; Wl[nbmax] = L
    constexpr int T = kConsumerWarps * 32;
    for (int i = tid; i < 2 * nb; i += T) {
      const ll_t* src = i < nb ? part_m + (size_t)h * nbmax + i : part_l + (size_t)h * nbmax + (i - nb);
      ll_t x = ll_load(src);
      if (ll_wait(src, ew, x, p, ctl)) (i < nb ? Wm[i] : Wl[i - nb]) = ll_value(x);
    }
    consumer_sync();
    if (tid == 0) stamp(p, c, P.index, 10);
    // Every block's maximum and sum has arrived, and each block publishes its outputs before
    // them, so the outputs almost surely have too: all consumer threads load them (eight words in
    // flight each, [block][dim]) into shared memory as fp32, while warp 0, whose own loads are in
    // flight, forms the weights.  Blocks beyond what the staging area holds come in further batches.
    float* So = xbuf + ((2 * nbmax + 2 + 3) & ~3);
    const int batch = (int)(((size_t)p.xbuf_floats - (size_t)((2 * nbmax + 2 + 3) & ~3)) / (size_t)HS);
    bool ok = true;
    auto weights = [&]() {
      float M = __int_as_float(0xFF800000);
      for (int bb = lane; bb < nb; bb += 32) M = fmaxf(M, Wm[bb]);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
      for (int bb = lane; bb < nb; bb += 32) Wm[bb] = exp_c(__fsub_rn(Wm[bb], M));
      __syncwarp();
      if (lane == 0) {
        float Ls = 0.0f;
        int bb = 0;
        for (; bb + 8 <= nb; bb += 8) {
          float wv[8], lv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            wv[k] = Wm[bb + k];
            lv[k] = Wl[bb + k];
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) Ls = fmaf(wv[k], lv[k], Ls);
        }
        for (; bb < nb; ++bb) Ls = fmaf(Wm[bb], Wl[bb], Ls);
        Wl[nbmax] = Ls;
        stamp(p, c, P.index, 12);
      }
    };
    float O = 0.0f;
    for (int b0 = 0; b0 < nb; b0 += batch) {
      const int nbk = min(batch, nb - b0);
      const ll_t* src = part_o + ((size_t)h * nbmax + b0) * HD + hs;  // word i: block i / HS, dim hs + i % HS
      auto word = [&](int i) { return src + (size_t)(i >> hs_log) * HD + (i & (HS - 1)); };
      const int nw = nbk * HS;
      constexpr int B = 8, T = kConsumerWarps * 32;
      bool first = b0 == 0;
      for (int base = tid; base < nw; base += B * T) {
        ll_t w[B];
#pragma unroll
        for (int k = 0; k < B; ++k) {
          const int i = base + k * T;
          w[k] = i < nw ? ll_load(word(i)) : 0ull;
        }
        if (first && cw == 0) weights();  // warp 0's loads are in flight meanwhile
        first = false;
#pragma unroll
        for (int k = 0; k < B; ++k) {
          const int i = base + k * T;
          if (i < nw) {
            if (ll_epoch(w[k]) != ew) {
              if (!ll_wait(word(i), ew, w[k], p, ctl)) { ok = false; break; }
#pragma unroll
              for (int j = k + 1; j < B; ++j) {  // reload the rest together (see ll_fetch)
                const int ij = base + j * T;
                if (ij < nw && ll_epoch(w[j]) != ew) w[j] = ll_load(word(ij));
              }
            }
            So[i] = ll_value(w[k]);
          }
        }
      }
      if (first && cw == 0) weights();  // a batch with fewer words than threads
      consumer_sync();
      if (tid < HS) {
        int t2 = 0;
        for (; t2 + 8 <= nbk; t2 += 8) {
          float ov[8], wv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            ov[k] = So[(size_t)(t2 + k) * HS + tid];
            wv[k] = Wm[b0 + t2 + k];
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) O = fmaf(wv[k], ov[k], O);
        }
        for (; t2 < nbk; ++t2) O = fmaf(Wm[b0 + t2], So[(size_t)t2 * HS + tid], O);
      }
      if (b0 + nbk < nb) consumer_sync();  // the staging area is reused by the next batch
    }
    ok = ok && !aborted(ctl);
    if (tid == 0) stamp(p, c, P.index, 13);
    if (ok && tid < HS) ll_store(attn + (size_t)h * HD + hs + tid, ll_pack(__fdiv_rn(O, Wl[nbmax]), ew));
    if (tid == 0) stamp(p, c, P.index, 11);
  }
  att_uses_io = att_uses;
}

// ---------------------------------------------------------------- sampling phase

__device__ __forceinline__ void sample_phase(const Params& p, Ctl* ctl, const Step& st, uint32_t c, uint32_t G, int cw, int lane) {
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
    const float Sb = warp_fold(acc);
    if (lane == 0) __stcg(p.sblock + it, Sb);
    __threadfence();
    __syncwarp();
    uint32_t last = 0;
    if (lane == 0) last = atomicAdd(p.sample_ctr, 1u) == (uint32_t)(nblk - 1) ? 1u : 0u;
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    __threadfence();
    // inverse CDF over the block sums (staged in shared memory), then within the chosen block
    float* S = ctl->stage;
    for (int b = lane; b < nblk; b += 32) S[b] = __ldcg(p.sblock + b);
    __syncwarp();
    float Z = 0.0f;
    for (int b = 0; b < nblk; ++b) Z = __fadd_rn(Z, S[b]);
    const float tau = __fmul_rn(st.u, Z);
    float P = 0.0f;
    int bstar = -1;
    for (int b = 0; b < nblk; ++b) {
      const float Pn = __fadd_rn(P, S[b]);
      if (Pn > tau) { bstar = b; break; }
      P = Pn;
    }
    bool from_end = false;
    if (bstar < 0) {  // tau rounded up to Z: take the last token with nonzero weight
      from_end = true;
      bstar = 0;
      for (int b = nblk - 1; b >= 0; --b)
        if (S[b] > 0.0f) { bstar = b; break; }
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
      *p.argkey = 0ull;
      *p.sample_ctr = 0u;
      finalize_token(p, st, token);
    }
  }
}

// ---------------------------------------------------------------- the kernel


template <int WDT>
__device__ void run_gemv(const Params& p, Ctl* ctl, uint8_t* ring, float* xbuf, const PhaseDesc& P, const Step& st,
                         uint32_t c, uint32_t G, int cw, int lane, uint32_t& t, uint32_t ew) {
  switch (P.kind) {
    case PK_QKV:
    case PK_GU:
    case PK_WO:
    case PK_DOWN:
      gemv_phase<2, 1, WDT, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
      break;
    case PK_LM:
      gemv_phase<4, 1, WDT, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
      break;
    default:
      break;
  }
}

template <int SLOTS>
__device__ void run_expert(const Params& p, Ctl* ctl, uint8_t* ring, float* xbuf, const PhaseDesc& P, const Step& st,
                           uint32_t c, uint32_t G, int cw, int lane, uint32_t& t, uint32_t ew) {
  if (P.kind == PK_EGU)
    gemv_phase<2, SLOTS, DT_E4M3, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
  else
    gemv_phase<1, SLOTS, DT_E4M3, true>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
}

// A model's specialisation: its head width, KV-cache type and the 16-bit type of its dense weights
// (16-bit models) or of its embedding and LM head (the others), fixed at compile time so that a
// kernel instantiation holds only the attention and GEMV code that model runs (SPEC 0: chosen at
// run time from the parameters, for every other combination).
constexpr int spec_code(int hd, int kvdt, int t16) { return (1 << 30) | hd | (kvdt << 16) | (t16 << 20); }
template <int SPEC>
struct Spec {
  static constexpr bool on = SPEC != 0;
  static constexpr int hd = SPEC & 0xFFFF, kvdt = (SPEC >> 16) & 0xF, t16 = (SPEC >> 20) & 0xF;
};

template <int KIND, int SPEC>
__device__ void consumer(const Params& p, Ctl* ctl, uint8_t* ring, float* xbuf, Step st, uint32_t c,
                         uint32_t G, int ph0, int ph1, bool use_barrier, int cw, int lane) {
  using S = Spec<SPEC>;
  uint32_t t = 0;
  int bidx = 0;
  int sel_layer = -1;
  uint32_t att_uses = 0;
  const int tid = cw * 32 + lane;
  constexpr bool MOE = KIND == KK_MOE;
  for (int step = 0; step < p.n_steps; ++step) {
    if (step > 0) {
      // the next step of this launch: its position, epochs and inputs follow from the last one,
      // except the token, which the step's last CTA publishes
      st.ebase += (uint32_t)p.n_phases;
      st.pos += 1;
      st.seq_index += 1;
      if (p.u_seq) st.u = __ldcg(p.u_seq + st.seq_index);
      if (p.tok_seq) {
        st.token = __ldcg(p.tok_seq + st.seq_index);
      } else {
        if (tid == 0) {
          ll_t w = ll_load(p.tok_word);
          ctl->bcast_tok = ll_wait(p.tok_word, st.ebase, w, p, ctl) ? (int32_t)(uint32_t)w : 0;
        }
        consumer_sync();
        st.token = ctl->bcast_tok;
      }
      sel_layer = -1;
    }
    for (int ph = ph0; ph < ph1; ++ph) {
      // every warp of this CTA has left the previous phase before this one reuses the shared input
      // vector, the staging areas and the staged residual rows
      if (ph > ph0 || step > 0) consumer_sync();
      const PhaseDesc P = phase_table(ctl)[ph];
      const int L = P.layer;
      const bool ab = aborted(ctl);
      // epochs: what this phase publishes (0 = withheld by the test hook) and what it reads
      const uint32_t ew = ((int)c == p.skip_cta && ph == p.skip_phase) ? 0u : st.ebase + 1 + (uint32_t)ph;
      const uint32_t e_src = st.ebase + 1 + (uint32_t)P.src_ph;
      const uint32_t e_res = st.ebase + 1 + (uint32_t)P.res_ph;
      const uint32_t e_sel = st.ebase + 1 + (uint32_t)P.sel_ph;
      int32_t u0, n;
      cta_share(p, ctl, P, u0, n);
      if (cw == 0 && lane == 0) stamp(p, c, ph, 0);
      // ---- prologue: the GEMV input vector into shared memory (skipped by CTAs without units)
      switch (P.kind) {
        case PK_QKV: {
          const void* emb = L == 0 ? (const uint8_t*)p.tok_emb + (size_t)st.token * p.d * 2 : nullptr;
          if (L == 0 && !ab) {  // the residual starts as the embedding row: publish this CTA's slice
            const int a = (int)((long long)c * p.d / G), b = (int)((long long)(c + 1) * p.d / G);
            for (int i = a + tid; i < b; i += kConsumerWarps * 32)
              ll_store(p.x + i, ll_pack(load_elem(emb, (size_t)i, p.edt), ew));
          }
          if (cw == kConsumerWarps - 1 && lane == 0 && !ab) {
            if (!(p.pf_flags & PF_KV_AHEAD)) {
              prefetch_attention_kv(p, L, st.pos + 1, c, G);
            } else {  // one layer early: this layer's blocks were requested during the previous layer
              if (L == 0 && step == 0) prefetch_attention_kv(p, 0, st.pos + 1, c, G);
              if (L + 1 < p.L) prefetch_attention_kv(p, L + 1, st.pos + 1, c, G);
              else if (step + 1 < p.n_steps && st.pos + 2 <= p.max_ctx) prefetch_attention_kv(p, 0, st.pos + 2, c, G);
            }
          }
          if (n > 0) {
            const int half = p.hd / 2;  // the RoPE row of this position, for the epilogue
            if (tid < half) {
              ctl->rope_cs[tid] = __ldg(p.rope_cos + (size_t)st.pos * half + tid);
              ctl->rope_sn[tid] = __ldg(p.rope_sin + (size_t)st.pos * half + tid);
            }
            rmsnorm_prologue(p, ctl, xbuf, p.attn_norm[L], emb, e_src, L, c, cw, lane);
          }
          break;
        }
        case PK_WO:
          if (n > 0) {
            ll_fetch(p, ctl, xbuf, p.attn, p.hq * p.hd, p.hq * p.hd, 0, e_src, tid,
                     residual_word(p, ctl, P, 2, e_res, tid));
          }
          break;
        case PK_DOWN:
          if (n > 0) {
            ll_fetch(p, ctl, xbuf, p.h, p.ff, p.ff, 0, e_src, tid, residual_word(p, ctl, P, 2, e_res, tid));
          }
          break;
        case PK_EDOWN:
          if constexpr (MOE) {
            if (sel_layer != L) {
              if (cw == 0) {
                select_experts(p, ctl, L, e_sel, lane, false);
                if (lane == 0) mbar_arrive(&ctl->sel_bar);
              }
              sel_layer = L;
            }
            if (n > 0) {
              ll_fetch(p, ctl, xbuf, p.h, p.topk * p.fexp, p.fexp, (p.fexp + 255) & ~255, e_src, tid,
                       residual_word(p, ctl, P, 1, e_res, tid));
            } else {
              consumer_sync();  // the choice (shared memory) is read by every warp's epilogue
            }
          }
          break;
        case PK_GU:
        case PK_ROUTER:
          if (n > 0) rmsnorm_prologue(p, ctl, xbuf, p.ffn_norm[L], nullptr, e_src, -1, c, cw, lane);
          break;
        case PK_EGU:
          if constexpr (MOE) {
            // the router phase ran in this launch: its logits are in shared memory, and the input
            // vector still holds rmsnorm(x, ffn_norm), the router's input and this phase's
            const bool local = P.sel_ph >= ph0;
            if (cw == 0) {
              select_experts(p, ctl, L, e_sel, lane, local);
              if (lane == 0) {
                if (c == 0 && !ab) for (int i = 0; i < p.topk; ++i) p.sel_out[L * p.topk + i] = ctl->sel[i];
                mbar_arrive(&ctl->sel_bar);  // release the choice to the producer
              }
            }
            sel_layer = L;
            if (!local && n > 0) rmsnorm_prologue(p, ctl, xbuf, p.ffn_norm[L], nullptr, e_src, -1, c, cw, lane);
            else consumer_sync();
          }
          break;
        case PK_LM:
          if (n > 0) rmsnorm_prologue(p, ctl, xbuf, p.final_norm, nullptr, e_src, p.L, c, cw, lane);
          break;
        default: break;
      }
      // ---- body
      if (cw == 0 && lane == 0) stamp(p, c, ph, 1);
      if (P.kind == PK_ATTN) {
        if constexpr (S::on) {
          attention_phase<S::hd, S::kvdt>(p, ctl, xbuf, P, st, c, G, cw, lane, att_uses, ew);
        } else if (p.kvdt == DT_BF16) {
          if (p.hd == 128) attention_phase<128, DT_BF16>(p, ctl, xbuf, P, st, c, G, cw, lane, att_uses, ew);
          else if (p.hd == 64) attention_phase<64, DT_BF16>(p, ctl, xbuf, P, st, c, G, cw, lane, att_uses, ew);
          else attention_phase<256, DT_BF16>(p, ctl, xbuf, P, st, c, G, cw, lane, att_uses, ew);
        } else {
          if (p.hd == 128) attention_phase<128, DT_F16>(p, ctl, xbuf, P, st, c, G, cw, lane, att_uses, ew);
          else if (p.hd == 64) attention_phase<64, DT_F16>(p, ctl, xbuf, P, st, c, G, cw, lane, att_uses, ew);
          else attention_phase<256, DT_F16>(p, ctl, xbuf, P, st, c, G, cw, lane, att_uses, ew);
        }
      } else if (P.kind == PK_SAMPLE) {
        if (st.temperature > 0.0f) sample_phase(p, ctl, st, c, G, cw, lane);
      } else if (P.kind == PK_EGU || P.kind == PK_EDOWN) {
        if constexpr (MOE) {
          switch (p.topk) {
            case 1: run_expert<1>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew); break;
            case 2: run_expert<2>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew); break;
            case 4: run_expert<4>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew); break;
            default: run_expert<8>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew); break;
          }
        }
      } else if (P.kind == PK_ROUTER) {
        if constexpr (MOE) {
          if (P.unit_rows == 4) {
            if (p.rdt == DT_BF16) gemv_phase<4, 1, DT_BF16, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
            else gemv_phase<4, 1, DT_F16, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
          } else {
            if (p.rdt == DT_BF16) gemv_phase<1, 1, DT_BF16, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
            else gemv_phase<1, 1, DT_F16, false>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
          }
        }
      } else {
        if constexpr (KIND == KK_DENSE8 || KIND == KK_DENSE4) {
          if (P.kind != PK_LM)
            run_gemv<KIND == KK_DENSE8 ? DT_E4M3 : DT_NVFP4>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
          else if constexpr (S::on) run_gemv<S::t16>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
          else if (p.edt == DT_BF16) run_gemv<DT_BF16>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
          else run_gemv<DT_F16>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
        } else {
          if constexpr (S::on) run_gemv<S::t16>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
          else if (p.wdt == DT_BF16) run_gemv<DT_BF16>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
          else run_gemv<DT_F16>(p, ctl, ring, xbuf, P, st, c, G, cw, lane, t, ew);
        }
      }
      // ---- the LM head's last CTA picks the greedy token
      if (P.kind == PK_LM && ctl->flag && st.temperature <= 0.0f && cw == 0 && lane == 0) {
        __threadfence();
        const unsigned long long key = atomicAdd(p.argkey, 0ull);
        *p.argkey = 0ull;
        *p.lm_ctr = 0u;
        finalize_token(p, st, (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull)));
      } else if (P.kind == PK_LM && ctl->flag && cw == 0 && lane == 0) {
        *p.lm_ctr = 0u;  // sampling: the maximum stays in argkey for the sampling phase
      }
      if (cw == 0 && lane == 0) stamp(p, c, ph, 2);
      // ---- dependent phases wait on the epochs of their inputs; only sampling, which needs the
      // maximum over every CTA's logits, takes a grid barrier
      if (use_barrier && ph + 1 < ph1 && ((P.kind == PK_LM && st.temperature > 0.0f) || p.debug_barriers))
        grid_barrier(p, ctl, c, G, bidx);
      if (cw == 0 && lane == 0) stamp(p, c, ph, 3);
    }
  }
}

// KIND: KK_DENSE (16-bit weights), KK_MOE (top-k expert models), KK_DENSE8 (e4m3 layer
// matrices), KK_DENSE4 (NVFP4 layer matrices): each model runs the instantiation that carries
// only its own code paths.
template <int KIND, int SPEC>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ Params p, int32_t ph0, int32_t ph1, int32_t use_barrier,
                  int32_t xbuf_floats) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* xbuf = reinterpret_cast<float*>(smem + (size_t)p.nslots * kSlotBytes);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)p.nslots * kSlotBytes + (((size_t)xbuf_floats * 4 + 127) & ~(size_t)127));
  const uint32_t c = blockIdx.x, G = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cta_setup(p, ctl);
  if (*(volatile int32_t*)&ctl->abort) return;  // sticky device error: nothing runs until reset
  Step st;
  {
    const StepState* s = p.state;
    st.pos = __ldcg(&s->pos);
    st.seq_index = __ldcg(&s->seq_index);
    st.temperature = __ldcg(&s->temperature);
    st.token = p.tok_seq ? __ldcg(p.tok_seq + st.seq_index) : __ldcg(&s->token);
    st.u = p.u_seq ? __ldcg(p.u_seq + st.seq_index) : __ldcg(&s->u);
    st.ebase = __ldcg(p.epoch);
  }
  if (warp == kConsumerWarps) {
    if (lane == 0) producer(p, ctl, ring, c, G, ph0, ph1);
  } else {
    consumer<KIND, SPEC>(p, ctl, ring, xbuf, st, c, G, ph0, ph1, use_barrier != 0, warp, lane);
  }
}

}  // namespace adp

namespace adp {

// Host-side launchers of the decode kernel: the instantiation of a model's kind and, for the
// full-size workloads' combinations (head width 128; f16 or bf16 KV and 16-bit weights), its
// specialisation; every other model runs the kind's run-time-dispatching instantiation.
template <int KIND>
static const void* kernel_spec(int hd, int kvdt, int t16) {
  if (hd == 128 && kvdt == DT_F16 && t16 == DT_F16)
    return (const void*)decode_kernel<KIND, spec_code(128, DT_F16, DT_F16)>;
  if (hd == 128 && kvdt == DT_BF16 && t16 == DT_BF16)
    return (const void*)decode_kernel<KIND, spec_code(128, DT_BF16, DT_BF16)>;
  return (const void*)decode_kernel<KIND, 0>;
}

static const void* kernel_of(int kind, int hd, int kvdt, int t16) {
  switch (kind) {
    case KK_MOE: return kernel_spec<KK_MOE>(hd, kvdt, t16);
    case KK_DENSE8: return kernel_spec<KK_DENSE8>(hd, kvdt, t16);
    case KK_DENSE4: return kernel_spec<KK_DENSE4>(hd, kvdt, t16);
    default: return kernel_spec<KK_DENSE>(hd, kvdt, t16);
  }
}

cudaError_t decode_prepare(size_t smem_bytes, int kind, int hd, int kvdt, int t16, int* blocks_per_sm) {
  const void* k = kernel_of(kind, hd, kvdt, t16);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, kThreads, smem_bytes);
}

cudaError_t decode_launch(const Params& p, int ph0, int ph1, bool persistent, int grid, size_t smem_bytes,
                          int xbuf_floats, cudaStream_t stream) {
  int32_t a0 = ph0, a1 = ph1, ub = persistent ? 1 : 0, xf = xbuf_floats;
  void* args[] = {(void*)&p, &a0, &a1, &ub, &xf};
  const int kind = p.E > 0 ? KK_MOE : p.wdt == DT_E4M3 ? KK_DENSE8 : p.wdt == DT_NVFP4 ? KK_DENSE4 : KK_DENSE;
  const void* k = kernel_of(kind, p.hd, p.kvdt, kind == KK_DENSE ? p.wdt : p.edt);
  if (persistent) return cudaLaunchCooperativeKernel(k, dim3(grid), dim3(kThreads), args, smem_bytes, stream);
  return cudaLaunchKernel(k, dim3(grid), dim3(kThreads), args, smem_bytes, stream);
}

}  // namespace adp

namespace adp {
size_t ctl_bytes(int n_phases) { return kCtlPad + (size_t)n_phases * (sizeof(PhaseDesc) + sizeof(int2)); }
}  // namespace adp

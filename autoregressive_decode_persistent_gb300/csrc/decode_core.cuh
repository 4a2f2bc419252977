// Device code shared by the single-request and the batched decode kernels: the CTA's control
// block in shared memory, the per-CTA phase table, the producer (TMA) warp that streams the
// weight tiles, the epoch-tagged exchange helpers and the grid barrier.
//
// Pages followed (title, section): "標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒",
// "Kog Inference Engineの特徴とイノベーション" (one GPU-resident program that controls its own
// synchronisation, prefetch and ordering).
#pragma once
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace adp {


struct Ctl {
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint64_t sel_bar;
  int32_t abort;
  int32_t pad;
  unsigned long long red_k[kConsumerWarps];
  float bcast;
  int32_t flag;
  int32_t sel[kMaxTopK];
  float gate[kMaxTopK];
  float stage[1024];  // router logits or sampling block sums, loaded in one batch
  uint64_t att_bar[kAttnSlots];  // TMA completion of each attention slot's K/V block
  uint64_t merge_bar;            // TMA completion of the attention merge's block outputs
  int32_t bcast_tok;             // the token of the next step of a multi-step launch
  float rope_cs[128], rope_sn[128];  // RoPE row of this step's position (QKV epilogue)
  float xres[64];                    // residual rows this CTA updates (Wo / down epilogues)
};

struct Step {
  int32_t pos, token, seq_index;
  float temperature, u;
  uint32_t ebase;  // epoch of phase ph in this step = ebase + 1 + ph
};

__device__ __forceinline__ void set_error(const Params& p, Ctl* ctl, int32_t code) {
  atomicCAS(p.err, 0, code);
  *(volatile int32_t*)&ctl->abort = 1;
}

__device__ __forceinline__ bool aborted(Ctl* ctl) { return *(volatile int32_t*)&ctl->abort != 0; }

// SM cycle counter for the timeline's cycle breakdowns (entries 12..15), compiled in only with
// -DADP_CYCLE_STAMPS: the reads sit in the GEMV chunk loop.
#ifdef ADP_CYCLE_STAMPS
__device__ __forceinline__ long long cyc_now() { return clock64(); }
#else
__device__ __forceinline__ long long cyc_now() { return 0; }
#endif

// Timeline stamp k of phase ph for this CTA (debug hook; one thread writes each slot).
__device__ __forceinline__ void stamp(const Params& p, uint32_t c, int ph, int k) {
  if (p.timeline) p.timeline[((size_t)c * p.n_phases + ph) * kStamps + k] = globaltimer();
}

// Per-CTA share of a phase: units [u0, u0 + n); a replicated phase gives every CTA all units.  (c + 1) * n_units stays below 2^32: the model
// checks n_units * G < 2^32 at creation.
__device__ __forceinline__ void cta_units(const PhaseDesc& P, uint32_t c, uint32_t G, int32_t& u0, int32_t& n) {
  if (P.replicated) {  // every CTA streams the phase's one region and computes every unit
    u0 = 0;
    n = P.n_units;
    return;
  }
  const uint32_t nu = (uint32_t)P.n_units;
  const uint32_t a = c * nu / G, b = (c + 1) * nu / G;
  u0 = (int32_t)a;
  n = (int32_t)(b - a);
}

// The step's phase table, copied into shared memory after the control block at kernel start
// (every phase begins by reading its descriptor: from global memory that would be a round trip
// to L2 on the critical path of every phase), followed by this CTA's unit range of each phase.
constexpr size_t kCtlPad = (sizeof(Ctl) + 15) & ~(size_t)15;
__device__ __forceinline__ const PhaseDesc* phase_table(const Ctl* ctl) {
  return reinterpret_cast<const PhaseDesc*>(reinterpret_cast<const uint8_t*>(ctl) + kCtlPad);
}
__device__ __forceinline__ int2* share_table(const Ctl* ctl, int n_phases) {
  return const_cast<int2*>(reinterpret_cast<const int2*>(phase_table(ctl) + n_phases));
}
// This CTA's units [u0, u0 + n) of phase P, as computed at kernel start.
__device__ __forceinline__ void cta_share(const Params& p, const Ctl* ctl, const PhaseDesc& P, int32_t& u0,
                                          int32_t& n) {
  const int2 v = share_table(ctl, p.n_phases)[P.index];
  u0 = v.x;
  n = v.y;
}

// ---------------------------------------------------------------- producer (TMA) warp

constexpr uint32_t kL2Chunk = 32 * 1024;

// Cursor over this CTA's weight stream for L2 prefetch.  Positions count bytes of the dense
// phases' shares (each contiguous in the image) in consumption order.  The cursor runs up to
// p.l2_lookahead bytes beyond the TMA issue position and stops at an expert phase until routing
// has chosen the experts.
// With p.l2_rate set, the prefetches are paced by a token bucket (p.l2_rate bytes per microsecond,
// at most p.l2_burst at once), so that the lookahead keeps HBM streaming without queueing a burst
// of requests ahead of the step's latency-bound accesses.
struct L2Cursor {
  int ph;
  uint64_t off;  // within the current phase's share
  uint64_t pos;  // stream position of the cursor
};

struct L2Pace {
  uint64_t t;       // %globaltimer of the last refill
  uint64_t tokens;  // bytes that may be prefetched now
};

__device__ __forceinline__ void l2_advance(const Params& p, const Ctl* ctl, L2Cursor& cur, uint64_t issue_pos, int ph1, uint32_t c,
                                           uint32_t G, uint64_t wpol, L2Pace& pace) {
  if (p.l2_rate) {
    const uint64_t now = globaltimer();
    const uint64_t add = (now - pace.t) * p.l2_rate / 1000u;
    pace.tokens = min((uint64_t)p.l2_burst, pace.tokens + add);
    pace.t = now;
  }
  while (cur.pos < issue_pos + p.l2_lookahead && cur.ph < ph1) {
    const PhaseDesc& Q = phase_table(ctl)[cur.ph];
    if (!Q.has_weights) { ++cur.ph; cur.off = 0; continue; }
    if (Q.kind == PK_EGU || Q.kind == PK_EDOWN) return;  // experts not chosen yet
    int32_t u0, n;
    cta_share(p, ctl, Q, u0, n);
    const uint64_t unit_bytes = wbytes(Q, (uint64_t)Q.unit_rows * Q.K);
    const uint64_t len = (uint64_t)n * unit_bytes;
    if (cur.off >= len) { ++cur.ph; cur.off = 0; continue; }
    const uint64_t left = len - cur.off;
    const uint32_t chunk = left < kL2Chunk ? (uint32_t)left : kL2Chunk;
    if (p.l2_rate && cur.pos >= issue_pos) {
      if (pace.tokens < chunk) return;
      pace.tokens -= chunk;
    }
    if (cur.pos >= issue_pos) {
      const uint8_t* src = p.image + Q.region + (uint64_t)u0 * unit_bytes + cur.off;
      if (p.pf_flags & PF_W_LAST) prefetch_l2_hint(src, chunk, wpol);
      else prefetch_l2(src, chunk);
    }
    cur.off += chunk;
    cur.pos += chunk;
  }
}

static __device__ void producer(const Params& p, Ctl* ctl, uint8_t* ring, uint32_t c, uint32_t G, int ph0, int ph1) {
  const uint64_t pol = policy_evict_first();
  const uint64_t wpol = policy_evict_last();
  const uint32_t ns = (uint32_t)p.nslots;
  uint32_t t = 0;               // tiles issued
  uint32_t pslot = 0, puse = 0;  // ring slot of the next tile and how often it was filled before
  uint32_t sel_uses = 0;
  int sel_layer = -1;
  bool stop = false;
  L2Cursor cur{ph0, 0, 0};
  L2Pace pace{globaltimer(), 0};
  uint64_t issue_pos = 0;  // stream position of the next dense tile
  for (int step = 0; step < p.n_steps && !stop; ++step) {  // the launch's decode steps
    sel_layer = -1;
    cur = L2Cursor{ph0, 0, issue_pos};
    for (int ph = ph0; ph < ph1 && !stop; ++ph) {
      const PhaseDesc P = phase_table(ctl)[ph];
      if (!P.has_weights) continue;
      int32_t u0, n;
      cta_share(p, ctl, P, u0, n);
      const bool expert = P.kind == PK_EGU || P.kind == PK_EDOWN;
      if (!expert && cur.ph < ph) cur = L2Cursor{ph, 0, issue_pos};  // behind, or waited at the experts
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
      const uint64_t unit_bytes = wbytes(P, (uint64_t)P.unit_rows * P.K);
      const uint8_t* base = p.image + P.region + (uint64_t)u0 * unit_bytes;
      const int rounds = (n + P.upr - 1) / P.upr;
      bool first = true;
      uint64_t blocked = 0;  // ns spent with the ring full (timeline only)
      for (int r = 0; r < rounds && !stop; ++r) {
        const int m = min(P.upr, n - r * P.upr);
        const uint64_t round_off = (uint64_t)r * P.upr * unit_bytes;
        for (int ck = 0; ck < P.n_chunks; ++ck) {
          if (aborted(ctl)) { stop = true; break; }
          const int kck = min(P.KC, P.K - ck * P.KC);
          const uint32_t bytes = (uint32_t)wbytes(P, (uint64_t)m * P.unit_rows * kck);
          const uint64_t off = round_off + wbytes(P, (uint64_t)m * P.unit_rows * ck * P.KC);
          const uint32_t slot = pslot, use = puse;
          if (use > 0) {
            if (!mbar_try_wait(&ctl->empty[slot], (use - 1) & 1)) {
              const uint64_t tb = p.timeline ? globaltimer() : 0;
              l2_advance(p, ctl, cur, issue_pos, ph1, c, G, wpol, pace);  // keep HBM busy while the consumers catch up
              bool ok;
              if (p.l2_rate && p.l2_lookahead) {
                // paced: refill and prefetch while waiting for the slot (bounded like every wait)
                const uint64_t t0 = globaltimer();
                for (;;) {
                  if ((ok = mbar_try_wait(&ctl->empty[slot], (use - 1) & 1))) break;
                  if (aborted(ctl) || globaltimer() - t0 > p.wait_ns) break;
                  l2_advance(p, ctl, cur, issue_pos, ph1, c, G, wpol, pace);
                }
              } else {
                ok = mbar_wait(&ctl->empty[slot], (use - 1) & 1, &ctl->abort, p.wait_ns);
              }
              if (!ok) {
                if (!aborted(ctl)) set_error(p, ctl, DE_PIPELINE_TIMEOUT);
                stop = true;
                break;
              }
              if (p.timeline) blocked += globaltimer() - tb;
            }
          }
          if (first) {
            stamp(p, c, ph, 4);
            first = false;
          }
          mbar_arrive_expect_tx(&ctl->full[slot], bytes * P.slots);
          uint8_t* dst = ring + (size_t)slot * kSlotBytes;
          for (int s = 0; s < P.slots; ++s) {
            const uint8_t* src = base + off;
            if (expert) src += (uint64_t)(*(volatile int32_t*)&ctl->sel[s]) * P.expert_stride;
            tma_load_1d(dst + (size_t)s * bytes, src, bytes, &ctl->full[slot], pol);
          }
          if (!expert) {
            issue_pos += bytes;
            if (p.l2_lookahead) l2_advance(p, ctl, cur, issue_pos, ph1, c, G, wpol, pace);
          }
          ++t;
          if (++pslot == ns) {
            pslot = 0;
            ++puse;
          }
        }
      }
      stamp(p, c, ph, 5);
      if (p.timeline) p.timeline[((size_t)c * p.n_phases + ph) * kStamps + 7] = blocked;
    }
  }
  // No bulk copy may still be writing this CTA's shared memory when it exits.
  int32_t never = 0;
  for (uint32_t i = (t > ns ? t - ns : 0); i < t; ++i) mbar_wait(&ctl->full[i % ns], (i / ns) & 1, &never, p.wait_ns);
}

// ---------------------------------------------------------------- consumer helpers

__device__ __forceinline__ void load_x8(const float* xs, float (&x)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(xs);
  const float4 b = *reinterpret_cast<const float4*>(xs + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// A GEMV input vector sits in shared memory in a split layout, so that 32 lanes reading 32
// consecutive 8-element vectors hit every bank once per 16-byte load: element e (0..7) of vector
// v is stored at (v / 32) * 256 + (e / 4) * 128 + (v % 32) * 4 + e % 4.  Vectors of n elements
// take n rounded up to a multiple of 256 floats.
__device__ __forceinline__ int xpos(int i) {
  const int v = i >> 3, e = i & 7;
  return ((v >> 5) << 8) + ((e >> 2) << 7) + ((v & 31) << 2) + (e & 3);
}

__device__ __forceinline__ void load_xs8(const float* xb, int v, float (&x)[8]) {
  const float* a = xb + ((v >> 5) << 8) + ((v & 31) << 2);
  const float4 lo = *reinterpret_cast<const float4*>(a);
  const float4 hi = *reinterpret_cast<const float4*>(a + 128);
  x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
  x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
}

__device__ __forceinline__ void ldcg_x8(const float* g, float (&x)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(g));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(g) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

constexpr int kPrologueRegs = 16;  // d_model <= 16 * 15 * 32 = 7680 (checked at model creation)

// Wait until *src carries `epoch` (w holds the word already loaded).  Bounded; on timeout the
// CTA records a dependency-wait error and stops waiting.
__device__ __forceinline__ bool ll_wait(const ll_t* src, uint32_t epoch, ll_t& w, const Params& p, Ctl* ctl) {
  if (ll_epoch(w) == epoch) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    w = ll_load(src);
    if (ll_epoch(w) == epoch) return true;
    if ((it & 15) == 15) {
      if (aborted(ctl)) return false;
      if (globaltimer() - t0 > p.wait_ns) {
        set_error(p, ctl, DE_BARRIER_TIMEOUT);
        return false;
      }
    }
  }
}

// One more epoch-tagged word a thread fetches alongside an ll_fetch batch (src null: none): it is
// loaded before the batch and stored to *dst once it carries `epoch`, before the batch's closing
// consumer_sync, so that its round trip overlaps the batch's instead of preceding it.
struct SideWord {
  const ll_t* src;
  float* dst;
  uint32_t epoch;
};

// The values of src[0..n) once each carries `epoch`, into dst in the split layout: n/seg vectors
// of seg elements, each taking segp floats (all consumer threads, eight loads in flight per
// thread; ends with consumer_sync).
static __device__ void ll_fetch(const Params& p, Ctl* ctl, float* dst, const ll_t* src, int n, int seg, int segp,
                         uint32_t epoch, int tid, SideWord side = SideWord{nullptr, nullptr, 0}) {
  constexpr int B = 8, T = kConsumerWarps * 32;
  ll_t sw = side.src ? ll_load(side.src) : 0ull;
  for (int base = tid; base < n; base += B * T) {
    ll_t w[B];
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int i = base + k * T;
      w[k] = i < n ? ll_load(src + i) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int i = base + k * T;
      if (i < n) {
        if (ll_epoch(w[k]) != epoch) {
          if (!ll_wait(src + i, epoch, w[k], p, ctl)) break;
          // the later words of the batch were loaded before this one arrived: reload those
          // still behind together, so the batch costs one more round trip, not one per word
#pragma unroll
          for (int j = k + 1; j < B; ++j) {
            const int ij = base + j * T;
            if (ij < n && ll_epoch(w[j]) != epoch) w[j] = ll_load(src + ij);
          }
        }
        dst[seg == n ? xpos(i) : (i / seg) * segp + xpos(i % seg)] = ll_value(w[k]);
      }
    }
  }
  if (side.src && ll_wait(side.src, side.epoch, sw, p, ctl)) *side.dst = ll_value(sw);
  consumer_sync();
}

// Heads [h0, h1) read KV head g: floor(h * hkv / hq) == g.
__device__ __forceinline__ void group_heads(int g, int hq, int hkv, int& h0, int& h1) {
  h0 = (g * hq + hkv - 1) / hkv;
  h1 = ((g + 1) * hq + hkv - 1) / hkv;
}

// 8 KV-cache values (16 bytes) -> fp32 (exact).
template <int KVDT>
__device__ __forceinline__ void kv8(const uint4 w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (KVDT == DT_BF16) {
      f[2 * i] = __uint_as_float(u[i] << 16);
      f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    } else {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

// DPL consecutive KV values of one row (one lane's share of the PV pass) from shared memory.
template <int KVDT, int DPL>
__device__ __forceinline__ void kv_dims_smem(const uint16_t* src, float (&f)[DPL]) {
  if constexpr (DPL == 8) {
    kv8<KVDT>(*reinterpret_cast<const uint4*>(src), f);
  } else {
    uint32_t u[DPL / 2];
    if constexpr (DPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      u[0] = w.x;
      u[1] = w.y;
    } else {
      u[0] = *reinterpret_cast<const uint32_t*>(src);
    }
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) {
      if constexpr (KVDT == DT_BF16) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
      } else {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
      }
    }
  }
}

static __device__ bool grid_barrier(const Params& p, Ctl* ctl, uint32_t c, uint32_t G, int& bidx) {
  consumer_sync();
  if (threadIdx.x == 0) {
    const bool was_aborted = aborted(ctl);
    if (!grid_arrive_wait(p.bar_ctr, G, true, !was_aborted, p.wait_ns)) set_error(p, ctl, DE_BARRIER_TIMEOUT);
    if (!aborted(ctl) && *(volatile int32_t*)p.err != 0) *(volatile int32_t*)&ctl->abort = 1;
  }
  ++bidx;
  consumer_sync();
  return !aborted(ctl);
}


// Kernel start, all threads of the CTA: the mbarriers, the phase table and this CTA's share of
// every phase in shared memory (ends with __syncthreads).
__device__ __forceinline__ void cta_setup(const Params& p, Ctl* ctl) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nslots; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], kConsumerWarps);
    }
    mbar_init(&ctl->sel_bar, 1);
    mbar_init(&ctl->merge_bar, 1);
    for (int w = 0; w < kAttnSlots; ++w) mbar_init(&ctl->att_bar[w], 1);
    ctl->abort = *(volatile int32_t*)p.err != 0 ? 1 : 0;
    ctl->flag = 0;
    mbar_fence_init();
  }
  {
    static_assert(sizeof(PhaseDesc) % 8 == 0, "phase descriptors are copied as 8-byte words");
    const uint2* src = reinterpret_cast<const uint2*>(p.phases);
    uint2* dst = reinterpret_cast<uint2*>(const_cast<PhaseDesc*>(phase_table(ctl)));
    const int nv = p.n_phases * (int)(sizeof(PhaseDesc) / 8);
    for (int i = threadIdx.x; i < nv; i += kThreads) dst[i] = __ldg(src + i);
    int2* shares = share_table(ctl, p.n_phases);
    for (int i = threadIdx.x; i < p.n_phases; i += kThreads) {
      int32_t u0, n;
      cta_units(p.phases[i], blockIdx.x, gridDim.x, u0, n);
      shares[i] = make_int2(u0, n);
    }
  }
  __syncthreads();
}

}  // namespace adp

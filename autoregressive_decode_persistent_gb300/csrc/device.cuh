// Device primitives of the decode kernel (sm_103a): mbarriers, TMA bulk copies, a bounded
// grid barrier, the arithmetic contract (exp, dot-product lanes, RoPE), and storage types.
//
// The pages ask the GPU program to control synchronisation, prefetch and execution order
// itself ("標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒", hakusoku.com,
// section "Kog Inference Engineの特徴とイノベーション"); these are the pieces it is built from.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "plan.h"

namespace adp {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier + TMA bulk copy

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete.  Gives up (returns false) when *abort becomes
// nonzero or after limit_ns; every wait in the kernel is bounded.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int32_t* abort, uint64_t limit_ns) {
  if (mbar_try_wait(b, parity)) return true;
  uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// 1-D TMA bulk copy global -> this CTA's shared memory, completing on an mbarrier.
// Not multicast. dst, src and bytes are multiples of 16.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Bulk prefetch of global memory into L2 (no completion; bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The same with an L2 eviction-priority policy for the prefetched lines.
__device__ __forceinline__ void prefetch_l2_hint(const void* src, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(policy)
               : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Named barrier over the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// ---------------------------------------------------------------- grid barrier

// Monotonic 64-bit arrival counter shared by all launches of a model: barrier instance k of
// a step completes when the counter reaches the next multiple of the grid size.  Arrival is a
// release RMW (cumulative over the CTA's writes ordered before it by the preceding CTA barrier),
// the wait an acquire load; the wait is bounded by limit_ns.  Returns false on timeout.  Called
// by one thread per CTA, between two consumer_sync()s.
__device__ __forceinline__ bool grid_arrive_wait(unsigned long long* ctr, uint32_t G, bool arrive, bool wait,
                                                 uint64_t limit_ns) {
  unsigned long long old = 0;
  if (arrive) {
    asm volatile("atom.add.release.gpu.u64 %0, [%1], 1;" : "=l"(old) : "l"(ctr) : "memory");
  } else {
    asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(old) : "l"(ctr) : "memory");
  }
  if (!wait) return true;
  const unsigned long long target = (old / G + 1) * G;
  uint64_t t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
    if (v >= target) break;
    if ((it & 31) == 31 && globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- epoch-tagged words

using ll_t = unsigned long long;

__device__ __forceinline__ ll_t ll_pack(float v, uint32_t epoch) {
  return ((ll_t)epoch << 32) | (ll_t)__float_as_uint(v);
}
__device__ __forceinline__ ll_t ll_pack_bits(uint32_t bits, uint32_t epoch) { return ((ll_t)epoch << 32) | bits; }
__device__ __forceinline__ uint32_t ll_epoch(ll_t w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ float ll_value(ll_t w) { return __uint_as_float((uint32_t)w); }

// One 64-bit store / load: value and epoch become visible together.
__device__ __forceinline__ void ll_store(ll_t* p, ll_t w) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ ll_t ll_load(const ll_t* p) {
  ll_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}

// ---------------------------------------------------------------- storage types

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// 8 consecutive weights (16 bytes for 16-bit types, 8 bytes for e4m3) -> fp32 (exact).
template <int WDT>
__device__ __forceinline__ void load8(const uint8_t* p, float (&w)[8]) {
  if constexpr (WDT == DT_F16) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h2 = *reinterpret_cast<const __half2*>(&u[i]);
      float2 f = __half22float2(h2);
      w[2 * i] = f.x;
      w[2 * i + 1] = f.y;
    }
  } else if constexpr (WDT == DT_BF16) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[2 * i] = __uint_as_float(u[i] << 16);
      w[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  } else {  // DT_E4M3
    uint2 v = *reinterpret_cast<const uint2*>(p);
    const uint32_t u[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(u[i] & 0xFFFFu), __NV_E4M3);
      __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(u[i] >> 16), __NV_E4M3);
      float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
      float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
      w[4 * i + 0] = a.x;
      w[4 * i + 1] = a.y;
      w[4 * i + 2] = b.x;
      w[4 * i + 3] = b.y;
    }
  }
}

// 8 NVFP4 elements from one 32-bit word of codes (element 2i in the low nibble of byte i) -> fp32
// (exact: every E2M1 value is an fp16 value).
__device__ __forceinline__ void load8_e2m1(uint32_t q, float (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((q >> (8 * i)) & 0xFFu), __NV_E2M1);
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    w[2 * i] = f.x;
    w[2 * i + 1] = f.y;
  }
}

// One e4m3 code -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&h));
}

__device__ __forceinline__ float load_elem(const void* base, size_t i, int dt) {
  if (dt == DT_F16) return __half2float(reinterpret_cast<const __half*>(base)[i]);
  if (dt == DT_BF16) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(base)[i]);
  if (dt == DT_E4M3) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(reinterpret_cast<const __nv_fp8_storage_t*>(base)[i], __NV_E4M3);
    return __half2float(*reinterpret_cast<__half*>(&h));
  }
  return reinterpret_cast<const float*>(base)[i];
}

// KV store: fp32 -> storage type, round to nearest even.
__device__ __forceinline__ uint16_t round_kv(float v, int kvdt) {
  if (kvdt == DT_BF16) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&b);
  }
  __half h = __float2half_rn(v);
  return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ float kv_to_f32(uint16_t b, int kvdt) {
  if (kvdt == DT_BF16) return bf16_bits_to_f32(b);
  __half h = *reinterpret_cast<__half*>(&b);
  return __half2float(h);
}

// ---------------------------------------------------------------- arithmetic contract

// exp of the contract: Cody & Waite argument reduction ("Software Manual for the
// Elementary Functions", 1980) with ln 2 split into a 15-bit head and a tail, a degree-7
// Taylor polynomial in Horner form with fused multiply-adds, and an exact 2^n scale.
// 0 for x <= -87, +inf for x >= 88.  Deterministic IEEE operations only, so the CPU
// oracle's independent implementation of the same steps returns identical bits.
__device__ __forceinline__ float exp_c(float x) {
  if (x != x) return x;
  if (x <= -87.0f) return 0.0f;
  if (x >= 88.0f) return __int_as_float(0x7F800000);
  const float kLog2e = 1.44269502162933349609375f;
  const float kLn2Hi = 0.693145751953125f;
  const float kLn2Lo = 1.428606765330187e-06f;
  float n = rintf(__fmul_rn(x, kLog2e));
  float r = fmaf(-n, kLn2Hi, x);
  r = fmaf(-n, kLn2Lo, r);
  float p = 1.98412701138295233249664306640625e-4f;
  p = fmaf(p, r, 1.38888892251998186111450195312e-3f);
  p = fmaf(p, r, 8.33333376795053482055664062500e-3f);
  p = fmaf(p, r, 4.16666679084300994873046875000e-2f);
  p = fmaf(p, r, 1.66666671633720397949218750000e-1f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  const float scale = __int_as_float(((int)n + 127) << 23);
  return __fmul_rn(p, scale);
}

// One lane's share of a contract dot product: 8 fused multiply-adds in element order.
__device__ __forceinline__ float fma8(const float (&w)[8], const float (&x)[8], float acc) {
#pragma unroll
  for (int e = 0; e < 8; ++e) acc = fmaf(w[e], x[e], acc);
  return acc;
}

// The same for two rows against one input vector, as packed fp32 FMAs: lane .x is row a's chain,
// lane .y row b's, each an IEEE fused multiply-add in element order (bit-identical to fma8 per row).
__device__ __forceinline__ float2 fma8x2(const float (&wa)[8], const float (&wb)[8], const float (&x)[8],
                                         float2 acc) {
#pragma unroll
  for (int e = 0; e < 8; ++e) acc = __ffma2_rn(make_float2(wa[e], wb[e]), make_float2(x[e], x[e]), acc);
  return acc;
}

// Fold the 32 lane partials of a contract dot product: pairs (i, i+16), (i, i+8), ... (i, i+1).
// Every lane ends with the same bits (addition is commutative in IEEE arithmetic).
__device__ __forceinline__ float warp_fold(float a) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) a = __fadd_rn(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
  return a;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  const float t = exp_c(-g);
  const float den = __fadd_rn(1.0f, t);
  return __fmul_rn(__fdiv_rn(g, den), u);
}

// Order-preserving map of fp32 to uint32 (larger float -> larger integer).
__device__ __forceinline__ uint32_t float_order(float v) {
  uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_float(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}
// Key whose maximum is the largest value, and among equal values the lowest index.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  return ((unsigned long long)float_order(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

}  // namespace adp

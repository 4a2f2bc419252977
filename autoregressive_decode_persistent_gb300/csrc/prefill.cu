// Tensor-core prefill: the weight contractions of a whole prompt as dense GEMMs and its causal
// attention as flash-style MMAs, both on the fifth-generation tensor cores (tcgen05,
// accumulators in TMEM), with the norms, RoPE / KV write and SwiGLU between them as plain CUDA
// kernels.
//
// The pages time-to-first-token as a metric of their own ("標準GPUによるリアルタイムLLM推論：
// リクエストあたり3,000トークン/秒", "単一リクエストLLMデコード速度の重要性") and give no prefill
// algorithm.  Prefill over P prompt tokens is, per layer, matrix-matrix work ([P, d] x [d, n]):
// unlike a decode step it is a dense contraction, so it belongs on the tensor cores.
//
// GEMM: C[M, N] (fp32) = A[M, K] W[N, K]^T with A and W 16-bit (f16 or bf16), both K-major.
// Operands live in global memory already in the tensor cores' shared-memory layout (tc.cuh),
// tile by tile: A as 128-row x 64-K tiles, W as 256-row x 64-K tiles, each contiguous, so one
// 1-D bulk copy stages a tile.  One CTA computes one 256 x 256 output tile as two 128-row halves:
// warp 0 streams the K-tiles (two A tiles and one W tile, 64 KB) through a 3-stage ring, one
// thread of warp 1 issues 8 MMAs (2 halves x K = 16 x 4) per stage into two 128-lane x 256-column
// fp32 accumulators in TMEM (all 512 columns) and commits each stage back to the producer, and
// all four warps read the accumulators out (lane = row) when the last MMA has completed.  Each
// staged W tile thus serves 256 output rows, which halves the bytes staged per flop for W.
#include <cuda_runtime.h>

#include <algorithm>

#include "launch.h"
#include "tc.cuh"

namespace adp {

constexpr int kTcBM = 128, kTcBN = 256, kTcStages = 3;
constexpr uint32_t kTcABytes = kTcBM * kTcBK * 2;  // 16 KB: one 128-row A tile
constexpr uint32_t kTcBBytes = kTcBN * kTcBK * 2;  // 32 KB
// a CTA's output tile: HALVES x 128 rows x 256 columns (HALVES 2: each staged weight tile serves
// 256 rows; HALVES 1: twice the CTAs, for grids that would otherwise end in a nearly empty wave)
template <int HALVES>
__host__ __device__ constexpr uint32_t tc_stage_bytes() { return HALVES * kTcABytes + kTcBBytes; }
template <int HALVES>
constexpr size_t tc_gemm_smem() { return (size_t)kTcStages * tc_stage_bytes<HALVES>() + 256; }

// 16-bit storage of an fp32 value (RNE): bf16 or f16.
__device__ __forceinline__ uint16_t tc_store16(float v, int bf16) {
  if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}


// MODE TC_SWIGLU: C is the A-operand tile buffer of the next GEMM (K = n_valid / 2) and ldc its
// number of 64-wide K tiles; output columns 2i and 2i + 1 are gate_i and up_i.
template <int BF16, int MODE, int HALVES>
__global__ void __launch_bounds__(128, 1)
    tc_gemm_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ W, float* C, int ldc, int m_valid,
                   int n_valid, int k_tiles, int32_t* err, uint64_t wait_ns, const __grid_constant__ TcQkvEpi qe,
                   const float* __restrict__ cs) {
  constexpr uint32_t kTcStageBytes = tc_stage_bytes<HALVES>();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kTcStages * kTcStageBytes);
  uint64_t* empty = full + kTcStages;
  uint64_t* done = empty + kTcStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int32_t* abort_flag = reinterpret_cast<int32_t*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // M-blocks vary fastest across the grid, so the CTAs running together share few weight tiles
  // (each read from DRAM once, then from L2) and every A tile stays in L2
  const int mb = blockIdx.x, nb = blockIdx.y;  // rows 128 HALVES mb .., columns 256 nb ..
  const uint8_t* Ab = A + (size_t)(HALVES * mb) * k_tiles * kTcABytes;  // 128-row tile HALVES mb (and the next)
  const uint8_t* Wb = W + (size_t)nb * k_tiles * kTcBBytes;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, HALVES * kTcBN);  // HALVES 128 x 256 fp32 accumulators
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int32_t* ab = abort_flag;
  if (warp == 0 && lane == 0) {
    // producer: K-tile ks into stage ks % S once the MMAs of its previous use have completed
    const uint64_t pol = policy_evict_first();
    int issued = 0;
    for (int ks = 0; ks < k_tiles; ++ks) {
      const int s = ks % kTcStages;
      if (ks >= kTcStages && !mbar_wait(&empty[s], ((ks / kTcStages) - 1) & 1, ab, wait_ns)) {
        *ab = 1;
        break;
      }
      uint8_t* dst = smem + (size_t)s * kTcStageBytes;
      mbar_arrive_expect_tx(&full[s], kTcStageBytes);
      for (int hh = 0; hh < HALVES; ++hh)
        tma_load_1d(dst + hh * kTcABytes, Ab + ((size_t)hh * k_tiles + ks) * kTcABytes, kTcABytes, &full[s], pol);
      tma_load_1d(dst + HALVES * kTcABytes, Wb + (size_t)ks * kTcBBytes, kTcBBytes, &full[s], pol);
      issued = ks + 1;
    }
    // no bulk copy may still be writing this CTA's shared memory when it exits
    int32_t never = 0;
    for (int ks = issued > kTcStages ? issued - kTcStages : 0; ks < issued; ++ks)
      mbar_wait(&full[ks % kTcStages], (ks / kTcStages) & 1, &never, wait_ns);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = tc_idesc_f16(BF16, kTcBM, kTcBN);
    for (int ks = 0; ks < k_tiles; ++ks) {
      const int s = ks % kTcStages;
      if (!mbar_wait(&full[s], (ks / kTcStages) & 1, ab, wait_ns)) {
        *ab = 1;
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(smem + (size_t)s * kTcStageBytes);
      const uint32_t b0 = a0 + HALVES * kTcABytes;
#pragma unroll
      for (int hh = 0; hh < HALVES; ++hh)
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk)
          tc_mma_f16(tmem + hh * kTcBN, tc_smem_desc(a0 + hh * kTcABytes + kk * 256, 128, 1024),
                     tc_smem_desc(b0 + kk * 256, 128, 1024), idesc, ks > 0 || kk > 0);
      tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
    }
    tc_commit(done);
  }
  __syncwarp();
  // epilogue: warp w holds rows 32 w .. 32 w + 31 of the tile (TMEM lanes), 32 columns at a time.
  // The issuer commits `done` on every path, so this wait ends once no MMA is in flight.
  int32_t never = 0;
  const bool ok = mbar_wait(done, 0, &never, wait_ns) && !*ab;
  tc_fence_after();
  if (ok) {
   for (int hh = 0; hh < HALVES; ++hh) {
    const int row = (HALVES * mb + hh) * kTcBM + warp * 32 + lane;
    if (MODE == TC_QKV) {
      // whole heads lie in one 256-column tile; RoPE pairs (i, i + hd/2) of q and k, then q into
      // the query tiles and k, v into the cache rows of position pos0 + row
      const int hd = qe.hd, half = hd / 2;
      const int pos = qe.pos0 + row;
      const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(hh * kTcBN);
      for (int hb = 0; hb < kTcBN; hb += hd) {
        const int head = (nb * kTcBN + hb) / hd;  // of the q heads, then the k heads, then the v heads
        if (head >= qe.hq + 2 * qe.hkv) break;
        for (int ci = 0; ci < half; ci += 32) {
          float a[32], b[32];
          tmem_ld32(tbase + (uint32_t)(hb + ci), a);
          tmem_ld32(tbase + (uint32_t)(hb + half + ci), b);
          if (row >= m_valid) continue;
          if (cs) {  // quantised weights: the row scale of each output column
            const float* ca = cs + nb * kTcBN + hb + ci;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              a[j] *= __ldg(ca + j);
              b[j] *= __ldg(ca + half + j);
            }
          }
          uint16_t ea[32], eb[32];
          if (head >= qe.hq + qe.hkv) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              ea[j] = round_kv(a[j], qe.kvdt);
              eb[j] = round_kv(b[j], qe.kvdt);
            }
          } else {
            const float* cs = qe.rope_cos + (size_t)pos * half + ci;
            const float* sn = qe.rope_sin + (size_t)pos * half + ci;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float c = __ldg(cs + j), s = __ldg(sn + j);
              const float y0 = fmaf(a[j], c, -(b[j] * s)), y1 = fmaf(b[j], c, a[j] * s);
              ea[j] = round_kv(y0, qe.kvdt);
              eb[j] = round_kv(y1, qe.kvdt);
            }
          }
          if (head < qe.hq) {
            uint8_t* qb = qe.qt + ((size_t)head * qe.n_tb + row / kTcBM) * (size_t)(hd / kTcBK) * kTcABytes;
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              const int ka = ci + j, kb = ci + half + j;
              *reinterpret_cast<uint4*>(qb + (ka / kTcBK) * kTcABytes + tc_tile_offset(row % kTcBM, ka % kTcBK)) =
                  make_uint4(ea[j] | ((uint32_t)ea[j + 1] << 16), ea[j + 2] | ((uint32_t)ea[j + 3] << 16),
                             ea[j + 4] | ((uint32_t)ea[j + 5] << 16), ea[j + 6] | ((uint32_t)ea[j + 7] << 16));
              *reinterpret_cast<uint4*>(qb + (kb / kTcBK) * kTcABytes + tc_tile_offset(row % kTcBM, kb % kTcBK)) =
                  make_uint4(eb[j] | ((uint32_t)eb[j + 1] << 16), eb[j + 2] | ((uint32_t)eb[j + 3] << 16),
                             eb[j + 4] | ((uint32_t)eb[j + 5] << 16), eb[j + 6] | ((uint32_t)eb[j + 7] << 16));
            }
          } else {
            const bool is_v = head >= qe.hq + qe.hkv;
            const int g = is_v ? head - qe.hq - qe.hkv : head - qe.hq;
            uint16_t* dst = (is_v ? qe.vc : qe.kc) + (((size_t)qe.L * qe.hkv + g) * qe.max_ctx + pos) * hd;
            // and the attention's tiles, by position: K rows like the query tiles, V transposed
            const int kb = pos / kTcBM, r = pos % kTcBM;
            uint8_t* kbase = qe.kt + ((size_t)g * qe.n_kb + kb) * (size_t)(hd / kTcBK) * kTcABytes;
            uint8_t* vbase = qe.vt + ((size_t)g * qe.n_kb + kb) * 2 * (size_t)hd * kTcBK * 2 +
                             (r / kTcBK) * (size_t)hd * kTcBK * 2;
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              const uint4 wa = make_uint4(ea[j] | ((uint32_t)ea[j + 1] << 16), ea[j + 2] | ((uint32_t)ea[j + 3] << 16),
                                          ea[j + 4] | ((uint32_t)ea[j + 5] << 16), ea[j + 6] | ((uint32_t)ea[j + 7] << 16));
              const uint4 wb = make_uint4(eb[j] | ((uint32_t)eb[j + 1] << 16), eb[j + 2] | ((uint32_t)eb[j + 3] << 16),
                                          eb[j + 4] | ((uint32_t)eb[j + 5] << 16), eb[j + 6] | ((uint32_t)eb[j + 7] << 16));
              *reinterpret_cast<uint4*>(dst + ci + j) = wa;
              *reinterpret_cast<uint4*>(dst + ci + half + j) = wb;
              if (!is_v) {
                const int ka = ci + j, kb2 = ci + half + j;
                *reinterpret_cast<uint4*>(kbase + (ka / kTcBK) * kTcABytes + tc_tile_offset(r, ka % kTcBK)) = wa;
                *reinterpret_cast<uint4*>(kbase + (kb2 / kTcBK) * kTcABytes + tc_tile_offset(r, kb2 % kTcBK)) = wb;
              }
            }
            if (is_v) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                *reinterpret_cast<uint16_t*>(vbase + tc_tile_offset(ci + j, r % kTcBK)) = ea[j];
                *reinterpret_cast<uint16_t*>(vbase + tc_tile_offset(ci + half + j, r % kTcBK)) = eb[j];
              }
            }
          }
        }
      }
      continue;
    }
    for (int c0 = 0; c0 < kTcBN; c0 += 32) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(hh * kTcBN + c0), v);
      const int col0 = nb * kTcBN + c0;
      if (cs) {  // quantised weights: the row scale of each output column (columns past N read 0)
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= col0 + j < n_valid ? __ldg(cs + col0 + j) : 0.0f;
      }
      if (MODE == TC_SWIGLU) {
        // 16 (gate, up) pairs -> h = silu(g) u, two 16-byte runs of the next GEMM's A tile row
        const int i0 = col0 / 2, ffw = n_valid / 2;
        if (row < m_valid) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            if (i0 + 8 * q >= ffw) continue;
            uint16_t e[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float g = v[16 * q + 2 * k], u = v[16 * q + 2 * k + 1];
              e[k] = tc_store16(g / (1.0f + __expf(-g)) * u, BF16);
            }
            const int i = i0 + 8 * q;
            uint8_t* H = reinterpret_cast<uint8_t*>(C);
            *reinterpret_cast<uint4*>(H + ((size_t)(row / kTcBM) * ldc + i / kTcBK) * kTcABytes +
                                      tc_tile_offset(row % kTcBM, i % kTcBK)) =
                make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16),
                           e[4] | ((uint32_t)e[5] << 16), e[6] | ((uint32_t)e[7] << 16));
          }
        }
        continue;
      }
      if (row < m_valid) {
        float* dst = C + (size_t)row * ldc + col0;
        if (col0 + 32 <= n_valid && (ldc & 3) == 0) {  // whole 16-byte groups
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4 o = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            if (MODE == TC_ADD) {
              const float4 a = *reinterpret_cast<const float4*>(dst + j);
              o = make_float4(__fadd_rn(a.x, o.x), __fadd_rn(a.y, o.y), __fadd_rn(a.z, o.z), __fadd_rn(a.w, o.w));
              *reinterpret_cast<float4*>(dst + j) = o;
            } else {
              // streaming store: the output should not evict the operand tiles other CTAs still read
              __stcs(reinterpret_cast<float4*>(dst + j), o);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col0 + j < n_valid) dst[j] = MODE == TC_ADD ? __fadd_rn(dst[j], v[j]) : v[j];
        }
      }
    }
   }
  } else if (threadIdx.x == 0) {
    atomicCAS(err, 0, DE_PIPELINE_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, HALVES * kTcBN);
}

// Row-major 16-bit [rows, K] (row stride ld elements) -> tiles of `tile_rows` x 64 in the
// tensor-core layout, zero outside [rows, K): one thread per 16-byte chunk.
__global__ void tc_tile_kernel(const uint16_t* __restrict__ src, int rows, int K, int ld, uint8_t* dst,
                               int rows_pad, int k_tiles, int tile_rows) {
  const long long nchunks = (long long)rows_pad * k_tiles * 8;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nchunks;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / ((long long)k_tiles * 8));
    const int k = (int)(i % ((long long)k_tiles * 8)) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows && k < K) {
      uint16_t e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) e[j] = (k + j < K) ? src[(size_t)r * ld + k + j] : (uint16_t)0;
      v = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16), e[4] | ((uint32_t)e[5] << 16),
                     e[6] | ((uint32_t)e[7] << 16));
    }
    const size_t tile = (size_t)(r / tile_rows) * k_tiles + k / kTcBK;
    *reinterpret_cast<uint4*>(dst + tile * (size_t)tile_rows * kTcBK * 2 + tc_tile_offset(r % tile_rows, k % kTcBK)) = v;
  }
}

cudaError_t tc_tile(const uint16_t* src, int rows, int K, int ld, uint8_t* dst, int tile_rows, cudaStream_t st) {
  const int rows_pad = (rows + tile_rows - 1) / tile_rows * tile_rows;
  const int k_tiles = (K + kTcBK - 1) / kTcBK;
  const long long n = (long long)rows_pad * k_tiles * 8;
  const int grid = (int)std::min<long long>((n + 255) / 256, 152 * 16);
  tc_tile_kernel<<<grid, 256, 0, st>>>(src, rows, K, ld, dst, rows_pad, k_tiles, tile_rows);
  return cudaGetLastError();
}

// Whole waves of CTAs each kernel would take on this GPU, in units of a 256-row tile's work: 128-row
// tiles (HALVES 1) when they finish sooner, e.g. 2 waves of 256-row tiles whose second is nearly
// empty against 3 waves of half the work.
static int tc_halves_for(int M, int N) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      sms = 1;
  }
  const long long nt = (N + kTcBN - 1) / kTcBN;
  const long long c2 = (long long)((M + 2 * kTcBM - 1) / (2 * kTcBM)) * nt, c1 = (long long)((M + kTcBM - 1) / kTcBM) * nt;
  const long long w2 = 2 * ((c2 + sms - 1) / sms), w1 = (c1 + sms - 1) / sms;  // in half-tile units
  return w1 < w2 ? 1 : 2;
}

cudaError_t tc_gemm(int bf16, int mode, const uint8_t* A_tiled, const uint8_t* W_tiled, float* C, int ldc, int M,
                    int N, int K, int32_t* err, uint64_t wait_ns, cudaStream_t st, const TcQkvEpi* qkv,
                    const float* colscale) {
  const int k_tiles = (K + kTcBK - 1) / kTcBK;
  const int halves = tc_halves_for(M, N);
  const dim3 grid((M + halves * kTcBM - 1) / (halves * kTcBM), (N + kTcBN - 1) / kTcBN);
  const void* kernels[2][2][4] = {
      {{(const void*)tc_gemm_kernel<0, TC_STORE, 1>, (const void*)tc_gemm_kernel<0, TC_ADD, 1>,
        (const void*)tc_gemm_kernel<0, TC_SWIGLU, 1>, (const void*)tc_gemm_kernel<0, TC_QKV, 1>},
       {(const void*)tc_gemm_kernel<1, TC_STORE, 1>, (const void*)tc_gemm_kernel<1, TC_ADD, 1>,
        (const void*)tc_gemm_kernel<1, TC_SWIGLU, 1>, (const void*)tc_gemm_kernel<1, TC_QKV, 1>}},
      {{(const void*)tc_gemm_kernel<0, TC_STORE, 2>, (const void*)tc_gemm_kernel<0, TC_ADD, 2>,
        (const void*)tc_gemm_kernel<0, TC_SWIGLU, 2>, (const void*)tc_gemm_kernel<0, TC_QKV, 2>},
       {(const void*)tc_gemm_kernel<1, TC_STORE, 2>, (const void*)tc_gemm_kernel<1, TC_ADD, 2>,
        (const void*)tc_gemm_kernel<1, TC_SWIGLU, 2>, (const void*)tc_gemm_kernel<1, TC_QKV, 2>}}};
  TcQkvEpi qe{};
  if (mode == TC_QKV) {
    if (!qkv) return cudaErrorInvalidValue;
    qe = *qkv;
  }
  const void* k = kernels[halves - 1][bf16 ? 1 : 0][mode];
  const size_t smem = halves == 1 ? tc_gemm_smem<1>() : tc_gemm_smem<2>();
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&A_tiled, (void*)&W_tiled, (void*)&C,   (void*)&ldc,     (void*)&M, (void*)&N,
                  (void*)&k_tiles, (void*)&err,    (void*)&wait_ns, (void*)&qe, (void*)&colscale};
  return cudaLaunchKernel(k, grid, dim3(128), args, smem, st);
}

// (A operands are allocated with their rows padded to 256 (tc_tiled_bytes(rows, K, 256)): a CTA stages
// two 128-row tiles.)
size_t tc_tiled_bytes(int rows, int K, int tile_rows) {
  const size_t rows_pad = (size_t)(rows + tile_rows - 1) / tile_rows * tile_rows;
  const size_t k_tiles = (size_t)(K + kTcBK - 1) / kTcBK;
  return rows_pad * k_tiles * kTcBK * 2;
}

}  // namespace adp

// ---------------------------------------------------------------- the prefill pipeline

namespace adp {

// Logical row of the prefill GEMM's weight matrix for row j of decode unit u of phase P:
// QKV -> [q rows; k rows; v rows] (head-major, as the caller's wq/wk/wv), gate|up -> [gate; up],
// Wo and down -> their own rows.
__device__ __forceinline__ int tc_logical_row(const PhaseDesc& P, int u, int j, int hd, int hq, int hkv, int ff) {
  if (P.kind == PK_QKV) {
    const int half = hd / 2, nq = hq * half, nk = hkv * half;
    int base = 0, uu = u;
    if (u >= nq + nk) {
      base = (hq + hkv) * hd;
      uu = u - nq - nk;
    } else if (u >= nq) {
      base = hq * hd;
      uu = u - nq;
    }
    return base + (uu / half) * hd + uu % half + j * half;
  }
  if (P.kind == PK_GU) return 2 * u + j;  // gate_u, up_u side by side: the GEMM's SwiGLU epilogue pairs them
  return u * P.unit_rows + j;
}

// Per-row scale of an e4m3 layer matrix for logical row `row` of phase P's GEMM operand (the
// scale tables of the matrices the rows come from: q, k, v; gate, up; or the one matrix).
__device__ __forceinline__ float tc_row_scale(const PhaseDesc& P, int row, int hd, int hq, int hkv, int ff,
                                              const float* sa, const float* sb, const float* sc) {
  if (P.kind == PK_QKV) {
    if (row < hq * hd) return sa[row];
    if (row < (hq + hkv) * hd) return sb[row - hq * hd];
    return sc[row - (hq + hkv) * hd];
  }
  if (P.kind == PK_GU) return (row & 1) ? sb[row >> 1] : sa[row >> 1];
  return sa[row];
}

// The decode image's tiles of phase P back into one tiled GEMM operand (256-row tiles): the
// inverse of the repack, walked the same way (CTA c's units, rounds, K-chunks).  16-bit weights
// are copied as they are; e4m3 weights become their codes and NVFP4 weights block scale x code,
// both exact in either 16-bit type (4 and 2 + 4 significant bits); the row scales are applied to
// the GEMM's output columns instead (tc_colscale_kernel), so the operand carries no rounding.
__global__ void tc_unpack_kernel(const uint8_t* __restrict__ image, PhaseDesc P, uint8_t* dst, int k_tiles, int hd,
                                 int hq, int hkv, int ff, int out_bf16) {
  const uint32_t c = blockIdx.x, G = gridDim.x;
  const long long a0 = (long long)c * P.n_units / G, a1 = (long long)(c + 1) * P.n_units / G;
  const int u0 = (int)a0, n = (int)(a1 - a0);
  if (n <= 0) return;
  const int eb = P.eb;
  const uint64_t unit_bytes = wbytes(P, (uint64_t)P.unit_rows * P.K);
  const uint8_t* src_cta = image + P.region + (uint64_t)u0 * unit_bytes;
  const int nv8 = P.K / 8;
  const long long total = (long long)n * P.unit_rows * nv8;
  for (long long idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int lu = (int)(idx / ((long long)P.unit_rows * nv8));
    const int rem = (int)(idx % ((long long)P.unit_rows * nv8));
    const int j = rem / nv8, cv = rem % nv8;
    const int col = cv * 8;
    const int ck = col / P.KC;
    const int kck = min(P.KC, P.K - ck * P.KC);
    const int r = lu / P.upr, i = lu % P.upr;
    const int m = min(P.upr, n - r * P.upr);
    const uint64_t tile_off = (uint64_t)r * P.upr * unit_bytes + wbytes(P, (uint64_t)m * P.unit_rows * ck * P.KC);
    const uint64_t prow = (uint64_t)i * P.unit_rows + j, kc0 = (uint64_t)(col - ck * P.KC);
    const uint64_t off = tile_off + (prow * kck + kc0) * eb;
    const int row = tc_logical_row(P, u0 + lu, j, hd, hq, hkv, ff);
    const size_t tile = (size_t)(row / kTcBN) * k_tiles + col / kTcBK;
    uint4 v;
    if (P.wdt != DT_NVFP4 && eb == 2) {
      v = *reinterpret_cast<const uint4*>(src_cta + off);
    } else {
      float w[8];
      if (P.wdt == DT_NVFP4) {
        load8_e2m1(*reinterpret_cast<const uint32_t*>(src_cta + tile_off + prow * (kck / 2) + kc0 / 2), w);
        const float bs = e4m3_to_f32(src_cta[tile_off + (uint64_t)m * P.unit_rows * (kck / 2) + prow * (kck / 16) +
                                             kc0 / 16]);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = bs * w[k];  // exact: 2 + 4 significant bits
      } else {
        load8<DT_E4M3>(src_cta + off, w);
      }
      uint16_t e[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) e[k] = tc_store16(w[k], out_bf16);  // exact
      v = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16), e[4] | ((uint32_t)e[5] << 16),
                     e[6] | ((uint32_t)e[7] << 16));
    }
    *reinterpret_cast<uint4*>(dst + tile * kTcBBytes + tc_tile_offset(row % kTcBN, col % kTcBK)) = v;
  }
}

cudaError_t tc_unpack(const uint8_t* image, const PhaseDesc& P, int G, int hd, int hq, int hkv, int ff, uint8_t* dst,
                      int out_bf16, cudaStream_t st) {
  const int k_tiles = (P.K + kTcBK - 1) / kTcBK;
  tc_unpack_kernel<<<G, 256, 0, st>>>(image, P, dst, k_tiles, hd, hq, hkv, ff, out_bf16);
  return cudaGetLastError();
}

// out[row] = the row scale of logical row `row` of phase P's GEMM operand (e4m3 and NVFP4 layer
// matrices: the q, k, v; gate, up; or single matrix's table), for rows [0, rows).
__global__ void tc_colscale_kernel(PhaseDesc P, int rows, int hd, int hq, int hkv, int ff, const float* sa,
                                   const float* sb, const float* sc, float* out) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row < rows) out[row] = tc_row_scale(P, row, hd, hq, hkv, ff, sa, sb, sc);
}

cudaError_t tc_colscale(const PhaseDesc& P, int rows, int hd, int hq, int hkv, int ff, const float* sa,
                        const float* sb, const float* sc, float* out, cudaStream_t st) {
  tc_colscale_kernel<<<(rows + 255) / 256, 256, 0, st>>>(P, rows, hd, hq, hkv, ff, sa, sb, sc, out);
  return cudaGetLastError();
}

__device__ __forceinline__ size_t tc_a_offset(int t, int k, int k_tiles) {
  return ((size_t)(t / kTcBM) * k_tiles + k / kTcBK) * kTcABytes + tc_tile_offset(t % kTcBM, k % kTcBK);
}

// x[t] = embedding row of token t (exact widening).
__global__ void tc_embed_kernel(const int32_t* __restrict__ tok, const uint16_t* __restrict__ emb, int d, int bf16,
                                float* x) {
  const int t = blockIdx.x;
  const uint16_t* row = emb + (size_t)tok[t] * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x)
    x[(size_t)t * d + i] = bf16 ? bf16_bits_to_f32(row[i]) : __half2float(__ushort_as_half(row[i]));
}

// A[t] = rmsnorm(x[t]) * gain, rounded to the weights' 16-bit type, in the A-operand tiles (one
// warp per token; the padding columns up to the tile edge stay zero from the buffer's clear).
__global__ void tc_rmsnorm_kernel(const float* __restrict__ x, const uint16_t* __restrict__ gain, int P, int d,
                                  float eps, int bf16, uint8_t* A, int k_tiles) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= P) return;
  const float* xr = x + (size_t)t * d;
  float ss = 0.0f;
  for (int i = lane; i < d; i += 32) ss = fmaf(xr[i], xr[i], ss);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  const float r = 1.0f / sqrtf(ss / (float)d + eps);
  for (int i = lane; i < d; i += 32) {
    const float g = bf16 ? bf16_bits_to_f32(gain[i]) : __half2float(__ushort_as_half(gain[i]));
    *reinterpret_cast<uint16_t*>(A + tc_a_offset(t, i, k_tiles)) = tc_store16(xr[i] * r * g, bf16);
  }
}

cudaError_t tc_flash(const TcPrefill& a, int qkv_n, int L, int kt_att, cudaStream_t st);

cudaError_t tc_prefill(const TcPrefill& a, cudaStream_t st) {
  const int P = a.P;
  const int qkv_n = (a.hq + 2 * a.hkv) * a.hd;
  const int kt_d = (a.d + kTcBK - 1) / kTcBK, kt_att = (a.hq * a.hd + kTcBK - 1) / kTcBK,
            kt_ff = (a.ff + kTcBK - 1) / kTcBK;
  cudaError_t e;
  tc_embed_kernel<<<P, 256, 0, st>>>(a.tokens, (const uint16_t*)a.tok_emb, a.d, a.bf16, a.x);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  for (int L = 0; L < a.n_layers; ++L) {
    tc_rmsnorm_kernel<<<(P + 7) / 8, 256, 0, st>>>(a.x, (const uint16_t*)a.attn_norm[L], P, a.d, a.eps, a.bf16, a.A,
                                                   kt_d);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // QKV with RoPE and the cache writes in the epilogue; queries into the attention's tiles
    const TcQkvEpi qe{a.rope_cos, a.rope_sin, a.kc,   a.vc,     a.Qt,      a.Kt,  a.Vt,   a.pos0,
                      L,          a.hq,       a.hkv, a.hd, a.max_ctx, a.kvdt, (P + kTcBM - 1) / kTcBM, a.n_kb};
    if ((e = tc_gemm(a.bf16, TC_QKV, a.A, a.wqkv[L], nullptr, 0, P, qkv_n, a.d, a.err, a.wait_ns, st, &qe,
                     a.sqkv ? a.sqkv[L] : nullptr)) != cudaSuccess)
      return e;
    if ((e = tc_flash(a, qkv_n, L, kt_att, st)) != cudaSuccess) return e;
    if ((e = tc_gemm(a.bf16, TC_ADD, a.A, a.wo[L], a.x, a.d, P, a.d, a.hq * a.hd, a.err, a.wait_ns, st, nullptr,
                     a.swo ? a.swo[L] : nullptr)) != cudaSuccess)
      return e;
    tc_rmsnorm_kernel<<<(P + 7) / 8, 256, 0, st>>>(a.x, (const uint16_t*)a.ffn_norm[L], P, a.d, a.eps, a.bf16, a.A,
                                                   kt_d);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // gate|up with SwiGLU in the epilogue: h goes straight into the down GEMM's A tiles (A2)
    if ((e = tc_gemm(a.bf16, TC_SWIGLU, a.A, a.wgu[L], reinterpret_cast<float*>(a.A2), kt_ff, P, 2 * a.ff, a.d,
                     a.err, a.wait_ns, st, nullptr, a.sgu ? a.sgu[L] : nullptr)) != cudaSuccess)
      return e;
    if ((e = tc_gemm(a.bf16, TC_ADD, a.A2, a.wdown[L], a.x, a.d, P, a.d, a.ff, a.err, a.wait_ns, st, nullptr,
                     a.sdown ? a.sdown[L] : nullptr)) != cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

}  // namespace adp

namespace adp {

// Key and value rows of positions [0, npos) of layer L from the cache into the attention's tiles
// (the rows a prefill after a cached prefix attends to but does not compute): K as 128-key blocks of
// hd/64 tiles of 128 x 64 (the query tiles' layout), V transposed, as blocks of two hd x 64-key
// tiles.  One thread per (KV head, position, 8-element chunk).
__global__ void tc_kv_tile_kernel(const uint16_t* __restrict__ kc, const uint16_t* __restrict__ vc, int L, int hkv,
                                  int max_ctx, int hd, int npos, int n_kb, uint8_t* kt, uint8_t* vt) {
  const int nch = hd / 8;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)hkv * npos * nch) return;
  const int ch = (int)(i % nch), pos = (int)((i / nch) % npos), g = (int)(i / ((long long)nch * npos));
  const size_t row = (((size_t)L * hkv + g) * max_ctx + pos) * hd + ch * 8;
  const uint4 k8 = __ldg(reinterpret_cast<const uint4*>(kc + row));
  const uint4 v8 = __ldg(reinterpret_cast<const uint4*>(vc + row));
  const int kb = pos / kTcBM, r = pos % kTcBM, k = ch * 8;
  uint8_t* kbase = kt + ((size_t)g * n_kb + kb) * (size_t)(hd / kTcBK) * kTcABytes;
  *reinterpret_cast<uint4*>(kbase + (k / kTcBK) * kTcABytes + tc_tile_offset(r, k % kTcBK)) = k8;
  uint8_t* vbase = vt + ((size_t)g * n_kb + kb) * 2 * (size_t)hd * kTcBK * 2 + (r / kTcBK) * (size_t)hd * kTcBK * 2;
  const uint32_t w4[4] = {v8.x, v8.y, v8.z, v8.w};
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint16_t*>(vbase + tc_tile_offset(k + j, r % kTcBK)) = (uint16_t)(w4[j >> 1] >> ((j & 1) * 16));
}

// Causal attention of the prompt on the tensor cores, flash style, as a warp-specialised pipeline.
// CTA = query head h x 128 consecutive prompt tokens, 192 threads, two CTAs per SM:
//  - warps 0-3: the softmax, thread t = query row t = TMEM lane t;
//  - warp 4 (one thread): bulk copies of the query tiles and of each 64-key block (its halves of
//    the K tiles and its transposed V tile, laid out by the QKV GEMM's epilogue) into a two-stage
//    ring;
//  - warp 5 (one thread): the MMAs.  S_j = Q K_j^T (128 x 64) goes into one of two TMEM buffers
//    (columns [0, 64) and [64, 128)), so S_{j+1} is computed while the softmax works on S_j;
//    O += P_j V_j accumulates in columns [128, 128 + head_dim).
// The softmax keeps a running maximum m (base-2 exponent units) and sum l per row in fp32 and
// writes the block's probabilities exp2(s log2(e) scale - m), rounded to the KV type, into the P
// tile in shared memory.  A larger block maximum replaces m only when it exceeds m by more than 8
// (decided per warp): until then the probabilities stay below 2^8, the same m scales l and O, so
// the result O / l is unchanged, and O in TMEM is rescaled only on those blocks.  At the end O / l
// is rounded into the A-operand tiles of Wo.
constexpr int kFlashBK = 64;  // keys per block

// 2^x by the hardware's approximate base-2 exponential (results below 2^-126 flush to zero, which
// a probability may).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two probabilities rounded (RNE) to the KV type, packed low | high << 16.
template <int BF16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  if constexpr (BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

template <int HD, int KVDT>
__global__ void __launch_bounds__(192, 2)
    tc_flash_kernel(const uint8_t* __restrict__ qt, int n_tb, const uint8_t* __restrict__ kt,
                    const uint8_t* __restrict__ vt, int n_kb, int P, int pos0, int hq, int hkv, float scale_log2,
                    int out_bf16, uint8_t* A, int k_tiles, int32_t* err, uint64_t wait_ns) {
  constexpr int KT = HD / kTcBK;                    // 64-wide K tiles of Q and K
  constexpr int BK = kFlashBK;
  constexpr uint32_t QK_TILE = 128 * kTcBK * 2;     // 16 KB: 128 rows x 64 (a query tile; a global K tile)
  constexpr uint32_t QBLK = KT * QK_TILE;
  constexpr uint32_t KH_TILE = BK * kTcBK * 2;      // 8 KB: 64 keys x 64 (half of a global K tile)
  constexpr uint32_t KBLK = KT * KH_TILE;           // a K block: 64 keys x head_dim
  constexpr uint32_t VT_TILE = HD * kTcBK * 2;      // a V^T block: head_dim rows x 64 keys
  constexpr uint32_t STAGE = KBLK + VT_TILE;
  constexpr uint32_t P_TILE = 128 * BK * 2;         // 16 KB: 128 queries x 64 keys
  constexpr int KV_BF16 = KVDT == DT_BF16 ? 1 : 0;
  constexpr float kRescale = 8.0f;                  // base-2 growth of the maximum that forces a rescale
  constexpr uint32_t kCols = 256;                   // TMEM: S0, S1 (64 columns each), O (head_dim <= 128)
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* Qs = smem;
  uint8_t* ring = Qs + QBLK;                        // 2 stages: K block, then V^T block
  uint8_t* Ps = ring + 2 * STAGE;
  uint64_t* bar = reinterpret_cast<uint64_t*>(Ps + P_TILE);
  uint64_t* qfull = bar;
  uint64_t* kvfull = bar + 1;                       // [2]
  uint64_t* kvempty = bar + 3;                      // [2]
  uint64_t* sfull = bar + 5;                        // [2]
  uint64_t* pready = bar + 7;
  uint64_t* odone = bar + 8;
  uint64_t* done = bar + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 10);
  int32_t* abort_flag = reinterpret_cast<int32_t*>(tmem_slot + 1);
  // the longest causal rows (last query blocks) start first
  const int h = blockIdx.x, qb = gridDim.y - 1 - blockIdx.y, t0 = qb * 128;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int g = h * hkv / hq;
  const int kmax = pos0 + min(t0 + 127, P - 1);    // the tile's last key position
  const int nkb = kmax / BK + 1;                    // key blocks 0 .. kmax / 64
  if (t == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], 1);
      mbar_init(&sfull[s], 1);
    }
    mbar_init(pready, 128);
    mbar_init(odone, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int32_t* ab = abort_flag;
  int32_t never = 0;
  if (warp == 4) {
    if (lane == 0) {
      // producer: the query tiles once, then key block j into stage j % 2 when the MMAs of block
      // j - 2 have released it.  Block j is half j % 2 of 128-key block j / 2 in global memory: the
      // first or last 8 KB of each of its K tiles (8-row groups are 1 KB apart) and one V^T tile.
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();  // every query tile of the KV group reads them
      mbar_arrive_expect_tx(qfull, QBLK);
      tma_load_1d(Qs, qt + ((size_t)h * n_tb + qb) * QBLK, QBLK, qfull, pol_q);
      int issued = 0;
      for (int j = 0; j < nkb; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&kvempty[s], ((j >> 1) - 1) & 1, ab, wait_ns)) {
          *ab = 1;
          break;
        }
        uint8_t* dst = ring + s * STAGE;
        const size_t blk = (size_t)g * n_kb + (j >> 1);
        mbar_arrive_expect_tx(&kvfull[s], STAGE);
#pragma unroll
        for (int q = 0; q < KT; ++q)
          tma_load_1d(dst + q * KH_TILE, kt + (blk * KT + q) * QK_TILE + (j & 1) * KH_TILE, KH_TILE, &kvfull[s],
                      pol_kv);
        tma_load_1d(dst + KBLK, vt + blk * 2 * VT_TILE + (j & 1) * VT_TILE, VT_TILE, &kvfull[s], pol_kv);
        issued = j + 1;
      }
      // no bulk copy may still be writing this CTA's shared memory when it exits
      mbar_wait(qfull, 0, &never, wait_ns);
      for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j) mbar_wait(&kvfull[j & 1], (j >> 1) & 1, &never, wait_ns);
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idS = tc_idesc_f16(KV_BF16, 128, BK);
      constexpr uint32_t idO = tc_idesc_f16(KV_BF16, 128, HD);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(&kvfull[s], (j >> 1) & 1, ab, wait_ns)) return false;
        tc_fence_after();
        const uint32_t q0 = smem_u32(Qs), k0 = smem_u32(ring + s * STAGE);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma_f16(tmem + (uint32_t)(s * BK), tc_smem_desc(q0 + (kk / 4) * QK_TILE + (kk % 4) * 256, 128, 1024),
                     tc_smem_desc(k0 + (kk / 4) * KH_TILE + (kk % 4) * 256, 128, 1024), idS, kk > 0);
        tc_commit(&sfull[s]);
        return true;
      };
      bool ok = mbar_wait(qfull, 0, ab, wait_ns) && issue_s(0);
      for (int j = 0; ok && j < nkb; ++j) {
        // S_{j+1} into the other buffer (the softmax of block j - 1 has released it), then O += P_j V_j
        if (j + 1 < nkb && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(pready, j & 1, ab, wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t p0 = smem_u32(Ps), v0 = smem_u32(ring + (j & 1) * STAGE + KBLK);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_f16(tmem + 2 * BK, tc_smem_desc(p0 + kk * 256, 128, 1024), tc_smem_desc(v0 + kk * 256, 128, 1024), idO,
                     j > 0 || kk > 0);
        tc_commit(odone);
        tc_commit(&kvempty[j & 1]);
      }
      if (!ok) *ab = 1;
      tc_commit(done);  // on every path: arrives once no MMA of this CTA is in flight
    }
    __syncwarp();
  } else {
    // ---- softmax warps
    const int qpos = pos0 + min(t0 + t, P - 1);     // this row's position (padding rows: the last)
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + 2 * BK;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    // every wait's outcome is made warp-uniform: the TMEM loads and stores are warp-collective
    auto wait_all = [&](uint64_t* b, uint32_t parity) {
      return __all_sync(0xFFFFFFFFu, mbar_wait(b, parity, ab, wait_ns));
    };
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      if (!wait_all(&sfull[s], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[BK];
      tmem_ld64(tmem + lane_base + (uint32_t)(s * BK), v);
      const int lim = qpos - j * BK;                // keys c <= lim of this block are visible to the row
      const bool full = lim >= BK - 1;
      // (eight independent partial maxima and sums: no long dependent chains)
      float mq[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mq[q] = -INFINITY;
      if (full) {
#pragma unroll
        for (int c = 0; c < BK; ++c) mq[c & 7] = fmaxf(mq[c & 7], v[c]);
      } else {
#pragma unroll
        for (int c = 0; c < BK; ++c) mq[c & 7] = c <= lim ? fmaxf(mq[c & 7], v[c]) : mq[c & 7];
      }
      const float mb = fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])), fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7])));
      const float mbs = mb * scale_log2;
      const bool grow = mbs > m + kRescale || (m == -INFINITY && mbs > -INFINITY);
      const bool rescale = __any_sync(0xFFFFFFFFu, grow);
      float corr = 1.0f;
      if (rescale) {
        const float mn = fmaxf(m, mbs);
        corr = m == -INFINITY ? 0.0f : ex2_approx(m - mn);
        m = mn;
      }
      // probabilities of the block, rounded to the KV type, two per 32-bit word
      uint32_t pw[BK / 2];
      float sq[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) sq[q] = 0.0f;
#pragma unroll
      for (int c = 0; c < BK; c += 2) {
        float p0 = ex2_approx(fmaf(v[c], scale_log2, -m)), p1 = ex2_approx(fmaf(v[c + 1], scale_log2, -m));
        if (!full) {
          p0 = c <= lim ? p0 : 0.0f;
          p1 = c + 1 <= lim ? p1 : 0.0f;
        }
        sq[(c >> 1) & 7] += p0 + p1;
        pw[c / 2] = pack16x2<KV_BF16>(p0, p1);
      }
      const float ps = ((sq[0] + sq[1]) + (sq[2] + sq[3])) + ((sq[4] + sq[5]) + (sq[6] + sq[7]));
      l = l * corr + ps;
      // P_{j-1} V_{j-1} must have completed before P is overwritten and O rescaled
      if (j > 0) {
        if (!wait_all(odone, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (rescale) {
#pragma unroll
          for (int c0 = 0; c0 < HD; c0 += 32) {
            float o[32];
            tmem_ld32(tO + c0, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] *= corr;
            tmem_st32(tO + c0, o);
          }
        }
      }
#pragma unroll
      for (int c = 0; c < BK; c += 8)
        *reinterpret_cast<uint4*>(Ps + tc_tile_offset(t, c)) = make_uint4(pw[c / 2], pw[c / 2 + 1], pw[c / 2 + 2], pw[c / 2 + 3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(pready);
    }
    // ---- O / l into the Wo GEMM's A tiles
    if (ok) ok = wait_all(odone, (nkb - 1) & 1);
    tc_fence_after();
    const int tok = t0 + t;
    if (ok) {
      const float inv = 1.0f / l;
#pragma unroll
      for (int c0 = 0; c0 < HD; c0 += 32) {
        float o[32];
        tmem_ld32(tO + c0, o);
        if (tok < P) {
#pragma unroll
          for (int q = 0; q < 32; q += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = (uint32_t)tc_store16(o[q + 2 * e] * inv, out_bf16) |
                     ((uint32_t)tc_store16(o[q + 2 * e + 1] * inv, out_bf16) << 16);
            *reinterpret_cast<uint4*>(A + tc_a_offset(tok, h * HD + c0 + q, k_tiles)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    } else {
      *ab = 1;
      if (t == 0) atomicCAS(err, 0, DE_PIPELINE_TIMEOUT);
    }
  }
  // no MMA may be in flight (nor TMEM in use) when the accumulators are freed
  mbar_wait(done, 0, &never, wait_ns);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, kCols);
}

template <int HD>
constexpr size_t tc_flash_smem() {
  // query tiles + two ring stages (K block, V^T block) + the P tile + barriers; at least 80 KB, so
  // that at most two CTAs (256 TMEM columns each) run per SM
  constexpr size_t q = (size_t)(HD / kTcBK) * 128 * kTcBK * 2;
  constexpr size_t stage = (size_t)(HD / kTcBK) * kFlashBK * kTcBK * 2 + (size_t)HD * kTcBK * 2;
  constexpr size_t need = q + 2 * stage + 128 * kFlashBK * 2 + 128;
  return need > 80 * 1024 ? need : 80 * 1024;
}

template <int HD, int KVDT>
cudaError_t tc_flash_launch(const TcPrefill& a, int kt_att, cudaStream_t st) {
  constexpr size_t smem = tc_flash_smem<HD>();
  const void* k = (const void*)tc_flash_kernel<HD, KVDT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_flash_kernel<HD, KVDT><<<dim3(a.hq, (a.P + 127) / 128), 192, smem, st>>>(
      a.Qt, (a.P + 127) / 128, a.Kt, a.Vt, a.n_kb, a.P, a.pos0, a.hq, a.hkv, a.scale * 1.4426950408889634f, a.bf16,
      a.A, kt_att, a.err, a.wait_ns);
  return cudaGetLastError();
}

cudaError_t tc_flash(const TcPrefill& a, int qkv_n, int L, int kt_att, cudaStream_t st) {
  (void)qkv_n;
  if (a.pos0 > 0) {
    // the cached prefix's rows into the attention's tiles (the QKV epilogue writes the prompt's)
    const long long n = (long long)a.hkv * a.pos0 * (a.hd / 8);
    tc_kv_tile_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a.kc, a.vc, L, a.hkv, a.max_ctx, a.hd, a.pos0,
                                                                    a.n_kb, a.Kt, a.Vt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.kvdt == DT_BF16)
    return a.hd == 128 ? tc_flash_launch<128, DT_BF16>(a, kt_att, st) : tc_flash_launch<64, DT_BF16>(a, kt_att, st);
  return a.hd == 128 ? tc_flash_launch<128, DT_F16>(a, kt_att, st) : tc_flash_launch<64, DT_F16>(a, kt_att, st);
}

}  // namespace adp

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
constexpr int kTcHalves = 2;                        // a CTA's output tile: 2 x 128 rows x 256 columns
constexpr uint32_t kTcABytes = kTcBM * kTcBK * 2;  // 16 KB: one 128-row A tile
constexpr uint32_t kTcBBytes = kTcBN * kTcBK * 2;  // 32 KB
constexpr uint32_t kTcStageBytes = kTcHalves * kTcABytes + kTcBBytes;  // 64 KB
constexpr size_t kTcSmem = (size_t)kTcStages * kTcStageBytes + 256;

// 16-bit storage of an fp32 value (RNE): bf16 or f16.
__device__ __forceinline__ uint16_t tc_store16(float v, int bf16) {
  if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}


// MODE TC_SWIGLU: C is the A-operand tile buffer of the next GEMM (K = n_valid / 2) and ldc its
// number of 64-wide K tiles; output columns 2i and 2i + 1 are gate_i and up_i.
template <int BF16, int MODE>
__global__ void __launch_bounds__(128, 1)
    tc_gemm_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ W, float* C, int ldc, int m_valid,
                   int n_valid, int k_tiles, int32_t* err, uint64_t wait_ns, const __grid_constant__ TcQkvEpi qe) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kTcStages * kTcStageBytes);
  uint64_t* empty = full + kTcStages;
  uint64_t* done = empty + kTcStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int32_t* abort_flag = reinterpret_cast<int32_t*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // M-blocks vary fastest across the grid, so the CTAs running together share few weight tiles
  // (each read from DRAM once, then from L2) and every A tile stays in L2
  const int mb = blockIdx.x, nb = blockIdx.y;  // rows 256 mb .., columns 256 nb ..
  const uint8_t* Ab = A + (size_t)(kTcHalves * mb) * k_tiles * kTcABytes;  // 128-row tile 2 mb (2 mb + 1 follows)
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
    tmem_alloc(tmem_slot, kTcHalves * kTcBN);  // two 128 x 256 fp32 accumulators: all 512 columns
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
      for (int hh = 0; hh < kTcHalves; ++hh)
        tma_load_1d(dst + hh * kTcABytes, Ab + ((size_t)hh * k_tiles + ks) * kTcABytes, kTcABytes, &full[s], pol);
      tma_load_1d(dst + kTcHalves * kTcABytes, Wb + (size_t)ks * kTcBBytes, kTcBBytes, &full[s], pol);
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
      const uint32_t b0 = a0 + kTcHalves * kTcABytes;
#pragma unroll
      for (int hh = 0; hh < kTcHalves; ++hh)
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
   for (int hh = 0; hh < kTcHalves; ++hh) {
    const int row = (kTcHalves * mb + hh) * kTcBM + warp * 32 + lane;
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
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              *reinterpret_cast<uint4*>(dst + ci + j) =
                  make_uint4(ea[j] | ((uint32_t)ea[j + 1] << 16), ea[j + 2] | ((uint32_t)ea[j + 3] << 16),
                             ea[j + 4] | ((uint32_t)ea[j + 5] << 16), ea[j + 6] | ((uint32_t)ea[j + 7] << 16));
              *reinterpret_cast<uint4*>(dst + ci + half + j) =
                  make_uint4(eb[j] | ((uint32_t)eb[j + 1] << 16), eb[j + 2] | ((uint32_t)eb[j + 3] << 16),
                             eb[j + 4] | ((uint32_t)eb[j + 5] << 16), eb[j + 6] | ((uint32_t)eb[j + 7] << 16));
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
  if (warp == 2) tmem_dealloc(tmem, kTcHalves * kTcBN);
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

cudaError_t tc_gemm(int bf16, int mode, const uint8_t* A_tiled, const uint8_t* W_tiled, float* C, int ldc, int M,
                    int N, int K, int32_t* err, uint64_t wait_ns, cudaStream_t st, const TcQkvEpi* qkv) {
  const int k_tiles = (K + kTcBK - 1) / kTcBK;
  const dim3 grid((M + kTcHalves * kTcBM - 1) / (kTcHalves * kTcBM), (N + kTcBN - 1) / kTcBN);
  const void* kernels[2][4] = {
      {(const void*)tc_gemm_kernel<0, TC_STORE>, (const void*)tc_gemm_kernel<0, TC_ADD>,
       (const void*)tc_gemm_kernel<0, TC_SWIGLU>, (const void*)tc_gemm_kernel<0, TC_QKV>},
      {(const void*)tc_gemm_kernel<1, TC_STORE>, (const void*)tc_gemm_kernel<1, TC_ADD>,
       (const void*)tc_gemm_kernel<1, TC_SWIGLU>, (const void*)tc_gemm_kernel<1, TC_QKV>}};
  TcQkvEpi qe{};
  if (mode == TC_QKV) {
    if (!qkv) return cudaErrorInvalidValue;
    qe = *qkv;
  }
  const void* k = kernels[bf16 ? 1 : 0][mode];
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&A_tiled, (void*)&W_tiled, (void*)&C,   (void*)&ldc,     (void*)&M, (void*)&N,
                  (void*)&k_tiles, (void*)&err,    (void*)&wait_ns, (void*)&qe};
  return cudaLaunchKernel(k, grid, dim3(128), args, kTcSmem, st);
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
// are copied as they are; e4m3 weights become scale x code and NVFP4 weights row scale x (block
// scale x code) (fp32, then RNE to the operand type).
__global__ void tc_unpack_kernel(const uint8_t* __restrict__ image, PhaseDesc P, uint8_t* dst, int k_tiles, int hd,
                                 int hq, int hkv, int ff, const float* sa, const float* sb, const float* sc,
                                 int out_bf16) {
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
      const float s = tc_row_scale(P, row, hd, hq, hkv, ff, sa, sb, sc);
      uint16_t e[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) e[k] = tc_store16(s * w[k], out_bf16);
      v = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16), e[4] | ((uint32_t)e[5] << 16),
                     e[6] | ((uint32_t)e[7] << 16));
    }
    *reinterpret_cast<uint4*>(dst + tile * kTcBBytes + tc_tile_offset(row % kTcBN, col % kTcBK)) = v;
  }
}

cudaError_t tc_unpack(const uint8_t* image, const PhaseDesc& P, int G, int hd, int hq, int hkv, int ff, uint8_t* dst,
                      const float* sa, const float* sb, const float* sc, int out_bf16, cudaStream_t st) {
  const int k_tiles = (P.K + kTcBK - 1) / kTcBK;
  tc_unpack_kernel<<<G, 256, 0, st>>>(image, P, dst, k_tiles, hd, hq, hkv, ff, sa, sb, sc, out_bf16);
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
    const TcQkvEpi qe{a.rope_cos, a.rope_sin, a.kc, a.vc, a.Qt, a.pos0, L, a.hq, a.hkv, a.hd, a.max_ctx, a.kvdt,
                      (P + kTcBM - 1) / kTcBM};
    if ((e = tc_gemm(a.bf16, TC_QKV, a.A, a.wqkv[L], nullptr, 0, P, qkv_n, a.d, a.err, a.wait_ns, st, &qe)) !=
        cudaSuccess)
      return e;
    if ((e = tc_flash(a, qkv_n, L, kt_att, st)) != cudaSuccess) return e;
    if ((e = tc_gemm(a.bf16, TC_ADD, a.A, a.wo[L], a.x, a.d, P, a.d, a.hq * a.hd, a.err, a.wait_ns, st)) != cudaSuccess)
      return e;
    tc_rmsnorm_kernel<<<(P + 7) / 8, 256, 0, st>>>(a.x, (const uint16_t*)a.ffn_norm[L], P, a.d, a.eps, a.bf16, a.A,
                                                   kt_d);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // gate|up with SwiGLU in the epilogue: h goes straight into the down GEMM's A tiles (A2)
    if ((e = tc_gemm(a.bf16, TC_SWIGLU, a.A, a.wgu[L], reinterpret_cast<float*>(a.A2), kt_ff, P, 2 * a.ff, a.d,
                     a.err, a.wait_ns, st)) != cudaSuccess)
      return e;
    if ((e = tc_gemm(a.bf16, TC_ADD, a.A2, a.wdown[L], a.x, a.d, P, a.d, a.ff, a.err, a.wait_ns, st)) != cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

}  // namespace adp

namespace adp {

// Causal attention of the prompt on the tensor cores, flash style.  CTA = query head h x 128
// consecutive prompt tokens (thread t = token t0 + t = TMEM lane t), 128 threads; its queries come
// ready in the core-matrix layout from the QKV GEMM's epilogue.  Per block of
// 128 cached keys: the K block and the V block (transposed) are staged in shared memory in the
// K-major core-matrix layout; S = Q K^T (128 x 128, K = head_dim) accumulates in TMEM columns
// [0, 128); each thread turns its row of S into the online softmax (scale, causal mask, running
// max m and sum l in fp32, the block's probabilities rounded to the KV type into the P tile) and
// rescales its row of O (TMEM columns [128, 128 + head_dim)) by exp(m_old - m_new); then
// O += P V (K = 128 keys).  At the end O / l is rounded into the A-operand tiles of Wo.
template <int HD, int KVDT>
__global__ void __launch_bounds__(128) tc_flash_kernel(const uint8_t* __restrict__ qt, int n_tb, int P, int pos0, int L,
                                                      int hq, int hkv, int max_ctx, float scale,
                                                      const uint16_t* __restrict__ kc,
                                                      const uint16_t* __restrict__ vc, int out_bf16, uint8_t* A,
                                                      int k_tiles, int32_t* err, uint64_t wait_ns) {
  constexpr int KT = HD / kTcBK;                        // 64-wide K tiles of Q and K
  constexpr uint32_t QK_TILE = 128 * kTcBK * 2;         // 16 KB: 128 rows x 64
  constexpr uint32_t VT_TILE = HD * kTcBK * 2;          // V^T tile: head_dim rows x 64 keys
  constexpr int KV_BF16 = KVDT == DT_BF16 ? 1 : 0;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* Qs = smem;                                   // KT tiles
  uint8_t* Ks = Qs + KT * QK_TILE;                      // max(KT, 2) tiles
  uint8_t* Ps = Ks;                                     // P reuses the K block once S is computed
  uint8_t* Vt = Ks + (KT > 2 ? KT : 2) * QK_TILE;       // 2 tiles (keys 0..63, 64..127)
  uint64_t* bar = reinterpret_cast<uint64_t*>(Vt + 2 * VT_TILE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  // the longest causal rows (last query blocks) start first
  const int h = blockIdx.x, t0 = (gridDim.y - 1 - blockIdx.y) * 128;
  const int t = threadIdx.x, warp = t >> 5;
  const int g = h * hkv / hq;
  if (t == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  // the query tiles of (head h, tokens t0 ..), written by the QKV GEMM's epilogue (post-RoPE, KV type)
  {
    const uint4* src = reinterpret_cast<const uint4*>(qt + ((size_t)h * n_tb + t0 / 128) * KT * QK_TILE);
    uint4* dst = reinterpret_cast<uint4*>(Qs);
#pragma unroll 4
    for (int i = t; i < KT * (int)QK_TILE / 16; i += 128) dst[i] = __ldg(src + i);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tmem + lane_base, tO = tmem + lane_base + 128;
  const int pos = pos0 + min(t0 + t, P - 1);            // this row's position (padding rows: the last)
  const int kmax = pos0 + min(t0 + 127, P - 1);
  const size_t head0 = ((size_t)L * hkv + g) * max_ctx;
  constexpr uint32_t idS = tc_idesc_f16(KV_BF16, 128, 128);
  constexpr uint32_t idO = tc_idesc_f16(KV_BF16, 128, HD);
  float m = -INFINITY, l = 0.0f;
  uint32_t phase = 0;
  bool ok = true;
  int32_t never = 0;
  // this thread's key row of the block at kb: K and V, 16-byte chunks (zero past kmax)
  constexpr int NC = HD / 8;
  uint4 kreg[NC], vreg[NC];
  auto load_rows = [&](int kb) {
    const int kp = kb + t;
    const bool in = kp <= kmax;
    const uint4* kr = reinterpret_cast<const uint4*>(kc + (head0 + (in ? kp : 0)) * HD);
    const uint4* vr = reinterpret_cast<const uint4*>(vc + (head0 + (in ? kp : 0)) * HD);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      kreg[c] = in ? __ldg(kr + c) : make_uint4(0, 0, 0, 0);
      vreg[c] = in ? __ldg(vr + c) : make_uint4(0, 0, 0, 0);
    }
  };
  load_rows(0);
  for (int kb0 = 0; kb0 <= kmax && ok; kb0 += 128) {
    // ---- stage key rows kb0 + t (held in registers since the previous block): K as a B operand
    // (keys x head_dim), V transposed (head_dim x keys); then start loading the next block's rows,
    // which arrive while this block's MMAs and softmax run
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int k = c * 8;
      *reinterpret_cast<uint4*>(Ks + (k / kTcBK) * QK_TILE + tc_tile_offset(t, k % kTcBK)) = kreg[c];
      const uint32_t w4[4] = {vreg[c].x, vreg[c].y, vreg[c].z, vreg[c].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint16_t e = (uint16_t)(w4[j >> 1] >> ((j & 1) * 16));
        *reinterpret_cast<uint16_t*>(Vt + (t / kTcBK) * VT_TILE + tc_tile_offset(k + j, t % kTcBK)) = e;
      }
    }
    load_rows(kb0 + 128);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- S = Q K^T
    if (t == 0) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk / 4) * QK_TILE + (kk % 4) * 256;
        tc_mma_f16(tmem, tc_smem_desc(smem_u32(Qs) + off, 128, 1024), tc_smem_desc(smem_u32(Ks) + off, 128, 1024),
                   idS, kk > 0);
      }
      tc_commit(bar);
    }
    __syncwarp();
    ok = mbar_wait(bar, phase, &never, wait_ns);
    phase ^= 1u;
    tc_fence_after();
    // ---- online softmax of row t (its probabilities overwrite the K block, which S no longer needs)
    float mb = -INFINITY;
#pragma unroll
    for (int c0 = 0; c0 < 128; c0 += 32) {
      float v[32];
      tmem_ld32(tS + c0, v);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (kb0 + c0 + j <= pos) mb = fmaxf(mb, v[j] * scale);
    }
    // exponentials by CUDA's fast intrinsic (ex2-based; this path is checked within tolerances)
    const float mn = fmaxf(m, mb);
    const float corr = __expf(m - mn);
    float ps = 0.0f;
#pragma unroll
    for (int c0 = 0; c0 < 128; c0 += 32) {
      float v[32];
      tmem_ld32(tS + c0, v);
      uint16_t e[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float p = kb0 + c0 + j <= pos ? __expf(v[j] * scale - mn) : 0.0f;
        ps += p;
        e[j] = tc_store16(p, KV_BF16);
      }
#pragma unroll
      for (int j = 0; j < 32; j += 8)
        *reinterpret_cast<uint4*>(Ps + ((c0 + j) / kTcBK) * QK_TILE + tc_tile_offset(t, (c0 + j) % kTcBK)) =
            make_uint4(e[j] | ((uint32_t)e[j + 1] << 16), e[j + 2] | ((uint32_t)e[j + 3] << 16),
                       e[j + 4] | ((uint32_t)e[j + 5] << 16), e[j + 6] | ((uint32_t)e[j + 7] << 16));
    }
    l = l * corr + ps;
    m = mn;
    if (kb0 > 0) {  // O *= exp(m_old - m_new) before this block's products are added
#pragma unroll
      for (int c0 = 0; c0 < HD; c0 += 32) {
        float v[32];
        tmem_ld32(tO + c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= corr;
        tmem_st32(tO + c0, v);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- O += P V
    if (t == 0) {
#pragma unroll
      for (int kk = 0; kk < 128 / 16; ++kk) {
        const uint32_t pa = smem_u32(Ps) + (kk / 4) * QK_TILE + (kk % 4) * 256;
        const uint32_t vb = smem_u32(Vt) + (kk / 4) * VT_TILE + (kk % 4) * 256;
        tc_mma_f16(tmem + 128, tc_smem_desc(pa, 128, 1024), tc_smem_desc(vb, 128, 1024), idO, kb0 > 0 || kk > 0);
      }
      tc_commit(bar);
    }
    __syncwarp();
    ok = mbar_wait(bar, phase, &never, wait_ns) && ok;
    phase ^= 1u;
    tc_fence_after();
  }
  // ---- O / l into the Wo GEMM's A tiles
  const int tok = t0 + t;
  if (ok) {
    const float inv = 1.0f / l;
#pragma unroll
    for (int c0 = 0; c0 < HD; c0 += 32) {
      float v[32];
      tmem_ld32(tO + c0, v);
      if (tok < P) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          *reinterpret_cast<uint16_t*>(A + tc_a_offset(tok, h * HD + c0 + j, k_tiles)) =
              tc_store16(v[j] * inv, out_bf16);
      }
    }
  } else if (t == 0) {
    atomicCAS(err, 0, DE_PIPELINE_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

template <int HD, int KVDT>
cudaError_t tc_flash_launch(const TcPrefill& a, int qkv_n, int L, int kt_att, cudaStream_t st) {
  constexpr int KT = HD / kTcBK;
  constexpr size_t smem = (size_t)(KT + (KT > 2 ? KT : 2)) * 128 * kTcBK * 2 + 2 * (size_t)HD * kTcBK * 2 + 64;
  const void* k = (const void*)tc_flash_kernel<HD, KVDT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_flash_kernel<HD, KVDT><<<dim3(a.hq, (a.P + 127) / 128), 128, smem, st>>>(
      a.Qt, (a.P + 127) / 128, a.P, a.pos0, L, a.hq, a.hkv, a.max_ctx, a.scale, a.kc, a.vc, a.bf16, a.A, kt_att,
      a.err, a.wait_ns);
  return cudaGetLastError();
}

cudaError_t tc_flash(const TcPrefill& a, int qkv_n, int L, int kt_att, cudaStream_t st) {
  if (a.kvdt == DT_BF16)
    return a.hd == 128 ? tc_flash_launch<128, DT_BF16>(a, qkv_n, L, kt_att, st)
                       : tc_flash_launch<64, DT_BF16>(a, qkv_n, L, kt_att, st);
  return a.hd == 128 ? tc_flash_launch<128, DT_F16>(a, qkv_n, L, kt_att, st)
                     : tc_flash_launch<64, DT_F16>(a, qkv_n, L, kt_att, st);
}

}  // namespace adp

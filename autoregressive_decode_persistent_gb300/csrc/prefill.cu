// Tensor-core prefill: the weight contractions of a whole prompt as dense GEMMs on the
// fifth-generation tensor cores (tcgen05, accumulators in TMEM), with the norms, RoPE, causal
// attention and SwiGLU between them as plain CUDA kernels.
//
// The pages time-to-first-token as a metric of their own ("標準GPUによるリアルタイムLLM推論：
// リクエストあたり3,000トークン/秒", "単一リクエストLLMデコード速度の重要性") and give no prefill
// algorithm.  Prefill over P prompt tokens is, per layer, matrix-matrix work ([P, d] x [d, n]):
// unlike a decode step it is a dense contraction, so it belongs on the tensor cores.
//
// GEMM: C[M, N] (fp32) = A[M, K] W[N, K]^T with A and W 16-bit (f16 or bf16), both K-major.
// Operands live in global memory already in the tensor cores' shared-memory layout (tc.cuh),
// tile by tile: A as 128-row x 64-K tiles, W as 256-row x 64-K tiles, each contiguous, so one
// 1-D bulk copy stages a tile.  One CTA computes one 128 x 256 output tile: warp 0 streams the
// K-tiles through a 4-stage ring, one thread of warp 1 issues 4 MMAs (K = 16 each) per stage into
// a 128-lane x 256-column fp32 accumulator in TMEM and commits each stage back to the producer,
// and all four warps read the accumulator out (lane = row) when the last MMA has completed.
#include <cuda_runtime.h>

#include <algorithm>

#include "launch.h"
#include "tc.cuh"

namespace adp {

constexpr int kTcBM = 128, kTcBN = 256, kTcStages = 4;
constexpr uint32_t kTcABytes = kTcBM * kTcBK * 2;  // 16 KB
constexpr uint32_t kTcBBytes = kTcBN * kTcBK * 2;  // 32 KB
constexpr uint32_t kTcStageBytes = kTcABytes + kTcBBytes;
constexpr size_t kTcSmem = (size_t)kTcStages * kTcStageBytes + 256;

template <int BF16, bool ADD>
__global__ void __launch_bounds__(128, 1)
    tc_gemm_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ W, float* C, int ldc, int m_valid,
                   int n_valid, int k_tiles, int32_t* err, uint64_t wait_ns) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kTcStages * kTcStageBytes);
  uint64_t* empty = full + kTcStages;
  uint64_t* done = empty + kTcStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int32_t* abort_flag = reinterpret_cast<int32_t*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = blockIdx.x, mb = blockIdx.y;
  const uint8_t* Ab = A + (size_t)mb * k_tiles * kTcABytes;
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
    tmem_alloc(tmem_slot, kTcBN);
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
      tma_load_1d(dst, Ab + (size_t)ks * kTcABytes, kTcABytes, &full[s], pol);
      tma_load_1d(dst + kTcABytes, Wb + (size_t)ks * kTcBBytes, kTcBBytes, &full[s], pol);
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
      const uint32_t b0 = a0 + kTcABytes;
#pragma unroll
      for (int kk = 0; kk < kTcBK / 16; ++kk)
        tc_mma_f16(tmem, tc_smem_desc(a0 + kk * 256, 128, 1024), tc_smem_desc(b0 + kk * 256, 128, 1024), idesc,
                   ks > 0 || kk > 0);
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
    const int row = mb * kTcBM + warp * 32 + lane;
    for (int c0 = 0; c0 < kTcBN; c0 += 32) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
      const int col0 = nb * kTcBN + c0;
      if (row < m_valid) {
        float* dst = C + (size_t)row * ldc + col0;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < n_valid) dst[j] = ADD ? __fadd_rn(dst[j], v[j]) : v[j];
      }
    }
  } else if (threadIdx.x == 0) {
    atomicCAS(err, 0, DE_PIPELINE_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, kTcBN);
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

cudaError_t tc_gemm(int bf16, bool add, const uint8_t* A_tiled, const uint8_t* W_tiled, float* C, int ldc, int M,
                    int N, int K, int32_t* err, uint64_t wait_ns, cudaStream_t st) {
  const int k_tiles = (K + kTcBK - 1) / kTcBK;
  const dim3 grid((N + kTcBN - 1) / kTcBN, (M + kTcBM - 1) / kTcBM);
  const void* k = bf16 ? (add ? (const void*)tc_gemm_kernel<1, true> : (const void*)tc_gemm_kernel<1, false>)
                       : (add ? (const void*)tc_gemm_kernel<0, true> : (const void*)tc_gemm_kernel<0, false>);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&A_tiled, (void*)&W_tiled, (void*)&C, (void*)&ldc, (void*)&M, (void*)&N, (void*)&k_tiles,
                  (void*)&err, (void*)&wait_ns};
  return cudaLaunchKernel(k, grid, dim3(128), args, kTcSmem, st);
}

size_t tc_tiled_bytes(int rows, int K, int tile_rows) {
  const size_t rows_pad = (size_t)(rows + tile_rows - 1) / tile_rows * tile_rows;
  const size_t k_tiles = (size_t)(K + kTcBK - 1) / kTcBK;
  return rows_pad * k_tiles * kTcBK * 2;
}

}  // namespace adp

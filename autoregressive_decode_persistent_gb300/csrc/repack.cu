// Copy the caller's row-major weight matrices into the model-owned image, in the order each
// persistent CTA consumes them: for CTA c, its units [u0, u0 + n) in rounds of `upr` units,
// each round as K-chunks, each chunk as [unit][row][KC elements] (NVFP4: the chunk's codes as
// [unit][row][KC / 2 bytes], then its block scales as [unit][row][KC / 16 bytes]).  One TMA bulk
// copy then moves one tile.  Runs once, at model creation.
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace adp {

// Source row (as a byte pointer) of row j of unit u of phase P, expert e, in the phase's
// matrices a, b, c whose rows are row_bytes long.
__device__ __forceinline__ const uint8_t* source_row(const PhaseDesc& P, const RepackSrc& S, const uint8_t* a,
                                                     const uint8_t* b, const uint8_t* c, uint64_t row_bytes, int u,
                                                     int j, int e) {
  switch (P.kind) {
    case PK_QKV: {
      const int half = S.hd / 2, nq = S.hq * half, nk = S.hkv * half;
      const uint8_t* m = a;
      int uu = u;
      if (u >= nq + nk) { m = c; uu = u - nq - nk; }
      else if (u >= nq) { m = b; uu = u - nq; }
      const int head = uu / half, i = uu % half;
      return m + (uint64_t)(head * S.hd + i + j * half) * row_bytes;
    }
    case PK_GU:
      return (j == 0 ? a : b) + (uint64_t)u * row_bytes;
    case PK_EGU:
      return (j == 0 ? a : b) + (uint64_t)e * S.expert_src_stride + (uint64_t)u * row_bytes;
    case PK_EDOWN:
      return a + (uint64_t)e * S.expert_src_stride + (uint64_t)(u * P.unit_rows + j) * row_bytes;
    default:  // PK_WO, PK_DOWN, PK_LM, PK_ROUTER: row groups
      return a + (uint64_t)(u * P.unit_rows + j) * row_bytes;
  }
}

__global__ void repack_kernel(uint8_t* image, PhaseDesc P, RepackSrc S) {
  const uint32_t c = blockIdx.x, G = gridDim.x;
  const int e = blockIdx.y;
  const long long a0 = (long long)c * P.n_units / G, a1 = (long long)(c + 1) * P.n_units / G;
  const int u0 = (int)a0, n = (int)(a1 - a0);
  if (n <= 0) return;
  const uint64_t unit_bytes = (uint64_t)P.unit_rows * P.K * P.eb;
  uint8_t* dst_cta = image + P.region + (uint64_t)e * P.expert_stride + (uint64_t)u0 * unit_bytes;
  const int per16 = 16 / P.eb;               // elements per 16-byte vector
  const int nv16 = P.K / per16;               // vectors per row
  const long long total = (long long)n * P.unit_rows * nv16;
  for (long long idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int lu = (int)(idx / ((long long)P.unit_rows * nv16));
    const int rem = (int)(idx % ((long long)P.unit_rows * nv16));
    const int j = rem / nv16, cv = rem % nv16;
    const int col = cv * per16;
    const int ck = col / P.KC;
    const int kck = min(P.KC, P.K - ck * P.KC);
    const int r = lu / P.upr, i = lu % P.upr;
    const int m = min(P.upr, n - r * P.upr);
    const uint64_t off = (uint64_t)r * P.upr * unit_bytes + (uint64_t)m * P.unit_rows * ck * P.KC * P.eb +
                         ((uint64_t)(i * P.unit_rows + j) * kck + (col - ck * P.KC)) * P.eb;
    const uint8_t* src = source_row(P, S, S.a, S.b, S.c, (uint64_t)P.K * P.eb, u0 + lu, j, e) + (uint64_t)col * P.eb;
    *reinterpret_cast<uint4*>(dst_cta + off) = *reinterpret_cast<const uint4*>(src);
  }
}

// NVFP4 layer matrices (dense phases only): per 16-element block of a row, its 8 code bytes and
// its scale byte, each into its part of the tile (codes of all the tile's rows, then their scales).
__global__ void repack_nvfp4_kernel(uint8_t* image, PhaseDesc P, RepackSrc S) {
  const uint32_t c = blockIdx.x, G = gridDim.x;
  const long long a0 = (long long)c * P.n_units / G, a1 = (long long)(c + 1) * P.n_units / G;
  const int u0 = (int)a0, n = (int)(a1 - a0);
  if (n <= 0) return;
  const uint64_t unit_bytes = wbytes(P, (uint64_t)P.unit_rows * P.K);
  uint8_t* dst_cta = image + P.region + (uint64_t)u0 * unit_bytes;
  const int nb16 = P.K / 16;  // blocks per row
  const long long total = (long long)n * P.unit_rows * nb16;
  for (long long idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int lu = (int)(idx / ((long long)P.unit_rows * nb16));
    const int rem = (int)(idx % ((long long)P.unit_rows * nb16));
    const int j = rem / nb16, cb = rem % nb16;
    const int col = cb * 16;
    const int ck = col / P.KC;
    const int kck = min(P.KC, P.K - ck * P.KC);
    const int r = lu / P.upr, i = lu % P.upr;
    const int m = min(P.upr, n - r * P.upr);
    const uint64_t tile = (uint64_t)r * P.upr * unit_bytes + wbytes(P, (uint64_t)m * P.unit_rows * ck * P.KC);
    const uint64_t row = (uint64_t)i * P.unit_rows + j, kc0 = (uint64_t)(col - ck * P.KC);
    const uint8_t* src = source_row(P, S, S.a, S.b, S.c, (uint64_t)P.K / 2, u0 + lu, j, 0) + (uint64_t)cb * 8;
    const uint8_t* srs = source_row(P, S, S.sa, S.sb, S.sc, (uint64_t)P.K / 16, u0 + lu, j, 0) + cb;
    *reinterpret_cast<uint2*>(dst_cta + tile + row * (kck / 2) + kc0 / 2) = *reinterpret_cast<const uint2*>(src);
    dst_cta[tile + (uint64_t)m * P.unit_rows * (kck / 2) + row * (kck / 16) + kc0 / 16] = *srs;
  }
}

cudaError_t repack_launch(uint8_t* image, const PhaseDesc& P, const RepackSrc& S, int grid, int experts,
                          cudaStream_t stream) {
  if (P.wdt == DT_NVFP4)
    repack_nvfp4_kernel<<<dim3(grid, 1), 256, 0, stream>>>(image, P, S);
  else
    repack_kernel<<<dim3(grid, experts), 256, 0, stream>>>(image, P, S);
  return cudaGetLastError();
}

}  // namespace adp

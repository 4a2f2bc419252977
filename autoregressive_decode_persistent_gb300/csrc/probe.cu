// Read-bandwidth probe: streams a caller-given device buffer through the SMs with 16-byte loads
// and reports GB/s, so that a decode measurement can be set against the read bandwidth this GPU
// delivers in the same process (the bound on batch-1 decode is read bandwidth: every weight is
// read once per token; "標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒",
// hakusoku.com, section "GPU推論の速度制限要因：メモリ帯域幅").
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/adp.h"

namespace {

// Each thread reads four 16-byte vectors per iteration (grid-stride), folds them with xor and
// stores the fold only if it equals a value no buffer of this probe is expected to produce, so the
// loads cannot be removed and (in practice) nothing is written.
__global__ void read_probe_kernel(const uint4* __restrict__ src, uint64_t n16, uint32_t* sink) {
  uint32_t acc = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(v[k].x), "=r"(v[k].y), "=r"(v[k].z), "=r"(v[k].w)
                   : "l"(src + i + k * stride));
#pragma unroll
    for (int k = 0; k < 4; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = src[i];
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9E3779B9u) sink[0] = acc;
}

}  // namespace

extern "C" int adp_measure_read_bandwidth(const void* dev_buf, uint64_t bytes, int32_t reps, void* cuda_stream,
                                          double* gb_per_s) {
  if (!dev_buf || bytes < 16 || reps < 1 || !gb_per_s || ((uintptr_t)dev_buf & 15)) return ADP_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
    return ADP_ERR_CUDA;
  const uint64_t n16 = bytes / 16;
  const dim3 grid((unsigned)(sms * 4)), block(512);
  auto* src = static_cast<const uint4*>(dev_buf);
  auto* sink = const_cast<uint32_t*>(static_cast<const uint32_t*>(dev_buf));
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return ADP_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return ADP_ERR_CUDA;
  }
  read_probe_kernel<<<grid, block, 0, st>>>(src, n16, sink);  // warm-up
  cudaEventRecord(e0, st);
  for (int r = 0; r < reps; ++r) read_probe_kernel<<<grid, block, 0, st>>>(src, n16, sink);
  cudaEventRecord(e1, st);
  cudaError_t e = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e == cudaSuccess) e = cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess || ms <= 0.0f) return ADP_ERR_CUDA;
  *gb_per_s = (double)(n16 * 16) * reps / (ms * 1e-3) / 1e9;
  return ADP_OK;
}

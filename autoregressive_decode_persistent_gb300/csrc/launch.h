// Host-side entry points of the CUDA translation units (engine <-> kernels).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "plan.h"

namespace adp {

// Source matrices of one phase for the repack into the tile-ordered image.
struct RepackSrc {
  const uint8_t* a;            // wq / wo / w_gate / w_down / head / router / e_gate / e_down
  const uint8_t* b;            // wk / w_up / e_up
  const uint8_t* c;            // wv
  const uint8_t* sa;           // NVFP4 only: the block scales [rows][K / 16] of a, b, c
  const uint8_t* sb;
  const uint8_t* sc;
  uint64_t expert_src_stride;  // bytes of one expert's matrix in the caller's [E, rows, K] tensor
  int32_t hd, hq, hkv;
};

// kind: KernelKind; hd, kvdt and t16 (the 16-bit weight type of a 16-bit model, else the embedding's)
// select the kernel instantiation, as decode_launch does from the parameters
cudaError_t decode_prepare(size_t smem_bytes, int kind, int hd, int kvdt, int t16, int* blocks_per_sm);
cudaError_t decode_launch(const Params& p, int ph0, int ph1, bool persistent, int grid, size_t smem_bytes,
                          int xbuf_floats, cudaStream_t stream);
cudaError_t repack_launch(uint8_t* image, const PhaseDesc& P, const RepackSrc& S, int grid, int experts,
                          cudaStream_t stream);
size_t ctl_bytes(int n_phases);  // control block + phase table in shared memory
// The batched kernel (KK_BATCH): always one persistent cooperative launch.  Its shared memory
// adds batch_ctl_bytes() after ctl_bytes(n_phases).
cudaError_t decode_batch_prepare(size_t smem_bytes, int* blocks_per_sm);
// down_seg: elements of each request's down-projection input staged in shared memory at once
// (the FFN width: whole; less: segments, refetched as the GEMV reaches them).
cudaError_t decode_batch_launch(const Params& p, int ph0, int ph1, int grid, size_t smem_bytes, int xbuf_floats,
                                int down_seg, cudaStream_t stream);
size_t batch_ctl_bytes();

// Epilogues of the prefill GEMM: C = A W^T (fp32, streaming stores), C += A W^T (the fp32
// residual), or SwiGLU of interleaved (gate, up) output column pairs rounded into the next GEMM's
// A tiles (C is then that tile buffer and ldc its number of 64-wide K tiles).
enum TcMode : int { TC_STORE = 0, TC_ADD = 1, TC_SWIGLU = 2, TC_QKV = 3 };

// The QKV GEMM's epilogue (TC_QKV): RoPE on the q and k columns of each token (position pos0 + row),
// q rounded into the attention kernel's query tiles, k and v rounded into the KV cache rows.
struct TcQkvEpi {
  const float* rope_cos;  // [max_ctx][hd/2]
  const float* rope_sin;
  uint16_t* kc;           // [L][hkv][max_ctx][hd]
  uint16_t* vc;
  uint8_t* qt;            // [hq][ceil(P/128)][hd/64 tiles of 128 x 64]: queries in the core-matrix layout
  uint8_t* kt;            // [hkv][n_kb][hd/64 tiles of 128 keys x 64]: keys by position, the same layout
  uint8_t* vt;            // [hkv][n_kb][2 tiles of hd x 64 keys]: values by position, transposed
  int pos0, L, hq, hkv, hd, max_ctx, kvdt, n_tb, n_kb;
};

// Tensor-core GEMM of the prefill path (prefill.cu): A W^T with A and W in the tiled tensor-core
// layout (A: 128-row tiles, rows allocated in multiples of 256; W: 256-row tiles; 64 K-elements
// each), epilogue `mode`.
// colscale (optional, device [N]): every output column is multiplied by its entry first (the row
// scales of quantised weights, whose operand tiles hold the exact codes).
cudaError_t tc_gemm(int bf16, int mode, const uint8_t* A_tiled, const uint8_t* W_tiled, float* C, int ldc, int M,
                    int N, int K, int32_t* err, uint64_t wait_ns, cudaStream_t st, const TcQkvEpi* qkv = nullptr,
                    const float* colscale = nullptr);
// Row-major 16-bit [rows, K] (row stride ld) -> tiles of tile_rows x 64, zero-padded.
cudaError_t tc_tile(const uint16_t* src, int rows, int K, int ld, uint8_t* dst, int tile_rows, cudaStream_t st);
size_t tc_tiled_bytes(int rows, int K, int tile_rows);

// One tensor-core prefill of P prompt tokens at positions pos0 .. pos0 + P - 1 through every
// layer: K/V rows into the cache; x ends as the residual after the last layer.
struct TcPrefill {
  int P, pos0, n_layers, d, hq, hkv, hd, ff, max_ctx, bf16, kvdt;
  float eps, scale;
  const int32_t* tokens;        // device [P]
  const void* tok_emb;          // device [V, d] (16-bit)
  const void* const* attn_norm;  // host array [L] of device gains
  const void* const* ffn_norm;
  const uint8_t* const* wqkv;   // host arrays [L] of device tiled weights (256-row tiles)
  const uint8_t* const* wo;
  const uint8_t* const* wgu;
  const uint8_t* const* wdown;
  const float* const* sqkv;     // host arrays [L] of device column scales (quantised weights), or null
  const float* const* swo;
  const float* const* sgu;
  const float* const* sdown;
  uint16_t* kc;
  uint16_t* vc;
  const float* rope_cos;
  const float* rope_sin;
  float* x;        // device [P, d]
  uint8_t* A;      // device A-operand tiles, rows padded to 256, K up to max(d, hq*hd)
  uint8_t* A2;     // device A-operand tiles of the down GEMM (K = ff), written by gate|up's epilogue
  uint8_t* Qt;     // device query tiles written by the QKV GEMM's epilogue (see TcQkvEpi)
  uint8_t* Kt;     // device key and transposed value tiles of every position (see TcQkvEpi), zeroed
  uint8_t* Vt;     // at allocation so that positions never written read as finite values
  int n_kb;        // 128-key blocks in Kt and Vt: ceil(max_ctx / 128)
  int32_t* err;
  uint64_t wait_ns;
};
cudaError_t tc_prefill(const TcPrefill& a, cudaStream_t st);
// Phase P's tiles of the decode image -> one GEMM weight operand in 256-row tiles (dst cleared
// beforehand; rows in the order of the caller's matrices, except gate|up: gate_i and up_i
// interleaved as rows 2i and 2i + 1).
// 16-bit phases are copied; e4m3 codes and NVFP4 block scale x code are written exactly in the
// operand type (out_bf16), their row scales left to the GEMM's column scales (tc_colscale).
cudaError_t tc_unpack(const uint8_t* image, const PhaseDesc& P, int G, int hd, int hq, int hkv, int ff, uint8_t* dst,
                      int out_bf16, cudaStream_t st);
// The column scales of phase P's GEMM (rows of its operand): out[row] = the row scale of that row
// (sa, sb, sc: the q/k/v, gate/up or single matrix's tables).
cudaError_t tc_colscale(const PhaseDesc& P, int rows, int hd, int hq, int hkv, int ff, const float* sa,
                        const float* sb, const float* sc, float* out, cudaStream_t st);

}  // namespace adp

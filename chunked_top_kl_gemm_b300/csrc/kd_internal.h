// Internal interface between the C-ABI layer (kd_api.cu) and the kernels
// (kd_kernels.cu).  Not installed; not part of the public header.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kd_args.h"
#include "kd_ptx.cuh"

namespace kd {

// GEMM variants of the path (one template instantiation each).
enum GemmVariant {
  GV_FWD = 0,       // K1: hidden_c * W^T, forward epilogue (lse partials + gather)
  GV_DZ = 1,        // K3: hidden_c * W^T recomputed, dZ epilogue (bf16 store)
  GV_GRAD_H = 2,    // K4: (dZ W)^T = W^T dZ^T (A MN-major), fp32 split-K partials
  GV_GRAD_W = 3,    // K5: dZ^T * hidden (A and B MN-major), fp32 reduce-add
  GV_TEST_KK = 4,   // test GEMMs: fp32 store, all four major combinations
  GV_TEST_KM = 5,
  GV_TEST_MK = 6,
  GV_TEST_MM = 7,
  GV_TEST_KK192 = 8,   // the same four layouts with the other tile width
  GV_TEST_KM256 = 9,
  GV_TEST_MK256 = 10,
  GV_TEST_MM256 = 11,
  GV_TEST_KK2 = 12,    // the four layouts on a CTA pair (256 x 256 tiles)
  GV_TEST_KM2 = 13,
  GV_TEST_MK2 = 14,
  GV_TEST_MM2 = 15,
  GV_FWDZ = 16,        // K1 that also stores the chunk's fp32 logits
  GV_TEST_KK2S = 17,   // pair, K-major operands, two k-blocks per ring stage
  GV_DZFWD = 18,       // K3 of chunk j and K1 of chunk j+1 in one launch (W streamed once)
};

// Tile width of the N dimension of each variant.
int gemm_bn(int variant);
// M of one work unit of each variant (128, or 256 on a CTA pair).
int gemm_tile_m(int variant);
// Dynamic shared memory of each variant.
int gemm_smem(int variant);
// Work units of each variant that run at once on this device (SMs, or
// co-resident CTA pairs).
int gemm_width(int variant);

// Launch a persistent GEMM over the units of g (grid sized by the launcher).
cudaError_t launch_gemm(int variant, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& o, const GemmArgs& g, const EpiArgs& e,
                        cudaStream_t s);

cudaError_t launch_prep_topk(const int32_t* idx, const float* logit, long long N, int K, int V,
                             float T, int* sid, float* sp, int* perm, double* ent, double* psum,
                             DevStatus* st, cudaStream_t s);

cudaError_t launch_lse_loss(const float2* part, int n_tiles, int c_alloc, int rows_valid, int grow0,
                            const float* zg, const float* sp, const int* perm, const double* ent,
                            const double* psum, int K, float T, const uint8_t* mask, float* lse2,
                            double* loss_rows, float* dbg_lse, float* dbg_zg, cudaStream_t s);

cudaError_t launch_split_reduce_t(const float* part, int splits, long long split_stride,
                                  int c_alloc, int rows_valid, int H, float alpha,
                                  const float* alpha_dev, int accumulate, float* out,
                                  cudaStream_t s);

// dZ of rows [0, rows_cover) of a chunk from its stored fp32 logits z
// [rows][V] (rows >= rows_valid and masked rows get zeros), then the
// cached-id columns.
cudaError_t launch_dz_from_z(const float* z, int V, int rows_valid, int rows_cover,
                             const float* lse2, float scale2, const uint8_t* mask, int grow0,
                             const int* sid, const float* sp, int K, void* dz, cudaStream_t s);

// Top-K cache rows [0, rows_valid) of a chunk from its stored logits z
// [rows][V] and per-tile maxima part[n_tiles][c_alloc].x, written to rows
// row0.. of out_idx / out_val [N][K].  K <= 8192.  Scratch: tau and cnt
// [rows_valid], cand [rows_valid][SEL_GCAP].
constexpr int SEL_GCAP = 2048;   // candidates one row's list holds
cudaError_t launch_topk_select(const float* z, int V, const float2* part, int n_tiles,
                               int c_alloc, int rows_valid, int K, long long row0, float* tau,
                               uint32_t* cnt, unsigned long long* cand, int32_t* out_idx,
                               float* out_val, cudaStream_t s);

cudaError_t launch_mask_count(const uint8_t* mask, long long N, float T, DevStatus* st,
                              cudaStream_t s);


// Device-side results of an asynchronous call (loss == nullptr: none).
struct FinalOut {
  float* loss;        // the mean loss over N (masked: over the valid tokens)
  int* status;        // 0, or code_timeout / code_index from the error word
  int masked;
  int code_timeout, code_index;
};
cudaError_t launch_loss_final(const double* loss_rows, long long N, DevStatus* st,
                              const FinalOut& out, cudaStream_t s);

}  // namespace kd

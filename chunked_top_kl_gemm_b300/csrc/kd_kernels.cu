// Kernels of the fused chunked top-K KL loss (forward + backward) for sm_103a.
//
// The method (Multiverse Computing, "Efficient Knowledge Distillation for
// LLMs: Offline Top-K Logits and a Fused Chunked KL Loss", as summarised on
// glonce.com, body, and ainewsbank.com, "Two changes remove different
// bottlenecks"): per token chunk, project hidden states to logits, fold the
// chunk into the running loss and discard it; in the backward pass recompute
// each chunk's logits instead of storing them.  The teacher side is an offline
// cache of the K highest teacher logits and their ids per token (epoka.news,
// "The two proposed changes").
//
// Kernels (per call; chunk loop on the host, all launches on one stream):
//   prep_topk     teacher p = softmax(l/T) over the K cached entries, its
//                 sum p*log p, ids sorted per row (with p and the permutation)
//   GEMM FWD      z = h_c W^T on tcgen05, epilogue: online max/sum of
//                 2^(z log2e/T) per (row, 256-wide vocab tile) + gather of z
//                 at the cached ids          [kd_gemm.cuh]
//   lse_loss      combine the per-tile partials into logsumexp, fold the row's
//                 KL term  sum_k p (log p - z_idx/T + lse)
//   GEMM DZ       recompute z, G = softmax(z/T) - scatter(p) -> bf16 scratch
//   GEMM GRAD_H   split-K  G W  -> fp32 partials;  split_reduce sums them
//                 and scales by 1/(T N) into grad_hidden
//   GEMM GRAD_W   G^T h_c scaled by 1/(T N), TMA reduce-added into grad_W
//   loss_final    ordered sum of the per-token terms
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kd_gemm.cuh"
#include "kd_internal.h"

namespace kd {

using CfgFwd = GemmCfg<256, false, false, 4, EPI_FWD>;
using CfgDz = GemmCfg<256, false, false, 4, EPI_DZ>;
using CfgGradH = GemmCfg<192, false, true, 4, EPI_F32>;
using CfgGradW = GemmCfg<192, true, true, 4, EPI_ACC>;
using CfgTestKK = GemmCfg<256, false, false, 4, EPI_F32>;
using CfgTestKM = GemmCfg<192, false, true, 4, EPI_F32>;
using CfgTestMK = GemmCfg<192, true, false, 4, EPI_F32>;
using CfgTestMM = GemmCfg<192, true, true, 4, EPI_F32>;

template <class C>
static cudaError_t launch_cfg(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                              const GemmArgs& g, const EpiArgs& e, int grid, cudaStream_t s) {
  static bool attr_set = false;  // per instantiation; set once per process
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(kd_gemm_kernel<C>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  kd_gemm_kernel<C><<<grid, NUM_THREADS, C::SMEM_BYTES, s>>>(a, b, o, g, e);
  return cudaGetLastError();
}

int gemm_bn(int variant) {
  switch (variant) {
    case GV_FWD: return CfgFwd::BN;
    case GV_DZ: return CfgDz::BN;
    case GV_GRAD_H: return CfgGradH::BN;
    case GV_GRAD_W: return CfgGradW::BN;
    case GV_TEST_KK: return CfgTestKK::BN;
    case GV_TEST_KM: return CfgTestKM::BN;
    case GV_TEST_MK: return CfgTestMK::BN;
    case GV_TEST_MM: return CfgTestMM::BN;
  }
  return 0;
}

int gemm_smem(int variant) {
  switch (variant) {
    case GV_FWD: return CfgFwd::SMEM_BYTES;
    case GV_DZ: return CfgDz::SMEM_BYTES;
    case GV_GRAD_H: return CfgGradH::SMEM_BYTES;
    case GV_GRAD_W: return CfgGradW::SMEM_BYTES;
    case GV_TEST_KK: return CfgTestKK::SMEM_BYTES;
    case GV_TEST_KM: return CfgTestKM::SMEM_BYTES;
    case GV_TEST_MK: return CfgTestMK::SMEM_BYTES;
    case GV_TEST_MM: return CfgTestMM::SMEM_BYTES;
  }
  return 0;
}

cudaError_t launch_gemm(int variant, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& o, const GemmArgs& g, const EpiArgs& e, int grid,
                        cudaStream_t s) {
  switch (variant) {
    case GV_FWD: return launch_cfg<CfgFwd>(a, b, o, g, e, grid, s);
    case GV_DZ: return launch_cfg<CfgDz>(a, b, o, g, e, grid, s);
    case GV_GRAD_H: return launch_cfg<CfgGradH>(a, b, o, g, e, grid, s);
    case GV_GRAD_W: return launch_cfg<CfgGradW>(a, b, o, g, e, grid, s);
    case GV_TEST_KK: return launch_cfg<CfgTestKK>(a, b, o, g, e, grid, s);
    case GV_TEST_KM: return launch_cfg<CfgTestKM>(a, b, o, g, e, grid, s);
    case GV_TEST_MK: return launch_cfg<CfgTestMK>(a, b, o, g, e, grid, s);
    case GV_TEST_MM: return launch_cfg<CfgTestMM>(a, b, o, g, e, grid, s);
  }
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ prep
// One warp per token row.  Teacher distribution over the K cached entries:
// a_k = l_k / T, log p_k = a_k - logsumexp(a), p_k = exp(log p_k) (double).
// Writes the row's ids sorted ascending (ties by original position) with p
// and the original position alongside, sum_k p log p and sum_k p.  An id
// outside [0, V) raises DEV_ERR_INDEX.
__global__ void __launch_bounds__(256) kd_prep_topk(const int32_t* __restrict__ idx,
                                                    const float* __restrict__ logit, long long N,
                                                    int K, int V, double invT,
                                                    int* __restrict__ sid, float* __restrict__ sp,
                                                    int* __restrict__ perm,
                                                    double* __restrict__ ent,
                                                    double* __restrict__ psum, DevStatus* st) {
  extern __shared__ int s_ids[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + warp;
  if (r >= N) return;
  int* ids = s_ids + warp * K;
  const int32_t* id_row = idx + r * K;
  const float* l_row = logit + r * K;
  double m = -CUDART_INF;
  bool bad = false;
  for (int k = lane; k < K; k += 32) {
    const int id = id_row[k];
    ids[k] = id;
    bad |= (id < 0) || (id >= V);
    m = fmax(m, static_cast<double>(l_row[k]) * invT);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&st->err, DEV_ERR_INDEX);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, o));
  double s = 0.0;
  for (int k = lane; k < K; k += 32) s += exp(static_cast<double>(l_row[k]) * invT - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const double lse_t = m + log(s);
  __syncwarp();
  double e_acc = 0.0, p_acc = 0.0;
  for (int k = lane; k < K; k += 32) {
    const double lp = static_cast<double>(l_row[k]) * invT - lse_t;
    const double p = exp(lp);
    e_acc += p * lp;
    p_acc += p;
    const int idk = ids[k];
    int rank = 0;
    for (int j = 0; j < K; ++j) {
      const int idj = ids[j];
      rank += (idj < idk) || (idj == idk && j < k);
    }
    sid[r * K + rank] = idk;
    sp[r * K + rank] = static_cast<float>(p);
    perm[r * K + rank] = k;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    e_acc += __shfl_xor_sync(0xffffffffu, e_acc, o);
    p_acc += __shfl_xor_sync(0xffffffffu, p_acc, o);
  }
  if (lane == 0) {
    ent[r] = e_acc;
    psum[r] = p_acc;
  }
}

cudaError_t launch_prep_topk(const int32_t* idx, const float* logit, long long N, int K, int V,
                             float T, int* sid, float* sp, int* perm, double* ent, double* psum,
                             DevStatus* st, cudaStream_t s) {
  int wpb = 32768 / (K * 4);
  wpb = wpb < 1 ? 1 : (wpb > 8 ? 8 : wpb);
  const long long blocks = (N + wpb - 1) / wpb;
  const size_t smem = static_cast<size_t>(wpb) * K * 4;
  kd_prep_topk<<<static_cast<unsigned>(blocks), wpb * 32, smem, s>>>(
      idx, logit, N, K, V, 1.0 / static_cast<double>(T), sid, sp, perm, ent, psum, st);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ lse + loss fold
// One thread per chunk row: combine the (max, sum) partials of every vocab
// tile (log2 units) into lse2 = log2 sum_v 2^(z_v log2e / T), then the row's
// KL term  sum_k p_k (log p_k - z_k/T + lse)  with lse = lse2 * ln 2.
__global__ void __launch_bounds__(128) kd_lse_loss(
    const float2* __restrict__ part, int n_tiles, int c_alloc, int rows_valid, int grow0,
    const float* __restrict__ zg, const float* __restrict__ sp, const int* __restrict__ perm,
    const double* __restrict__ ent, const double* __restrict__ psum, int K, double invT,
    float* __restrict__ lse2_out, double* __restrict__ loss_rows, float* __restrict__ dbg_lse,
    float* __restrict__ dbg_zg) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows_valid) return;
  float M = -CUDART_INF_F;
  double S = 0.0;
  for (int t = 0; t < n_tiles; ++t) {
    const float2 v = part[static_cast<long long>(t) * c_alloc + r];
    if (v.x > M) {
      S = S * static_cast<double>(exp2f(M - v.x)) + static_cast<double>(v.y);
      M = v.x;
    } else {
      S += static_cast<double>(v.y) * static_cast<double>(exp2f(v.x - M));
    }
  }
  const double lse2 = static_cast<double>(M) + log2(S);
  lse2_out[r] = static_cast<float>(lse2);
  const double lse = lse2 * 0.69314718055994530942;  // ln 2
  const long long g = static_cast<long long>(grow0) + r;
  double dot = 0.0;
  for (int j = 0; j < K; ++j) {
    const float z = zg[static_cast<long long>(r) * K + j];
    dot += static_cast<double>(sp[g * K + j]) * static_cast<double>(z);
    if (dbg_zg) dbg_zg[g * K + perm[g * K + j]] = z;
  }
  loss_rows[g] = ent[g] + lse * psum[g] - dot * invT;
  if (dbg_lse) dbg_lse[g] = static_cast<float>(lse);
}

cudaError_t launch_lse_loss(const float2* part, int n_tiles, int c_alloc, int rows_valid, int grow0,
                            const float* zg, const float* sp, const int* perm, const double* ent,
                            const double* psum, int K, float T, float* lse2, double* loss_rows,
                            float* dbg_lse, float* dbg_zg, cudaStream_t s) {
  const int blocks = (rows_valid + 127) / 128;
  kd_lse_loss<<<blocks, 128, 0, s>>>(part, n_tiles, c_alloc, rows_valid, grow0, zg, sp, perm, ent,
                                     psum, K, 1.0 / static_cast<double>(T), lse2, loss_rows,
                                     dbg_lse, dbg_zg);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ split-K reduce
// out[r][h] = alpha * sum_s part[s][r][h] for r < rows_valid (fixed order).
__global__ void __launch_bounds__(256) kd_split_reduce(const float4* __restrict__ part, int splits,
                                                       int c_alloc, int rows_valid, int H4,
                                                       float alpha, float4* __restrict__ out) {
  const long long total = static_cast<long long>(rows_valid) * H4;
  const long long plane = static_cast<long long>(c_alloc) * H4;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = part[s * plane + i];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    a.x *= alpha; a.y *= alpha; a.z *= alpha; a.w *= alpha;
    out[i] = a;
  }
}

cudaError_t launch_split_reduce(const float* part, int splits, int c_alloc, int rows_valid, int H,
                                float alpha, float* out, cudaStream_t s) {
  const int H4 = H / 4;
  const long long total = static_cast<long long>(rows_valid) * H4;
  long long blocks = (total + 255) / 256;
  if (blocks > 148 * 8) blocks = 148 * 8;
  if (blocks < 1) blocks = 1;
  kd_split_reduce<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      reinterpret_cast<const float4*>(part), splits, c_alloc, rows_valid, H4, alpha,
      reinterpret_cast<float4*>(out));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ final loss
__global__ void __launch_bounds__(1024) kd_loss_final(const double* __restrict__ loss_rows,
                                                      long long N, DevStatus* st) {
  __shared__ double red[1024];
  double a = 0.0;
  for (long long i = threadIdx.x; i < N; i += 1024) a += loss_rows[i];
  red[threadIdx.x] = a;
  __syncthreads();
  for (int o = 512; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) st->loss_sum = red[0];
}

cudaError_t launch_loss_final(const double* loss_rows, long long N, DevStatus* st, cudaStream_t s) {
  kd_loss_final<<<1, 1024, 0, s>>>(loss_rows, N, st);
  return cudaGetLastError();
}

}  // namespace kd

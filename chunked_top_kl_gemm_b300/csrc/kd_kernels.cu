// Kernels of the fused chunked top-K KL loss (forward + backward) for sm_103a.
//
// The method (Multiverse Computing, "Efficient Knowledge Distillation for
// LLMs: Offline Top-K Logits and a Fused Chunked KL Loss", as summarised on
// glonce.com, body, and ainewsbank.com, "Two changes remove different
// bottlenecks"): a token chunk's logits are formed, reduced into the running
// loss and dropped, and the backward pass forms them again rather than
// keeping them.  The teacher side is an offline
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
//   GEMM GRAD_H   split-K  (G W)^T = W^T G^T -> fp32 partials [split][H][c];
//                 split_reduce_t sums them, transposes and scales by 1/(T N)
//                 into grad_hidden
//   GEMM GRAD_W   G^T h scaled by 1/(T N) over a pair of chunks' rows (h read
//                 MN-major), TMA reduce-added into grad_W
//   loss_final    ordered sum of the per-token terms
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <atomic>

#include "kd_gemm.cuh"
#include "kd_internal.h"

namespace kd {

// The loss's GEMMs run on CTA pairs (2-CTA MMA, 256 x 256 tiles): per SM
// they pull 32 KB of operands from L2 per 64-deep k-block instead of 48 KB.
// FWD and DZ stream L2-resident operands and are bound by the MMA issue:
// two 64-deep k-blocks per ring stage halve the issuer's waits and commits.
// The gradient GEMMs wait on DRAM-fed operands and keep finer stages.
using CfgFwd = GemmCfg<256, false, false, 3, EPI_FWD, true, 2>;
using CfgDz = GemmCfg<256, false, false, 3, EPI_DZ, true, 2>;
// the recompute of one chunk and the forward of the next in one launch
using CfgDzFwd = GemmCfg<256, false, false, 3, EPI_DZFWD, true, 2>;
using CfgGradH = GemmCfg<256, true, false, 6, EPI_F32, true>;   // grad_hidden^T = W^T dZ^T
using CfgGradW = GemmCfg<256, true, true, 6, EPI_ACC, true>;    // grad_W = dZ^T h_c (h_c MN-major)
// forward that also keeps the chunk's fp32 logits (backward without recompute)
using CfgFwdZ = GemmCfg<256, false, false, 3, EPI_FWDZ, true, 2>;
// single-CTA forms (128 x BN tiles), kept for the GEMM-core tests
using CfgTestKK = GemmCfg<256, false, false, 4, EPI_F32>;
using CfgTestKM = GemmCfg<192, false, true, 4, EPI_F32>;
using CfgTestMK = GemmCfg<192, true, false, 4, EPI_F32>;
using CfgTestMM = GemmCfg<192, true, true, 4, EPI_F32>;
using CfgTestKK192 = GemmCfg<192, false, false, 4, EPI_F32>;
using CfgTestKM256 = GemmCfg<256, false, true, 4, EPI_F32>;
using CfgTestMK256 = GemmCfg<256, true, false, 4, EPI_F32>;
using CfgTestMM256 = GemmCfg<256, true, true, 4, EPI_F32>;
// pair forms of the four operand layouts
using CfgTestKK2 = GemmCfg<256, false, false, 6, EPI_F32, true>;
using CfgTestKM2 = GemmCfg<256, false, true, 6, EPI_F32, true>;
using CfgTestMK2 = GemmCfg<256, true, false, 6, EPI_F32, true>;
using CfgTestMM2 = GemmCfg<256, true, true, 6, EPI_F32, true>;
// pair form with two k-blocks per stage (the FWD / DZ ring)
using CfgTestKK2S = GemmCfg<256, false, false, 3, EPI_F32, true, 2>;

// Work units that can run at once on the current device: one per SM, or one
// per co-resident CTA pair (queried once per instantiation and device).
template <class C>
static int resident_units() {
  constexpr int kMaxDev = 64;
  // host threads may query at once: relaxed atomics (every writer stores
  // the same value)
  static std::atomic<int> cached[kMaxDev];
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  if (dev >= 0 && dev < kMaxDev) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  if (dev >= 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 148;
  }
  int width = sms;
  if constexpr (C::CTA2) {
    width = sms / 2;
    if (cudaFuncSetAttribute(kd_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess) {
      cudaGetLastError();
      return width;     // no device: do not cache the guess
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kd_gemm_kernel<C>, &cfg) == cudaSuccess &&
        clusters > 0)
      width = clusters;
    else
      cudaGetLastError();
  }
  if (dev >= 0 && dev < kMaxDev) cached[dev].store(width, std::memory_order_relaxed);
  return width;
}

template <class C>
static cudaError_t launch_cfg(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                              const GemmArgs& g, const EpiArgs& e, cudaStream_t s) {
  static std::atomic<bool> attr_set[64];  // per instantiation and device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    err = cudaFuncSetAttribute(kd_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  const long long units = static_cast<long long>(g.m_tiles) * g.n_tiles * g.splits;
  if (units <= 0) return cudaSuccess;
  const int width = resident_units<C>();
  const int grid_units = static_cast<int>(units < width ? units : width);
  if constexpr (!C::CTA2) {
    kd_gemm_kernel<C><<<grid_units, NUM_THREADS, C::SMEM_BYTES, s>>>(a, b, o, g, e);
    return cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * grid_units, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kd_gemm_kernel<C>, a, b, o, g, e);
  }
}

#define KD_FOR_EACH_VARIANT(X)                                                          \
  X(GV_FWD, CfgFwd) X(GV_DZ, CfgDz) X(GV_GRAD_H, CfgGradH) X(GV_GRAD_W, CfgGradW)         \
  X(GV_TEST_KK, CfgTestKK) X(GV_TEST_KM, CfgTestKM) X(GV_TEST_MK, CfgTestMK)             \
  X(GV_TEST_MM, CfgTestMM) X(GV_TEST_KK192, CfgTestKK192) X(GV_TEST_KM256, CfgTestKM256) \
  X(GV_TEST_MK256, CfgTestMK256) X(GV_TEST_MM256, CfgTestMM256)                         \
  X(GV_TEST_KK2, CfgTestKK2) X(GV_TEST_KM2, CfgTestKM2) X(GV_TEST_MK2, CfgTestMK2)       \
  X(GV_TEST_MM2, CfgTestMM2) X(GV_FWDZ, CfgFwdZ) X(GV_TEST_KK2S, CfgTestKK2S)              \
  X(GV_DZFWD, CfgDzFwd)

int gemm_bn(int variant) {
#define X(V, C) case V: return C::BN;
  switch (variant) { KD_FOR_EACH_VARIANT(X) }
#undef X
  return 0;
}

int gemm_tile_m(int variant) {
#define X(V, C) case V: return C::TILE_M;
  switch (variant) { KD_FOR_EACH_VARIANT(X) }
#undef X
  return 0;
}

int gemm_smem(int variant) {
#define X(V, C) case V: return C::SMEM_BYTES;
  switch (variant) { KD_FOR_EACH_VARIANT(X) }
#undef X
  return 0;
}

int gemm_width(int variant) {
#define X(V, C) case V: return resident_units<C>();
  switch (variant) { KD_FOR_EACH_VARIANT(X) }
#undef X
  return 0;
}

cudaError_t launch_gemm(int variant, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& o, const GemmArgs& g, const EpiArgs& e,
                        cudaStream_t s) {
#define X(V, C) case V: return launch_cfg<C>(a, b, o, g, e, s);
  switch (variant) { KD_FOR_EACH_VARIANT(X) }
#undef X
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ prep
// One warp per token row.  Teacher distribution over the K cached entries:
// a_k = l_k / T, log p_k = a_k - logsumexp(a), p_k = exp(log p_k), in fp32
// (single-precision exp/log), with the row sums sum_k p log p and sum_k p
// accumulated in double.  Writes the row's ids sorted ascending (ties by
// original position) with p and the original position alongside: the warp
// sorts the keys (id << 32 | k) in shared memory with a bitonic network over
// P >= K slots (padding keys sort last).  An id outside [0, V) raises
// DEV_ERR_INDEX.
__global__ void __launch_bounds__(256) kd_prep_topk(const int32_t* __restrict__ idx,
                                                    const float* __restrict__ logit, long long N,
                                                    int K, int P, int V, float invT,
                                                    int* __restrict__ sid, float* __restrict__ sp,
                                                    int* __restrict__ perm,
                                                    double* __restrict__ ent,
                                                    double* __restrict__ psum, DevStatus* st) {
  extern __shared__ unsigned long long s_keys[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + warp;
  if (r >= N) return;
  unsigned long long* keys = s_keys + static_cast<long long>(warp) * P;
  const int32_t* id_row = idx + r * K;
  const float* l_row = logit + r * K;
  float m = -CUDART_INF_F;
  bool bad = false;
  for (int k = lane; k < P; k += 32) {
    unsigned long long key = ~0ull;
    if (k < K) {
      const int id = id_row[k];
      key = (static_cast<unsigned long long>(static_cast<uint32_t>(id)) << 32) |
            static_cast<uint32_t>(k);
      bad |= (id < 0) || (id >= V);
      m = fmaxf(m, l_row[k] * invT);
    }
    keys[k] = key;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&st->err, DEV_ERR_INDEX);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
  for (int k = lane; k < K; k += 32) s += expf(l_row[k] * invT - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float lse_t = m + logf(s);
  double e_acc = 0.0, p_acc = 0.0;
  for (int k = lane; k < K; k += 32) {
    const float lp = l_row[k] * invT - lse_t;
    const float p = expf(lp);
    e_acc += static_cast<double>(p) * static_cast<double>(lp);
    p_acc += static_cast<double>(p);
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
  // ascending bitonic sort of keys[0..P)
  __syncwarp();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = lane; i < P; i += 32) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long a = keys[i], b = keys[j];
          if ((a > b) == ((i & size) == 0)) {
            keys[i] = b;
            keys[j] = a;
          }
        }
      }
      __syncwarp();
    }
  }
  for (int q = lane; q < K; q += 32) {
    const unsigned long long key = keys[q];
    const int k = static_cast<int>(key & 0xffffffffu);
    sid[r * K + q] = static_cast<int>(key >> 32);
    sp[r * K + q] = expf(l_row[k] * invT - lse_t);
    perm[r * K + q] = k;
  }
}

cudaError_t launch_prep_topk(const int32_t* idx, const float* logit, long long N, int K, int V,
                             float T, int* sid, float* sp, int* perm, double* ent, double* psum,
                             DevStatus* st, cudaStream_t s) {
  int P = 32;
  while (P < K) P <<= 1;                       // K <= 8192: P <= 8192, 64 KB of keys
  int wpb = 65536 / (P * 8);
  wpb = wpb < 1 ? 1 : (wpb > 8 ? 8 : wpb);
  const size_t smem = static_cast<size_t>(wpb) * P * 8;
  static std::atomic<bool> attr_set[64];  // per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kd_prep_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  const long long blocks = (N + wpb - 1) / wpb;
  kd_prep_topk<<<static_cast<unsigned>(blocks), wpb * 32, smem, s>>>(
      idx, logit, N, K, P, V, static_cast<float>(1.0 / static_cast<double>(T)), sid, sp, perm,
      ent, psum, st);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ lse + loss fold
// One block per 8 chunk rows (32 warps).  Lane l of warp w takes row
// r0 + (l & 7) and the vocab tiles t = p + 4 (w + 32 i), p = l >> 3: it
// combines their (max, sum) partials (log2 units) in fp32 relative to its
// running max, a warp load covering 4 tiles x 8 consecutive rows; a lane's
// loads are issued LSE_BATCH at a time before any is folded.  Warp w < 8
// then merges row r0 + w's 128 partial pairs into
// lse2 = log2 sum_v 2^(z_v log2e / T) and forms the row's KL term
// sum_k p_k (log p_k - z_k/T + lse),  lse = lse2 ln 2,  with the lanes
// striding over the K cached entries.  The merges and the dot product run in
// fp32 with a fixed butterfly order (fp64 is a small fraction of fp32's rate
// on this part); only the last combination of the row's terms is in double.
constexpr int LSE_ROWS = 8;
constexpr int LSE_PHASES = 4;     // lanes per row in a warp
constexpr int LSE_WARPS = 32;
constexpr int LSE_SLOTS = LSE_WARPS * LSE_PHASES;   // partial pairs per row
constexpr int LSE_BATCH = 8;      // partial loads a lane has in flight

__device__ __forceinline__ void lse_fold(float& M, float& S, float2 v) {
  const float m_new = fmaxf(M, v.x);
  S = S * exp2f(M - m_new) + v.y * exp2f(v.x - m_new);
  M = m_new;
}

__global__ void __launch_bounds__(LSE_WARPS * 32) kd_lse_loss(
    const float2* __restrict__ part, int n_tiles, int c_alloc, int rows_valid, int grow0,
    const float* __restrict__ zg, const float* __restrict__ sp, const int* __restrict__ perm,
    const double* __restrict__ ent, const double* __restrict__ psum, int K, double invT,
    const uint8_t* __restrict__ mask, float* __restrict__ lse2_out,
    double* __restrict__ loss_rows, float* __restrict__ dbg_lse, float* __restrict__ dbg_zg) {
  __shared__ float sM[LSE_ROWS][LSE_SLOTS + 1];
  __shared__ float sS[LSE_ROWS][LSE_SLOTS + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * LSE_ROWS;
  const int rr = lane & (LSE_ROWS - 1), ph = lane / LSE_ROWS;
  const int r = r0 + rr;
  float M = -CUDART_INF_F, S = 0.f;
  if (r < rows_valid) {
    const float2* col = part + r;
    constexpr int STEP = LSE_PHASES * LSE_WARPS;
    for (int t0 = ph + LSE_PHASES * warp; t0 < n_tiles; t0 += LSE_BATCH * STEP) {
      float2 v[LSE_BATCH];
#pragma unroll
      for (int i = 0; i < LSE_BATCH; ++i) {
        const int t = t0 + i * STEP;
        v[i] = t < n_tiles ? col[static_cast<long long>(t) * c_alloc]
                           : make_float2(-CUDART_INF_F, 0.f);
      }
#pragma unroll
      for (int i = 0; i < LSE_BATCH; ++i)
        if (t0 + i * STEP < n_tiles) lse_fold(M, S, v[i]);
    }
  }
  const int slot = warp * LSE_PHASES + ph;
  sM[rr][slot] = M;
  sS[rr][slot] = S;
  __syncthreads();
  if (warp >= LSE_ROWS) return;
  const int row = r0 + warp;
  if (row >= rows_valid) return;                 // warp-uniform
  // merge the row's partial pairs: max over the lanes, then the sum in double
  float m4[LSE_SLOTS / 32], s4[LSE_SLOTS / 32];
  float Mr = -CUDART_INF_F;
#pragma unroll
  for (int i = 0; i < LSE_SLOTS / 32; ++i) {
    m4[i] = sM[warp][lane + 32 * i];
    s4[i] = sS[warp][lane + 32 * i];
    Mr = fmaxf(Mr, m4[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Mr = fmaxf(Mr, __shfl_xor_sync(0xffffffffu, Mr, o));
  float Sr = 0.f;
#pragma unroll
  for (int i = 0; i < LSE_SLOTS / 32; ++i)
    if (s4[i] > 0.f) Sr = fmaf(s4[i], exp2f(m4[i] - Mr), Sr);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Sr += __shfl_xor_sync(0xffffffffu, Sr, o);
  const float lse2 = Mr + log2f(Sr);
  const long long g = static_cast<long long>(grow0) + row;
  float dot = 0.f;
  for (int j = lane; j < K; j += 32) {
    const float z = zg[static_cast<long long>(row) * K + j];
    dot = fmaf(sp[g * K + j], z, dot);
    if (dbg_zg) dbg_zg[g * K + perm[g * K + j]] = z;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if (lane == 0) {
    const double lse = static_cast<double>(lse2) * 0.69314718055994530942;  // ln 2
    lse2_out[row] = lse2;
    const bool live = !mask || mask[g] != 0;
    loss_rows[g] = live ? ent[g] + lse * psum[g] - static_cast<double>(dot) * invT : 0.0;
    if (dbg_lse) dbg_lse[g] = static_cast<float>(lse);
  }
}

cudaError_t launch_lse_loss(const float2* part, int n_tiles, int c_alloc, int rows_valid, int grow0,
                            const float* zg, const float* sp, const int* perm, const double* ent,
                            const double* psum, int K, float T, const uint8_t* mask, float* lse2,
                            double* loss_rows, float* dbg_lse, float* dbg_zg, cudaStream_t s) {
  const int blocks = (rows_valid + LSE_ROWS - 1) / LSE_ROWS;
  kd_lse_loss<<<blocks, LSE_WARPS * 32, 0, s>>>(part, n_tiles, c_alloc, rows_valid, grow0, zg, sp,
                                                perm, ent, psum, K, 1.0 / static_cast<double>(T),
                                                mask, lse2, loss_rows, dbg_lse, dbg_zg);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ split-K reduce
// out[r][h] = alpha * sum_s part[s][h][r]  for r < rows_valid, h < H, i.e. the
// K splits of grad_hidden^T summed in a fixed order and transposed back
// (added to out instead when `accumulate`; alpha read from alpha_dev when
// that is given).
// Tiles of 32 h x 128 r through shared memory: float4 reads along r, 128-byte
// warp writes along h.
constexpr int SR_H = 32, SR_R = 128;

__global__ void __launch_bounds__(256) kd_split_reduce_t(const float* __restrict__ part,
                                                         int splits, long long split_stride,
                                                         int c_alloc, int rows_valid, int H,
                                                         float alpha_host,
                                                         const float* __restrict__ alpha_dev,
                                                         int accumulate, float* __restrict__ out) {
  __shared__ float tile[SR_H][SR_R + 1];
  const float alpha = alpha_dev ? *alpha_dev : alpha_host;
  const int r0 = blockIdx.x * SR_R, h0 = blockIdx.y * SR_H;
  const int t = threadIdx.x;
  const int r4 = (t & 31) * 4;
#pragma unroll
  for (int i = 0; i < SR_H / 8; ++i) {
    const int hh = (t >> 5) + 8 * i;
    const int h = h0 + hh;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h < H && r0 + r4 < c_alloc) {   // c_alloc is a multiple of 128
      const long long off = static_cast<long long>(h) * c_alloc + r0 + r4;
      a = *reinterpret_cast<const float4*>(part + off);
      for (int sp = 1; sp < splits; ++sp) {
        const float4 b = *reinterpret_cast<const float4*>(part + sp * split_stride + off);
        a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
      }
    }
    tile[hh][r4 + 0] = a.x * alpha;
    tile[hh][r4 + 1] = a.y * alpha;
    tile[hh][r4 + 2] = a.z * alpha;
    tile[hh][r4 + 3] = a.w * alpha;
  }
  __syncthreads();
  const int hh = t & 31;
#pragma unroll 4
  for (int j = 0; j < SR_R / 8; ++j) {
    const int rr = (t >> 5) + 8 * j;
    const int r = r0 + rr, h = h0 + hh;
    if (r < rows_valid && h < H) {
      float* o = out + static_cast<long long>(r) * H + h;
      *o = accumulate ? *o + tile[hh][rr] : tile[hh][rr];
    }
  }
}

cudaError_t launch_split_reduce_t(const float* part, int splits, long long split_stride,
                                  int c_alloc, int rows_valid, int H, float alpha,
                                  const float* alpha_dev, int accumulate, float* out,
                                  cudaStream_t s) {
  dim3 grid((rows_valid + SR_R - 1) / SR_R, (H + SR_H - 1) / SR_H);
  kd_split_reduce_t<<<grid, 256, 0, s>>>(part, splits, split_stride, c_alloc, rows_valid, H,
                                         alpha, alpha_dev, accumulate, out);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ dZ from stored logits
// The backward's dZ without recomputing the logits: for rows < rows_cover,
//   dZ[r][v] = bf16(2^(z[r][v] * scale2 - lse2[r]))      (0 for r >= rows_valid
// and for masked rows), eight columns per thread; kd_dz_fixup then rewrites
// the cached-id columns.  Both round exactly as the recompute GEMM's epilogue
// does, so the two backward forms give bitwise the same dZ.
__global__ void __launch_bounds__(256) kd_dz_from_z(const float* __restrict__ z, int V,
                                                    int rows_valid, int col_blocks,
                                                    const float* __restrict__ lse2,
                                                    float scale2, const uint8_t* __restrict__ mask,
                                                    int grow0, __nv_bfloat16* __restrict__ dz) {
  // one flat grid of rows x col_blocks (a chunk may hold more than 65,535 rows)
  const int r = static_cast<int>(blockIdx.x / static_cast<unsigned>(col_blocks));
  const int cb = static_cast<int>(blockIdx.x % static_cast<unsigned>(col_blocks));
  const int v = (cb * 256 + threadIdx.x) * 8;
  if (v >= V) return;                       // V is a multiple of 8
  const long long off = static_cast<long long>(r) * V + v;
  uint4 out = make_uint4(0u, 0u, 0u, 0u);
  const bool live = r < rows_valid && (!mask || mask[grow0 + r] != 0);
  if (live) {
    const float l2 = lse2[r];
    const float4 a = *reinterpret_cast<const float4*>(z + off);
    const float4 b = *reinterpret_cast<const float4*>(z + off + 4);
    out.x = pack_bf16x2(ex2_approx(fmaf(a.x, scale2, -l2)), ex2_approx(fmaf(a.y, scale2, -l2)));
    out.y = pack_bf16x2(ex2_approx(fmaf(a.z, scale2, -l2)), ex2_approx(fmaf(a.w, scale2, -l2)));
    out.z = pack_bf16x2(ex2_approx(fmaf(b.x, scale2, -l2)), ex2_approx(fmaf(b.y, scale2, -l2)));
    out.w = pack_bf16x2(ex2_approx(fmaf(b.z, scale2, -l2)), ex2_approx(fmaf(b.w, scale2, -l2)));
  }
  *reinterpret_cast<uint4*>(dz + off) = out;
}

// dZ at the cached ids: g - p for each distinct id of a live row, with the
// teacher masses of a repeated id subtracted one by one in sorted order.
__global__ void __launch_bounds__(256) kd_dz_fixup(const float* __restrict__ z, int V,
                                                   int rows_valid, int K,
                                                   const float* __restrict__ lse2, float scale2,
                                                   const uint8_t* __restrict__ mask, int grow0,
                                                   const int* __restrict__ sid,
                                                   const float* __restrict__ sp,
                                                   __nv_bfloat16* __restrict__ dz) {
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= static_cast<long long>(rows_valid) * K) return;
  const int r = static_cast<int>(i / K), k = static_cast<int>(i % K);
  const long long g = static_cast<long long>(grow0) + r;
  if (mask && mask[g] == 0) return;
  const int* ids = sid + g * K;
  const float* ps = sp + g * K;
  const int id = ids[k];
  if (id < 0 || id >= V) return;             // out of range: the call reports KD_ERR_INDEX
  if (k > 0 && ids[k - 1] == id) return;     // the run's first entry writes
  float val = ex2_approx(fmaf(z[static_cast<long long>(r) * V + id], scale2, -lse2[r]));
  for (int j = k; j < K && ids[j] == id; ++j) val -= ps[j];
  dz[static_cast<long long>(r) * V + id] = __float2bfloat16_rn(val);
}

cudaError_t launch_dz_from_z(const float* z, int V, int rows_valid, int rows_cover,
                             const float* lse2, float scale2, const uint8_t* mask, int grow0,
                             const int* sid, const float* sp, int K, void* dz, cudaStream_t s) {
  const int col_blocks = (V / 8 + 255) / 256;
  const long long blocks = static_cast<long long>(rows_cover) * col_blocks;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kd_dz_from_z<<<static_cast<unsigned>(blocks), 256, 0, s>>>(z, V, rows_valid, col_blocks, lse2,
                                                             scale2, mask, grow0,
                                                             static_cast<__nv_bfloat16*>(dz));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(rows_valid) * K;
  kd_dz_fixup<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
      z, V, rows_valid, K, lse2, scale2, mask, grow0, sid, sp, static_cast<__nv_bfloat16*>(dz));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ top-K cache select
// Offline teacher cache: per row of a chunk's stored fp32 logits z [rows][V],
// the K largest values in decreasing order with equal values ordered by
// increasing id.  Values are compared through an order-preserving 32-bit key;
// a candidate is the 64-bit (key << 32 | ~id), so sorting candidates in
// decreasing order sorts by value, then by increasing id.
//
// Four stream-ordered kernels per chunk:
//   kd_sel_tau     the K-th largest of the row's per-tile maxima (from the
//                  GEMM epilogue): a lower bound tau0 of the row's K-th
//                  largest value, since K tiles hold a value at least that
//                  large (-inf when K exceeds the tile count);
//   kd_sel_filter  one streaming pass over the whole chunk: every value
//                  >= tau0 is appended to its row's candidate list
//                  (typically about K of them; warp-aggregated counters);
//   kd_sel_sort    rows with at most SEL_GCAP candidates: bitonic sort of
//                  the list, the first K written out;
//   kd_sel_exact   every other row (its list overflowed; fewer than K
//                  candidates cannot happen, but would land here too): a three-pass radix select
//                  finds the K-th largest key, then the larger keys and, in
//                  increasing id order, enough of the equal keys are
//                  gathered and sorted.
// The filter is the only pass over the logits on the fast path, so it runs
// as a flat, evenly loaded stream at HBM speed; the per-row work (threshold,
// sort) is tiny and runs in kernels of its own.
constexpr int SEL_THREADS = 512;       // exact path
constexpr int SEL_CAP = 8192;          // exact path: keys a block holds (>= K)
constexpr int SEL_BINS = 2048;
constexpr int SEL_TAU_THREADS = 128;   // one row per warp
constexpr int SEL_TAU_MAX = 2048;      // tile maxima a warp holds (vocabularies <= 524,288)
constexpr int FLT_THREADS = 128;
constexpr int FLT_UNROLL = 8;          // 16-byte loads in flight per thread
constexpr int SORT_THREADS = 256;

__device__ __forceinline__ uint32_t sel_key(float f) {
  const uint32_t b = __float_as_uint(f + 0.0f);      // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float sel_val(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ unsigned long long sel_cand(uint32_t key, int id) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~id);
}
__device__ __forceinline__ int sel_pow2(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// Sort s[0..P) (P a power of two) in decreasing order; all threads call.
__device__ void sel_bitonic_desc(unsigned long long* s, int P) {
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = s[i], b = s[ixj];
          const bool first_half = (i & k) == 0;
          if (first_half ? (a < b) : (a > b)) { s[i] = b; s[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
}

// Write the first K sorted candidates of a row.
__device__ __forceinline__ void sel_write(const unsigned long long* s, int K, long long row,
                                          int32_t* out_idx, float* out_val) {
  const long long o = row * static_cast<long long>(K);
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const unsigned long long c = s[k];
    out_val[o + k] = sel_val(static_cast<uint32_t>(c >> 32));
    out_idx[o + k] = static_cast<int32_t>(~static_cast<uint32_t>(c));
  }
}

// tau0 of one row per warp, and the row's candidate count reset.  The K-th
// largest of the row's n_tiles tile-maximum keys, found bit by bit from the
// top: the largest key t with at least K keys >= t.
__global__ void __launch_bounds__(SEL_TAU_THREADS) kd_sel_tau(const float2* __restrict__ part,
                                                              int n_tiles, int c_alloc,
                                                              int rows_valid, int K,
                                                              float* __restrict__ tau,
                                                              uint32_t* __restrict__ cnt) {
  __shared__ uint32_t keys[SEL_TAU_THREADS / 32][SEL_TAU_MAX];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * (SEL_TAU_THREADS / 32) + warp;
  if (r >= rows_valid) return;                       // warp-uniform
  float t0 = -CUDART_INF_F;
  if (K <= n_tiles && n_tiles <= SEL_TAU_MAX) {
    uint32_t* k = keys[warp];
#pragma unroll 8
    for (int t = lane; t < n_tiles; t += 32)   // strided L2 reads: keep several in flight
      k[t] = sel_key(__ldg(&part[static_cast<long long>(t) * c_alloc + r].x));
    __syncwarp();
    uint32_t prefix = 0;
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t c = prefix | (1u << bit);
      uint32_t n = 0;
      for (int t = lane; t < n_tiles; t += 32) n += k[t] >= c;
      if (__reduce_add_sync(0xffffffffu, n) >= static_cast<uint32_t>(K)) prefix = c;
    }
    t0 = sel_val(prefix);
  }
  if (lane == 0) {
    tau[r] = t0;
    cnt[r] = 0;
  }
}

// Values >= tau0 of one row, columns of one segment of FLT_THREADS x
// FLT_UNROLL float4s: block b takes row b / segs, segment b % segs (a flat
// grid: a chunk may hold more than 65,535 rows).  A list holds SEL_GCAP
// candidates; the count goes on past it, so a count above SEL_GCAP marks an
// overflow.
__global__ void __launch_bounds__(FLT_THREADS) kd_sel_filter(const float* __restrict__ z, int V,
                                                             int segs,
                                                             const float* __restrict__ tau,
                                                             uint32_t* __restrict__ cnt,
                                                             unsigned long long* __restrict__ cand) {
  const int r = static_cast<int>(blockIdx.x / static_cast<unsigned>(segs));
  const int seg = static_cast<int>(blockIdx.x % static_cast<unsigned>(segs));
  const int lane = threadIdx.x & 31;
  const float t0 = __ldg(tau + r);
  const float4* z4 = reinterpret_cast<const float4*>(z + static_cast<long long>(r) * V);
  const int V4 = V >> 2;                      // V is a multiple of 8
  const int i0 = seg * (FLT_THREADS * FLT_UNROLL) + threadIdx.x;
  float4 x[FLT_UNROLL];
#pragma unroll
  for (int u = 0; u < FLT_UNROLL; ++u) {
    const int i = i0 + u * FLT_THREADS;
    x[u] = i < V4 ? __ldcs(z4 + i) : make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F,
                                                 -CUDART_INF_F);
  }
  unsigned long long* list = cand + static_cast<long long>(r) * SEL_GCAP;
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int u = 0; u < FLT_UNROLL; ++u) {
    const int i = i0 + u * FLT_THREADS;
    const float v4[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const bool pass = i < V4 && v4[c] >= t0;
      const unsigned m = __ballot_sync(0xffffffffu, pass);
      if (m == 0u) continue;                  // warp-uniform
      uint32_t base = 0;
      const int leader = __ffs(m) - 1;
      if (lane == leader) base = atomicAdd(cnt + r, static_cast<uint32_t>(__popc(m)));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (pass) {
        const uint32_t slot = base + __popc(m & lt);
        if (slot < SEL_GCAP) list[slot] = sel_cand(sel_key(v4[c]), 4 * i + c);
      }
    }
  }
}

// Rows whose list did not overflow: sort it and write the first K.
__global__ void __launch_bounds__(SORT_THREADS) kd_sel_sort(const uint32_t* __restrict__ cnt,
                                                            const unsigned long long* __restrict__ cand,
                                                            int K, long long row0,
                                                            int32_t* __restrict__ out_idx,
                                                            float* __restrict__ out_val) {
  __shared__ unsigned long long s[SEL_GCAP];
  const int r = blockIdx.x;
  const int n = static_cast<int>(cnt[r]);
  if (n > SEL_GCAP || n < K) return;          // kd_sel_exact takes this row
  const int P = sel_pow2(n);
  const unsigned long long* list = cand + static_cast<long long>(r) * SEL_GCAP;
  for (int i = threadIdx.x; i < P; i += SORT_THREADS) s[i] = i < n ? list[i] : 0ull;
  __syncthreads();
  sel_bitonic_desc(s, P);
  sel_write(s, K, row0 + r, out_idx, out_val);
}

// Rows whose list overflowed: exact K-th largest key by radix select
// (11 + 11 + 10 bits), then the keys above it and the lowest ids among the
// keys equal to it.
__global__ void __launch_bounds__(SEL_THREADS) kd_sel_exact(const float* __restrict__ z, int V,
                                                            const uint32_t* __restrict__ cnt,
                                                            int K, long long row0,
                                                            int32_t* __restrict__ out_idx,
                                                            float* __restrict__ out_val) {
  const int r = blockIdx.x, tid = threadIdx.x;
  const uint32_t n = cnt[r];
  if (n <= static_cast<uint32_t>(SEL_GCAP) && n >= static_cast<uint32_t>(K)) return;   // sorted
  extern __shared__ unsigned long long kcand[];                     // [SEL_CAP]
  uint32_t* hist = reinterpret_cast<uint32_t*>(kcand + SEL_CAP);    // [SEL_BINS]
  uint32_t* scan = hist + SEL_BINS;                                  // [SEL_THREADS]
  __shared__ uint32_t s_cnt, s_prefix, s_rank;
  const float* zr = z + static_cast<long long>(r) * V;

  uint32_t prefix = 0, pmask = 0, kk = static_cast<uint32_t>(K);
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass], nb = 1 << widths[pass];
    for (int b = tid; b < nb; b += SEL_THREADS) hist[b] = 0;
    __syncthreads();
    for (int v = tid; v < V; v += SEL_THREADS) {
      const uint32_t key = sel_key(zr[v]);
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t above = 0;
      int b = nb - 1;
      for (; b > 0; --b) {
        if (above + hist[b] >= kk) break;
        above += hist[b];
      }
      s_prefix = prefix | (static_cast<uint32_t>(b) << sh);
      s_rank = kk - above;
    }
    __syncthreads();
    prefix = s_prefix;
    kk = s_rank;
    pmask |= static_cast<uint32_t>(nb - 1) << sh;
    __syncthreads();
  }
  const uint32_t tau = prefix;                   // the K-th largest key
  const int need = static_cast<int>(kk);         // equal keys to take
  // the keys above tau (fewer than K)
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  for (int v = tid; v < V; v += SEL_THREADS) {
    const uint32_t key = sel_key(zr[v]);
    if (key > tau) kcand[atomicAdd(&s_cnt, 1u)] = sel_cand(key, v);
  }
  __syncthreads();
  const int n_gt = static_cast<int>(s_cnt);
  // the `need` lowest ids among the keys equal to tau: each thread scans a
  // contiguous id range; an exclusive scan of the counts orders them
  const int L = (V + SEL_THREADS - 1) / SEL_THREADS;
  const int v0 = tid * L, v1 = min(V, v0 + L);
  uint32_t mine = 0;
  for (int v = v0; v < v1; ++v) mine += sel_key(zr[v]) == tau;
  scan[tid] = mine;
  __syncthreads();
  if (tid == 0) {
    uint32_t acc = 0;
    for (int i = 0; i < SEL_THREADS; ++i) { const uint32_t c = scan[i]; scan[i] = acc; acc += c; }
  }
  __syncthreads();
  uint32_t rank = scan[tid];
  for (int v = v0; v < v1 && rank < static_cast<uint32_t>(need); ++v) {
    if (sel_key(zr[v]) == tau) { kcand[n_gt + rank] = sel_cand(tau, v); ++rank; }
  }
  __syncthreads();
  const int P = sel_pow2(K);
  for (int i = K + tid; i < P; i += SEL_THREADS) kcand[i] = 0ull;
  __syncthreads();
  sel_bitonic_desc(kcand, P);
  sel_write(kcand, K, row0 + r, out_idx, out_val);
}

cudaError_t launch_topk_select(const float* z, int V, const float2* part, int n_tiles,
                               int c_alloc, int rows_valid, int K, long long row0, float* tau,
                               uint32_t* cnt, unsigned long long* cand, int32_t* out_idx,
                               float* out_val, cudaStream_t s) {
  const size_t smem = SEL_CAP * sizeof(unsigned long long) + (SEL_BINS + SEL_THREADS) * 4;
  static std::atomic<bool> attr_set[64];  // per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kd_sel_exact, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  constexpr int rows_per_block = SEL_TAU_THREADS / 32;
  kd_sel_tau<<<(rows_valid + rows_per_block - 1) / rows_per_block, SEL_TAU_THREADS, 0, s>>>(
      part, n_tiles, c_alloc, rows_valid, K, tau, cnt);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int V4 = V / 4;
  const int segs = (V4 + FLT_THREADS * FLT_UNROLL - 1) / (FLT_THREADS * FLT_UNROLL);
  const long long fblocks = static_cast<long long>(rows_valid) * segs;
  if (fblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kd_sel_filter<<<static_cast<unsigned>(fblocks), FLT_THREADS, 0, s>>>(z, V, segs, tau, cnt, cand);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kd_sel_sort<<<rows_valid, SORT_THREADS, 0, s>>>(cnt, cand, K, row0, out_idx, out_val);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kd_sel_exact<<<rows_valid, SEL_THREADS, smem, s>>>(z, V, cnt, K, row0, out_idx, out_val);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ token mask
// n_valid = number of tokens whose mask byte is nonzero; alpha = 1/(T n_valid)
// (0 when no token is valid), the gradient scale of a masked call.
__global__ void __launch_bounds__(1024) kd_mask_count(const uint8_t* __restrict__ mask,
                                                      long long N, double T, DevStatus* st) {
  __shared__ long long red[32];
  long long c = 0;
  for (long long i = threadIdx.x; i < N; i += 1024) c += mask[i] != 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x < 32) {
    c = red[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (threadIdx.x == 0) {
      st->n_valid = c;
      st->alpha = c > 0 ? static_cast<float>(1.0 / (T * static_cast<double>(c))) : 0.f;
    }
  }
}

cudaError_t launch_mask_count(const uint8_t* mask, long long N, float T, DevStatus* st,
                              cudaStream_t s) {
  kd_mask_count<<<1, 1024, 0, s>>>(mask, N, static_cast<double>(T), st);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ final loss
// Sum of the per-token loss terms into the status block; for an asynchronous
// call also the mean loss and the status code, into the caller's device words.
__global__ void __launch_bounds__(1024) kd_loss_final(const double* __restrict__ loss_rows,
                                                      long long N, DevStatus* st,
                                                      const FinalOut out) {
  __shared__ double red[1024];
  double a = 0.0;
  for (long long i = threadIdx.x; i < N; i += 1024) a += loss_rows[i];
  red[threadIdx.x] = a;
  __syncthreads();
  for (int o = 512; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    st->loss_sum = red[0];
    if (out.loss) {
      // the mean in double, rounded once to float (as the host does it)
      const long long n = out.masked ? st->n_valid : N;
      *out.loss = n > 0 ? static_cast<float>(red[0] / static_cast<double>(n)) : 0.f;
      const int err = st->err;
      *out.status = (err & DEV_ERR_TIMEOUT) ? out.code_timeout
                    : (err & DEV_ERR_INDEX) ? out.code_index : 0;
    }
  }
}

cudaError_t launch_loss_final(const double* loss_rows, long long N, DevStatus* st,
                              const FinalOut& out, cudaStream_t s) {
  kd_loss_final<<<1, 1024, 0, s>>>(loss_rows, N, st, out);
  return cudaGetLastError();
}

}  // namespace kd

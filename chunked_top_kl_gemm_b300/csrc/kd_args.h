// Launch arguments shared by the host layer and the tcgen05 GEMM kernel.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace kd {

struct DevStatus;

enum EpiKind { EPI_FWD = 0, EPI_DZ = 1, EPI_F32 = 2, EPI_ACC = 3, EPI_FWDZ = 4, EPI_DZFWD = 5 };
enum Order { ORDER_M_FAST = 0, ORDER_N_FAST = 1, ORDER_SPLIT = 2 };
enum WaitSite { SITE_PROD = 1, SITE_MMA_FULL = 2, SITE_MMA_TEMPTY = 3, SITE_EPI = 4,
                SITE_INJECT = 5, SITE_DRAIN = 6 };

struct GemmArgs {
  int m_tiles, n_tiles, splits;
  int kb_total;          // k-blocks of the whole reduction
  int order;             // Order
  int a_row0;            // y offset of A's TMA coordinates
  int m_split;           // EPI_DZFWD: M tiles of the DZ part; tiles from m_split on are the FWD part
  int a_row0_b;          // EPI_DZFWD: y offset of A for the FWD part's tiles
  int b_row0;            // y offset of B's TMA coordinates
  uint64_t timeout_ns;
  DevStatus* status;
  int inject_timeout;    // test hook: the epilogue waits on a barrier nothing arrives at
};

struct EpiArgs {
  int rows_valid;        // valid rows of the M dimension of this launch
  int cols_valid;        // valid columns of the N dimension
  float scale2;          // log2(e) / T
  float alpha;           // EPI_F32 / EPI_ACC scale
  int out_row0;          // EPI_F32 / EPI_ACC / EPI_DZ: y offset of the output coordinates
  int split_rows;        // EPI_F32: y offset between the outputs of two K splits
  int first;             // EPI_ACC: store instead of add
  // EPI_FWD / EPI_DZ (EPI_DZFWD: grow0 / rows_valid for the DZ part, *_b for the FWD part)
  int K;                 // cached entries per token
  int grow0;             // global token index of chunk row 0
  int grow0_b;           // EPI_DZFWD: global token index of the FWD part's chunk row 0
  int rows_valid_b;      // EPI_DZFWD: valid rows of the FWD part's chunk
  int c_alloc;           // rows of the chunk scratch buffers
  const int* sid;        // [N][K] ids sorted ascending per row
  const float* sp;       // [N][K] teacher p in the same order
  const int* perm;       // [N][K] sorted position -> original k
  float2* part;          // EPI_FWD(Z): [n_tiles][c_alloc] (max, sum) in log2 units
  float* zg;             // EPI_FWD: [c_alloc][K] z at the sorted ids
  const float* lse2;     // EPI_DZ: [c_alloc] log2-sum-exp2 of z*log2e/T
  int* dbg_found;        // EPI_FWD: optional [N][K] column at which id k was found
  const uint8_t* mask;   // EPI_DZ: optional [N] token mask (0 = the token's dZ row is 0)
  const float* alpha_dev;  // EPI_ACC: optional device scale, read instead of alpha
};

}  // namespace kd

// Persistent warp-specialised tcgen05 GEMM with fused epilogues.
//
//   D[TILE_M x BN tile] = A[TILE_M x K] * B[BN x K]^T   (bf16 in, fp32 in TMEM)
//
// TILE_M is 128 (one CTA per tile) or 256 (a CTA pair per tile: each CTA
// loads 128 rows of A and BN/2 rows of B, the leader CTA issues 2-CTA MMAs
// and each CTA's TMEM holds its 128 rows of the accumulator).  The pair
// halves the operand bytes each SM pulls from L2 per MMA.
//
// Roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: fills a STAGES-deep ring of (A, B) k-blocks
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..5  epilogue: TMEM -> registers -> fused math -> global
// The accumulator is double-buffered in TMEM so the epilogue of one tile
// overlaps the MMAs of the next.  Every wait is bounded (see kd_ptx.cuh):
// on expiry the CTA raises an error bit, stops, drains what it issued,
// frees TMEM and returns.
//
// Operand layouts (128-byte swizzle, 64 bf16 = 128 B per smem row):
//   K-major  : one TMA box {64 k, rows}; rows of 128 B; 8-row atoms of 1 KB.
//   MN-major : boxes {64 mn, 64 k} placed 8 KB apart; a row is one k.
//
// Epilogue kinds:
//   EPI_FWD  : per (row, tile) online max / sum of 2^(z*log2e/T) over the
//              valid columns, plus the gather of z at the row's cached
//              teacher ids that fall in the tile (forward of the loss).
//   EPI_DZ   : G = 2^(z*log2e/T - lse2) - sum of teacher p at the row's ids
//              in the tile, stored as bf16 through TMA (backward recompute).
//   EPI_FWDZ : EPI_FWD, and z itself stored as fp32 through TMA (the
//              logits kept for a backward pass without recompute).
//   EPI_DZFWD: EPI_DZ on the M tiles below m_split (the recompute of one
//              chunk) and EPI_FWD on the others (the forward of the next
//              chunk): both multiply by all of W, which one launch then
//              streams from memory once for the two.
//   EPI_F32  : alpha * D stored as fp32 through TMA.
//   EPI_ACC  : alpha * D added into an fp32 tensor by TMA reduce-add
//              (plain store when `first`).
// EPI_FWDZ and EPI_ACC pace their TMA writes over the next unit's operand
// loads (see the epilogue).
#pragma once
#include "kd_args.h"
#include "kd_ptx.cuh"

namespace kd {

constexpr int BM = 128;          // rows of a tile (TMEM lanes)
constexpr int BK = 64;           // bf16 k per stage (128 B rows)
constexpr int UMMA_K = 16;       // k of one tcgen05.mma kind::f16
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_THREADS = 128;
constexpr int EPI_STAGE_BYTES = 4096;   // one 32-row x 128-byte staging box

template <int BN_, bool A_MN_, bool B_MN_, int STAGES_, int KIND_, bool CTA2_ = false,
          int KSUB_ = 1>
struct GemmCfg {
  static constexpr int BN = BN_;           // N of one accumulator tile (both CTAs of a pair)
  static constexpr bool A_MN = A_MN_;
  static constexpr bool B_MN = B_MN_;
  static constexpr int STAGES = STAGES_;
  static constexpr int KIND = KIND_;
  static constexpr bool CTA2 = CTA2_;      // 2-CTA MMA: tile 256 x BN over a CTA pair
  static constexpr int NCTA = CTA2 ? 2 : 1;
  static constexpr int TILE_M = BM * NCTA; // M of one work unit
  static constexpr int BN_CTA = BN / NCTA; // B rows one CTA loads and holds
  static constexpr int KSUB = KSUB_;       // 64-deep k-blocks per ring stage
  static constexpr int A_SUB = BM * BK * 2;          // one k-block of A
  static constexpr int B_SUB = BN_CTA * BK * 2;      // one k-block of B
  static constexpr int A_BYTES = KSUB * A_SUB;       // one stage
  static constexpr int B_BYTES = KSUB * B_SUB;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TX_BYTES = NCTA * STAGE_BYTES;   // one stage of the whole pair
  static constexpr int TMEM_COLS = (2 * BN <= 256) ? 256 : 512;
  // epilogues that write 128 KB of fp32 per CTA and tile pace those writes
  // over the next tile's operand loads (see the epilogue); DZ's 64 KB of
  // bf16 ran slower paced and is written at once
  static constexpr bool PACED = KIND == EPI_ACC || KIND == EPI_FWDZ;
  static constexpr int OUT_BOXES = BN / 32;   // fp32 32-column boxes per warp and tile
  static constexpr int EPI_BYTES = (KIND == EPI_FWD) ? 0 : 4 * 2 * EPI_STAGE_BYTES;
  static constexpr bool HAS_FWD = KIND == EPI_FWD || KIND == EPI_FWDZ || KIND == EPI_DZFWD;
  static constexpr bool HAS_DZ = KIND == EPI_DZ || KIND == EPI_DZFWD;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(!B_MN || BN_CTA % 64 == 0, "MN-major B boxes are 64 wide");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert((2 * STAGES + 6) * 8 + 4 * 4 <= BAR_BYTES, "barrier area");
};

struct Unit {
  int m, n, s, kb0, kb1;
};

__device__ __forceinline__ Unit unit_of(int u, const GemmArgs& g) {
  Unit t;
  if (g.order == ORDER_M_FAST) {
    t.m = u % g.m_tiles;
    t.n = u / g.m_tiles;
    t.s = 0;
    t.kb0 = 0;
    t.kb1 = g.kb_total;
  } else if (g.order == ORDER_N_FAST) {
    t.n = u % g.n_tiles;
    t.m = u / g.n_tiles;
    t.s = 0;
    t.kb0 = 0;
    t.kb1 = g.kb_total;
  } else {
    t.n = u % g.n_tiles;
    const int r = u / g.n_tiles;
    t.m = r % g.m_tiles;
    const int s = r / g.m_tiles;
    t.s = s;
    t.kb0 = static_cast<int>((static_cast<long long>(s) * g.kb_total) / g.splits);
    t.kb1 = static_cast<int>((static_cast<long long>(s + 1) * g.kb_total) / g.splits);
  }
  return t;
}

// Wait that ignores the abort word (used to drain work already issued).
static __device__ __noinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Number of ids of the sorted row `ids[0..K)` that are < v.
__device__ __forceinline__ int lower_bound_ids(const int* ids, int K, int v) {
  int lo = 0, hi = K;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ids + mid) < v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// r[j] for a runtime j in [0, 32) without dynamic register indexing.
__device__ __forceinline__ float select32(const uint32_t (&r)[32], int j) {
  float v = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) v = (i == j) ? __uint_as_float(r[i]) : v;
  return v;
}

// Write one 128-byte row (8 x 16 B chunks) of a 32-row staging box laid out
// with the TMA 128-byte swizzle: chunk c of row i lives at chunk c ^ (i & 7).
__device__ __forceinline__ void stage_row_128B(uint32_t box_base, int row, const uint32_t (&w)[32]) {
  const uint32_t rb = box_base + row * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    st_shared_v4(rb + ((c ^ (row & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  }
}

// Stage fills issued so far for ring slot s after `issued` k-blocks.
__device__ __forceinline__ uint32_t ring_fills(uint32_t issued, int s, int stages) {
  return issued > static_cast<uint32_t>(s) ? (issued - 1 - s) / stages + 1 : 0u;
}

template <class C>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    kd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO, const GemmArgs g, const EpiArgs e) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::STAGES * C::A_BYTES;
  uint8_t* sEpi = sB + C::STAGES * C::B_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + C::EPI_BYTES);
  uint64_t* full = bars;                     // [STAGES]  (pair: used in the leader only)
  uint64_t* empty = full + C::STAGES;        // [STAGES]
  uint64_t* tfull = empty + C::STAGES;       // [2]
  uint64_t* tempty = tfull + 2;              // [2]       (pair: used in the leader only)
  uint64_t* mma_done = tempty + 2;           // [1]
  uint64_t* inj_bar = mma_done + 1;          // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(inj_bar + 1);
  volatile int* abort_word = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
  volatile uint32_t* prod_progress = reinterpret_cast<volatile uint32_t*>(tmem_slot + 3);  // PACED

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int units = g.m_tiles * g.n_tiles * g.splits;
  // CTA pairs: rank 0 (the leader) issues the MMAs of the pair and owns the
  // ring's full barriers and the accumulators' empty barriers.
  const uint32_t rank = C::CTA2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit0 = C::CTA2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ustep = C::CTA2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * C::NCTA);   // one arrival per epilogue warp of the pair
    }
    mbar_init(mma_done, 1);
    mbar_init(inj_bar, 1);
    *abort_word = 0;
    *peer_issued = 0;
    *prod_progress = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (C::KIND != EPI_FWD) tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc<C::NCTA>(tmem_slot, C::TMEM_COLS);
    tmem_relinquish<C::NCTA>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (C::CTA2) cluster_sync_all();   // the peer's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx w{abort_word, g.status, g.timeout_ns};

  // valid columns of tile n, rounded to what the MMA may multiply
  auto tile_cols = [&](int n) {
    const int rem = e.cols_valid - n * C::BN;
    if (rem >= C::BN) return C::BN;
    const int q = C::CTA2 ? 32 : 16;           // pair: each half a multiple of 16 rows
    const int nn = rem <= q ? q : ((rem + q - 1) / q) * q;
    return nn < C::BN ? nn : C::BN;
  };

  uint32_t issued = 0;   // k-blocks this CTA's producer issued (ring position)
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int u = unit0; u < units; u += ustep) {
        const Unit t = unit_of(u, g);
        const int a_m0 = t.m * C::TILE_M + static_cast<int>(rank) * BM;
        const int a_y0 = (C::KIND == EPI_DZFWD && t.m >= g.m_split) ? g.a_row0_b : g.a_row0;
        const int b_n0 = t.n * C::BN + static_cast<int>(rank) * (tile_cols(t.n) / C::NCTA);
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; kb += C::KSUB) {
          if (*abort_word || !mbar_wait(&empty[stage], phase ^ 1u, w, SITE_PROD)) { ok = false; break; }
          // a stage always carries KSUB k-blocks (the byte count stays fixed); a
          // k-block past the unit's end is loaded but not multiplied
          if constexpr (!C::CTA2) mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          else if (leader) mbar_arrive_expect_tx(&full[stage], C::TX_BYTES);
          const uint32_t fb = C::CTA2 ? mapa_shared(smem_u32(&full[stage]), 0) : 0u;
#pragma unroll
          for (int j = 0; j < C::KSUB; ++j) {
            uint8_t* a = sA + stage * C::A_BYTES + j * C::A_SUB;
            uint8_t* b = sB + stage * C::B_BYTES + j * C::B_SUB;
            const int k0 = (kb + j) * BK;
            if constexpr (!C::CTA2) {
              if (!C::A_MN) {
                tma_load_2d(a, &tmA, &full[stage], k0, a_y0 + a_m0);
              } else {
                tma_load_2d(a, &tmA, &full[stage], a_m0, a_y0 + k0);
                tma_load_2d(a + 8192, &tmA, &full[stage], a_m0 + 64, a_y0 + k0);
              }
              if (!C::B_MN) {
                tma_load_2d(b, &tmB, &full[stage], k0, g.b_row0 + b_n0);
              } else {
#pragma unroll
                for (int jj = 0; jj < C::BN_CTA / 64; ++jj)
                  tma_load_2d(b + jj * 8192, &tmB, &full[stage], b_n0 + jj * 64, g.b_row0 + k0);
              }
            } else {
              // both CTAs' bytes complete on the leader's full barrier
              if (!C::A_MN) {
                tma_load_2d_pair(a, &tmA, fb, k0, a_y0 + a_m0);
              } else {
                tma_load_2d_pair(a, &tmA, fb, a_m0, a_y0 + k0);
                tma_load_2d_pair(a + 8192, &tmA, fb, a_m0 + 64, a_y0 + k0);
              }
              if (!C::B_MN) {
                tma_load_2d_pair(b, &tmB, fb, k0, g.b_row0 + b_n0);
              } else {
#pragma unroll
                for (int jj = 0; jj < C::BN_CTA / 64; ++jj)
                  tma_load_2d_pair(b + jj * 8192, &tmB, fb, b_n0 + jj * 64, g.b_row0 + k0);
              }
            }
          }
          ++issued;
          if constexpr (C::PACED) *prod_progress = issued;   // read by the epilogue's pacing
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      if constexpr (C::CTA2) {
        if (!leader) st_shared_cluster_u32(mapa_shared(smem_u32((const void*)peer_issued), 0), issued);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      bool ok = true;
      // Shared-memory descriptors of ring slot 0; slot s is slot 0 advanced by
      // s stage sizes in the 16-byte address field (smem < 256 KB: no carry).
      const uint64_t a_desc0 = C::A_MN ? sdesc_sw128(smem_u32(sA), 8192, 1024)
                                       : sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t b_desc0 = C::B_MN ? sdesc_sw128(smem_u32(sB), 8192, 1024)
                                       : sdesc_sw128(smem_u32(sB), 16, 1024);
      constexpr uint32_t A_STEP = C::A_BYTES >> 4, B_STEP = C::B_BYTES >> 4;
      constexpr uint32_t A_SUBD = C::A_SUB >> 4, B_SUBD = C::B_SUB >> 4;
      constexpr uint32_t A_KK = C::A_MN ? (2048 >> 4) : (32 >> 4);   // one UMMA_K slice
      constexpr uint32_t B_KK = C::B_MN ? (2048 >> 4) : (32 >> 4);
      uint64_t a_desc = a_desc0, b_desc = b_desc0;
      for (int u = unit0; u < units && ok; u += ustep, ++lt) {
        const Unit t = unit_of(u, g);
        const int acc = lt & 1;
        const uint32_t acc_par = (lt >> 1) & 1;
        if (!mbar_wait<C::CTA2>(&tempty[acc], acc_par ^ 1u, w, SITE_MMA_TEMPTY)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * C::BN;
        // a ragged last N tile multiplies only its valid columns
        const int nn = tile_cols(t.n);
        const uint32_t idesc_t = idesc_bf16(C::TILE_M, nn, C::A_MN, C::B_MN);
        uint32_t first = 0;   // the unit's first MMA overwrites the accumulator
        for (int kb = t.kb0; kb < t.kb1; kb += C::KSUB) {
          if (!mbar_wait(&full[stage], phase, w, SITE_MMA_FULL)) { ok = false; break; }
          tc_mma_bf16<C::NCTA>(d, a_desc, b_desc, idesc_t, first);
#pragma unroll
          for (int kk = 1; kk < BK / UMMA_K; ++kk)
            tc_mma_bf16_acc<C::NCTA>(d, a_desc + kk * A_KK, b_desc + kk * B_KK, idesc_t);
#pragma unroll
          for (int j = 1; j < C::KSUB; ++j) {
            if (kb + j < t.kb1) {
#pragma unroll
              for (int kk = 0; kk < BK / UMMA_K; ++kk)
                tc_mma_bf16_acc<C::NCTA>(d, a_desc + j * A_SUBD + kk * A_KK,
                                         b_desc + j * B_SUBD + kk * B_KK, idesc_t);
            }
          }
          first = 1;
          if constexpr (C::CTA2) tc_commit_pair(&empty[stage]);
          else tc_commit<1>(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
            a_desc = a_desc0;
            b_desc = b_desc0;
          } else {
            a_desc += A_STEP;
            b_desc += B_STEP;
          }
        }
        if (ok) {
          if constexpr (C::CTA2) tc_commit_pair(&tfull[acc]);
          else tc_commit<1>(&tfull[acc]);
        }
      }
      // drain: all MMAs issued by this thread complete before TMEM is freed
      tc_commit<C::NCTA>(mma_done);
      mbar_wait_drain(mma_done, 0, g.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int row = q * 32 + lane;          // row of this CTA's 128-row slab
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t stage_base = smem_u32(sEpi) + (warp - EPI_WARP0) * 2 * EPI_STAGE_BYTES;
    // where this warp reports a drained accumulator: the leader's tempty
    const uint32_t tempty_dst[2] = {C::CTA2 ? mapa_shared(smem_u32(&tempty[0]), 0) : 0u,
                                    C::CTA2 ? mapa_shared(smem_u32(&tempty[1]), 0) : 0u};
    auto release_acc = [&](int acc) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty[acc]);
        else mbar_arrive_remote(tempty_dst[acc]);
      }
    };
    uint32_t sub_ctr = 0;
    bool ok = true;
    if (g.inject_timeout) {
      ok = mbar_wait(inj_bar, 0, w, SITE_INJECT);
    }
    // Output pacing.  A tile's TMA writes issued as one burst (128 KB per
    // CTA) delay the next tile's operand loads, which share the TMA unit and
    // the L2 with them.  Box sb of a tile's OUT_BOXES therefore waits until
    // the producer has issued sb / OUT_BOXES of the first three quarters of
    // the next tile's ring stages.  The wait is bounded and gives up on
    // abort; the last tile of a CTA (no next tile) is not paced.
    uint32_t stages_done = 0;   // ring stages of the units up to this one
    uint32_t next_stages = 0;   // ring stages of the next unit (0: none)
    auto pace = [&](int sb) {
      if (sb > 0 && next_stages > 0) {
        const uint32_t target = stages_done + (3u * static_cast<uint32_t>(sb) * next_stages) /
                                                  (4u * static_cast<uint32_t>(C::OUT_BOXES));
        for (int it = 0; it < 512 && *prod_progress < target && !*abort_word; ++it)
          __nanosleep(64);
      }
    };
    int lt = 0;
    for (int u = unit0; u < units && ok; u += ustep, ++lt) {
      const Unit t = unit_of(u, g);
      if constexpr (C::PACED) {
        next_stages = 0;
        stages_done += static_cast<uint32_t>((t.kb1 - t.kb0 + C::KSUB - 1) / C::KSUB);
        if (u + ustep < units) {
          const Unit tn = unit_of(u + ustep, g);
          next_stages = static_cast<uint32_t>((tn.kb1 - tn.kb0 + C::KSUB - 1) / C::KSUB);
        }
      }
      const int acc = lt & 1;
      const uint32_t acc_par = (lt >> 1) & 1;
      const int slab0 = t.m * C::TILE_M + static_cast<int>(rank) * BM;   // first row of the slab
      const int box_row0 = slab0 + q * 32;              // first row of this warp's boxes
      // EPI_DZFWD: which part this tile belongs to, and its rows within that
      // part's chunk (the FWD part's tiles start at m_split)
      const bool fwd_part = C::KIND == EPI_DZFWD ? t.m >= g.m_split : C::HAS_FWD;
      const bool b_part = C::KIND == EPI_DZFWD && fwd_part;
      const int mrow = b_part ? slab0 + row - g.m_split * C::TILE_M : slab0 + row;
      const int grow0 = b_part ? e.grow0_b : e.grow0;
      const bool row_ok = mrow < (b_part ? e.rows_valid_b : e.rows_valid);

      // per-row teacher lookups, issued before waiting on the accumulator
      int hit = 0, hit_end = 0, hit_col = 1 << 30;
      const int* ids = nullptr;
      float lse2 = 0.f;
      const int v0 = t.n * C::BN;
      if constexpr (C::HAS_FWD || C::HAS_DZ) {
        if (row_ok) {
          ids = e.sid + static_cast<long long>(grow0 + mrow) * e.K;
          hit = lower_bound_ids(ids, e.K, v0);
          hit_end = lower_bound_ids(ids, e.K, v0 + C::BN);
          if (hit < hit_end) hit_col = __ldg(ids + hit) - v0;
          if (C::HAS_DZ && !fwd_part) lse2 = __ldg(e.lse2 + mrow);
        }
      }
      // DZ: a masked token's dZ row is zero
      bool row_live = row_ok;
      if constexpr (C::HAS_DZ) {
        if (!fwd_part && row_ok && e.mask && __ldg(e.mask + grow0 + mrow) == 0) {
          row_live = false;
          hit_col = 1 << 30;
        }
      }

      bool got = mbar_wait(&tfull[acc], acc_par, w, SITE_EPI);
      got = __all_sync(0xffffffffu, got);
      if (!got) { ok = false; break; }
      tc_fence_after();
      __syncwarp();
      const uint32_t tb = tmem_base + lane_off + acc * C::BN;

      if constexpr (C::HAS_FWD || C::HAS_DZ) {
        if (C::HAS_FWD && fwd_part) {
          float m_run = -INFINITY, s_run = 0.f;
#pragma unroll 1
          for (int b = 0; b < C::BN / 32; ++b) {
            uint32_t r[32];
            tmem_ld32(tb + b * 32, r);
            tmem_ld_wait();
            reg_fence(r);
            const int c0 = b * 32;
            // gather z at the cached ids that fall in these 32 columns
            while (hit_col < c0 + 32) {
              const float z = select32(r, hit_col - c0);
              e.zg[static_cast<long long>(mrow) * e.K + hit] = z;
              if (e.dbg_found) {
                const long long gr = static_cast<long long>(grow0 + mrow) * e.K;
                e.dbg_found[gr + __ldg(e.perm + gr + hit)] = v0 + hit_col;
              }
              ++hit;
              hit_col = (hit < hit_end) ? __ldg(ids + hit) - v0 : (1 << 30);
            }
            const int nvalid = e.cols_valid - (v0 + c0);   // warp-uniform
            if (nvalid <= 0) continue;
            if constexpr (C::KIND == EPI_FWDZ) {
              if (box_row0 < e.c_alloc) {                  // warp-uniform: inside the z tensor
                pace(b);
                const uint32_t box = stage_base + (sub_ctr & 1u) * EPI_STAGE_BYTES;
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                stage_row_128B(box, lane, r);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  tma_store_2d(&tmO, sEpi + (box - smem_u32(sEpi)), v0 + c0, box_row0);
                  bulk_commit();
                }
                ++sub_ctr;
              }
            }
            float bm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nvalid) bm = fmaxf(bm, __uint_as_float(r[j]));
            const float m_new = fmaxf(m_run, bm * e.scale2);
            float s = s_run * ex2_approx(m_run - m_new);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nvalid) s += ex2_approx(fmaf(__uint_as_float(r[j]), e.scale2, -m_new));
            s_run = s;
            m_run = m_new;
          }
          release_acc(acc);
          if (row_ok) e.part[static_cast<long long>(t.n) * e.c_alloc + mrow] = make_float2(m_run, s_run);
        } else if constexpr (C::HAS_DZ) {
          const bool box_ok = box_row0 < e.c_alloc;       // warp-uniform: inside the dZ tensor
#pragma unroll 1
          for (int sb = 0; sb < C::BN / 64; ++sb) {
            const int c0 = sb * 64;
            if (v0 + c0 >= e.cols_valid) break;            // warp-uniform
            uint32_t r0[32], r1[32];
            tmem_ld32(tb + c0, r0);
            tmem_ld32(tb + c0 + 32, r1);
            tmem_ld_wait();
            reg_fence(r0);
            reg_fence(r1);
            if (!box_ok) continue;
            float gv[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              gv[j] = row_live ? ex2_approx(fmaf(__uint_as_float(r0[j]), e.scale2, -lse2)) : 0.f;
              gv[32 + j] = row_live ? ex2_approx(fmaf(__uint_as_float(r1[j]), e.scale2, -lse2)) : 0.f;
            }
            while (hit_col < c0 + 64) {
              const float p = __ldg(e.sp + static_cast<long long>(grow0 + mrow) * e.K + hit);
              const int jj = hit_col - c0;
#pragma unroll
              for (int j = 0; j < 64; ++j) gv[j] -= (j == jj) ? p : 0.f;
              ++hit;
              hit_col = (hit < hit_end) ? __ldg(ids + hit) - v0 : (1 << 30);
            }
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) pk[j] = pack_bf16x2(gv[2 * j], gv[2 * j + 1]);
            const uint32_t box = stage_base + (sub_ctr & 1u) * EPI_STAGE_BYTES;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            stage_row_128B(box, lane, pk);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmO, sEpi + (box - smem_u32(sEpi)), v0 + c0, e.out_row0 + box_row0);
              bulk_commit();
            }
            ++sub_ctr;
          }
          release_acc(acc);
        }
      } else {
        // EPI_F32 / EPI_ACC: alpha * D -> fp32, 32-column boxes
        const bool box_ok = box_row0 < e.rows_valid;    // warp-uniform
        const float alpha = e.alpha_dev ? __ldg(e.alpha_dev) : e.alpha;
#pragma unroll 1
        for (int sb = 0; sb < C::BN / 32; ++sb) {
          const int c0 = sb * 32;
          if (!box_ok || t.n * C::BN + c0 >= e.cols_valid) break;   // warp-uniform
          pace(sb);
          uint32_t r[32];
          tmem_ld32(tb + c0, r);
          tmem_ld_wait();
          reg_fence(r);
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
          const uint32_t box = stage_base + (sub_ctr & 1u) * EPI_STAGE_BYTES;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          stage_row_128B(box, lane, r);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const void* src = sEpi + (box - smem_u32(sEpi));
            const int x = t.n * C::BN + c0;
            const int y = e.out_row0 + t.s * e.split_rows + box_row0;
            if (C::KIND == EPI_ACC && !e.first) tma_reduce_add_2d(&tmO, src, x, y);
            else tma_store_2d(&tmO, src, x, y);
            bulk_commit();
          }
          ++sub_ctr;
        }
        release_acc(acc);
      }
    }
    if (C::KIND != EPI_FWD && lane == 0) bulk_wait_all();
  }

  // ---------------------------------------------------------------- teardown
  // Every TMA load issued must have landed before either CTA may exit.  A
  // pair's loads complete on the leader's full barriers: the leader waits for
  // the last phase of each ring slot, arming a phase that only the peer
  // filled (it stopped early) or cancelling the peer's share of a phase that
  // the peer never filled (the peer stopped early).
  tc_fence_before();
  if constexpr (C::CTA2) cluster_sync_all(); else __syncthreads();
  if (warp == 0 && lane == 0 && leader) {
    const uint32_t mine = issued;
    const uint32_t peer = C::CTA2 ? *peer_issued : issued;
    for (int s = 0; s < C::STAGES; ++s) {
      const uint32_t a = ring_fills(mine, s, C::STAGES);
      const uint32_t b = ring_fills(peer, s, C::STAGES);
      uint32_t last = a;                       // number of the phases to wait for
      if (C::CTA2 && b == a + 1) {
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        last = b;
      } else if (C::CTA2 && a > 0 && b + 1 == a) {
        mbar_complete_tx(&full[s], C::STAGE_BYTES);
      }
      if (last > 0) mbar_wait_drain(&full[s], (last - 1) & 1u, g.timeout_ns);
    }
  }
  if constexpr (C::CTA2) cluster_sync_all(); else __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<C::NCTA>(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace kd

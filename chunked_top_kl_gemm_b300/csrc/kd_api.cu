// C ABI of the fused chunked top-K KL loss: argument validation, workspace
// plan, TMA descriptors and the chunk loop (all launches on one stream).
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "kd_internal.h"
#include "../../include/kd_topk_kl.h"

namespace {

using kd::DevStatus;

thread_local char g_last_cuda_error[256] = "";

kd_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", where,
                cudaGetErrorString(e));
  return KD_ERR_CUDA;
}

#define KD_CUDA(call)                                  \
  do {                                                 \
    cudaError_t e_ = (call);                           \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

constexpr uint64_t kDefaultTimeoutNs = 5ull * 1000 * 1000 * 1000;
constexpr int kMaxK = 8192;
constexpr unsigned kAllFlags = KD_FLAG_ACCUMULATE | KD_FLAG_STORE_LOGITS | KD_FLAG_MIN_SCRATCH;

// ---------------------------------------------------------------- profiler
// Optional per-kernel timing: when enabled, every launch of run() is
// bracketed by two CUDA events on the launch stream; after the call's final
// synchronisation the elapsed times are added to per-kind totals.
enum ProfKind { PK_PREP = 0, PK_FWD, PK_LSE, PK_DZ, PK_GRAD_H, PK_SPLIT_RED, PK_GRAD_W,
                PK_FINAL, PK_MASK, PK_DZ_EW, PK_CACHE_GEMM, PK_CACHE_SELECT,
                PK_DZ_FWD, PK_COUNT };
const char* const kProfNames[PK_COUNT] = {"prep_topk", "gemm_fwd_lse_gather", "lse_loss_fold",
                                          "gemm_bwd_dz", "gemm_grad_hidden", "split_reduce",
                                          "gemm_grad_W", "loss_final",
                                          "mask_count", "dz_from_logits", "cache_gemm_logits",
                                          "cache_topk_select", "gemm_dz_and_next_fwd"};

struct Profiler {
  std::mutex mu;
  std::atomic<bool> on{false};   // read by every call, profiling or not
  double total_ms[PK_COUNT] = {};
  long long launches[PK_COUNT] = {};
  // events of the call in flight (reused across calls)
  std::vector<cudaEvent_t> ev;
  std::vector<int> kinds;
  size_t used = 0;
};
Profiler& prof() {
  static Profiler p;
  return p;
}
// Set while an asynchronous call enqueues: its launches are not timed (the
// events could only be read after a synchronisation the call does not do).
thread_local bool t_prof_off = false;

// A call starts with no event pairs in flight (touched only while profiling,
// which is documented as single-threaded).
void prof_reset_call() {
  Profiler& P = prof();
  if (P.on.load(std::memory_order_relaxed) && !t_prof_off) P.used = 0;
}

// Bracket one launch.  Returns the index of its event pair or -1.
struct ProfScope {
  Profiler* p = nullptr;
  cudaStream_t s = nullptr;
  int slot = -1;
  ProfScope(int kind, cudaStream_t st) {
    Profiler& P = prof();
    if (!P.on || t_prof_off) return;
    p = &P;
    s = st;
    if (P.ev.size() < 2 * (P.used + 1)) {
      cudaEvent_t a, b;
      if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) { p = nullptr; return; }
      P.ev.push_back(a);
      P.ev.push_back(b);
    }
    slot = static_cast<int>(P.used++);
    if (P.kinds.size() < P.used) P.kinds.resize(P.used);
    P.kinds[slot] = kind;
    cudaEventRecord(P.ev[2 * slot], s);
  }
  ~ProfScope() {
    if (p && slot >= 0) cudaEventRecord(p->ev[2 * slot + 1], s);
  }
};

// After the stream has been synchronised: fold the call's event pairs in.
void prof_collect() {
  Profiler& P = prof();
  if (!P.on) return;
  for (size_t i = 0; i < P.used; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, P.ev[2 * i], P.ev[2 * i + 1]) == cudaSuccess) {
      P.total_ms[P.kinds[i]] += ms;
      P.launches[P.kinds[i]] += 1;
    }
  }
  P.used = 0;
}

// ---------------------------------------------------------------- TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The tensor-map encoder is a driver-API call and needs a context current on
// the calling thread; a thread that has made no context-binding runtime call
// yet has none (a new host thread).  Every entry point therefore binds the
// current device's primary context before encoding, unless the thread
// already has a context current (a caller's own context is left alone).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

bool bind_current_device() {
  CtxGetCurrentFn get = ctx_get_current_fn();
  CUcontext cur = nullptr;
  if (get && get(&cur) == CUDA_SUCCESS && cur != nullptr) return true;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                  "could not make the current device's context current");
    return false;
  }
  return true;
}

// 2-D row-major tensor [outer][inner], 128-byte swizzled boxes of
// box_inner x box_outer elements.  On failure the driver's result code is
// left in the thread's last-error text.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
              uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                  "cuTensorMapEncodeTiled: no driver entry point");
    return false;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(esize)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                  "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return false;
  }
  return true;
}

// Rows of the B operand's TMA box of a GEMM variant (K-major B): the rows one
// CTA holds, i.e. the tile width, halved on a CTA pair.
uint32_t b_box_rows(int variant) {
  return static_cast<uint32_t>(kd::gemm_bn(variant) / (kd::gemm_tile_m(variant) / 128));
}

// ---------------------------------------------------------------- plan
inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }
constexpr long long kMaxChunk = 1LL << 30;   // rows of one chunk at most
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Plan {
  long long N;
  int H, V, K;
  int chunk;      // rows per chunk, multiple of 128
  int n_chunks;
  int vt;         // vocab tiles of the forward / recompute GEMMs
  int ht;         // hidden tiles (N) of the grad_W GEMM
  int mth;        // hidden tiles (M) of the grad_hidden^T GEMM
  int hp;         // mth * its tile M: rows of one split's grad_hidden^T partial
  int splits;     // K splits of the grad_hidden^T GEMM
  int gg;         // chunks whose dZ one grad_W GEMM reduces over (1 or 2)
  int sms;
  bool store_z;   // keep each chunk's fp32 logits instead of recomputing them
  size_t off_status, off_sid, off_sp, off_perm, off_ent, off_psum, off_loss_rows, off_lse2,
      off_zg, off_part, off_dz, off_k4, off_z, total;
};

bool sizes_ok(long long N, int H, int V, int K, int chunk) {
  return N >= 1 && N <= 0x7fffffffLL && H >= 8 && H % 8 == 0 && V >= 8 && V % 8 == 0 && K >= 1 &&
         K <= V && K <= kMaxK && chunk >= 1;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 148;
  return sms;
}

// Smallest split count whose work units fill the machine to >= 94 %, else
// the best one, among 1..16 (and never more than the k-blocks).
int pick_splits(int units, int kb_total, int sms) {
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 16 && s <= kb_total; ++s) {
    const long long u = static_cast<long long>(units) * s;
    const double eff = static_cast<double>(u) / (cdiv(u, sms) * sms);
    if (eff >= 0.94) return s;
    if (eff > best_eff + 1e-9) { best_eff = eff; best = s; }
  }
  return best;
}

// The grad_W GEMM reduces over the dZ rows of gg consecutive chunks at once
// (K = gg x chunk): its fp32 read-modify-write of all of grad_W, 8 V H bytes
// per launch, then happens once per gg chunks.  gg = 2 holds two chunks' dZ
// (2 x chunk x V bf16); KD_FLAG_MIN_SCRATCH keeps one (gg = 1).
Plan make_plan(long long N, int H, int V, int K, int chunk, int sms, bool store_z = false,
               bool min_scratch = false) {
  Plan p{};
  p.N = N; p.H = H; p.V = V; p.K = K; p.sms = sms; p.store_z = store_z;
  long long c = cdiv(chunk, 128) * 128;
  const long long cmax = cdiv(N, 128) * 128;
  if (c > cmax) c = cmax;
  if (c > kMaxChunk) c = kMaxChunk;   // row coordinates of the chunk buffers stay in int
  p.chunk = static_cast<int>(c);
  p.n_chunks = static_cast<int>(cdiv(N, c));
  p.gg = (min_scratch || p.n_chunks < 2) ? 1 : 2;
  p.vt = static_cast<int>(cdiv(V, kd::gemm_bn(kd::GV_FWD)));
  p.ht = static_cast<int>(cdiv(H, kd::gemm_bn(kd::GV_GRAD_W)));
  p.mth = static_cast<int>(cdiv(H, kd::gemm_tile_m(kd::GV_GRAD_H)));
  p.hp = p.mth * kd::gemm_tile_m(kd::GV_GRAD_H);
  p.splits = pick_splits(p.mth * static_cast<int>(cdiv(c, kd::gemm_bn(kd::GV_GRAD_H))),
                         static_cast<int>(cdiv(V, 64)), kd::gemm_width(kd::GV_GRAD_H));
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes, 256); return at; };
  p.off_status = take(sizeof(DevStatus));
  p.off_sid = take(sizeof(int) * N * K);
  p.off_sp = take(sizeof(float) * N * K);
  p.off_perm = take(sizeof(int) * N * K);
  p.off_ent = take(sizeof(double) * N);
  p.off_psum = take(sizeof(double) * N);
  p.off_loss_rows = take(sizeof(double) * N);
  p.off_lse2 = take(sizeof(float) * c);
  p.off_zg = take(sizeof(float) * c * K);
  p.off_part = take(sizeof(float2) * p.vt * c);
  p.off_dz = take(2ull * p.gg * c * V);
  p.off_k4 = take(4ull * p.splits * p.hp * c);
  p.off_z = store_z ? take(4ull * c * V) : 0;
  p.total = o;
  return p;
}

// Device memory of the current device, or managed memory.
bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  if (a.type != cudaMemoryTypeDevice) return false;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.device == dev;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kd_status validate(const void* hidden, const void* W, const int32_t* idx, const float* logit,
                   long long N, int H, int V, int K, float T, int chunk, const float* loss,
                   const float* gh, const float* gW) {
  if (!hidden || !W || !idx || !logit || !loss || !gh || !gW) return KD_ERR_INVALID_ARG;
  if (!sizes_ok(N, H, V, K, chunk)) return KD_ERR_INVALID_ARG;
  if (!(T > 0.f) || !std::isfinite(T)) return KD_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(gh, 16) || !aligned(gW, 16) ||
      !aligned(idx, 4) || !aligned(logit, 4))
    return KD_ERR_ALIGNMENT;
  if (!is_device_ptr(hidden) || !is_device_ptr(W) || !is_device_ptr(idx) ||
      !is_device_ptr(logit) || !is_device_ptr(gh) || !is_device_ptr(gW))
    return KD_ERR_INVALID_ARG;
  return KD_OK;
}

// The whole path on stream s.  mask (optional, device [N]): nonzero = the
// token counts; the mean runs over the valid tokens and masked tokens get
// zero gradient rows.  flags: KD_FLAG_ACCUMULATE adds into grad_hidden /
// grad_W; KD_FLAG_STORE_LOGITS keeps each chunk's fp32 logits from the
// forward GEMM and forms dZ from them instead of recomputing the GEMM.
// async (loss_dev and status_dev device words): nothing waits for the
// stream; the last kernel writes the loss and the status code.
// n_norm > 0 (a shard of a larger batch): the gradients are scaled by
// 1/(T n_norm) and the returned loss is the shard's sum of per-token terms
// divided by n_norm, so that shards' results add up to the whole batch's.
kd_status run_impl(const void* hidden, const void* W, const int32_t* idx, const float* logit,
                   long long N, int H, int V, int K, float T, int chunk, float* loss, float* gh,
                   float* gW, void* ws, size_t ws_bytes, cudaStream_t s,
                   const kd_debug_opts* opts, const uint8_t* mask, unsigned flags,
                   float* loss_dev = nullptr, int32_t* status_dev = nullptr,
                   double n_norm = 0.0) {
  const bool async = loss_dev != nullptr;
  const int accumulate = (flags & KD_FLAG_ACCUMULATE) ? 1 : 0;
  const bool store_z = (flags & KD_FLAG_STORE_LOGITS) != 0;
  const bool min_scratch = (flags & KD_FLAG_MIN_SCRATCH) != 0;
  if (flags & ~kAllFlags) return KD_ERR_INVALID_ARG;
  kd_status st = validate(hidden, W, idx, logit, N, H, V, K, T, chunk, async ? loss_dev : loss,
                          gh, gW);
  if (st != KD_OK) return st;
  if (mask && !is_device_ptr(mask)) return KD_ERR_INVALID_ARG;
  if (async) {
    if (!status_dev) return KD_ERR_INVALID_ARG;
    if (!aligned(loss_dev, 4) || !aligned(status_dev, 4)) return KD_ERR_ALIGNMENT;
    if (!is_device_ptr(loss_dev) || !is_device_ptr(status_dev)) return KD_ERR_INVALID_ARG;
  }
  const Plan p = make_plan(N, H, V, K, chunk, device_sms(), store_z, min_scratch);
  if (!ws || ws_bytes < p.total) return KD_ERR_OOM;
  prof_reset_call();
  if (!aligned(ws, 256)) return KD_ERR_ALIGNMENT;
  if (!is_device_ptr(ws)) return KD_ERR_INVALID_ARG;

  uint8_t* base = static_cast<uint8_t*>(ws);
  DevStatus* dst = reinterpret_cast<DevStatus*>(base + p.off_status);
  int* sid = reinterpret_cast<int*>(base + p.off_sid);
  float* sp = reinterpret_cast<float*>(base + p.off_sp);
  int* perm = reinterpret_cast<int*>(base + p.off_perm);
  double* ent = reinterpret_cast<double*>(base + p.off_ent);
  double* psum = reinterpret_cast<double*>(base + p.off_psum);
  double* loss_rows = reinterpret_cast<double*>(base + p.off_loss_rows);
  float* lse2 = reinterpret_cast<float*>(base + p.off_lse2);
  float* zg = reinterpret_cast<float*>(base + p.off_zg);
  float2* part = reinterpret_cast<float2*>(base + p.off_part);
  void* dz = base + p.off_dz;
  float* k4 = reinterpret_cast<float*>(base + p.off_k4);
  float* zbuf = store_z ? reinterpret_cast<float*>(base + p.off_z) : nullptr;

  const uint64_t timeout = (opts && opts->timeout_ns) ? opts->timeout_ns : kDefaultTimeoutNs;
  float* dbg_lse = opts ? opts->lse : nullptr;
  float* dbg_zg = opts ? opts->zg : nullptr;
  int* dbg_found = opts ? opts->found_idx : nullptr;
  const int inject = opts ? opts->inject_timeout : 0;

  // TMA descriptors
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUtensorMap tm_hid_k, tm_w_k, tm_dz_st, tm_dz_k256, tm_w_mn, tm_k4_st, tm_dz_mn, tm_hid_mn, tm_gw;
  if (!bind_current_device()) return KD_ERR_CUDA;
  bool ok = true;
  ok &= make_map(&tm_hid_k, BF16, 2, hidden, H, N, 64, 128);
  ok &= make_map(&tm_w_k, BF16, 2, W, H, V, 64, b_box_rows(kd::GV_FWD));
  const uint64_t dz_rows = static_cast<uint64_t>(p.gg) * p.chunk;   // dZ of gg chunks
  ok &= make_map(&tm_dz_st, BF16, 2, dz, V, dz_rows, 64, 32);
  ok &= make_map(&tm_dz_k256, BF16, 2, dz, V, dz_rows, 64, b_box_rows(kd::GV_GRAD_H));
  ok &= make_map(&tm_w_mn, BF16, 2, W, H, V, 64, 64);
  ok &= make_map(&tm_k4_st, F32, 4, k4, p.chunk, static_cast<uint64_t>(p.splits) * p.hp, 32, 32);
  ok &= make_map(&tm_dz_mn, BF16, 2, dz, V, dz_rows, 64, 64);
  ok &= make_map(&tm_hid_mn, BF16, 2, hidden, H, N, 64, 64);       // MN-major B of grad_W
  ok &= make_map(&tm_gw, F32, 4, gW, H, V, 32, 32);
  CUtensorMap tm_z_st;
  if (store_z) ok &= make_map(&tm_z_st, F32, 4, zbuf, V, p.chunk, 32, 32);
  if (!ok) return KD_ERR_CUDA;   // make_map left the driver's result in the last-error text

  const bool sharded = n_norm > 0.0;
  const float scale2 = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  const float alpha = static_cast<float>(
      1.0 / (static_cast<double>(T) * (sharded ? n_norm : static_cast<double>(N))));

  KD_CUDA(cudaMemsetAsync(dst, 0, sizeof(DevStatus), s));
  // masked calls: n_valid and the gradient scale 1/(T n_valid) on the device
  // (a shard's scale is the host's 1/(T n_norm) instead)
  const float* alpha_dev = nullptr;
  if (mask) {
    ProfScope ps_(PK_MASK, s);
    KD_CUDA(kd::launch_mask_count(mask, N, T, dst, s));
    if (!sharded) alpha_dev = &dst->alpha;
  }
  { ProfScope ps_(PK_PREP, s); KD_CUDA(kd::launch_prep_topk(idx, logit, N, K, V, T, sid, sp, perm, ent, psum, dst, s)); }

  for (int j = 0; j < p.n_chunks; ++j) {
    const int row0 = j * p.chunk;
    const int cj = static_cast<int>(std::min<long long>(p.chunk, N - row0));
    const int mt = static_cast<int>(cdiv(cj, kd::gemm_tile_m(kd::GV_FWD)));
    // this chunk's dZ rows: slot `slot` of its grad_W group
    const int slot = j % p.gg;
    const int slot_row0 = slot * p.chunk;
    uint8_t* dz_slot = static_cast<uint8_t*>(dz) + 2ull * slot_row0 * V;

    kd::GemmArgs g{};
    g.m_tiles = mt; g.n_tiles = p.vt; g.splits = 1;
    g.kb_total = static_cast<int>(cdiv(H, 64));
    g.order = kd::ORDER_M_FAST; g.a_row0 = row0; g.b_row0 = 0;
    g.timeout_ns = timeout; g.status = dst; g.inject_timeout = (j == 0 && inject == 1);
    kd::EpiArgs e{};
    e.rows_valid = cj; e.cols_valid = V; e.scale2 = scale2; e.alpha = 1.f;
    e.K = K; e.grow0 = row0; e.c_alloc = p.chunk;
    e.sid = sid; e.sp = sp; e.perm = perm; e.part = part; e.zg = zg; e.lse2 = lse2;
    e.dbg_found = dbg_found;
    e.mask = mask;
    // chunk j's forward: its own launch for the first chunk (and for every
    // chunk when the logits are stored); otherwise it ran inside the previous
    // chunk's recompute launch
    auto lse_of = [&](int r0, int rows) {
      return kd::launch_lse_loss(part, p.vt, p.chunk, rows, r0, zg, sp, perm, ent, psum, K, T,
                                 mask, lse2, loss_rows, dbg_lse, dbg_zg, s);
    };
    if (store_z || j == 0) {
      if (store_z) {
        ProfScope ps_(PK_FWD, s);
        KD_CUDA(kd::launch_gemm(kd::GV_FWDZ, tm_hid_k, tm_w_k, tm_z_st, g, e, s));
      } else {
        ProfScope ps_(PK_FWD, s);
        KD_CUDA(kd::launch_gemm(kd::GV_FWD, tm_hid_k, tm_w_k, tm_dz_st, g, e, s));
      }
      { ProfScope ps_(PK_LSE, s); KD_CUDA(lse_of(row0, cj)); }
    }

    g.inject_timeout = (j == 0 && inject == 2);
    if (store_z) {
      // rows up to the GEMMs' reach get a dZ row (zeros past the chunk)
      const int cover = static_cast<int>(std::min<long long>(p.chunk, cdiv(cj, 256) * 256));
      ProfScope ps_(PK_DZ_EW, s);
      KD_CUDA(kd::launch_dz_from_z(zbuf, V, cj, cover, lse2, scale2, mask, row0, sid, sp, K,
                                   dz_slot, s));
    } else if (j + 1 < p.n_chunks) {
      // the recompute of chunk j (tiles below m_split) and the forward of
      // chunk j+1 (the tiles after) in one launch: W is streamed once for both
      const int row1 = row0 + p.chunk;
      const int cj1 = static_cast<int>(std::min<long long>(p.chunk, N - row1));
      const int tm = kd::gemm_tile_m(kd::GV_DZFWD);
      g.m_split = mt;
      g.m_tiles = mt + static_cast<int>(cdiv(cj1, tm));
      g.a_row0_b = row1 - mt * tm;                   // tile m_split starts at row1
      e.out_row0 = slot_row0;                        // dZ rows of chunk j's slot
      e.grow0_b = row1; e.rows_valid_b = cj1;
      { ProfScope ps_(PK_DZ_FWD, s);
        KD_CUDA(kd::launch_gemm(kd::GV_DZFWD, tm_hid_k, tm_w_k, tm_dz_st, g, e, s)); }
      // chunk j+1's logsumexp and loss terms (chunk j's lse2 is consumed)
      { ProfScope ps_(PK_LSE, s); KD_CUDA(lse_of(row1, cj1)); }
    } else {
      e.out_row0 = slot_row0;                        // dZ rows of this chunk's slot
      ProfScope ps_(PK_DZ, s);
      KD_CUDA(kd::launch_gemm(kd::GV_DZ, tm_hid_k, tm_w_k, tm_dz_st, g, e, s));
    }

    // grad_hidden rows of this chunk: (dZ W)^T = W^T dZ^T, split-K over the
    // vocabulary, then an ordered transposing reduction of the splits
    kd::GemmArgs g2{};
    g2.m_tiles = p.mth; g2.n_tiles = static_cast<int>(cdiv(cj, kd::gemm_bn(kd::GV_GRAD_H)));
    g2.splits = p.splits;
    g2.kb_total = static_cast<int>(cdiv(V, 64));
    g2.order = kd::ORDER_SPLIT; g2.a_row0 = 0; g2.b_row0 = slot_row0;
    g2.timeout_ns = timeout; g2.status = dst; g2.inject_timeout = (j == 0 && inject == 3);
    kd::EpiArgs e2{};
    e2.rows_valid = H; e2.cols_valid = cj; e2.alpha = 1.f; e2.out_row0 = 0;
    e2.split_rows = p.hp;
    { ProfScope ps_(PK_GRAD_H, s); KD_CUDA(kd::launch_gemm(kd::GV_GRAD_H, tm_w_mn, tm_dz_k256, tm_k4_st, g2, e2, s)); }
    { ProfScope ps_(PK_SPLIT_RED, s); KD_CUDA(kd::launch_split_reduce_t(k4, p.splits,
                                    static_cast<long long>(p.hp) * p.chunk, p.chunk, cj, H, alpha, alpha_dev, accumulate,
                                    gh + static_cast<long long>(row0) * H, s)); }

    // grad_W += dZ_g^T h_g over the group's rows, once its last chunk is in.
    // B is the group's hidden rows read MN-major; k-blocks past the group's
    // rows meet zero dZ rows, or hidden rows past N (zero-filled)
    if (slot + 1 < p.gg && j + 1 < p.n_chunks) continue;
    const int grp_rows = slot_row0 + cj;   // only the call's last chunk is partial
    kd::GemmArgs g3{};
    g3.m_tiles = static_cast<int>(cdiv(V, kd::gemm_tile_m(kd::GV_GRAD_W))); g3.n_tiles = p.ht;
    g3.splits = 1;
    g3.kb_total = static_cast<int>(cdiv(grp_rows, 64));
    g3.order = kd::ORDER_N_FAST; g3.a_row0 = 0; g3.b_row0 = row0 - slot_row0;
    g3.timeout_ns = timeout; g3.status = dst; g3.inject_timeout = (j == p.gg - 1 && inject == 4);
    kd::EpiArgs e3{};
    e3.rows_valid = V; e3.cols_valid = H; e3.alpha = alpha; e3.out_row0 = 0;
    e3.alpha_dev = alpha_dev;
    e3.first = (j - slot == 0) && !accumulate;
    { ProfScope ps_(PK_GRAD_W, s); KD_CUDA(kd::launch_gemm(kd::GV_GRAD_W, tm_dz_mn, tm_hid_mn, tm_gw, g3, e3, s)); }
  }
  kd::FinalOut fo{};
  if (async) fo = kd::FinalOut{loss_dev, status_dev, mask ? 1 : 0, KD_ERR_TIMEOUT, KD_ERR_INDEX};
  { ProfScope ps_(PK_FINAL, s); KD_CUDA(kd::launch_loss_final(loss_rows, N, dst, fo, s)); }

  if (opts && opts->loss_rows)
    KD_CUDA(cudaMemcpyAsync(opts->loss_rows, loss_rows, sizeof(double) * N,
                            cudaMemcpyDeviceToDevice, s));
  if (async) return KD_OK;
  DevStatus hs{};
  KD_CUDA(cudaMemcpyAsync(&hs, dst, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
  KD_CUDA(cudaStreamSynchronize(s));
  prof_collect();
  if (hs.err & kd::DEV_ERR_TIMEOUT) return KD_ERR_TIMEOUT;
  if (hs.err & kd::DEV_ERR_INDEX) return KD_ERR_INDEX;
  const double n_mean = sharded ? n_norm : static_cast<double>(mask ? hs.n_valid : N);
  *loss = n_mean > 0 ? static_cast<float>(hs.loss_sum / n_mean) : 0.f;
  return KD_OK;
}

// run_impl, and after a CUDA error part-way through the chunk loop, a
// best-effort synchronisation: the call never returns while its own kernels
// may still use the caller's workspace or outputs.
kd_status run(const void* hidden, const void* W, const int32_t* idx, const float* logit,
              long long N, int H, int V, int K, float T, int chunk, float* loss, float* gh,
              float* gW, void* ws, size_t ws_bytes, cudaStream_t s, const kd_debug_opts* opts,
              const uint8_t* mask = nullptr, unsigned flags = 0, double n_norm = 0.0) {
  const kd_status st = run_impl(hidden, W, idx, logit, N, H, V, K, T, chunk, loss, gh, gW, ws,
                                ws_bytes, s, opts, mask, flags, nullptr, nullptr, n_norm);
  if (st == KD_ERR_CUDA) {
    cudaStreamSynchronize(s);
    cudaGetLastError();
  }
  return st;
}

}  // namespace

extern "C" {

size_t kd_topk_kl_workspace_size(int64_t N, int H, int V, int K, int chunk) {
  if (!sizes_ok(N, H, V, K, chunk)) return 0;
  return make_plan(N, H, V, K, chunk, device_sms()).total;
}

kd_status kd_topk_kl_fwd_bwd_ex(const void* hidden, const void* W, const int32_t* topk_idx,
                                const float* topk_logit, int64_t N, int H, int V, int K, float T,
                                int chunk, float* loss, float* grad_hidden, float* grad_W,
                                void* workspace, size_t workspace_bytes, void* stream) {
  return run(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden, grad_W,
             workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr);
}

kd_status kd_topk_kl_fwd_bwd_masked(const void* hidden, const void* W, const int32_t* topk_idx,
                                    const float* topk_logit, const uint8_t* token_mask,
                                    int64_t N, int H, int V, int K, float T, int chunk,
                                    int accumulate, float* loss, float* grad_hidden,
                                    float* grad_W, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  return run(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden, grad_W,
             workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr, token_mask,
             accumulate ? KD_FLAG_ACCUMULATE : 0u);
}

size_t kd_topk_kl_workspace_size_flags(int64_t N, int H, int V, int K, int chunk,
                                       unsigned flags) {
  if (!sizes_ok(N, H, V, K, chunk)) return 0;
  if (flags & ~kAllFlags) return 0;
  return make_plan(N, H, V, K, chunk, device_sms(), (flags & KD_FLAG_STORE_LOGITS) != 0,
                   (flags & KD_FLAG_MIN_SCRATCH) != 0).total;
}

kd_status kd_topk_kl_fwd_bwd_flags(const void* hidden, const void* W, const int32_t* topk_idx,
                                   const float* topk_logit, const uint8_t* token_mask,
                                   int64_t N, int H, int V, int K, float T, int chunk,
                                   unsigned flags, float* loss, float* grad_hidden, float* grad_W,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  return run(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden, grad_W,
             workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr, token_mask,
             flags);
}

kd_status kd_topk_kl_fwd_bwd_sharded(const void* hidden, const void* W, const int32_t* topk_idx,
                                     const float* topk_logit, const uint8_t* token_mask,
                                     int64_t N, int H, int V, int K, float T, int chunk,
                                     unsigned flags, int64_t n_norm, float* loss,
                                     float* grad_hidden, float* grad_W, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (n_norm < 1) return KD_ERR_INVALID_ARG;
  return run(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden, grad_W,
             workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr, token_mask,
             flags, static_cast<double>(n_norm));
}

kd_status kd_topk_kl_fwd_bwd_async(const void* hidden, const void* W, const int32_t* topk_idx,
                                   const float* topk_logit, const uint8_t* token_mask,
                                   int64_t N, int H, int V, int K, float T, int chunk,
                                   unsigned flags, float* loss_dev, int32_t* status_dev,
                                   float* grad_hidden, float* grad_W, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  t_prof_off = true;
  const kd_status st = run_impl(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, nullptr,
                                grad_hidden, grad_W, workspace, workspace_bytes, s, nullptr,
                                token_mask, flags, loss_dev, status_dev);
  t_prof_off = false;
  if (st == KD_ERR_CUDA) {
    // outside a capture, wait for what was enqueued before the failure
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusActive;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone)
      cudaStreamSynchronize(s);
    cudaGetLastError();
  }
  return st;
}

kd_status kd_topk_kl_debug(const void* hidden, const void* W, const int32_t* topk_idx,
                           const float* topk_logit, int64_t N, int H, int V, int K, float T,
                           int chunk, float* loss, float* grad_hidden, float* grad_W,
                           void* workspace, size_t workspace_bytes, void* stream,
                           const kd_debug_opts* opts) {
  if (opts) {
    if ((opts->lse && !is_device_ptr(opts->lse)) || (opts->zg && !is_device_ptr(opts->zg)) ||
        (opts->found_idx && !is_device_ptr(opts->found_idx)) ||
        (opts->loss_rows && !is_device_ptr(opts->loss_rows)))
      return KD_ERR_INVALID_ARG;
  }
  return run(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden, grad_W,
             workspace, workspace_bytes, static_cast<cudaStream_t>(stream), opts);
}

kd_status kd_topk_kl_fwd_bwd(const void* hidden, const void* W, const int32_t* topk_idx,
                             const float* topk_logit, int64_t N, int H, int V, int K, float T,
                             int chunk, float* loss, float* grad_hidden, float* grad_W) {
  kd_status st = validate(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden,
                          grad_W);
  if (st != KD_OK) return st;
  const size_t bytes = kd_topk_kl_workspace_size(N, H, V, K, chunk);
  void* ws = nullptr;
  cudaStream_t s = nullptr;
  if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return KD_ERR_OOM;
  }
  st = run(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden, grad_W, ws,
           bytes, s, nullptr);
  cudaError_t fe = cudaFreeAsync(ws, s);
  if (st == KD_OK && fe != cudaSuccess) return cuda_fail(fe, "cudaFreeAsync");
  if (st == KD_OK) {
    cudaError_t se = cudaStreamSynchronize(s);
    if (se != cudaSuccess) return cuda_fail(se, "cudaStreamSynchronize");
  }
  return st;
}

kd_status kd_gemm_bf16_test(const void* A, const void* B, float* C, int M, int N, int K, int a_mn,
                            int b_mn, int bn, int pair, void* stream) {
  if (!A || !B || !C) return KD_ERR_INVALID_ARG;
  if (M < 8 || N < 8 || K < 8 || M % 8 || N % 8 || K % 8) return KD_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return KD_ERR_ALIGNMENT;
  if (!is_device_ptr(A) || !is_device_ptr(B) || !is_device_ptr(C)) return KD_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int variant = a_mn ? (b_mn ? kd::GV_TEST_MM : kd::GV_TEST_MK)
                     : (b_mn ? kd::GV_TEST_KM : kd::GV_TEST_KK);
  if (pair == 2) {
    if ((bn != 0 && bn != 256) || a_mn || b_mn) return KD_ERR_INVALID_ARG;
    variant = kd::GV_TEST_KK2S;
  } else if (pair) {
    if (bn != 0 && bn != 256) return KD_ERR_INVALID_ARG;
    variant = a_mn ? (b_mn ? kd::GV_TEST_MM2 : kd::GV_TEST_MK2)
                   : (b_mn ? kd::GV_TEST_KM2 : kd::GV_TEST_KK2);
  } else if (bn != 0 && bn != kd::gemm_bn(variant)) {
    if (bn != 192 && bn != 256) return KD_ERR_INVALID_ARG;
    variant = a_mn ? (b_mn ? kd::GV_TEST_MM256 : kd::GV_TEST_MK256)
                   : (b_mn ? kd::GV_TEST_KM256 : kd::GV_TEST_KK192);
  }
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap ta, tb, tc;
  if (!bind_current_device()) return KD_ERR_CUDA;
  bool ok = true;
  ok &= a_mn ? make_map(&ta, BF16, 2, A, M, K, 64, 64) : make_map(&ta, BF16, 2, A, K, M, 64, 128);
  ok &= b_mn ? make_map(&tb, BF16, 2, B, N, K, 64, 64)
              : make_map(&tb, BF16, 2, B, K, N, 64, b_box_rows(variant));
  ok &= make_map(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, N, M, 32, 32);
  if (!ok) return KD_ERR_CUDA;
  DevStatus* dst = nullptr;
  KD_CUDA(cudaMallocAsync(&dst, sizeof(DevStatus), s));
  KD_CUDA(cudaMemsetAsync(dst, 0, sizeof(DevStatus), s));
  kd::GemmArgs g{};
  g.m_tiles = static_cast<int>(cdiv(M, kd::gemm_tile_m(variant)));
  g.n_tiles = static_cast<int>(cdiv(N, kd::gemm_bn(variant)));
  g.splits = 1; g.kb_total = static_cast<int>(cdiv(K, 64)); g.order = kd::ORDER_M_FAST;
  g.timeout_ns = kDefaultTimeoutNs; g.status = dst;
  kd::EpiArgs e{};
  e.rows_valid = M; e.cols_valid = N; e.alpha = 1.f;
  KD_CUDA(kd::launch_gemm(variant, ta, tb, tc, g, e, s));
  DevStatus hs{};
  KD_CUDA(cudaMemcpyAsync(&hs, dst, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
  KD_CUDA(cudaFreeAsync(dst, s));
  KD_CUDA(cudaStreamSynchronize(s));
  if (hs.err & kd::DEV_ERR_TIMEOUT) return KD_ERR_TIMEOUT;
  return KD_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- top-K cache builder
namespace {

struct CachePlan {
  int chunk, n_chunks, vt;
  size_t off_status, off_part, off_z, off_tau, off_cnt, off_cand, total;
};

CachePlan make_cache_plan(long long N, int V, int chunk) {
  CachePlan p{};
  long long c = cdiv(chunk, 128) * 128;
  const long long cmax = cdiv(N, 128) * 128;
  if (c > cmax) c = cmax;
  if (c > kMaxChunk) c = kMaxChunk;   // row coordinates of the chunk buffers stay in int
  p.chunk = static_cast<int>(c);
  p.n_chunks = static_cast<int>(cdiv(N, c));
  p.vt = static_cast<int>(cdiv(V, kd::gemm_bn(kd::GV_FWDZ)));
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes, 256); return at; };
  p.off_status = take(sizeof(DevStatus));
  p.off_part = take(sizeof(float2) * p.vt * c);
  p.off_z = take(4ull * c * V);
  p.off_tau = take(sizeof(float) * c);
  p.off_cnt = take(sizeof(uint32_t) * c);
  p.off_cand = take(sizeof(unsigned long long) * c * kd::SEL_GCAP);
  p.total = o;
  return p;
}

bool cache_sizes_ok(long long N, int H, int V, int K, int chunk) {
  return N >= 1 && N <= 0x7fffffffLL && H >= 8 && H % 8 == 0 && V >= 8 && V % 8 == 0 &&
         K >= 1 && K <= V && K <= 8192 && chunk >= 1;
}

kd_status cache_build_impl(const void* hidden, const void* W, int64_t N, int H, int V, int K,
                           int chunk, int32_t* topk_idx, float* topk_logit, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (!hidden || !W || !topk_idx || !topk_logit || !workspace) return KD_ERR_INVALID_ARG;
  if (!cache_sizes_ok(N, H, V, K, chunk)) return KD_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(topk_idx, 4) ||
      !aligned(topk_logit, 4) || !aligned(workspace, 256))
    return KD_ERR_ALIGNMENT;
  if (!is_device_ptr(hidden) || !is_device_ptr(W) || !is_device_ptr(topk_idx) ||
      !is_device_ptr(topk_logit) || !is_device_ptr(workspace))
    return KD_ERR_INVALID_ARG;
  const CachePlan p = make_cache_plan(N, V, chunk);
  if (workspace_bytes < p.total) return KD_ERR_OOM;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prof_reset_call();
  uint8_t* base = static_cast<uint8_t*>(workspace);
  DevStatus* dst = reinterpret_cast<DevStatus*>(base + p.off_status);
  float2* part = reinterpret_cast<float2*>(base + p.off_part);
  float* zbuf = reinterpret_cast<float*>(base + p.off_z);
  float* tau = reinterpret_cast<float*>(base + p.off_tau);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(base + p.off_cnt);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(base + p.off_cand);

  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tm_hid_k, tm_w_k, tm_z_st;
  if (!bind_current_device()) return KD_ERR_CUDA;
  bool ok = true;
  ok &= make_map(&tm_hid_k, BF16, 2, hidden, H, N, 64, 128);
  ok &= make_map(&tm_w_k, BF16, 2, W, H, V, 64, b_box_rows(kd::GV_FWDZ));
  ok &= make_map(&tm_z_st, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, zbuf, V, p.chunk, 32, 32);
  if (!ok) return KD_ERR_CUDA;   // make_map left the driver's result in the last-error text
  KD_CUDA(cudaMemsetAsync(dst, 0, sizeof(DevStatus), s));
  for (int j = 0; j < p.n_chunks; ++j) {
    const int row0 = j * p.chunk;
    const int cj = static_cast<int>(std::min<long long>(p.chunk, N - row0));
    kd::GemmArgs g{};
    g.m_tiles = static_cast<int>(cdiv(cj, kd::gemm_tile_m(kd::GV_FWDZ)));
    g.n_tiles = p.vt; g.splits = 1;
    g.kb_total = static_cast<int>(cdiv(H, 64));
    g.order = kd::ORDER_M_FAST; g.a_row0 = row0; g.b_row0 = 0;
    g.timeout_ns = kDefaultTimeoutNs; g.status = dst;
    kd::EpiArgs e{};
    // the forward epilogue with scale 1 and no cached ids: part[.].x is the
    // exact maximum of each (row, 256-wide vocab tile), z is stored in fp32
    e.rows_valid = cj; e.cols_valid = V; e.scale2 = 1.f; e.alpha = 1.f;
    e.K = 0; e.grow0 = row0; e.c_alloc = p.chunk; e.part = part;
    { ProfScope ps_(PK_CACHE_GEMM, s);
      KD_CUDA(kd::launch_gemm(kd::GV_FWDZ, tm_hid_k, tm_w_k, tm_z_st, g, e, s)); }
    { ProfScope ps_(PK_CACHE_SELECT, s);
      KD_CUDA(kd::launch_topk_select(zbuf, V, part, p.vt, p.chunk, cj, K, row0, tau, cnt, cand,
                                     topk_idx, topk_logit, s)); }
  }
  DevStatus hs{};
  KD_CUDA(cudaMemcpyAsync(&hs, dst, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
  KD_CUDA(cudaStreamSynchronize(s));
  prof_collect();
  if (hs.err & kd::DEV_ERR_TIMEOUT) return KD_ERR_TIMEOUT;
  return KD_OK;
}

}  // namespace

extern "C" {

size_t kd_topk_cache_workspace_size(int64_t N, int H, int V, int K, int chunk) {
  if (!cache_sizes_ok(N, H, V, K, chunk)) return 0;
  return make_cache_plan(N, V, chunk).total;
}

kd_status kd_topk_cache_build(const void* hidden, const void* W, int64_t N, int H, int V, int K,
                              int chunk, int32_t* topk_idx, float* topk_logit, void* workspace,
                              size_t workspace_bytes, void* stream) {
  const kd_status st = cache_build_impl(hidden, W, N, H, V, K, chunk, topk_idx, topk_logit,
                                        workspace, workspace_bytes, stream);
  if (st == KD_ERR_CUDA) {   // never return while its kernels may still run
    cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    cudaGetLastError();
  }
  return st;
}

}  // extern "C"

// ---------------------------------------------------------------- no-alloc entry
// The scratch of kd_topk_kl_fwd_bwd_noalloc: a fixed device buffer owned by
// the library, so that callers who may not allocate device memory can still
// run the loss.  Host code must not pass the symbol itself to a kernel (on the
// host it only names a stand-in object); it passes the device address looked
// up once per device below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KD_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up on
// the first call per device).  nullptr and *st set on failure.
void* noalloc_scratch(kd_status* st) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *st = cuda_fail(e, "cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *st = KD_ERR_INVALID_ARG;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    // the first lookup on a device loads the module that holds the buffer
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e == cudaErrorMemoryAllocation) {
      cuda_fail(e, "cudaGetSymbolAddress");
      cudaGetLastError();
      *st = KD_ERR_OOM;
      return nullptr;
    }
    if (e != cudaSuccess || p == nullptr) {
      *st = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol, "cudaGetSymbolAddress");
      return nullptr;
    }
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" {

kd_status kd_topk_kl_fwd_bwd_noalloc(const void* hidden, const void* W, const int32_t* topk_idx,
                                     const float* topk_logit, int64_t N, int H, int V, int K,
                                     float T, int chunk, float* loss, float* grad_hidden,
                                     float* grad_W, void* stream) {
  kd_status st = validate(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden,
                          grad_W);
  if (st != KD_OK) return st;
  const size_t need = kd_topk_kl_workspace_size(N, H, V, K, chunk);
  if (need == 0) return KD_ERR_INVALID_ARG;
  if (need > KD_NOALLOC_SCRATCH_BYTES) return KD_ERR_TOO_LARGE;
  void* ws = noalloc_scratch(&st);
  if (!ws) return st;
  // run() resets the status word it needs zeroed; the rest of the workspace
  // is fully written before it is read, whatever the previous call left.
  return run(hidden, W, topk_idx, topk_logit, N, H, V, K, T, chunk, loss, grad_hidden, grad_W,
             ws, KD_NOALLOC_SCRATCH_BYTES, static_cast<cudaStream_t>(stream), nullptr);
}

const char* kd_status_string(kd_status s) {
  switch (s) {
    case KD_OK: return "ok";
    case KD_ERR_INVALID_ARG: return "invalid argument";
    case KD_ERR_ALIGNMENT: return "misaligned pointer";
    case KD_ERR_INDEX: return "teacher id outside [0, V)";
    case KD_ERR_OOM: return "out of device memory (or workspace too small)";
    case KD_ERR_CUDA: return "CUDA error";
    case KD_ERR_TIMEOUT: return "device-side wait timed out";
    case KD_ERR_NOT_IMPLEMENTED: return "not implemented";
    case KD_ERR_TOO_LARGE: return "problem needs more scratch than KD_NOALLOC_SCRATCH_BYTES";
  }
  return "unknown status";
}

const char* kd_last_cuda_error(void) { return g_last_cuda_error; }

void kd_profile_enable(int on) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  if (on && !P.on) {
    for (int k = 0; k < PK_COUNT; ++k) { P.total_ms[k] = 0.0; P.launches[k] = 0; }
  }
  P.on = on != 0;
  P.used = 0;
}

int kd_profile_read(double* total_ms, long long* launches, int max_kinds) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  const int n = max_kinds < PK_COUNT ? max_kinds : PK_COUNT;
  for (int k = 0; k < n; ++k) {
    if (total_ms) total_ms[k] = P.total_ms[k];
    if (launches) launches[k] = P.launches[k];
  }
  return PK_COUNT;
}

const char* kd_profile_kind_name(int kind) {
  return (kind >= 0 && kind < PK_COUNT) ? kProfNames[kind] : "";
}

int kd_abi_version(void) { return 2; }

#ifndef KD_BUILD_ID
#define KD_BUILD_ID "unknown"
#endif
const char* kd_build_id(void) { return KD_BUILD_ID; }

}  // extern "C"

// Host side of the C ABI declared in include/flce.h: argument checks, workspace
// layout, TMA tensor maps, launch sequence and the optional per-kernel timing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "flce.h"
#include "flce_kernels.cuh"

namespace {

using namespace flce;

thread_local char g_last_error[512] = "";

flce_status fail(flce_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

#define CUDA_TRY(expr)                                                                            \
  do {                                                                                            \
    cudaError_t e_ = (expr);                                                                      \
    if (e_ != cudaSuccess) return fail(FLCE_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));  \
  } while (0)

constexpr size_t kHeaderBytes = 256;  // status word and spare scalars at the start of each workspace
constexpr size_t kUnitCounterOff = 32;  // forward header: the logit kernel's work-unit counter (int32, zeroed per call)
constexpr int kMaxSplit = 16;         // forward: vocab ranges per token block
constexpr int64_t kDefaultChunk = 8192;
constexpr int32_t kMaxShards = 64;    // vocab shards one combine call merges
// T and V bound: tile coordinates (block * 128 + row) stay inside int32 with room to spare.
constexpr int64_t kMaxRows = int64_t(1) << 30;

std::atomic<uint64_t> g_timeout_ns{4000000000ull};
std::atomic<bool> g_timeout_fixed{false};  // set by flce_set_wait_timeout_ns

// Limit of the bounded waits of one GEMM launch whose longest tile has a K loop of
// `k_max`.  The longest wait inside the kernels is the epilogue's wait for one
// tile's whole K loop: a 256 x 256 pair tile needs 8 SM-pair clocks per unit of K
// (131,072 FLOP at 16,384 dense bf16 FLOP per pair per clock), so 16 ns per unit of
// K covers it twice over at 1 GHz.  A limit the caller fixed is used as it is.
uint64_t wait_limit_ns(int64_t k_max) {
  const uint64_t base = g_timeout_ns.load();
  if (g_timeout_fixed.load()) return base;
  return std::max<uint64_t>(base, 16ull * static_cast<uint64_t>(std::max<int64_t>(k_max, 0)));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The kernels read and write the per-token arrays with plain typed loads and
// stores, so each pointer must carry its type's natural alignment (checked on the
// host: a misaligned access would fault the device instead of returning an error).
template <typename E>
bool misaligned(const E* p) {
  return (reinterpret_cast<uintptr_t>(p) % alignof(E)) != 0;
}
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ device info
struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int major = 0, minor = 0;
  bool attrs_set = false;
  int pairs[4] = {0, 0, 0, 0};  // co-resident CTA pairs (clusters of 2) per GEMM mode
};

template <int MODE>
flce_status query_pairs(DeviceInfo& d) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * std::max(d.sms / 2, 1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for(MODE);
  int n = 0;
  CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, gemm_kernel<MODE>, &cfg));
  d.pairs[MODE] = std::max(1, std::min(n, d.sms / 2));
  return FLCE_OK;
}
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

flce_status device_info(DeviceInfo** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(FLCE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    CUDA_TRY(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
    CUDA_TRY(cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev));
    CUDA_TRY(cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev));
    d.init = true;
  }
  if (!(d.major == 10 && d.minor == 3))
    return fail(FLCE_ERR_UNSUPPORTED, "this library is built for sm_103a; device is sm_%d%d", d.major, d.minor);
  if (!d.attrs_set) {
    CUDA_TRY(cudaFuncSetAttribute(gemm_kernel<MODE_FWD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem_bytes_for(MODE_FWD)));
    CUDA_TRY(cudaFuncSetAttribute(gemm_kernel<MODE_DZ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem_bytes_for(MODE_DZ)));
    CUDA_TRY(cudaFuncSetAttribute(gemm_kernel<MODE_DHW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem_bytes_for(MODE_DHW)));
    CUDA_TRY(cudaFuncSetAttribute(gemm_kernel<MODE_SCORE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem_bytes_for(MODE_SCORE)));
    flce_status st;
    if ((st = query_pairs<MODE_FWD>(d)) != FLCE_OK) return st;
    if ((st = query_pairs<MODE_DZ>(d)) != FLCE_OK) return st;
    if ((st = query_pairs<MODE_DHW>(d)) != FLCE_OK) return st;
    if ((st = query_pairs<MODE_SCORE>(d)) != FLCE_OK) return st;
    d.attrs_set = true;
  }
  *out = &d;
  return FLCE_OK;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

flce_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(FLCE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  return FLCE_OK;
}

// 2-D map over a row-major matrix: `inner` contiguous elements per row,
// `outer` rows, `pitch` bytes between rows; box {box_inner, box_outer};
// 128-byte swizzle; out-of-range elements read as zero, stores are clipped.
flce_status make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
                     uint64_t pitch, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FLCE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for dims {%llu, %llu} pitch %llu box {%u, %u}",
                static_cast<int>(r), static_cast<unsigned long long>(inner), static_cast<unsigned long long>(outer),
                static_cast<unsigned long long>(pitch), box_inner, box_outer);
  return FLCE_OK;
}

// 3-D map over the dZ block stored as 64-column panels: {64 columns, rows,
// panels}, rows of 128 bytes, panels `rows` x 128 bytes apart; box {64,
// box_rows, 1}; 128-byte swizzle.  Out-of-range panels read as zero, stores
// there are clipped.
flce_status make_panel_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t panels, uint32_t box_rows) {
  cuuint64_t dims[3] = {64, rows, panels};
  cuuint64_t strides[2] = {128, 128 * rows};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FLCE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for panels {64, %llu, %llu} box rows %u",
                static_cast<int>(r), static_cast<unsigned long long>(rows), static_cast<unsigned long long>(panels),
                box_rows);
  return FLCE_OK;
}

// ------------------------------------------------------------------ profiling
struct LaunchRecord {
  int kind;
  cudaEvent_t start, stop;
  double flops, bytes;
  // Launches over the backward's row list add rows * (flops, bytes) per row, the
  // rows read from the workspace when the records are collected.
  const int32_t* rows_dev;
  int64_t index0, cap;
  double flops_per_row, bytes_per_row;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<LaunchRecord> g_records;
std::vector<cudaEvent_t> g_event_pool;

// An event from the pool, or a new one; nullptr if none can be created.
cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one launch with an NVTX range named after the kernel (seen by any
// attached profiler) and, while profiling is enabled, with events on its stream.
struct KernelScope {
  bool on = false;
  bool nvtx = true;
  LaunchRecord rec{};
  cudaStream_t stream;
  KernelScope(int kind, cudaStream_t s, double flops, double bytes, const int32_t* rows_dev = nullptr,
              int64_t index0 = 0, int64_t cap = 0, double flops_per_row = 0.0, double bytes_per_row = 0.0)
      : stream(s) {
    nvtxRangePushA(flce_kernel_name(kind));
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    on = true;
    rec.kind = kind;
    rec.flops = flops;
    rec.bytes = bytes;
    rec.rows_dev = rows_dev;
    rec.index0 = index0;
    rec.cap = cap;
    rec.flops_per_row = flops_per_row;
    rec.bytes_per_row = bytes_per_row;
    rec.start = take_event();
    rec.stop = take_event();
    if (!rec.start || !rec.stop || cudaEventRecord(rec.start, s) != cudaSuccess) {
      // no timing for this launch (the profile is an aid; the launch itself goes
      // ahead, and the failed call's error is cleared so that it is not taken for
      // the launch's)
      (void)cudaGetLastError();
      release_events();
    }
  }
  ~KernelScope() {
    if (nvtx) nvtxRangePop();
    if (on) {  // an error return before done(): the events go back to the pool
      std::lock_guard<std::mutex> lk(g_prof_mu);
      release_events();
    }
  }
  // Caller holds g_prof_mu.
  void release_events() {
    if (rec.start) g_event_pool.push_back(rec.start);
    if (rec.stop) g_event_pool.push_back(rec.stop);
    rec.start = rec.stop = nullptr;
    on = false;
  }
  void done() {
    if (nvtx) {
      nvtxRangePop();
      nvtx = false;
    }
    if (!on) return;
    const bool ok = cudaEventRecord(rec.stop, stream) == cudaSuccess;
    if (!ok) (void)cudaGetLastError();
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (ok) {
      g_records.push_back(rec);
      on = false;
    } else {
      release_events();
    }
  }
};

flce_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FLCE_ERR_CUDA, "launch of %s failed: %s", what, cudaGetErrorString(e));
  return FLCE_OK;
}

// ------------------------------------------------------------------ workspace layouts
struct FwdLayout {
  int n_split;
  int64_t part_stride;
  size_t partials_off, zy_off, bsum_off, bcnt_off, total;
  int num_fin_blocks;
};

FwdLayout fwd_layout(int64_t T, int n_split) {
  FwdLayout L{};
  L.n_split = n_split;
  L.part_stride = static_cast<int64_t>(align_up(static_cast<size_t>(std::max<int64_t>(T, 1)), 128));
  L.num_fin_blocks = static_cast<int>(std::max<int64_t>(cdiv(T, kFinalizeThreads), 1));
  size_t off = kHeaderBytes;
  L.partials_off = off;
  off = align_up(off + sizeof(float2) * static_cast<size_t>(n_split) * L.part_stride, 256);
  L.zy_off = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(L.part_stride), 256);
  L.bsum_off = off;
  off = align_up(off + sizeof(double) * L.num_fin_blocks, 256);
  L.bcnt_off = off;
  off = align_up(off + sizeof(int64_t) * L.num_fin_blocks, 256);
  L.total = off;
  return L;
}

// flce_forward_valid: the forward layout (all kMaxSplit ranges), then the row
// list [T] and each token's list position [T] (int32), then the listed rows of
// H [T, Hd] bf16.  The list length sits in the header.
struct FwdValidLayout {
  size_t idx_off, pos_off, hc_off, total;
};

FwdValidLayout fwd_valid_layout(int64_t T, int64_t Hd) {
  FwdValidLayout L{};
  const size_t t1 = static_cast<size_t>(std::max<int64_t>(T, 1));
  size_t off = align_up(fwd_layout(T, kMaxSplit).total, 256);
  L.idx_off = off;
  off = align_up(off + sizeof(int32_t) * t1, 256);
  L.pos_off = off;
  off = align_up(off + sizeof(int32_t) * t1, 1024);
  L.hc_off = off;
  off = align_up(off + 2ull * t1 * static_cast<size_t>(Hd), 256);
  L.total = off;
  return L;
}

struct BwdLayout {
  int64_t chunk;
  int64_t v_pad;
  int64_t max_chunks;
  size_t cnt_off, g_off, idx_off, hc_off, dz_off, total;
};

constexpr size_t kRowCountOff = 16;  // backward header: length of the row list (int32)

// Header (status word, row count) | tile counters (one per possible chunk) |
// g [T] | row list [T] | H rows of the chunk [chunk, Hd] | dZ chunk: V_pad / 64
// panels of [chunk, 64] (DzPanels).  The dH rows go straight to the caller's dH.
BwdLayout bwd_layout(int64_t T, int64_t Hd, int64_t V, int64_t chunk) {
  BwdLayout L{};
  L.chunk = chunk;
  L.v_pad = static_cast<int64_t>(align_up(static_cast<size_t>(V), 64));
  L.max_chunks = cdiv(std::max<int64_t>(T, 1), 128);
  const size_t t1 = static_cast<size_t>(std::max<int64_t>(T, 1));
  size_t off = kHeaderBytes;
  L.cnt_off = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(L.max_chunks), 256);
  L.g_off = off;
  off = align_up(off + sizeof(float) * t1, 256);
  L.idx_off = off;
  off = align_up(off + sizeof(int32_t) * t1, 1024);
  L.hc_off = off;
  off = align_up(off + 2ull * static_cast<size_t>(chunk) * static_cast<size_t>(Hd), 1024);
  L.dz_off = off;
  off = align_up(off + 2ull * static_cast<size_t>(chunk) * L.v_pad, 256);
  L.total = off;
  return L;
}

int64_t default_chunk(int64_t T) {
  // Up to 256 rows: one chunk (fewest launches).  Above: at most T / 2, so dZ
  // residency stays [chunk x V] <= [T/2 x V] and the whole workspace below one
  // [T x V] bf16 tensor whenever Hd < V / 2.
  if (T <= 256) return T <= 128 ? 128 : 256;
  const int64_t c = std::max<int64_t>(T / 2 / 128 * 128, 128);
  return std::min<int64_t>(c, kDefaultChunk);
}

// Vocab ranges per token pair for the forward: the even count whose units
// spread most evenly over `grid` persistent SM pairs, ties going to fewer
// ranges; 1 when V has a single tile.
int pick_split(int64_t m_blocks, int64_t n_blocks, int grid) {
  int best = 1;
  double best_eff = -1.0;
  const int max_split = static_cast<int>(std::min<int64_t>(kMaxSplit, n_blocks));
  for (int ns = 2; ns <= max_split; ns += 2) {
    const int64_t units = m_blocks * ns;
    const int64_t per_unit = cdiv(n_blocks, ns);
    const int64_t waves = cdiv(units, grid);
    // every SM counts, also those left without a unit
    const double eff = static_cast<double>(m_blocks * n_blocks) / static_cast<double>(grid * waves * per_unit);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = ns;
    }
  }
  return best;
}

// The forward's unit schedule: range-major units from the work-index ring when
// the H blocks of all in-flight token pairs (pairs of them, 512 * Hd bytes each)
// fit in about 80 MB of L2, else units strided over the pairs with the vocab
// ranges taken four at a time (two, or one, when n_split does not divide by
// four).  Both from measurements at Hd = 2048 and 4096 (see the kernel's
// decode_unit).
struct FwdSchedule {
  int split_group;
  int dynamic;
};
FwdSchedule fwd_schedule(int n_split, int64_t Hd, int64_t pairs) {
  constexpr double kL2Budget = 80.0 * 1024 * 1024;
  if (static_cast<double>(pairs) * 512.0 * static_cast<double>(Hd) <= kL2Budget) return {1, 1};
  return {n_split % 4 == 0 ? 4 : (n_split % 2 == 0 ? 2 : 1), 0};
}

flce_status check_common(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd, int64_t V,
                         int64_t ignore_index, int32_t reduction) {
  if (T < 0 || T >= kMaxRows) return fail(FLCE_ERR_INVALID_ARG, "T = %lld out of range", (long long)T);
  if (V < 1 || V >= kMaxRows) return fail(FLCE_ERR_INVALID_ARG, "V = %lld out of range", (long long)V);
  if (Hd < 1 || Hd >= (int64_t(1) << 24)) return fail(FLCE_ERR_INVALID_ARG, "Hd = %lld out of range", (long long)Hd);
  if (Hd % 64 != 0) return fail(FLCE_ERR_UNSUPPORTED, "Hd = %lld is not a multiple of 64", (long long)Hd);
  if (reduction < 0 || reduction > 2) return fail(FLCE_ERR_INVALID_ARG, "unknown reduction %d", reduction);
  if (ignore_index >= 0 && ignore_index < V)
    return fail(FLCE_ERR_INVALID_ARG, "ignore_index %lld lies inside [0, V)", (long long)ignore_index);
  if (!W) return fail(FLCE_ERR_INVALID_ARG, "W is NULL");
  if (T > 0 && (!H || !targets)) return fail(FLCE_ERR_INVALID_ARG, "H or targets is NULL");
  if ((reinterpret_cast<uintptr_t>(H) | reinterpret_cast<uintptr_t>(W)) & 15)
    return fail(FLCE_ERR_ALIGNMENT, "H and W must be 16-byte aligned");
  if (misaligned(targets)) return fail(FLCE_ERR_ALIGNMENT, "targets must be 8-byte aligned");
  return FLCE_OK;
}

// ------------------------------------------------------------------ built-in scratch
// Scratch of flce_forward_noalloc(): a device array of fixed size in this
// library's module.  Host code must not use the symbol as a pointer; the
// device address comes from cudaGetSymbolAddress with the device current.
// The address belongs to the module as loaded into one context, so it is
// remembered per (device, current context): a context created after
// cudaDeviceReset, or another context made current on the same device, loads
// the module again and gets its address looked up again.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];
std::mutex g_scratch_mu;
struct ScratchSlot {
  CUcontext ctx = nullptr;
  void* addr = nullptr;
};
ScratchSlot g_scratch_slot[64];
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;

flce_status static_scratch_address(void** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(FLCE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_ctx_get_current) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    if (!g_ctx_get_current) return fail(FLCE_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
  }
  auto lookup = [&](void** p) -> flce_status {
    const cudaError_t e = cudaGetSymbolAddress(p, g_static_scratch);
    if (e != cudaSuccess || !*p)
      return fail(FLCE_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch failed on device %d: %s", dev,
                  cudaGetErrorString(e));
    return FLCE_OK;
  };
  ScratchSlot& slot = g_scratch_slot[dev];
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  if (!ctx) {
    // No context yet on this thread: the runtime call below makes the device's
    // primary context current, and the address is remembered for that context.
    void* p = nullptr;
    flce_status st = lookup(&p);
    if (st != FLCE_OK) return st;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx)
      return fail(FLCE_ERR_CUDA, "no current CUDA context on device %d", dev);
    slot.ctx = ctx;
    slot.addr = p;
  } else if (slot.ctx != ctx || !slot.addr) {
    void* p = nullptr;
    flce_status st = lookup(&p);
    if (st != FLCE_OK) return st;
    slot.ctx = ctx;
    slot.addr = p;
  }
  *out = slot.addr;
  return FLCE_OK;
}

// ------------------------------------------------------------------ shared launch sequences
// Logit tiles of H against W rows [0, V) (global ids vocab_offset + row): per
// row and vocab range, the running max / sum-exp partials and the target
// logit (when these rows own the target) go to the workspace layout L.
// With `best_val` / `best_idx` set (scoring), the argmax variant also records
// each row's largest logit and its global id per vocab range.
// Over a row list (rows_dev, row_index set), H holds the listed rows in list
// order and the partials are written at list positions.
flce_status launch_logits_lse(DeviceInfo* dev, cudaStream_t s, const void* H, const void* W, const int64_t* targets,
                              int64_t T, int64_t Hd, int64_t V, int64_t vocab_offset, int64_t ignore_index,
                              uint8_t* ws, FwdLayout* L_out, float* best_val = nullptr,
                              int32_t* best_idx = nullptr, const int32_t* rows_dev = nullptr,
                              const int32_t* row_index = nullptr) {
  flce_status st;
  const int64_t m_pairs = cdiv(T, 2 * BM);
  const int64_t n_blocks = cdiv(V, BN);
  const int n_split = pick_split(m_pairs, n_blocks, dev->pairs[MODE_FWD]);
  const FwdLayout L = fwd_layout(T, n_split);
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  if ((st = make_map(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, H, Hd, T, Hd * 2, BK, BM)) != FLCE_OK) return st;
  if ((st = make_map(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, Hd, V, Hd * 2, BK, BN_HALF)) != FLCE_OK) return st;
  p.num_m_pairs = static_cast<int32_t>(m_pairs);
  p.num_n_blocks = static_cast<int32_t>(n_blocks);
  p.num_k_blocks = static_cast<int32_t>(Hd / BK);
  p.n_split = n_split;
  const FwdSchedule sched = fwd_schedule(n_split, Hd, std::min<int64_t>(dev->pairs[MODE_FWD], m_pairs * n_split));
  p.split_group = sched.split_group;
  p.dynamic_units = sched.dynamic;
  p.num_units = static_cast<int32_t>(m_pairs * n_split);
  p.row0 = 0;
  p.rows = static_cast<int32_t>(T);
  p.T = static_cast<int32_t>(T);
  p.V = static_cast<int32_t>(V);
  p.part_stride = static_cast<int32_t>(L.part_stride);
  p.vocab_offset = vocab_offset;
  p.ignore_index = ignore_index;
  p.targets = targets;
  p.partials = reinterpret_cast<float2*>(ws + L.partials_off);
  p.zy = reinterpret_cast<float*>(ws + L.zy_off);
  p.best_val = best_val;
  p.best_idx = best_idx;
  p.status = reinterpret_cast<int32_t*>(ws);
  p.tile_counter = reinterpret_cast<int32_t*>(ws + kUnitCounterOff);  // zeroed with the header by every caller
  p.timeout_ns = wait_limit_ns(Hd);
  p.rows_dev = rows_dev;
  p.row_index = row_index;
  const bool score = best_val != nullptr;
  const int grid = 2 * static_cast<int>(std::min<int64_t>(dev->pairs[score ? MODE_SCORE : MODE_FWD], p.num_units));
  // Over a row list the work is counted on the listed rows (read at collection).
  const double per_row_bytes = 2.0 * Hd + (score ? 16.0 : 8.0) * n_split + 4.0;
  KernelScope ks(FLCE_KERNEL_FWD_LOGITS_LSE, s, rows_dev ? 0.0 : 2.0 * T * Hd * V,
                 2.0 * V * Hd + (rows_dev ? 0.0 : per_row_bytes * T), rows_dev, 0, T, rows_dev ? 2.0 * Hd * V : 0.0,
                 rows_dev ? per_row_bytes : 0.0);
  if (score)
    gemm_kernel<MODE_SCORE><<<grid, kThreads, smem_bytes_for(MODE_SCORE), s>>>(p);
  else
    gemm_kernel<MODE_FWD><<<grid, kThreads, smem_bytes_for(MODE_FWD), s>>>(p);
  ks.done();
  if ((st = check_launch("fwd_logits_lse")) != FLCE_OK) return st;
  *L_out = L;
  return FLCE_OK;
}

// Partials of layout L (n_split ranges, z_y) -> lse, logp, loss, n_valid.
flce_status launch_finalize_reduce(cudaStream_t s, uint8_t* ws, const FwdLayout& L, const int64_t* targets, int64_t T,
                                   int64_t V_total, int64_t ignore_index, int32_t reduction, float* loss, float* lse,
                                   float* logp, int64_t* n_valid, const int32_t* pos = nullptr) {
  flce_status st;
  FinalizeParams f;
  f.partials = reinterpret_cast<const float2*>(ws + L.partials_off);
  f.zy = reinterpret_cast<const float*>(ws + L.zy_off);
  f.targets = targets;
  f.lse = lse;
  f.logp = logp;
  f.loss_rows = reduction == FLCE_REDUCTION_NONE ? loss : nullptr;
  f.block_sum = reinterpret_cast<double*>(ws + L.bsum_off);
  f.block_count = reinterpret_cast<int64_t*>(ws + L.bcnt_off);
  f.status = reinterpret_cast<int32_t*>(ws);
  f.pos = pos;
  f.ignore_index = ignore_index;
  f.T = static_cast<int32_t>(T);
  f.V = static_cast<int32_t>(V_total);
  f.n_split = L.n_split;
  f.part_stride = static_cast<int32_t>(L.part_stride);
  {
    KernelScope ks(FLCE_KERNEL_FWD_FINALIZE, s, 0.0, (8.0 * L.n_split + 4 + 8 + 12) * T);
    fwd_finalize_kernel<<<L.num_fin_blocks, kFinalizeThreads, 0, s>>>(f);
    ks.done();
    if ((st = check_launch("fwd_finalize")) != FLCE_OK) return st;
  }
  {
    KernelScope ks(FLCE_KERNEL_FWD_REDUCE, s, 0.0, 16.0 * L.num_fin_blocks);
    fwd_reduce_kernel<<<1, kReduceThreads, 0, s>>>(f.block_sum, f.block_count, L.num_fin_blocks, reduction, loss,
                                                   n_valid);
    ks.done();
    if ((st = check_launch("fwd_reduce")) != FLCE_OK) return st;
  }
  return FLCE_OK;
}

flce_status check_shard(int64_t V_shard, int64_t vocab_offset, int64_t V_total, int64_t ignore_index) {
  if (V_total < 1 || V_total >= kMaxRows)
    return fail(FLCE_ERR_INVALID_ARG, "V_total = %lld out of range", (long long)V_total);
  if (V_shard < 1 || vocab_offset < 0 || vocab_offset + V_shard > V_total)
    return fail(FLCE_ERR_INVALID_ARG, "shard [%lld, %lld) does not lie inside [0, V_total = %lld)",
                (long long)vocab_offset, (long long)(vocab_offset + V_shard), (long long)V_total);
  if (ignore_index >= 0 && ignore_index < V_total)
    return fail(FLCE_ERR_INVALID_ARG, "ignore_index %lld lies inside [0, V_total)", (long long)ignore_index);
  return FLCE_OK;
}

// The backward over W rows [0, V) with global ids vocab_offset + row; g_t is
// computed against the full vocabulary [0, V_total).
flce_status backward_impl(const float* dloss, const float* dlogp, const void* H, const void* W,
                          const int64_t* targets, const float* lse, int64_t T, int64_t Hd, int64_t V,
                          int64_t vocab_offset, int64_t V_total, int64_t ignore_index, int32_t reduction, void* dH,
                          float* dW, void* workspace, size_t workspace_bytes, void* stream) {
  flce_status st;
  if (!dW || (T > 0 && ((!dloss && !dlogp) || !lse || !dH)))
    return fail(FLCE_ERR_INVALID_ARG, "dloss (or dlogp), lse, dH or dW is NULL");
  if ((reinterpret_cast<uintptr_t>(dH) | reinterpret_cast<uintptr_t>(dW)) & 15)
    return fail(FLCE_ERR_ALIGNMENT, "dH and dW must be 16-byte aligned");
  if (misaligned(dloss) || misaligned(dlogp) || misaligned(lse))
    return fail(FLCE_ERR_ALIGNMENT, "dloss, dlogp and lse must be 4-byte aligned");
  if (!workspace) return fail(FLCE_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(FLCE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  const int64_t chunk = flce_backward_chunk_tokens(T, Hd, V, workspace_bytes);
  if (chunk <= 0)
    return fail(FLCE_ERR_WORKSPACE, "workspace of %zu bytes is too small (need %zu)", workspace_bytes,
                flce_backward_workspace_size(T, Hd, V));
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FLCE_OK) return st;
  if ((st = get_encoder()) != FLCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  CUDA_TRY(cudaMemsetAsync(ws, 0, kHeaderBytes, s));

  if (T == 0) {
    CUDA_TRY(cudaMemsetAsync(dW, 0, sizeof(float) * static_cast<size_t>(V) * Hd, s));
    return FLCE_OK;
  }
  const BwdLayout L = bwd_layout(T, Hd, V, chunk);
  float* g = reinterpret_cast<float*>(ws + L.g_off);
  int32_t* row_index = reinterpret_cast<int32_t*>(ws + L.idx_off);
  int32_t* row_count = reinterpret_cast<int32_t*>(ws + kRowCountOff);
  void* Hc = ws + L.hc_off;
  void* dz = ws + L.dz_off;

  // Rows whose g_t is zero have zero dZ rows: their dH rows are zero and they add
  // nothing to dW, so the contractions run over the list of the other rows only.
  CUDA_TRY(cudaMemsetAsync(dH, 0, 2 * static_cast<size_t>(T) * Hd, s));
  {
    KernelScope ks(FLCE_KERNEL_BWD_PREP, s, 0.0, 20.0 * T);
    bwd_prep_kernel<<<1, kReduceThreads, 0, s>>>(dloss, dlogp, targets, static_cast<int>(T),
                                                 static_cast<int>(V_total), ignore_index, reduction, g, row_index,
                                                 row_count, status);
    ks.done();
    if ((st = check_launch("bwd_prep")) != FLCE_OK) return st;
  }
  const int64_t n_hd_blocks = cdiv(Hd, BN);
  CUtensorMap tm_Hc_k, tm_W_k, tm_W_mn, tm_Hc_mn, tm_dW_out, tm_dz_store, tm_dz_k, tm_dz_mn;
  if ((st = make_map(&tm_Hc_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Hc, Hd, chunk, Hd * 2, BK, BM)) != FLCE_OK) return st;
  if ((st = make_map(&tm_W_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, Hd, V, Hd * 2, BK, BN_HALF)) != FLCE_OK) return st;
  if ((st = make_map(&tm_W_mn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, Hd, V, Hd * 2, 64, 64)) != FLCE_OK) return st;
  if ((st = make_map(&tm_Hc_mn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Hc, Hd, chunk, Hd * 2, 64, 64)) != FLCE_OK) return st;
  if ((st = make_map(&tm_dW_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dW, Hd, V, Hd * 4, 32, 32)) != FLCE_OK) return st;
  // dZ block: V_pad / 64 panels of [chunk x 64] (the kernels' DzPanels layout)
  const uint64_t dz_panels = static_cast<uint64_t>(L.v_pad / 64);
  if ((st = make_panel_map(&tm_dz_store, dz, chunk, dz_panels, 32)) != FLCE_OK) return st;
  if ((st = make_panel_map(&tm_dz_k, dz, chunk, dz_panels, BM)) != FLCE_OK) return st;
  if ((st = make_panel_map(&tm_dz_mn, dz, chunk, dz_panels, 64)) != FLCE_OK) return st;

  const int64_t n_chunks = cdiv(T, chunk);
  int32_t* counters = reinterpret_cast<int32_t*>(ws + L.cnt_off);
  CUDA_TRY(cudaMemsetAsync(counters, 0, sizeof(int32_t) * static_cast<size_t>(n_chunks), s));
  const int row_vecs = static_cast<int>(Hd / 8);  // 16-byte pieces of a bf16 row
  const int copy_grid =
      static_cast<int>(std::min<int64_t>(cdiv(chunk * row_vecs, kCopyThreads), 8 * static_cast<int64_t>(dev->sms)));
  const int64_t cap_pairs = cdiv(chunk, 2 * BM);

  for (int64_t c = 0; c < n_chunks; ++c) {
    const int64_t c0 = c * chunk;  // list position of the chunk's first row
    {
      KernelScope ks(FLCE_KERNEL_BWD_GATHER, s, 0.0, 0.0, row_count, c0, chunk, 0.0, 4.0 * Hd + 4.0);
      gather_rows_kernel<<<copy_grid, kCopyThreads, 0, s>>>(static_cast<const uint4*>(H), row_index, row_count,
                                                            static_cast<int>(c0), static_cast<int>(chunk), row_vecs,
                                                            static_cast<uint4*>(Hc));
      ks.done();
      if ((st = check_launch("bwd_gather")) != FLCE_OK) return st;
    }

    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.row0 = 0;
    p.rows = static_cast<int32_t>(chunk);  // capacity; the kernels take the chunk's share of the list
    p.rows_dev = row_count;
    p.row_index = row_index;
    p.index0 = static_cast<int32_t>(c0);
    p.T = static_cast<int32_t>(T);
    p.V = static_cast<int32_t>(V);
    p.vocab_offset = vocab_offset;
    p.ignore_index = ignore_index;
    p.targets = targets;
    p.lse = lse;
    p.g = g;
    p.status = status;
    p.timeout_ns = wait_limit_ns(Hd);
    p.n_split = 1;

    // (1) recomputed logit tiles -> dZ chunk
    p.tmA = tm_Hc_k;
    p.tmB = tm_W_k;
    p.tmOut = tm_dz_store;
    p.num_m_pairs = static_cast<int32_t>(cap_pairs);
    p.num_n_blocks = static_cast<int32_t>(cdiv(V, BN));
    p.num_k_blocks = static_cast<int32_t>(Hd / BK);
    p.num_units = p.num_m_pairs * p.num_n_blocks;
    {
      const int grid = 2 * static_cast<int>(std::min<int64_t>(dev->pairs[MODE_DZ], p.num_units));
      KernelScope ks(FLCE_KERNEL_BWD_DZ, s, 0.0, 2.0 * V * Hd, row_count, c0, chunk, 2.0 * Hd * V,
                     2.0 * Hd + 2.0 * V + 16.0);
      gemm_kernel<MODE_DZ><<<grid, kThreads, smem_bytes_for(MODE_DZ), s>>>(p);
      ks.done();
      if ((st = check_launch("bwd_dz")) != FLCE_OK) return st;
    }
    // (2) dH rows of the chunk = dZ W and dW (+)= dZ^T H[chunk] in one launch;
    //     the first chunk stores dW, later chunks add to it, in chunk order.
    p.tmA = tm_dz_k;
    p.tmB = tm_W_mn;
    p.tmA2 = tm_dz_mn;
    p.tmB2 = tm_Hc_mn;
    p.tmOut2 = tm_dW_out;
    p.num_n_blocks = static_cast<int32_t>(n_hd_blocks);
    p.num_k_blocks = static_cast<int32_t>(cdiv(V, BK));
    p.num_k_blocks2 = static_cast<int32_t>(cdiv(chunk, BK));
    // dH tiles 256 x 512 when the hidden size splits into 512-column blocks: one
    // A block (dZ rows) feeds two N = 256 MMAs, so each SM moves 25 % fewer
    // operand bytes per FLOP than with 256 x 256 tiles.
    p.dh_wide = (Hd % (2 * BN) == 0) ? 1 : 0;
    p.n_dh_tiles = static_cast<int32_t>(cap_pairs * (p.dh_wide ? n_hd_blocks / 2 : n_hd_blocks));
    p.n_dw_tiles = static_cast<int32_t>(cdiv(V, 2 * BM) * n_hd_blocks);
    p.reduce_out = c > 0 ? 1 : 0;
    p.tile_counter = counters + c;
    p.dH_out = static_cast<uint16_t*>(dH);
    p.dH_ld = Hd;
    p.Hd = static_cast<int32_t>(Hd);
    p.dW_zero = dW;
    p.dW_elems = V * Hd;
    // dH tiles: K = V (twice the work per unit of K when wide); dW tiles: K = the chunk
    p.timeout_ns = wait_limit_ns(std::max<int64_t>(p.dh_wide ? 2 * V : V, chunk));
    {
      const int grid = 2 * static_cast<int>(std::min<int64_t>(dev->pairs[MODE_DHW], p.n_dh_tiles + p.n_dw_tiles));
      KernelScope ks(FLCE_KERNEL_BWD_DH_DW, s, 0.0, 2.0 * V * Hd + (c > 0 ? 8.0 : 4.0) * V * Hd, row_count, c0,
                     chunk, 4.0 * Hd * V, 4.0 * V + 4.0 * Hd);
      gemm_kernel<MODE_DHW><<<grid, kThreads, smem_bytes_for(MODE_DHW), s>>>(p);
      ks.done();
      if ((st = check_launch("bwd_dh_dw")) != FLCE_OK) return st;
    }
  }
  return FLCE_OK;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

int32_t flce_abi_version(void) { return FLCE_ABI_VERSION; }

const char* flce_last_error(void) { return g_last_error; }

const char* flce_status_string(int32_t st) {
  switch (st) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED";
    case FLCE_ERR_ALIGNMENT: return "FLCE_ERR_ALIGNMENT";
    case FLCE_ERR_WORKSPACE: return "FLCE_ERR_WORKSPACE";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA";
    case FLCE_ERR_TARGET_RANGE: return "FLCE_ERR_TARGET_RANGE";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT";
    default: return "FLCE_ERR_UNKNOWN";
  }
}

void flce_set_wait_timeout_ns(uint64_t ns) {
  g_timeout_ns.store(std::max<uint64_t>(ns, 1000000ull));
  g_timeout_fixed.store(true);
}

const char* flce_kernel_name(int32_t kind) {
  switch (kind) {
    case FLCE_KERNEL_FWD_LOGITS_LSE: return "fwd_logits_lse";
    case FLCE_KERNEL_FWD_FINALIZE: return "fwd_finalize";
    case FLCE_KERNEL_FWD_REDUCE: return "fwd_reduce";
    case FLCE_KERNEL_BWD_PREP: return "bwd_prep";
    case FLCE_KERNEL_BWD_DZ: return "bwd_dz";
    case FLCE_KERNEL_BWD_DH_DW: return "bwd_dh_dw";
    case FLCE_KERNEL_BWD_GATHER: return "bwd_gather";
    case FLCE_KERNEL_BWD_SCATTER: return "bwd_scatter";
    case FLCE_KERNEL_FWD_LIST: return "fwd_list";
    default: return "unknown";
  }
}

void flce_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
}

flce_status flce_profile_collect(flce_kernel_stats* out, int32_t max_entries, int32_t* n_out) {
  std::vector<LaunchRecord> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_records);
  }
  flce_kernel_stats agg[FLCE_KERNEL_KINDS];
  for (int k = 0; k < FLCE_KERNEL_KINDS; ++k) agg[k] = flce_kernel_stats{k, 0, 0.0, 0.0, 0.0};
  flce_status st = FLCE_OK;
  for (auto& r : recs) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      st = fail(FLCE_ERR_CUDA, "event query failed");
    double flops = r.flops, bytes = r.bytes;
    if (r.rows_dev) {
      int32_t n = 0;
      if (cudaMemcpy(&n, r.rows_dev, sizeof(n), cudaMemcpyDeviceToHost) != cudaSuccess)
        st = fail(FLCE_ERR_CUDA, "reading a row count failed");
      const double rows = static_cast<double>(std::min<int64_t>(std::max<int64_t>(n - r.index0, 0), r.cap));
      flops += rows * r.flops_per_row;
      bytes += rows * r.bytes_per_row;
    }
    agg[r.kind].launches += 1;
    agg[r.kind].total_ms += ms;
    agg[r.kind].flops += flops;
    agg[r.kind].bytes += bytes;
  }
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& r : recs) {
      g_event_pool.push_back(r.start);
      g_event_pool.push_back(r.stop);
    }
  }
  int n = 0;
  for (int k = 0; k < FLCE_KERNEL_KINDS; ++k)
    if (agg[k].launches > 0 && n < max_entries && out) out[n++] = agg[k];
  if (n_out) *n_out = n;
  return st;
}

size_t flce_forward_workspace_size(int64_t T, int64_t Hd, int64_t V) {
  (void)Hd;
  if (T < 0 || V < 1) return 0;
  return fwd_layout(T, kMaxSplit).total;
}

size_t flce_backward_workspace_size(int64_t T, int64_t Hd, int64_t V) {
  if (T < 0 || V < 1 || Hd < 1) return 0;
  return bwd_layout(T, Hd, V, default_chunk(T)).total;
}

size_t flce_backward_workspace_size_for_chunk(int64_t T, int64_t Hd, int64_t V, int64_t chunk) {
  if (T < 0 || V < 1 || Hd < 1 || chunk < 128 || chunk % 128 != 0) return 0;
  const int64_t cap = static_cast<int64_t>(align_up(static_cast<size_t>(std::max<int64_t>(T, 1)), 128));
  return bwd_layout(T, Hd, V, std::min(chunk, cap)).total;
}

int64_t flce_backward_chunk_tokens(int64_t T, int64_t Hd, int64_t V, size_t workspace_bytes) {
  if (T < 0 || V < 1 || Hd < 1) return 0;
  const int64_t cap = static_cast<int64_t>(align_up(static_cast<size_t>(std::max<int64_t>(T, 1)), 128));
  const BwdLayout L0 = bwd_layout(T, Hd, V, 0);
  if (workspace_bytes < L0.total) return 0;
  // per chunk row: its dZ row and its H row; the regions' alignment padding (a
  // few KB) can cost one step of 128 rows
  const size_t per_row = 2ull * static_cast<size_t>(L0.v_pad) + 2ull * static_cast<size_t>(Hd);
  int64_t c = static_cast<int64_t>((workspace_bytes - L0.hc_off) / per_row);
  c = std::min(c / 128 * 128, cap);
  while (c >= 128 && bwd_layout(T, Hd, V, c).total > workspace_bytes) c -= 128;
  return c < 128 ? 0 : c;
}

flce_status flce_selftest_wait_timeout(void* workspace, uint64_t timeout_ns, void* stream) {
  if (!workspace) return fail(FLCE_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(FLCE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (timeout_ns < 1000000ull || timeout_ns > 10000000000ull)
    return fail(FLCE_ERR_INVALID_ARG, "timeout_ns must lie in [1e6, 1e10]");
  DeviceInfo* dev = nullptr;
  flce_status st = device_info(&dev);
  if (st != FLCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemsetAsync(workspace, 0, kHeaderBytes, s));
  wait_selftest_kernel<<<1, 1, 0, s>>>(static_cast<int32_t*>(workspace), timeout_ns);
  return check_launch("wait_selftest");
}

flce_status flce_read_device_status(const void* workspace, void* stream, int32_t* out) {
  if (!workspace || !out) return fail(FLCE_ERR_INVALID_ARG, "workspace or out is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  CUDA_TRY(cudaMemcpyAsync(&v, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  *out = v;
  return FLCE_OK;
}

flce_status flce_forward(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd, int64_t V,
                         int64_t ignore_index, int32_t reduction, float* loss, float* lse, float* logp,
                         int64_t* n_valid, void* workspace, size_t workspace_bytes, void* stream) {
  flce_status st = check_common(H, W, targets, T, Hd, V, ignore_index, reduction);
  if (st != FLCE_OK) return st;
  if (!loss || (T > 0 && (!lse || !logp))) return fail(FLCE_ERR_INVALID_ARG, "loss, lse or logp is NULL");
  if (misaligned(loss) || misaligned(lse) || misaligned(logp) || misaligned(n_valid))
    return fail(FLCE_ERR_ALIGNMENT, "loss, lse, logp (4 bytes) or n_valid (8 bytes) misaligned");
  if (!workspace) return fail(FLCE_ERR_WORKSPACE, "workspace is NULL");
  if (workspace_bytes < flce_forward_workspace_size(T, Hd, V))
    return fail(FLCE_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes,
                flce_forward_workspace_size(T, Hd, V));
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(FLCE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FLCE_OK) return st;
  if ((st = get_encoder()) != FLCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  CUDA_TRY(cudaMemsetAsync(ws, 0, kHeaderBytes, s));

  if (T == 0) {
    if (reduction != FLCE_REDUCTION_NONE) CUDA_TRY(cudaMemsetAsync(loss, 0, sizeof(float), s));
    if (n_valid) CUDA_TRY(cudaMemsetAsync(n_valid, 0, sizeof(int64_t), s));
    return FLCE_OK;
  }
  FwdLayout L;
  if ((st = launch_logits_lse(dev, s, H, W, targets, T, Hd, V, 0, ignore_index, ws, &L)) != FLCE_OK) return st;
  return launch_finalize_reduce(s, ws, L, targets, T, V, ignore_index, reduction, loss, lse, logp, n_valid);
}

size_t flce_forward_valid_workspace_size(int64_t T, int64_t Hd, int64_t V) {
  if (T < 0 || V < 1 || Hd < 1) return 0;
  return fwd_valid_layout(T, Hd).total;
}

flce_status flce_forward_valid(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd,
                               int64_t V, int64_t ignore_index, int32_t reduction, float* loss, float* lse,
                               float* logp, int64_t* n_valid, void* workspace, size_t workspace_bytes,
                               void* stream) {
  flce_status st = check_common(H, W, targets, T, Hd, V, ignore_index, reduction);
  if (st != FLCE_OK) return st;
  if (!loss || (T > 0 && (!lse || !logp))) return fail(FLCE_ERR_INVALID_ARG, "loss, lse or logp is NULL");
  if (misaligned(loss) || misaligned(lse) || misaligned(logp) || misaligned(n_valid))
    return fail(FLCE_ERR_ALIGNMENT, "loss, lse, logp (4 bytes) or n_valid (8 bytes) misaligned");
  if (!workspace) return fail(FLCE_ERR_WORKSPACE, "workspace is NULL");
  if (workspace_bytes < flce_forward_valid_workspace_size(T, Hd, V))
    return fail(FLCE_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes,
                flce_forward_valid_workspace_size(T, Hd, V));
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(FLCE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FLCE_OK) return st;
  if ((st = get_encoder()) != FLCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  CUDA_TRY(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
  if (T == 0) {
    if (reduction != FLCE_REDUCTION_NONE) CUDA_TRY(cudaMemsetAsync(loss, 0, sizeof(float), s));
    if (n_valid) CUDA_TRY(cudaMemsetAsync(n_valid, 0, sizeof(int64_t), s));
    return FLCE_OK;
  }
  const FwdValidLayout LV = fwd_valid_layout(T, Hd);
  int32_t* row_index = reinterpret_cast<int32_t*>(ws + LV.idx_off);
  int32_t* pos = reinterpret_cast<int32_t*>(ws + LV.pos_off);
  int32_t* row_count = reinterpret_cast<int32_t*>(ws + kRowCountOff);
  void* Hc = ws + LV.hc_off;
  {
    KernelScope ks(FLCE_KERNEL_FWD_LIST, s, 0.0, 16.0 * T);
    fwd_list_kernel<<<1, kReduceThreads, 0, s>>>(targets, static_cast<int>(T), static_cast<int>(V), ignore_index,
                                                 row_index, pos, row_count, reinterpret_cast<int32_t*>(ws));
    ks.done();
    if ((st = check_launch("fwd_list")) != FLCE_OK) return st;
  }
  {
    const int row_vecs = static_cast<int>(Hd / 8);
    const int grid =
        static_cast<int>(std::min<int64_t>(cdiv(T * row_vecs, kCopyThreads), 8 * static_cast<int64_t>(dev->sms)));
    KernelScope ks(FLCE_KERNEL_BWD_GATHER, s, 0.0, 0.0, row_count, 0, T, 0.0, 4.0 * Hd + 4.0);
    gather_rows_kernel<<<grid, kCopyThreads, 0, s>>>(static_cast<const uint4*>(H), row_index, row_count, 0,
                                                     static_cast<int>(T), row_vecs, static_cast<uint4*>(Hc));
    ks.done();
    if ((st = check_launch("fwd_gather")) != FLCE_OK) return st;
  }
  FwdLayout L;
  if ((st = launch_logits_lse(dev, s, Hc, W, targets, T, Hd, V, 0, ignore_index, ws, &L, nullptr, nullptr, row_count,
                              row_index)) != FLCE_OK)
    return st;
  return launch_finalize_reduce(s, ws, L, targets, T, V, ignore_index, reduction, loss, lse, logp, n_valid, pos);
}

size_t flce_score_workspace_size(int64_t T, int64_t Hd, int64_t V) {
  (void)Hd;
  if (T < 0 || V < 1) return 0;
  const FwdLayout L = fwd_layout(T, kMaxSplit);
  return L.total + 2 * align_up(sizeof(float) * kMaxSplit * static_cast<size_t>(L.part_stride), 256);
}

flce_status flce_score(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd, int64_t V,
                       int64_t ignore_index, float* logp, float* lse, int64_t* argmax, void* workspace,
                       size_t workspace_bytes, void* stream) {
  flce_status st = check_common(H, W, targets, T, Hd, V, ignore_index, FLCE_REDUCTION_NONE);
  if (st != FLCE_OK) return st;
  if (T > 0 && !logp) return fail(FLCE_ERR_INVALID_ARG, "logp is NULL");
  if (misaligned(logp) || misaligned(lse) || misaligned(argmax))
    return fail(FLCE_ERR_ALIGNMENT, "logp, lse (4 bytes) or argmax (8 bytes) misaligned");
  if (!workspace) return fail(FLCE_ERR_WORKSPACE, "workspace is NULL");
  if (workspace_bytes < flce_score_workspace_size(T, Hd, V))
    return fail(FLCE_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes,
                flce_score_workspace_size(T, Hd, V));
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(FLCE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FLCE_OK) return st;
  if ((st = get_encoder()) != FLCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  CUDA_TRY(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
  if (T == 0) return FLCE_OK;
  const FwdLayout Lmax = fwd_layout(T, kMaxSplit);
  const size_t best_bytes = align_up(sizeof(float) * kMaxSplit * static_cast<size_t>(Lmax.part_stride), 256);
  float* best_val = reinterpret_cast<float*>(ws + Lmax.total);
  int32_t* best_idx = reinterpret_cast<int32_t*>(ws + Lmax.total + best_bytes);
  FwdLayout L;
  if ((st = launch_logits_lse(dev, s, H, W, targets, T, Hd, V, 0, ignore_index, ws, &L, best_val, best_idx)) !=
      FLCE_OK)
    return st;
  KernelScope ks(FLCE_KERNEL_FWD_FINALIZE, s, 0.0, (16.0 * L.n_split + 4 + 8 + 4 + 4 + 8) * T);
  score_finalize_kernel<<<L.num_fin_blocks, kFinalizeThreads, 0, s>>>(
      reinterpret_cast<const float2*>(ws + L.partials_off), reinterpret_cast<const float*>(ws + L.zy_off), best_val,
      best_idx, targets, static_cast<int>(T), static_cast<int>(V), ignore_index, L.n_split,
      static_cast<int>(L.part_stride), lse, logp, argmax, reinterpret_cast<int32_t*>(ws), nullptr);
  ks.done();
  return check_launch("score_finalize");
}

// flce_score_valid: the scoring workspace, then the row list, the position map
// and the listed rows of H, as in the flce_forward_valid layout.
static FwdValidLayout score_valid_layout(int64_t T, int64_t Hd, int64_t V) {
  FwdValidLayout L{};
  const size_t t1 = static_cast<size_t>(std::max<int64_t>(T, 1));
  size_t off = align_up(flce_score_workspace_size(T, Hd, V), 256);
  L.idx_off = off;
  off = align_up(off + sizeof(int32_t) * t1, 256);
  L.pos_off = off;
  off = align_up(off + sizeof(int32_t) * t1, 1024);
  L.hc_off = off;
  off = align_up(off + 2ull * t1 * static_cast<size_t>(Hd), 256);
  L.total = off;
  return L;
}

size_t flce_score_valid_workspace_size(int64_t T, int64_t Hd, int64_t V) {
  if (T < 0 || V < 1 || Hd < 1) return 0;
  return score_valid_layout(T, Hd, V).total;
}

flce_status flce_score_valid(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd, int64_t V,
                             int64_t ignore_index, float* logp, float* lse, int64_t* argmax, void* workspace,
                             size_t workspace_bytes, void* stream) {
  flce_status st = check_common(H, W, targets, T, Hd, V, ignore_index, FLCE_REDUCTION_NONE);
  if (st != FLCE_OK) return st;
  if (T > 0 && !logp) return fail(FLCE_ERR_INVALID_ARG, "logp is NULL");
  if (misaligned(logp) || misaligned(lse) || misaligned(argmax))
    return fail(FLCE_ERR_ALIGNMENT, "logp, lse (4 bytes) or argmax (8 bytes) misaligned");
  if (!workspace) return fail(FLCE_ERR_WORKSPACE, "workspace is NULL");
  if (workspace_bytes < flce_score_valid_workspace_size(T, Hd, V))
    return fail(FLCE_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes,
                flce_score_valid_workspace_size(T, Hd, V));
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(FLCE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FLCE_OK) return st;
  if ((st = get_encoder()) != FLCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  CUDA_TRY(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
  if (T == 0) return FLCE_OK;
  const FwdValidLayout LV = score_valid_layout(T, Hd, V);
  int32_t* row_index = reinterpret_cast<int32_t*>(ws + LV.idx_off);
  int32_t* pos = reinterpret_cast<int32_t*>(ws + LV.pos_off);
  int32_t* row_count = reinterpret_cast<int32_t*>(ws + kRowCountOff);
  void* Hc = ws + LV.hc_off;
  {
    KernelScope ks(FLCE_KERNEL_FWD_LIST, s, 0.0, 16.0 * T);
    fwd_list_kernel<<<1, kReduceThreads, 0, s>>>(targets, static_cast<int>(T), static_cast<int>(V), ignore_index,
                                                 row_index, pos, row_count, reinterpret_cast<int32_t*>(ws));
    ks.done();
    if ((st = check_launch("fwd_list")) != FLCE_OK) return st;
  }
  {
    const int row_vecs = static_cast<int>(Hd / 8);
    const int grid =
        static_cast<int>(std::min<int64_t>(cdiv(T * row_vecs, kCopyThreads), 8 * static_cast<int64_t>(dev->sms)));
    KernelScope ks(FLCE_KERNEL_BWD_GATHER, s, 0.0, 0.0, row_count, 0, T, 0.0, 4.0 * Hd + 4.0);
    gather_rows_kernel<<<grid, kCopyThreads, 0, s>>>(static_cast<const uint4*>(H), row_index, row_count, 0,
                                                     static_cast<int>(T), row_vecs, static_cast<uint4*>(Hc));
    ks.done();
    if ((st = check_launch("fwd_gather")) != FLCE_OK) return st;
  }
  const FwdLayout Lmax = fwd_layout(T, kMaxSplit);
  const size_t best_bytes = align_up(sizeof(float) * kMaxSplit * static_cast<size_t>(Lmax.part_stride), 256);
  float* best_val = reinterpret_cast<float*>(ws + Lmax.total);
  int32_t* best_idx = reinterpret_cast<int32_t*>(ws + Lmax.total + best_bytes);
  FwdLayout L;
  if ((st = launch_logits_lse(dev, s, Hc, W, targets, T, Hd, V, 0, ignore_index, ws, &L, best_val, best_idx,
                              row_count, row_index)) != FLCE_OK)
    return st;
  KernelScope ks(FLCE_KERNEL_FWD_FINALIZE, s, 0.0, (16.0 * L.n_split + 4 + 8 + 4 + 4 + 8) * T);
  score_finalize_kernel<<<L.num_fin_blocks, kFinalizeThreads, 0, s>>>(
      reinterpret_cast<const float2*>(ws + L.partials_off), reinterpret_cast<const float*>(ws + L.zy_off), best_val,
      best_idx, targets, static_cast<int>(T), static_cast<int>(V), ignore_index, L.n_split,
      static_cast<int>(L.part_stride), lse, logp, argmax, reinterpret_cast<int32_t*>(ws), pos);
  ks.done();
  return check_launch("score_finalize");
}

size_t flce_combine_workspace_size(int64_t T, int32_t n_shards) {
  if (T < 0 || n_shards < 1 || n_shards > kMaxShards) return 0;
  return fwd_layout(T, n_shards).total;
}

flce_status flce_forward_shard(const void* H, const void* W_shard, const int64_t* targets, int64_t T, int64_t Hd,
                               int64_t V_shard, int64_t vocab_offset, int64_t V_total, int64_t ignore_index,
                               float* shard_lse, float* shard_zy, void* workspace, size_t workspace_bytes,
                               void* stream) {
  flce_status st = check_shard(V_shard, vocab_offset, V_total, ignore_index);
  if (st != FLCE_OK) return st;
  if ((st = check_common(H, W_shard, targets, T, Hd, V_shard, -1, FLCE_REDUCTION_SUM)) != FLCE_OK) return st;
  if (T > 0 && (!shard_lse || !shard_zy)) return fail(FLCE_ERR_INVALID_ARG, "shard_lse or shard_zy is NULL");
  if (misaligned(shard_lse) || misaligned(shard_zy))
    return fail(FLCE_ERR_ALIGNMENT, "shard_lse and shard_zy must be 4-byte aligned");
  if (!workspace) return fail(FLCE_ERR_WORKSPACE, "workspace is NULL");
  if (workspace_bytes < flce_forward_workspace_size(T, Hd, V_shard))
    return fail(FLCE_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes,
                flce_forward_workspace_size(T, Hd, V_shard));
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(FLCE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FLCE_OK) return st;
  if ((st = get_encoder()) != FLCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  CUDA_TRY(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
  if (T == 0) return FLCE_OK;
  FwdLayout L;
  if ((st = launch_logits_lse(dev, s, H, W_shard, targets, T, Hd, V_shard, vocab_offset, ignore_index, ws, &L)) !=
      FLCE_OK)
    return st;
  KernelScope ks(FLCE_KERNEL_FWD_FINALIZE, s, 0.0, (8.0 * L.n_split + 4 + 8 + 8) * T);
  fwd_shard_finalize_kernel<<<L.num_fin_blocks, kFinalizeThreads, 0, s>>>(
      reinterpret_cast<const float2*>(ws + L.partials_off), reinterpret_cast<const float*>(ws + L.zy_off), targets,
      static_cast<int>(T), vocab_offset, static_cast<int>(V_shard), L.n_split, static_cast<int>(L.part_stride),
      shard_lse, shard_zy);
  ks.done();
  return check_launch("fwd_shard_finalize");
}

flce_status flce_combine_shards(const float* shard_lse, const float* shard_zy, int32_t n_shards,
                                const int64_t* targets, int64_t T, int64_t V_total, int64_t ignore_index,
                                int32_t reduction, float* loss, float* lse, float* logp, int64_t* n_valid,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (n_shards < 1 || n_shards > kMaxShards)
    return fail(FLCE_ERR_INVALID_ARG, "n_shards = %d outside [1, %d]", n_shards, kMaxShards);
  if (T < 0 || T >= kMaxRows) return fail(FLCE_ERR_INVALID_ARG, "T = %lld out of range", (long long)T);
  if (V_total < 1 || V_total >= kMaxRows)
    return fail(FLCE_ERR_INVALID_ARG, "V_total = %lld out of range", (long long)V_total);
  if (reduction < 0 || reduction > 2) return fail(FLCE_ERR_INVALID_ARG, "unknown reduction %d", reduction);
  if (ignore_index >= 0 && ignore_index < V_total)
    return fail(FLCE_ERR_INVALID_ARG, "ignore_index %lld lies inside [0, V_total)", (long long)ignore_index);
  if (!loss || (T > 0 && (!shard_lse || !shard_zy || !targets || !lse || !logp)))
    return fail(FLCE_ERR_INVALID_ARG, "a required pointer is NULL");
  if (misaligned(shard_lse) || misaligned(shard_zy) || misaligned(loss) || misaligned(lse) || misaligned(logp) ||
      misaligned(n_valid) || misaligned(targets))
    return fail(FLCE_ERR_ALIGNMENT, "a float array is not 4-byte or an int64 array not 8-byte aligned");
  if (!workspace) return fail(FLCE_ERR_WORKSPACE, "workspace is NULL");
  if (workspace_bytes < flce_combine_workspace_size(T, n_shards))
    return fail(FLCE_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes,
                flce_combine_workspace_size(T, n_shards));
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(FLCE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  CUDA_TRY(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
  if (T == 0) {
    if (reduction != FLCE_REDUCTION_NONE) CUDA_TRY(cudaMemsetAsync(loss, 0, sizeof(float), s));
    if (n_valid) CUDA_TRY(cudaMemsetAsync(n_valid, 0, sizeof(int64_t), s));
    return FLCE_OK;
  }
  const FwdLayout L = fwd_layout(T, n_shards);
  {
    KernelScope ks(FLCE_KERNEL_FWD_FINALIZE, s, 0.0, (8.0 * n_shards + 12.0 * n_shards + 4) * T);
    combine_shards_kernel<<<L.num_fin_blocks, kFinalizeThreads, 0, s>>>(
        shard_lse, shard_zy, n_shards, static_cast<int>(T), reinterpret_cast<float2*>(ws + L.partials_off),
        static_cast<int>(L.part_stride), reinterpret_cast<float*>(ws + L.zy_off));
    ks.done();
    flce_status st = check_launch("combine_shards");
    if (st != FLCE_OK) return st;
  }
  return launch_finalize_reduce(s, ws, L, targets, T, V_total, ignore_index, reduction, loss, lse, logp, n_valid);
}

flce_status flce_forward_noalloc(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd,
                                 int64_t V, int64_t ignore_index, int32_t reduction, float* loss, float* lse,
                                 float* logp, int64_t* n_valid, int32_t* device_status, void* stream) {
  if (T < 0 || V < 1) return fail(FLCE_ERR_INVALID_ARG, "T = %lld or V = %lld out of range", (long long)T, (long long)V);
  flce_status st = check_common(H, W, targets, T, Hd, V, ignore_index, reduction);
  if (st != FLCE_OK) return st;
  const size_t need = flce_forward_workspace_size(T, Hd, V);
  if (need > kStaticScratchBytes)
    return fail(FLCE_ERR_WORKSPACE,
                "T = %lld needs %zu bytes of scratch; the built-in scratch holds %zu bytes (T <= 253952)",
                (long long)T, need, kStaticScratchBytes);
  if (misaligned(device_status)) return fail(FLCE_ERR_ALIGNMENT, "device_status must be 4-byte aligned");
  void* scratch = nullptr;
  st = static_scratch_address(&scratch);
  if (st != FLCE_OK) return st;
  st = flce_forward(H, W, targets, T, Hd, V, ignore_index, reduction, loss, lse, logp, n_valid, scratch,
                    kStaticScratchBytes, stream);
  if (st != FLCE_OK) return st;
  if (device_status)
    CUDA_TRY(cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                             static_cast<cudaStream_t>(stream)));
  return FLCE_OK;
}

flce_status flce_backward(const float* dloss, const void* H, const void* W, const int64_t* targets, const float* lse,
                          int64_t T, int64_t Hd, int64_t V, int64_t ignore_index, int32_t reduction, void* dH,
                          float* dW, void* workspace, size_t workspace_bytes, void* stream) {
  flce_status st = check_common(H, W, targets, T, Hd, V, ignore_index, reduction);
  if (st != FLCE_OK) return st;
  return backward_impl(dloss, nullptr, H, W, targets, lse, T, Hd, V, 0, V, ignore_index, reduction, dH, dW,
                       workspace, workspace_bytes, stream);
}

flce_status flce_backward_logp(const float* dloss, const float* dlogp, const void* H, const void* W,
                               const int64_t* targets, const float* lse, int64_t T, int64_t Hd, int64_t V,
                               int64_t ignore_index, int32_t reduction, void* dH, float* dW, void* workspace,
                               size_t workspace_bytes, void* stream) {
  flce_status st = check_common(H, W, targets, T, Hd, V, ignore_index, reduction);
  if (st != FLCE_OK) return st;
  return backward_impl(dloss, dlogp, H, W, targets, lse, T, Hd, V, 0, V, ignore_index, reduction, dH, dW,
                       workspace, workspace_bytes, stream);
}

flce_status flce_backward_shard(const float* dloss, const void* H, const void* W_shard, const int64_t* targets,
                                const float* lse, int64_t T, int64_t Hd, int64_t V_shard, int64_t vocab_offset,
                                int64_t V_total, int64_t ignore_index, int32_t reduction, void* dH_partial,
                                float* dW_shard, void* workspace, size_t workspace_bytes, void* stream) {
  flce_status st = check_shard(V_shard, vocab_offset, V_total, ignore_index);
  if (st != FLCE_OK) return st;
  if ((st = check_common(H, W_shard, targets, T, Hd, V_shard, -1, reduction)) != FLCE_OK) return st;
  return backward_impl(dloss, nullptr, H, W_shard, targets, lse, T, Hd, V_shard, vocab_offset, V_total,
                       ignore_index, reduction, dH_partial, dW_shard, workspace, workspace_bytes, stream);
}

}  // extern "C"

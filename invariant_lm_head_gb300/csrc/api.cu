// C ABI of liblmhead.so: argument checks, workspace layout, TMA descriptors
// and the launch sequence of each entry point. Declarations and contracts are
// in include/lmhead.h.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "lmhead.h"
#include "ptx.cuh"

// Device-side status word (bit lmh::LMH_DEVSTAT_TIMEOUT) and the self-test's result.
__device__ unsigned g_lmh_status_word;
__device__ int g_lmh_selftest_result;

namespace {

thread_local char t_err[512];

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  t_err[0] = '\0';
  return LMH_OK;
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int major = 0, minor = 0;
  unsigned* status = nullptr;
  int* selftest = nullptr;
  void* noalloc_scratch = nullptr;  // lmhead_logprob_fwd_noalloc's array on this device
};

std::mutex g_mu;
std::atomic<unsigned long long> g_launches{0};
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// ------------------------------------------------------------ backward side stream
// Per device: a second stream of the library's own (non-blocking, created by
// the device's first call of any entry point, so that no later call under
// stream capture creates it) and two events. The backward runs grad_hidden
// on it beside grad_weight: both read the chunk's dl and write different
// outputs. Fork and join are an event record plus a stream wait each way, so
// under stream capture the two become parallel branches of the graph. The
// mutex keeps one call's records and waits together when several host
// threads call at once.
struct SideStream {
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};
SideStream g_side[kMaxDevices];

int side_stream_init(SideStream& sd) {
  cudaError_t e = cudaSuccess;
  if (!sd.st && (e = cudaStreamCreateWithFlags(&sd.st, cudaStreamNonBlocking)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "cudaStreamCreate: %s", cudaGetErrorString(e));
  if (!sd.fork && (e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "cudaEventCreate: %s", cudaGetErrorString(e));
  if (!sd.join && (e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "cudaEventCreate: %s", cudaGetErrorString(e));
  return LMH_OK;
}

// Per-device facts, queried once with that device current.
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(LMH_ERR_LAUNCH, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(LMH_ERR_UNSUPPORTED_DEVICE, "device %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return fail(LMH_ERR_LAUNCH, "device query: %s", cudaGetErrorString(e));
    if (d.major != 10 || d.minor != 3)
      return fail(LMH_ERR_UNSUPPORTED_DEVICE,
                  "device %d is sm_%d%d; this library is built for sm_103 (GB300) only", dev,
                  d.major, d.minor);
    if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_lmh_status_word)) !=
            cudaSuccess ||
        (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.selftest),
                                  g_lmh_selftest_result)) != cudaSuccess)
      return fail(LMH_ERR_LAUNCH, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    const int rc = lmh::noalloc_scratch_lookup(&d.noalloc_scratch);
    if (rc != LMH_OK) return rc;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(LMH_ERR_LAUNCH, "cuTensorMapEncodeTiled unavailable");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const int rc_side = side_stream_init(g_side[dev]);
    if (rc_side != LMH_OK) return rc_side;
    d.ready = true;
  }
  *out = &d;
  return LMH_OK;
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// rows `row_bytes` apart; box `box_inner` x `box_outer` with 128-byte swizzle.
// Out-of-range elements of a box read as zero.
int make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(LMH_ERR_LAUNCH, "cuTensorMapEncodeTiled failed (%d) for %llu x %llu", (int)r,
                (unsigned long long)inner, (unsigned long long)outer);
  return LMH_OK;
}

// Output map of a store epilogue: `cols` x `rows` elements, rows `row_bytes`
// apart. fp32: 32 x 128 box, 128-byte swizzle; bf16: 32 x 128 box, 64-byte
// swizzle (the staging layouts the epilogue writes). Stores outside the
// tensor are clipped by TMA.
int make_out_tmap(CUtensorMap* map, void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                  bool f32, bool transposed = false) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  // fp32: the 128 x 32 chunk of an epilogue group; bf16: one epilogue warp's
  // 32 x 32 box
  cuuint32_t box[2] = {32, f32 ? 128u : 32u};
  if (transposed) {  // StoreF32T: 128 columns x 32 rows of fp32, no swizzle
    box[0] = 128;
    box[1] = 32;
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(LMH_ERR_LAUNCH, "cuTensorMapEncodeTiled (transposed output) failed (%d)", (int)r);
    return LMH_OK;
  }
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(LMH_ERR_LAUNCH, "cuTensorMapEncodeTiled (output) failed (%d) for %llu x %llu",
                (int)r, (unsigned long long)cols, (unsigned long long)rows);
  return LMH_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

constexpr size_t kRegionAlign = 256;

// Carves consecutive 256-byte-aligned regions out of a workspace.
struct Carver {
  char* base;
  size_t off = 0;
  template <class T>
  T* take(int64_t count) {
    off = (off + kRegionAlign - 1) / kRegionAlign * kRegionAlign;
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += static_cast<size_t>(count) * sizeof(T);
    return p;
  }
};

int n_fwd_chunks(int64_t V) {
  const int64_t tiles = (V + lmh::kBN - 1) / lmh::kBN;
  return static_cast<int>((tiles + lmh::kFwdTilesPerChunk - 1) / lmh::kFwdTilesPerChunk);
}

struct FwdWs {
  float *pm, *ps, *pu, *pq, *pzl;
  unsigned* sched;  // the GEMMs' unit counter (dynamic schedule)
};

FwdWs carve_fwd(Carver& c, int64_t T, int64_t V) {
  const int64_t n = static_cast<int64_t>(n_fwd_chunks(V)) * T;
  FwdWs w;
  w.pm = c.take<float>(n);
  w.ps = c.take<float>(n);
  w.pu = c.take<float>(n);
  w.pq = c.take<float>(n);
  w.pzl = c.take<float>(T);
  w.sched = c.take<unsigned>(1);
  return w;
}

struct BwdWs {
  FwdWs fwd;
  float* lse;  // recomputed statistics when the caller passes none
  float* lp;
  float* ent;
  uint16_t* dl;  // [Tc][Vpad] bf16 dlogits of one row chunk
  uint16_t* ht;  // [H][Tcpad] bf16 transpose of one row chunk of hidden
  float* ghp;    // [2][ghp_rows][H] fp32 partials of grad_hidden, one per K segment
  unsigned* sched2;  // grad_hidden's unit counter when it runs beside grad_weight
  int64_t vpad, tc, tcpad, ghp_rows;
};

BwdWs carve_bwd(Carver& c, int64_t T, int64_t H, int64_t V,
                int64_t row_chunk = lmh::kBwdRowChunk) {
  BwdWs w;
  w.vpad = round_up(V, 8);
  w.tc = T < row_chunk ? T : row_chunk;
  w.fwd = carve_fwd(c, T, V);
  w.lse = c.take<float>(T);
  w.lp = c.take<float>(T);
  w.ent = c.take<float>(T);
  w.dl = c.take<uint16_t>(w.tc * w.vpad);
  w.tcpad = round_up(w.tc, 8);
  w.ht = c.take<uint16_t>(H * w.tcpad);
  w.ghp_rows = round_up(w.tc, lmh::kBM);
  w.ghp = c.take<float>(2 * w.ghp_rows * H);
  w.sched2 = c.take<unsigned>(1);
  return w;
}

int check_dims(int64_t T, int64_t H, int64_t V, bool need_h) {
  if (T < 0 || T > LMH_MAX_DIM) return fail(LMH_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  if (V < 1 || V > LMH_MAX_DIM) return fail(LMH_ERR_INVALID_ARG, "V=%lld out of range", (long long)V);
  if (need_h) {
    if (H < 8 || H > LMH_MAX_DIM) return fail(LMH_ERR_INVALID_ARG, "H=%lld out of range", (long long)H);
    if (H % 8 != 0)
      return fail(LMH_ERR_ALIGNMENT, "H=%lld must be a multiple of 8 (16-byte rows)", (long long)H);
  }
  return LMH_OK;
}

int check_temperature(float s) {
  if (!std::isfinite(s) || !(s > 0.f))
    return fail(LMH_ERR_INVALID_ARG, "inv_temperature must be finite and > 0");
  return LMH_OK;
}

int check_ptr(const void* p, uintptr_t align, const char* name, bool nullable = false) {
  if (!p) return nullable ? LMH_OK : fail(LMH_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, align))
    return fail(LMH_ERR_ALIGNMENT, "%s must be %u-byte aligned", name, (unsigned)align);
  return LMH_OK;
}

int launch_status(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(LMH_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
  return LMH_OK;
}

#define LMH_TRY(x)          \
  do {                      \
    int _rc = (x);          \
    if (_rc != LMH_OK) return _rc; \
  } while (0)

// ---------------------------------------------------------------- kernel timing
// Opt-in diagnostics: with timing enabled, every launch is bracketed by two
// CUDA events recorded on the launching stream; lmhead_timing_read() returns
// the kind and duration of each launch. Off by default (no events recorded).
const char* const kKindNames[lmh::K_COUNT] = {
    "fused_fwd_gemm", "fwd_merge",   "dlogits_gemm",  "grad_hidden_gemm",  "grad_weight_gemm",
    "logits_rowwise", "engine_gemm", "selftest_wait", "logits_rowwise_div",
    "hidden_transpose", "sum_parts_bf16", "grad_hidden_sum"};

struct TimingRec {
  int kind;
  cudaEvent_t b, e;
};
std::mutex g_tmu;
std::atomic<bool> g_timing{false};
std::vector<TimingRec> g_recs;
std::vector<cudaEvent_t> g_event_pool;

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

#define LMH_LAUNCH(kind, st, expr, what)                  \
  do {                                                    \
    lmh::KernelTimer _kt((kind), (st));                   \
    int _rc = launch_status((expr), (what));              \
    if (_rc != LMH_OK) return _rc;                        \
  } while (0)

// A run of vocab units [begin, end) of the forward GEMM; `ready` (or NULL) is
// an event the launch waits for first.
struct FwdSlice {
  int begin, end;
  cudaEvent_t ready;
};

// Forward statistics into `w`, merged into the outputs. out_sum_p2 may be NULL.
// With `slices`, the forward GEMM runs as one launch per slice, each after its
// event; every tile is computed exactly as in the single launch.
int run_forward(const DeviceInfo& dev, const uint16_t* hidden, const uint16_t* weight,
                const int32_t* labels, int64_t T, int64_t H, int64_t V, float s, float* out_lp,
                float* out_ent, float* out_lse, const FwdWs& w, cudaStream_t st,
                float* out_sum_p2 = nullptr, const std::vector<FwdSlice>* slices = nullptr) {
  CUtensorMap ta, tb;
  const int a_rows = lmh::short_a_rows(T);
  LMH_TRY(make_tmap(&ta, hidden, H, T, H * 2, lmh::kBK, a_rows ? a_rows : lmh::kBM));
  LMH_TRY(make_tmap(&tb, weight, H, V, H * 2, lmh::kBK, lmh::kBBoxRows));
  lmh::GemmParams p{};
  p.a_rows = a_rows;
  p.M = static_cast<int>(T);
  p.N = static_cast<int>(V);
  p.K = static_cast<int>(H);
  p.status = dev.status;
  p.scale2 = s * lmh::kLog2e;
  p.inv_temp = s;
  p.labels = labels;
  p.part_m = w.pm;
  p.part_s = w.ps;
  p.part_u = w.pu;
  p.part_q = out_sum_p2 ? w.pq : nullptr;
  p.part_zl = w.pzl;
  p.part_ld = T;
  p.sched = w.sched;
  if (!slices) {
    LMH_LAUNCH(lmh::K_FWD_GEMM, st,
               lmh::launch_gemm(lmh::Epi::FwdStats, ta, tb, p, lmh::kFwdTilesPerChunk, dev.sms, st),
               "fused forward");
  } else {
    for (const FwdSlice& sl : *slices) {
      if (sl.ready) {
        const cudaError_t e = cudaStreamWaitEvent(st, sl.ready, 0);
        if (e != cudaSuccess)
          return fail(LMH_ERR_LAUNCH, "cudaStreamWaitEvent: %s", cudaGetErrorString(e));
      }
      p.vunit_begin = sl.begin;
      p.vunit_end = sl.end;
      LMH_LAUNCH(lmh::K_FWD_GEMM, st,
                 lmh::launch_gemm(lmh::Epi::FwdStats, ta, tb, p, lmh::kFwdTilesPerChunk, dev.sms,
                                  st),
                 "fused forward (vocab slice)");
    }
  }
  LMH_LAUNCH(lmh::K_FWD_MERGE, st,
             lmh::launch_fwd_merge(w.pm, w.ps, w.pu, out_sum_p2 ? w.pq : nullptr, w.pzl, labels, T,
                                   n_fwd_chunks(V), V, out_lp, out_ent, out_lse, out_sum_p2, st),
             "forward merge");
  return LMH_OK;
}

int fwd_entry(const uint16_t* hidden, const uint16_t* weight, const int32_t* labels, int64_t T,
              int64_t H, int64_t V, float inv_temperature, float* out_logprob, float* out_entropy,
              float* out_lse, float* out_sum_p2, void* workspace, size_t workspace_bytes,
              struct CUstream_st* stream) {
  LMH_TRY(check_dims(T, H, V, true));
  LMH_TRY(check_temperature(inv_temperature));
  if (T == 0) return ok();  // nothing to read or write; pointers may be NULL
  LMH_TRY(check_ptr(hidden, 16, "hidden"));
  LMH_TRY(check_ptr(weight, 16, "weight"));
  LMH_TRY(check_ptr(labels, 4, "labels"));
  LMH_TRY(check_ptr(out_logprob, 4, "out_logprob"));
  LMH_TRY(check_ptr(out_entropy, 4, "out_entropy", true));
  LMH_TRY(check_ptr(out_lse, 4, "out_lse", true));
  LMH_TRY(check_ptr(out_sum_p2, 4, "out_sum_p2", true));
  const size_t need = lmhead_workspace_size(LMH_OP_FWD, T, H, V);
  if (!workspace || workspace_bytes < need)
    return fail(LMH_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);
  LMH_TRY(check_ptr(workspace, 16, "workspace"));
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  Carver c{static_cast<char*>(workspace)};
  const FwdWs w = carve_fwd(c, T, V);
  LMH_TRY(run_forward(*dev, hidden, weight, labels, T, H, V, inv_temperature, out_logprob,
                      out_entropy, out_lse, w, reinterpret_cast<cudaStream_t>(stream),
                      out_sum_p2));
  return ok();
}

// divide == false: temp_value is the inverse temperature s (z = x * s).
// divide == true: temp_value is the temperature t (z = x / t), or each row's
// t comes from row_temperature when that is not NULL.
int logits_entry(const uint16_t* logits, const int32_t* labels, int64_t T, int64_t V,
                 float temp_value, bool divide, const float* row_temperature, float* out_logprob,
                 float* out_entropy, float* out_lse, float* out_sum_p2,
                 struct CUstream_st* stream) {
  LMH_TRY(check_dims(T, 8, V, false));
  if (!row_temperature) {
    if (!std::isfinite(temp_value) || !(temp_value > 0.f))
      return fail(LMH_ERR_INVALID_ARG, "%s must be finite and > 0",
                  divide ? "temperature" : "inv_temperature");
  }
  if (T == 0) return ok();  // nothing to read or write; pointers may be NULL
  LMH_TRY(check_ptr(row_temperature, 4, "row_temperature", true));
  LMH_TRY(check_ptr(logits, (V % 8 == 0) ? 16 : 2, "logits"));
  LMH_TRY(check_ptr(labels, 4, "labels"));
  LMH_TRY(check_ptr(out_logprob, 4, "out_logprob"));
  LMH_TRY(check_ptr(out_entropy, 4, "out_entropy", true));
  LMH_TRY(check_ptr(out_lse, 4, "out_lse", true));
  LMH_TRY(check_ptr(out_sum_p2, 4, "out_sum_p2", true));
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LMH_LAUNCH(divide ? lmh::K_LOGITS_ROWWISE_DIV : lmh::K_LOGITS_ROWWISE, st,
             lmh::launch_logits_logprob(logits, labels, T, V, temp_value, divide,
                                        row_temperature, out_logprob, out_entropy, out_lse,
                                        out_sum_p2, dev->sms, dev->status, st),
             "logits log-prob");
  return ok();
}

// ------------------------------------------------------------ host-staged forward
// Per device: a copy stream of the library's own (non-blocking, created on
// first use) and a pool of events. Events are reused from call to call: a
// stream wait takes the record that is current when it is enqueued, so a later
// record cannot disturb an earlier wait. The mutex keeps one call's records and
// waits together when several host threads call at once.
struct Staging {
  cudaStream_t copy = nullptr;
  std::vector<cudaEvent_t> events;
  std::mutex mu;
};
Staging g_staging[kMaxDevices];

int staging_events(Staging& sg, size_t n) {
  while (sg.events.size() < n) {
    cudaEvent_t e = nullptr;
    const cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (r != cudaSuccess) return fail(LMH_ERR_LAUNCH, "cudaEventCreate: %s", cudaGetErrorString(r));
    sg.events.push_back(e);
  }
  return LMH_OK;
}

// Vocab slices of the host-staged forward, in 1024-column units. The first
// (1/32 of the vocabulary) is small, so the first GEMM launch starts soon
// after hidden has landed. Later slices grow by 3/2 up to a quarter of the
// vocabulary, and a tail shorter than the first slice joins the slice before
// it. At the 16384 x 3584 x 152064 step the GEMM uses a vocab unit (7.3 MB of
// W) in about 67 us and the copy link (about 211 GB/s) brings one in about
// 35 us, so slice i+1 (1.5x slice i) lands before the GEMM is done with slice
// i. (Against a schedule of n/16 doubling, the end-to-end step measured the
// same within run-to-run noise.)
std::vector<FwdSlice> staged_slices(int n_vunits) {
  std::vector<FwdSlice> out;
  const int first = n_vunits < 32 ? 1 : (n_vunits + 31) / 32;
  const int cap = std::max(first, (n_vunits + 3) / 4);
  int b = 0, size = first;
  while (b < n_vunits) {
    int e = std::min(n_vunits, b + size);
    if (n_vunits - e > 0 && n_vunits - e < first) e = n_vunits;
    out.push_back(FwdSlice{b, e, nullptr});
    b = e;
    size = std::min(cap, std::max(size + 1, size * 3 / 2));
  }
  return out;
}

int copy_async(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t st,
               const char* what) {
  if (bytes == 0) return LMH_OK;
  const cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, st);
  if (e != cudaSuccess) return fail(LMH_ERR_LAUNCH, "copy of %s: %s", what, cudaGetErrorString(e));
  return LMH_OK;
}

// Options of one backward call beyond the sizes and pointers.
struct BwdOpts {
  // A vocab shard: this call's weight holds rows [v_offset, v_offset + V) of
  // the whole head, labels index the whole vocabulary, and lse (and entropy)
  // are those of the whole distribution, so they cannot be recomputed here.
  int64_t v_offset = 0;
  bool shard = false;
  // Rows per chunk: dl and the transposed hidden hold this many rows.
  int64_t row_chunk = lmh::kBwdRowChunk;
};

// One fork of the side stream from `main`; the destructor joins a fork that
// an error left open, so `main` never runs ahead of the side stream's work.
struct SideBranch {
  SideStream* sd;
  cudaStream_t main;
  bool open = false;
  int fork() {
    cudaError_t e;
    if ((e = cudaEventRecord(sd->fork, main)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(sd->st, sd->fork, 0)) != cudaSuccess)
      return fail(LMH_ERR_LAUNCH, "side stream fork: %s", cudaGetErrorString(e));
    open = true;
    return LMH_OK;
  }
  int join() {
    open = false;
    cudaError_t e;
    if ((e = cudaEventRecord(sd->join, sd->st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(main, sd->join, 0)) != cudaSuccess)
      return fail(LMH_ERR_LAUNCH, "side stream join: %s", cudaGetErrorString(e));
    return LMH_OK;
  }
  ~SideBranch() {
    if (open && cudaEventRecord(sd->join, sd->st) == cudaSuccess)
      cudaStreamWaitEvent(main, sd->join, 0);
  }
};

// Row chunks up to this many rows run grad_hidden beside grad_weight. Alone
// at H = 3584, V = 152064, whole backward, one after the other / side by side
// (ms): 128 rows 0.935 / 0.743, 512 1.214 / 1.130, 1024 2.001 / 1.921, 2048
// 3.745 / 3.68, 4096 7.03 / 7.00, 16384 28.9 / 29.3; inside a long run at the
// power cap: 128 rows 1.065 / 0.785, 512 1.198 / 1.137, 1024 2.165 / 2.171,
// 2048 4.109 / 4.188. From 2048 rows grad_hidden spans more than one wave,
// and grad_weight then only fills its tail while disturbing its reads.
constexpr int64_t kBwdOverlapMaxRows = 1024;

// LMH_BWD_OVERLAP, read once (a diagnostic): "0" runs grad_hidden and
// grad_weight one after the other, "1" side by side; -1 when unset.
int bwd_overlap_mode() {
  static const int mode = [] {
    const char* v = std::getenv("LMH_BWD_OVERLAP");
    if (v && v[0] == '0') return 0;
    if (v && v[0] == '1') return 1;
    return -1;
  }();
  return mode;
}

// Backward of sum_t g[t] * logprob[t] (+ gH[t] * entropy[t]) for every row
// chunk of o.row_chunk rows, in ascending order:
//   dl   = recomputed logits -> dlogits (bf16 [rows][Vpad])
//   dH   = dl * W          (A = dl K-major, B = W MN-major); bf16, or fp32
//                          into grad_hidden_f32 (a vocab shard's partial)
//   hT   = hidden^T of the chunk (a transpose kernel, so the next A is K-major)
//   dW^T (+)= hT * dl      (A = hT K-major, B = dl MN-major; stored transposed)
// Chunks of up to kBwdOverlapMaxRows rows run dH on the side stream beside hT
// and dW^T.
int run_backward(const uint16_t* hidden, const uint16_t* weight, const int32_t* labels,
                 const float* grad_lp, const float* grad_ent, const float* lse, const float* ent,
                 int64_t T, int64_t H, int64_t V, float s, uint16_t* grad_hidden,
                 float* grad_hidden_f32, float* grad_weight, void* workspace,
                 size_t workspace_bytes, struct CUstream_st* stream, const BwdOpts& o = BwdOpts{}) {
  LMH_TRY(check_dims(T, H, V, true));
  LMH_TRY(check_temperature(s));
  if (o.v_offset < 0 || o.v_offset > LMH_MAX_DIM - V)
    return fail(LMH_ERR_INVALID_ARG, "v_offset=%lld out of range", (long long)o.v_offset);
  if (o.row_chunk < lmh::kBM || o.row_chunk % lmh::kBM != 0 || o.row_chunk > lmh::kBwdMaxRowChunk)
    return fail(LMH_ERR_INVALID_ARG, "row_chunk=%lld must be a multiple of %d in [%d, %lld]",
                (long long)o.row_chunk, lmh::kBM, lmh::kBM, (long long)lmh::kBwdMaxRowChunk);
  LMH_TRY(check_ptr(grad_weight, 16, "grad_weight"));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceInfo* dev = nullptr;
  if (T == 0) {  // only grad_weight is written (zeros); other pointers may be NULL
    LMH_TRY(device_info(&dev));
    LMH_TRY(launch_status(
        cudaMemsetAsync(grad_weight, 0, static_cast<size_t>(V) * H * sizeof(float), st),
        "zero grad_weight"));
    return ok();
  }
  LMH_TRY(check_ptr(hidden, 16, "hidden"));
  LMH_TRY(check_ptr(weight, 16, "weight"));
  LMH_TRY(check_ptr(labels, 4, "labels"));
  LMH_TRY(check_ptr(grad_lp, 4, "grad_logprob", true));
  LMH_TRY(check_ptr(grad_ent, 4, "grad_entropy", true));
  LMH_TRY(check_ptr(lse, 4, "lse", true));
  LMH_TRY(check_ptr(ent, 4, "entropy", true));
  if (grad_hidden_f32)
    LMH_TRY(check_ptr(grad_hidden_f32, 16, "grad_hidden_part"));
  else
    LMH_TRY(check_ptr(grad_hidden, 16, "grad_hidden"));
  if (!grad_lp && !grad_ent)
    return fail(LMH_ERR_INVALID_ARG, "grad_logprob and grad_entropy are both NULL");
  if (o.shard && (!lse || (grad_ent && !ent)))
    return fail(LMH_ERR_INVALID_ARG,
                "a vocab shard needs the whole vocabulary's lse (and entropy with grad_entropy)");
  Carver sizing{nullptr};
  carve_bwd(sizing, T, H, V, o.row_chunk);
  const size_t need = sizing.off + kRegionAlign;
  if (!workspace || workspace_bytes < need)
    return fail(LMH_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);
  LMH_TRY(check_ptr(workspace, 16, "workspace"));
  LMH_TRY(device_info(&dev));
  Carver c{static_cast<char*>(workspace)};
  const BwdWs w = carve_bwd(c, T, H, V, o.row_chunk);
  // grad_hidden beside grad_weight, on the side stream, for chunks of up to
  // kBwdOverlapMaxRows rows (LMH_BWD_OVERLAP forces it off or on)
  const int ov_mode = bwd_overlap_mode();
  auto overlap_for = [&](int64_t rows) {
    return ov_mode == 1 || (ov_mode < 0 && rows <= kBwdOverlapMaxRows);
  };
  const int64_t first_rows = T < o.row_chunk ? T : o.row_chunk;
  const int64_t last_rows = T % o.row_chunk == 0 ? first_rows : T % o.row_chunk;
  int dev_id = 0;
  cudaGetDevice(&dev_id);  // in range: device_info accepted it (and made the side stream)
  SideStream* side = &g_side[dev_id];
  std::unique_lock<std::mutex> side_lock(side->mu);
  LMH_TRY(side_stream_init(*side));
  if (!overlap_for(first_rows) && !overlap_for(last_rows)) {
    side_lock.unlock();
    side = nullptr;
  }

  if (!lse || (grad_ent && !ent)) {
    LMH_TRY(run_forward(*dev, hidden, weight, labels, T, H, V, s, w.lp, w.ent, w.lse, w.fwd, st));
    lse = w.lse;
    ent = w.ent;
  }
  CUtensorMap t_w_mn;
  LMH_TRY(make_tmap(&t_w_mn, weight, H, V, H * 2, 64, lmh::kBK));  // [K=V][N=H]

  for (int64_t c0 = 0; c0 < T; c0 += o.row_chunk) {
    const int64_t rows = (T - c0) < o.row_chunk ? (T - c0) : o.row_chunk;
    const uint16_t* h_c = hidden + c0 * H;
    CUtensorMap t_w, t_h, t_ht, t_dl, t_dl_mn;
    LMH_TRY(make_tmap(&t_w, weight, H, V, H * 2, lmh::kBK, lmh::kBBoxRows));   // [V][K=H]
    LMH_TRY(make_tmap(&t_h, h_c, H, rows, H * 2, lmh::kBK, lmh::kBM));        // [rows][K=H]
    LMH_TRY(make_tmap(&t_ht, w.ht, rows, H, w.tcpad * 2, lmh::kBK, lmh::kBM)); // [M=H][K=rows]
    LMH_TRY(make_tmap(&t_dl, w.dl, V, rows, w.vpad * 2, lmh::kBK, lmh::kBM)); // [rows][K=V]
    LMH_TRY(make_tmap(&t_dl_mn, w.dl, V, rows, w.vpad * 2, 64, lmh::kBK));    // [K=rows][N=V]

    lmh::GemmParams p{};
    p.status = dev->status;
    p.sched = w.fwd.sched;
    p.M = static_cast<int>(rows);
    p.N = static_cast<int>(V);
    p.K = static_cast<int>(H);
    p.scale2 = s * lmh::kLog2e;
    p.inv_temp = s;
    p.labels = labels + c0;
    p.label_base = o.v_offset;  // a label outside the shard gets no one-hot term
    p.grad = grad_lp ? grad_lp + c0 : nullptr;
    p.grad_ent = grad_ent ? grad_ent + c0 : nullptr;
    p.lse = lse + c0;
    p.ent = grad_ent ? ent + c0 : nullptr;
    CUtensorMap o_dl, o_gh, o_gw;
    LMH_TRY(make_out_tmap(&o_dl, w.dl, V, rows, w.vpad * 2, false));
    if (grad_hidden_f32)
      LMH_TRY(make_out_tmap(&o_gh, grad_hidden_f32 + c0 * H, H, rows, H * 4, true));
    else
      LMH_TRY(make_out_tmap(&o_gh, grad_hidden + c0 * H, H, rows, H * 2, false));
    LMH_TRY(make_out_tmap(&o_gw, grad_weight, H, V, H * 4, true, true));
    LMH_LAUNCH(lmh::K_DLOGITS_GEMM, st,
               lmh::launch_gemm(lmh::Epi::DLogits, t_h, t_w, p, 1, dev->sms, st, &o_dl),
               "dlogits");

    // grad_hidden sums dl * W over K = V in two fixed halves, P0 over the
    // first ceil(nk / 2) 64-wide K blocks and P1 over the rest, each walked in
    // order, then bf16(P0 + P1) (one K block: P0 alone). The split depends on
    // V only, so every row and every batch gets the same association; it
    // gives a short batch two independent MMA chains on two SMs per tile.
    const bool beside = side && overlap_for(rows);
    SideBranch branch{side, st};
    cudaStream_t gs = st;  // grad_hidden's stream
    if (beside) {
      LMH_TRY(branch.fork());
      gs = side->st;
    }
    lmh::GemmParams q{};
    q.status = dev->status;
    q.sched = beside ? w.sched2 : w.fwd.sched;
    q.corun = beside ? 1 : 0;
    q.M = static_cast<int>(rows);
    q.N = static_cast<int>(H);
    q.K = static_cast<int>(V);
    q.b_mn = 1;
    const int64_t nk = (V + lmh::kBK - 1) / lmh::kBK;
    if (nk >= 2) {
      q.k_split = static_cast<int>((nk + 1) / 2);
      q.seg_rows = static_cast<int>(w.ghp_rows);
      CUtensorMap o_ghp;
      LMH_TRY(make_out_tmap(&o_ghp, w.ghp, H, 2 * w.ghp_rows, H * 4, true));
      LMH_LAUNCH(lmh::K_DHIDDEN_GEMM, gs,
                 lmh::launch_gemm(lmh::Epi::StoreF32, t_dl, t_w_mn, q, 1, dev->sms, gs, &o_ghp),
                 "grad_hidden");
      void* gh_out = grad_hidden_f32 ? static_cast<void*>(grad_hidden_f32 + c0 * H)
                                     : static_cast<void*>(grad_hidden + c0 * H);
      LMH_LAUNCH(lmh::K_DHIDDEN_SUM, gs,
                 lmh::launch_sum_parts(w.ghp, 2, w.ghp_rows * H, rows * H, gh_out,
                                       grad_hidden_f32 == nullptr, dev->sms, gs),
                 "grad_hidden segments");
    } else {
      LMH_LAUNCH(lmh::K_DHIDDEN_GEMM, gs,
                 lmh::launch_gemm(grad_hidden_f32 ? lmh::Epi::StoreF32 : lmh::Epi::StoreBf16,
                                  t_dl, t_w_mn, q, 1, dev->sms, gs, &o_gh),
                 "grad_hidden");
    }

    // hidden^T of the chunk, so grad_weight reads its A operand K-major
    LMH_LAUNCH(lmh::K_HIDDEN_TRANSPOSE, st,
               lmh::launch_transpose_bf16(h_c, rows, H, H, w.ht, w.tcpad, st), "hidden transpose");

    lmh::GemmParams r{};
    r.status = dev->status;
    r.sched = w.fwd.sched;
    // grad_weight^T [H][V] = hidden^T * dl, stored transposed into grad_weight [V][H]
    r.M = static_cast<int>(H);
    r.N = static_cast<int>(V);
    r.K = static_cast<int>(rows);
    r.a_mn = 0;
    r.b_mn = 1;
    r.accumulate = c0 > 0 ? 1 : 0;  // later chunks: TMA reduce-add into grad_weight
    // Beside grad_hidden, grad_weight's CTAs start as SMs come free: claimed
    // units let the early ones take the work of those that start late. It
    // also takes wide pairs then, which changes its summation order (and so
    // its bits) against the run alone on 256-wide pairs.
    r.claim = beside ? 1 : 0;
    r.corun = beside ? 1 : 0;
    LMH_LAUNCH(lmh::K_DWEIGHT_GEMM, st,
               lmh::launch_gemm(lmh::Epi::StoreF32T, t_ht, t_dl_mn, r, 1, dev->sms, st, &o_gw),
               "grad_weight");
    // the next chunk overwrites dl and the partials
    if (beside) LMH_TRY(branch.join());
  }
  return ok();
}

}  // namespace

namespace lmh {
KernelTimer::KernelTimer(int kind, cudaStream_t st) : kind_(kind), st_(st) {
  if (!g_timing.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_tmu);
  b_ = take_event();
  if (b_) cudaEventRecord(b_, st_);
}

KernelTimer::~KernelTimer() {
  if (!b_) return;
  std::lock_guard<std::mutex> lk(g_tmu);
  cudaEvent_t e = take_event();
  if (!e) return;
  cudaEventRecord(e, st_);
  g_recs.push_back(TimingRec{kind_, b_, e});
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int api_set_error(int code, const char* msg) {
  if (code == LMH_OK) return ok();
  return fail(code, "%s", msg);
}

int api_device(int* sms, unsigned** status) {
  DeviceInfo* d = nullptr;
  const int rc = device_info(&d);
  if (rc != LMH_OK) return rc;
  *sms = d->sms;
  *status = d->status;
  return LMH_OK;
}

int api_noalloc_scratch(void** scratch) {
  DeviceInfo* d = nullptr;
  const int rc = device_info(&d);
  if (rc != LMH_OK) return rc;
  *scratch = d->noalloc_scratch;
  return LMH_OK;
}

int api_make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_tmap(map, base, inner, outer, row_bytes, box_inner, box_outer);
}
}  // namespace lmh

extern "C" {

unsigned long long lmhead_kernel_launches(void) { return g_launches.load(); }

int lmhead_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(g_tmu);
  for (const TimingRec& r : g_recs) {
    g_event_pool.push_back(r.b);
    g_event_pool.push_back(r.e);
  }
  g_recs.clear();
  g_timing.store(on != 0);
  return ok();
}

int lmhead_timing_read(int* kinds, float* ms, int capacity, int* count) {
  if (!count || capacity < 0 || (capacity > 0 && (!kinds || !ms)))
    return fail(LMH_ERR_INVALID_ARG, "lmhead_timing_read: bad arguments");
  std::lock_guard<std::mutex> lk(g_tmu);
  int n = 0;
  int rc = LMH_OK;
  for (const TimingRec& r : g_recs) {
    if (n < capacity) {
      float t = 0.f;
      cudaError_t e = cudaEventSynchronize(r.e);
      if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.b, r.e);
      if (e != cudaSuccess) rc = fail(LMH_ERR_LAUNCH, "timing: %s", cudaGetErrorString(e));
      kinds[n] = r.kind;
      ms[n] = t;
      ++n;
    }
    g_event_pool.push_back(r.b);
    g_event_pool.push_back(r.e);
  }
  g_recs.clear();
  *count = n;
  return rc == LMH_OK ? ok() : rc;
}

const char* lmhead_timing_kind_name(int kind) {
  return (kind >= 0 && kind < lmh::K_COUNT) ? kKindNames[kind] : "";
}

const char* lmhead_last_error_string(void) { return t_err; }

int lmhead_abi_version(void) { return 1; }

size_t lmhead_workspace_size(int op, int64_t T, int64_t H, int64_t V) {
  if (op == LMH_OP_LOGITS) {
    if (check_dims(T, 8, V, false) != LMH_OK) return SIZE_MAX;
    return 0;
  }
  if (op != LMH_OP_FWD && op != LMH_OP_BWD) {
    fail(LMH_ERR_INVALID_ARG, "unknown op %d", op);
    return SIZE_MAX;
  }
  if (check_dims(T, H, V, true) != LMH_OK) return SIZE_MAX;
  Carver c{nullptr};
  if (op == LMH_OP_FWD)
    carve_fwd(c, T, V);
  else
    carve_bwd(c, T, H, V);
  return c.off + kRegionAlign;
}

int lmhead_logprob_fwd(const uint16_t* hidden, const uint16_t* weight, const int32_t* labels,
                       int64_t T, int64_t H, int64_t V, float inv_temperature,
                       float* out_logprob, float* out_entropy, float* out_lse, void* workspace,
                       size_t workspace_bytes, struct CUstream_st* stream) {
  return fwd_entry(hidden, weight, labels, T, H, V, inv_temperature, out_logprob, out_entropy,
                   out_lse, nullptr, workspace, workspace_bytes, stream);
}

int lmhead_logprob_fwd_stats(const uint16_t* hidden, const uint16_t* weight, const int32_t* labels,
                             int64_t T, int64_t H, int64_t V, float inv_temperature,
                             float* out_logprob, float* out_entropy, float* out_lse,
                             float* out_sum_p2, void* workspace, size_t workspace_bytes,
                             struct CUstream_st* stream) {
  return fwd_entry(hidden, weight, labels, T, H, V, inv_temperature, out_logprob, out_entropy,
                   out_lse, out_sum_p2, workspace, workspace_bytes, stream);
}

int lmhead_logprob_bwd(const uint16_t* hidden, const uint16_t* weight, const int32_t* labels,
                       const float* grad_logprob, const float* lse, int64_t T, int64_t H,
                       int64_t V, float inv_temperature, uint16_t* grad_hidden,
                       float* grad_weight, void* workspace, size_t workspace_bytes,
                       struct CUstream_st* stream) {
  if (T > 0 && !grad_logprob) return fail(LMH_ERR_INVALID_ARG, "grad_logprob is NULL");
  return run_backward(hidden, weight, labels, grad_logprob, nullptr, lse, nullptr, T, H, V,
                      inv_temperature, grad_hidden, nullptr, grad_weight, workspace,
                      workspace_bytes, stream);
}

int lmhead_logprob_entropy_bwd(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* labels, const float* grad_logprob,
                               const float* grad_entropy, const float* lse, const float* entropy,
                               int64_t T, int64_t H, int64_t V, float inv_temperature,
                               uint16_t* grad_hidden, float* grad_weight, void* workspace,
                               size_t workspace_bytes, struct CUstream_st* stream) {
  return run_backward(hidden, weight, labels, grad_logprob, grad_entropy, lse, entropy, T, H, V,
                      inv_temperature, grad_hidden, nullptr, grad_weight, workspace,
                      workspace_bytes, stream);
}

int lmhead_logprob_bwd_chunked(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* labels, const float* grad_logprob,
                               const float* grad_entropy, const float* lse, const float* entropy,
                               int64_t T, int64_t H, int64_t V, float inv_temperature,
                               int64_t row_chunk, uint16_t* grad_hidden, float* grad_weight,
                               void* workspace, size_t workspace_bytes,
                               struct CUstream_st* stream) {
  BwdOpts o;
  o.row_chunk = row_chunk;
  return run_backward(hidden, weight, labels, grad_logprob, grad_entropy, lse, entropy, T, H, V,
                      inv_temperature, grad_hidden, nullptr, grad_weight, workspace,
                      workspace_bytes, stream, o);
}

size_t lmhead_workspace_size_bwd(int64_t T, int64_t H, int64_t V, int64_t row_chunk) {
  if (check_dims(T, H, V, true) != LMH_OK) return SIZE_MAX;
  if (row_chunk < lmh::kBM || row_chunk % lmh::kBM != 0 || row_chunk > lmh::kBwdMaxRowChunk) {
    fail(LMH_ERR_INVALID_ARG, "row_chunk=%lld must be a multiple of %d in [%d, %lld]",
         (long long)row_chunk, lmh::kBM, lmh::kBM, (long long)lmh::kBwdMaxRowChunk);
    return SIZE_MAX;
  }
  Carver c{nullptr};
  carve_bwd(c, T, H, V, row_chunk);
  return c.off + kRegionAlign;
}

int lmhead_logprob_bwd_shard(const uint16_t* hidden, const uint16_t* weight,
                             const int32_t* labels, const float* grad_logprob,
                             const float* grad_entropy, const float* lse, const float* entropy,
                             int64_t T, int64_t H, int64_t V, int64_t v_offset,
                             float inv_temperature, float* grad_hidden_part, float* grad_weight,
                             void* workspace, size_t workspace_bytes,
                             struct CUstream_st* stream) {
  BwdOpts o;
  o.v_offset = v_offset;
  o.shard = true;
  return run_backward(hidden, weight, labels, grad_logprob, grad_entropy, lse, entropy, T, H, V,
                      inv_temperature, nullptr, grad_hidden_part, grad_weight, workspace,
                      workspace_bytes, stream, o);
}

int lmhead_sum_ranks_bf16(const float* parts, int64_t n_parts, int64_t count, uint16_t* out,
                          struct CUstream_st* stream) {
  if (n_parts < 1 || n_parts > 65536)
    return fail(LMH_ERR_INVALID_ARG, "n_parts=%lld must be in [1, 65536]", (long long)n_parts);
  if (count < 0 || count > (int64_t(1) << 40))
    return fail(LMH_ERR_INVALID_ARG, "count=%lld out of range", (long long)count);
  if (count == 0) return ok();
  LMH_TRY(check_ptr(parts, 4, "parts"));
  LMH_TRY(check_ptr(out, 2, "out"));
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LMH_LAUNCH(lmh::K_SUM_PARTS, st,
             lmh::launch_sum_parts(parts, static_cast<int>(n_parts), count, count, out, true,
                                   dev->sms, st),
             "rank-ordered sum");
  return ok();
}

int logprob_from_logits(const uint16_t* logits, const int32_t* labels, int64_t T, int64_t V,
                        float inv_temperature, float* out_logprob, float* out_entropy,
                        float* out_lse, struct CUstream_st* stream) {
  return logits_entry(logits, labels, T, V, inv_temperature, false, nullptr, out_logprob,
                      out_entropy, out_lse, nullptr, stream);
}

int logprob_from_logits_stats(const uint16_t* logits, const int32_t* labels, int64_t T, int64_t V,
                              float inv_temperature, float* out_logprob, float* out_entropy,
                              float* out_lse, float* out_sum_p2, struct CUstream_st* stream) {
  return logits_entry(logits, labels, T, V, inv_temperature, false, nullptr, out_logprob,
                      out_entropy, out_lse, out_sum_p2, stream);
}

int logprob_from_logits_div(const uint16_t* logits, const int32_t* labels, int64_t T, int64_t V,
                            float temperature, const float* row_temperature, float* out_logprob,
                            float* out_entropy, float* out_lse, float* out_sum_p2,
                            struct CUstream_st* stream) {
  return logits_entry(logits, labels, T, V, temperature, true, row_temperature, out_logprob,
                      out_entropy, out_lse, out_sum_p2, stream);
}

int lmhead_logprob_fwd_partials(const uint16_t* hidden, const uint16_t* weight,
                                const int32_t* labels, int64_t T, int64_t H, int64_t V,
                                int64_t v_offset, float inv_temperature, float* part_m,
                                float* part_s, float* part_u, float* label_logit,
                                struct CUstream_st* stream) {
  LMH_TRY(check_dims(T, H, V, true));
  LMH_TRY(check_temperature(inv_temperature));
  const int64_t unit_cols = static_cast<int64_t>(lmh::kBN) * lmh::kFwdTilesPerChunk;
  if (v_offset < 0 || v_offset > LMH_MAX_DIM - V)
    return fail(LMH_ERR_INVALID_ARG, "v_offset=%lld out of range", (long long)v_offset);
  if (v_offset % unit_cols != 0)
    return fail(LMH_ERR_ALIGNMENT, "v_offset must be a multiple of %lld", (long long)unit_cols);
  if (T == 0) return ok();  // nothing to read or write; pointers may be NULL
  LMH_TRY(check_ptr(hidden, 16, "hidden"));
  LMH_TRY(check_ptr(weight, 16, "weight"));
  LMH_TRY(check_ptr(labels, 4, "labels"));
  LMH_TRY(check_ptr(part_m, 4, "part_m"));
  LMH_TRY(check_ptr(part_s, 4, "part_s"));
  LMH_TRY(check_ptr(part_u, 4, "part_u"));
  LMH_TRY(check_ptr(label_logit, 4, "label_logit"));
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // rows whose label lies in another shard keep 0, so the shards' buffers
  // can be summed
  LMH_TRY(launch_status(cudaMemsetAsync(label_logit, 0, static_cast<size_t>(T) * 4, st),
                        "zero label_logit"));
  CUtensorMap ta, tb;
  const int a_rows = lmh::short_a_rows(T);
  LMH_TRY(make_tmap(&ta, hidden, H, T, H * 2, lmh::kBK, a_rows ? a_rows : lmh::kBM));
  LMH_TRY(make_tmap(&tb, weight, H, V, H * 2, lmh::kBK, lmh::kBBoxRows));
  lmh::GemmParams p{};
  p.a_rows = a_rows;
  p.M = static_cast<int>(T);
  p.N = static_cast<int>(V);
  p.K = static_cast<int>(H);
  p.status = dev->status;
  p.scale2 = inv_temperature * lmh::kLog2e;
  p.inv_temp = inv_temperature;
  p.labels = labels;
  p.label_base = v_offset;
  p.part_m = part_m;
  p.part_s = part_s;
  p.part_u = part_u;
  p.part_q = nullptr;
  p.part_zl = label_logit;
  p.part_ld = T;
  LMH_LAUNCH(lmh::K_FWD_GEMM, st,
             lmh::launch_gemm(lmh::Epi::FwdStats, ta, tb, p, lmh::kFwdTilesPerChunk, dev->sms, st),
             "forward partials");
  return ok();
}

int lmhead_logprob_merge(const float* part_m, const float* part_s, const float* part_u,
                         const float* label_logit, const int32_t* labels, int64_t T, int64_t V,
                         float* out_logprob, float* out_entropy, float* out_lse,
                         struct CUstream_st* stream) {
  LMH_TRY(check_dims(T, 8, V, false));
  if (T == 0) return ok();
  LMH_TRY(check_ptr(part_m, 4, "part_m"));
  LMH_TRY(check_ptr(part_s, 4, "part_s"));
  LMH_TRY(check_ptr(part_u, 4, "part_u"));
  LMH_TRY(check_ptr(label_logit, 4, "label_logit"));
  LMH_TRY(check_ptr(labels, 4, "labels"));
  LMH_TRY(check_ptr(out_logprob, 4, "out_logprob"));
  LMH_TRY(check_ptr(out_entropy, 4, "out_entropy", true));
  LMH_TRY(check_ptr(out_lse, 4, "out_lse", true));
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LMH_LAUNCH(lmh::K_FWD_MERGE, st,
             lmh::launch_fwd_merge(part_m, part_s, part_u, nullptr, label_logit, labels, T,
                                   n_fwd_chunks(V), V, out_logprob, out_entropy, out_lse, nullptr,
                                   st),
             "partials merge");
  return ok();
}

int lmhead_logprob_fwd_host(const uint16_t* hidden_host, const uint16_t* weight_host,
                            const int32_t* labels_host, int64_t T, int64_t H, int64_t V,
                            float inv_temperature, uint16_t* hidden, uint16_t* weight,
                            int32_t* labels, float* out_logprob, float* out_entropy,
                            float* out_lse, float* out_logprob_host, float* out_entropy_host,
                            void* workspace, size_t workspace_bytes, struct CUstream_st* stream,
                            struct CUstream_st* copy_stream) {
  LMH_TRY(check_dims(T, H, V, true));
  LMH_TRY(check_temperature(inv_temperature));
  if (T == 0) return ok();  // nothing to copy, read or write; pointers may be NULL
  if (!hidden_host || !weight_host || !labels_host)
    return fail(LMH_ERR_INVALID_ARG, "a host input pointer is NULL");
  LMH_TRY(check_ptr(hidden, 16, "hidden"));
  LMH_TRY(check_ptr(weight, 16, "weight"));
  LMH_TRY(check_ptr(labels, 4, "labels"));
  LMH_TRY(check_ptr(out_logprob, 4, "out_logprob"));
  LMH_TRY(check_ptr(out_entropy, 4, "out_entropy", true));
  LMH_TRY(check_ptr(out_lse, 4, "out_lse", true));
  if (out_entropy_host && !out_entropy)
    return fail(LMH_ERR_INVALID_ARG, "out_entropy_host needs out_entropy");
  const size_t need = lmhead_workspace_size(LMH_OP_FWD, T, H, V);
  if (!workspace || workspace_bytes < need)
    return fail(LMH_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);
  LMH_TRY(check_ptr(workspace, 16, "workspace"));
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  Staging& sg = g_staging[dev_id];
  std::lock_guard<std::mutex> lk(sg.mu);
  cudaError_t e;
  if (!sg.copy && (e = cudaStreamCreateWithFlags(&sg.copy, cudaStreamNonBlocking)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "cudaStreamCreate: %s", cudaGetErrorString(e));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t cs = copy_stream ? reinterpret_cast<cudaStream_t>(copy_stream) : sg.copy;

  std::vector<FwdSlice> slices = staged_slices(n_fwd_chunks(V));
  LMH_TRY(staging_events(sg, slices.size() + 1));
  // The copies may overwrite the device inputs only after the caller's
  // earlier work on `stream` is done with them.
  if ((e = cudaEventRecord(sg.events[0], st)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(cs, sg.events[0], 0)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "stream ordering: %s", cudaGetErrorString(e));
  LMH_TRY(copy_async(hidden, hidden_host, static_cast<size_t>(T * H) * 2, cudaMemcpyHostToDevice,
                     cs, "hidden"));
  LMH_TRY(copy_async(labels, labels_host, static_cast<size_t>(T) * 4, cudaMemcpyHostToDevice, cs,
                     "labels"));
  const int64_t unit_cols = static_cast<int64_t>(lmh::kBN) * lmh::kFwdTilesPerChunk;
  for (size_t i = 0; i < slices.size(); ++i) {
    const int64_t r0 = slices[i].begin * unit_cols;
    const int64_t r1 = std::min<int64_t>(V, slices[i].end * unit_cols);
    LMH_TRY(copy_async(weight + r0 * H, weight_host + r0 * H, static_cast<size_t>((r1 - r0) * H) * 2,
                       cudaMemcpyHostToDevice, cs, "weight"));
    slices[i].ready = sg.events[1 + i];
    if ((e = cudaEventRecord(slices[i].ready, cs)) != cudaSuccess)
      return fail(LMH_ERR_LAUNCH, "cudaEventRecord: %s", cudaGetErrorString(e));
  }
  Carver c{static_cast<char*>(workspace)};
  const FwdWs w = carve_fwd(c, T, V);
  LMH_TRY(run_forward(*dev, hidden, weight, labels, T, H, V, inv_temperature, out_logprob,
                      out_entropy, out_lse, w, st, nullptr, &slices));
  if (out_logprob_host)
    LMH_TRY(copy_async(out_logprob_host, out_logprob, static_cast<size_t>(T) * 4,
                       cudaMemcpyDeviceToHost, st, "logprob"));
  if (out_entropy_host)
    LMH_TRY(copy_async(out_entropy_host, out_entropy, static_cast<size_t>(T) * 4,
                       cudaMemcpyDeviceToHost, st, "entropy"));
  return ok();
}

int lmhead_device_status(struct CUstream_st* stream, unsigned* bits) {
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(LMH_ERR_LAUNCH, "stream: %s", cudaGetErrorString(e));
  unsigned w = 0;
  if ((e = cudaMemcpyAsync(&w, dev->status, sizeof(w), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(dev->status, 0, sizeof(unsigned), st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "status word: %s", cudaGetErrorString(e));
  if (bits) *bits = w;
  if (w & lmh::LMH_DEVSTAT_TIMEOUT)
    return fail(LMH_ERR_DEVICE_TIMEOUT, "a bounded device wait ran out (status 0x%x)", w);
  return ok();
}

int lmhead_selftest_wait_timeout(uint64_t limit_ns, struct CUstream_st* stream) {
  if (limit_ns < 1000ull || limit_ns > 10000000000ull)
    return fail(LMH_ERR_INVALID_ARG, "limit_ns must be in [1e3, 1e10]");
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LMH_LAUNCH(lmh::K_SELFTEST, st, lmh::launch_wait_selftest(dev->status, limit_ns, dev->selftest, st),
             "wait self-test");
  int result = -1;
  cudaError_t e;
  if ((e = cudaMemcpyAsync(&result, dev->selftest, sizeof(int), cudaMemcpyDeviceToHost, st)) !=
          cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "wait self-test: %s", cudaGetErrorString(e));
  if (result == 0) return fail(LMH_ERR_DEVICE_TIMEOUT, "bounded wait gave up as expected");
  return fail(LMH_ERR_LAUNCH, "bounded wait self-test: unexpected result %d", result);
}

int lmhead_selftest_division(float temperature, int* mismatches, struct CUstream_st* stream) {
  if (!mismatches) return fail(LMH_ERR_INVALID_ARG, "mismatches is NULL");
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = cudaMemsetAsync(dev->selftest, 0, sizeof(int), st)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "division self-test: %s", cudaGetErrorString(e));
  LMH_LAUNCH(lmh::K_SELFTEST, st, lmh::launch_division_selftest(temperature, dev->selftest, st),
             "division self-test");
  int count = -1;
  if ((e = cudaMemcpyAsync(&count, dev->selftest, sizeof(int), cudaMemcpyDeviceToHost, st)) !=
          cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return fail(LMH_ERR_LAUNCH, "division self-test: %s", cudaGetErrorString(e));
  *mismatches = count;
  return ok();
}

int lmhead_engine_gemm(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                       int layout, float* D, struct CUstream_st* stream) {
  if (M < 0 || M > LMH_MAX_DIM || N < 8 || N > LMH_MAX_DIM || K < 8 || K > LMH_MAX_DIM)
    return fail(LMH_ERR_INVALID_ARG, "bad engine GEMM sizes");
  if (layout < 0 || layout > 3) return fail(LMH_ERR_INVALID_ARG, "layout must be 0..3");
  const bool a_mn = (layout & 1) != 0;
  const bool b_mn = (layout & 2) != 0;
  if (K % 8 != 0 || N % 8 != 0 || (a_mn && M % 8 != 0))
    return fail(LMH_ERR_ALIGNMENT, "K, N (and M when A is [K][M]) must be multiples of 8");
  LMH_TRY(check_ptr(A, 16, "A"));
  LMH_TRY(check_ptr(B, 16, "B"));
  LMH_TRY(check_ptr(D, 16, "D"));
  if (M == 0) return ok();
  DeviceInfo* dev = nullptr;
  LMH_TRY(device_info(&dev));
  CUtensorMap ta, tb;
  if (a_mn)
    LMH_TRY(make_tmap(&ta, A, M, K, M * 2, 64, lmh::kBK));
  else
    LMH_TRY(make_tmap(&ta, A, K, M, K * 2, lmh::kBK, lmh::kBM));
  if (b_mn)
    LMH_TRY(make_tmap(&tb, B, N, K, N * 2, 64, lmh::kBK));
  else
    LMH_TRY(make_tmap(&tb, B, K, N, K * 2, lmh::kBK, lmh::kBBoxRows));
  lmh::GemmParams p{};
  p.status = dev->status;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.a_mn = a_mn ? 1 : 0;
  p.b_mn = b_mn ? 1 : 0;
  p.accumulate = 0;
  CUtensorMap tc;
  LMH_TRY(make_out_tmap(&tc, D, N, M, N * 4, true));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LMH_LAUNCH(lmh::K_ENGINE_GEMM, st,
             lmh::launch_gemm(lmh::Epi::StoreF32, ta, tb, p, 1, dev->sms, st, &tc),
             "engine gemm");
  return ok();
}

}  // extern "C"

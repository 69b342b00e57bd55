// lmhead_logprob_fwd_noalloc: the fused forward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: for
// example a plugin whose host framework owns all device memory and offers no
// allocator, or a latency-critical loop that must not call an allocation
// routine because it can block and synchronise the device. For them this entry
// point keeps the forward's per-vocab-chunk partials in a fixed scratch array
// that is part of the library image itself (a file-scope __device__ array),
// so the call allocates nothing. The caller still passes every input and
// output buffer.
//
// Scratch rules:
//  * Size: LMH_NOALLOC_SCRATCH_BYTES (16 MiB). A call whose partials would not
//    fit is rejected with LMH_ERR_WORKSPACE before anything is launched.
//  * The array occupies that much memory on every GPU where the library's
//    device code is loaded, until the process exits.
//  * Set-up: the library's first call on each device (of any entry point)
//    looks up the array's device address with cudaGetSymbolAddress, with that
//    device current, and keeps it in the same per-device record as the status
//    word (the array's name in host code is only a host-side stand-in, never a
//    device address). Make that first call before any stream capture.
//  * Every call shares the one array, and it keeps the last call's contents.
//    Nothing in it has to start at zero: each call writes every partial it
//    later reads. Calls whose kernels overlap on the GPU (different streams, or
//    different host threads without ordering) race on the array and corrupt
//    each other's results; serialise them.
#include <cmath>
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "internal.h"
#include "lmhead.h"
#include "ptx.cuh"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(LMH_NOALLOC_SCRATCH_BYTES);
constexpr size_t kAlign = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

}  // namespace

namespace lmh {
// Called once per device, with that device current, when the library first
// sets the device up (api.cu keeps the result beside the status word). In
// host code g_noalloc_scratch names a host-side stand-in, never the device
// array, so its device address has to be looked up.
int noalloc_scratch_lookup(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    char msg[256];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(no-alloc scratch): %s", cudaGetErrorString(e));
    return api_set_error(LMH_ERR_LAUNCH, msg);
  }
  *out = p;
  return LMH_OK;
}
}  // namespace lmh

extern "C" int lmhead_logprob_fwd_noalloc(const uint16_t* hidden, const uint16_t* weight,
                                          const int32_t* labels, int64_t T, int64_t H, int64_t V,
                                          float inv_temperature, float* out_logprob,
                                          float* out_entropy, float* out_lse,
                                          struct CUstream_st* stream) {
  if (T < 0 || T > LMH_MAX_DIM || V < 1 || V > LMH_MAX_DIM || H < 8 || H > LMH_MAX_DIM)
    return lmh::api_set_error(LMH_ERR_INVALID_ARG, "T, H or V out of range");
  if (H % 8 != 0) return lmh::api_set_error(LMH_ERR_ALIGNMENT, "H must be a multiple of 8");
  if (!std::isfinite(inv_temperature) || !(inv_temperature > 0.f))
    return lmh::api_set_error(LMH_ERR_INVALID_ARG, "inv_temperature must be finite and > 0");
  if (T == 0) return lmh::api_set_error(LMH_OK, "");
  if (!hidden || !weight || !labels || !out_logprob)
    return lmh::api_set_error(LMH_ERR_INVALID_ARG, "hidden, weight, labels and out_logprob are required");
  if (misaligned(hidden, 16) || misaligned(weight, 16) || misaligned(labels, 4) ||
      misaligned(out_logprob, 4) || misaligned(out_entropy, 4) || misaligned(out_lse, 4))
    return lmh::api_set_error(LMH_ERR_ALIGNMENT, "hidden/weight need 16-byte, the rest 4-byte alignment");

  // Scratch layout: planes m, s, u of [n_chunks][T] floats, then zl [T].
  const int64_t n_tiles = (V + lmh::kBN - 1) / lmh::kBN;
  const int64_t n_chunks = (n_tiles + lmh::kFwdTilesPerChunk - 1) / lmh::kFwdTilesPerChunk;
  const size_t plane = round_up(static_cast<size_t>(n_chunks * T) * sizeof(float));
  const size_t need = 3 * plane + round_up(static_cast<size_t>(T) * sizeof(float));
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "T=%lld, V=%lld needs %zu bytes of forward scratch; the built-in scratch holds %zu "
             "(use lmhead_logprob_fwd with a workspace, or split the rows)",
             (long long)T, (long long)V, need, kScratchBytes);
    return lmh::api_set_error(LMH_ERR_WORKSPACE, msg);
  }

  int sms = 0;
  unsigned* status = nullptr;
  int rc = lmh::api_device(&sms, &status);
  if (rc != LMH_OK) return rc;
  void* base = nullptr;
  if ((rc = lmh::api_noalloc_scratch(&base)) != LMH_OK) return rc;
  char* b = static_cast<char*>(base);
  float* pm = reinterpret_cast<float*>(b);
  float* ps = reinterpret_cast<float*>(b + plane);
  float* pu = reinterpret_cast<float*>(b + 2 * plane);
  float* pzl = reinterpret_cast<float*>(b + 3 * plane);

  CUtensorMap ta, tb;
  const int a_rows = lmh::short_a_rows(T);
  if ((rc = lmh::api_make_tmap(&ta, hidden, H, T, H * 2, lmh::kBK, a_rows ? a_rows : lmh::kBM)) !=
      LMH_OK)
    return rc;
  if ((rc = lmh::api_make_tmap(&tb, weight, H, V, H * 2, lmh::kBK, lmh::kBBoxRows)) != LMH_OK) return rc;
  lmh::GemmParams p{};
  p.a_rows = a_rows;
  p.M = static_cast<int>(T);
  p.N = static_cast<int>(V);
  p.K = static_cast<int>(H);
  p.status = status;
  p.scale2 = inv_temperature * lmh::kLog2e;
  p.inv_temp = inv_temperature;
  p.labels = labels;
  p.part_m = pm;
  p.part_s = ps;
  p.part_u = pu;
  p.part_zl = pzl;
  p.part_ld = T;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  {
    lmh::KernelTimer timer(lmh::K_FWD_GEMM, st);
    e = lmh::launch_gemm(lmh::Epi::FwdStats, ta, tb, p, lmh::kFwdTilesPerChunk, sms, st);
  }
  if (e == cudaSuccess) {
    lmh::KernelTimer timer(lmh::K_FWD_MERGE, st);
    e = lmh::launch_fwd_merge(pm, ps, pu, nullptr, pzl, labels, T, static_cast<int>(n_chunks), V,
                              out_logprob, out_entropy, out_lse, nullptr, st);
  }
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "no-alloc forward launch: %s", cudaGetErrorString(e));
    return lmh::api_set_error(LMH_ERR_LAUNCH, msg);
  }
  return lmh::api_set_error(LMH_OK, "");
}

// Memory-bound kernels of the LM-head library (sm_103a):
//   * the sampler formula on materialised bf16 logits (one streaming pass per
//     row: fp32 scale by the temperature factor, online max / sum-exp /
//     entropy accumulator, optionally sum p^2, label gather),
//   * the fixed-order merge of the fused forward's per-vocab-chunk partials,
//   * a self-test of the bounded wait (a barrier that nothing completes).
//
// The sampler formula is the one of the verl pull request "batch-invariant
// actor forward and sampler log-prob formula" (fp32 log_softmax over the full
// vocabulary, then a gather of the label), with the temperature applied as an
// fp32 factor to the fp32 logits (same page, temperature-order comment) and
// the label outside [0, V) mapped to log-prob 0 (SkyRL pull request "Triton
// backend for fused LM-head log-prob", out-of-vocab fix).
#include <cstdint>

#include <cuda_bf16.h>

#include "internal.h"
#include "online_softmax.cuh"
#include "ptx.cuh"

namespace lmh {

namespace {

constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kVecPerIter = 4;  // 16-byte loads in flight per thread per step

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Fixed-order CTA reduction of per-thread states: shuffle-down tree inside
// each warp, then warp 0's lane 0 folds the warp results in warp order.
template <bool kQ>
__device__ __forceinline__ OnlineStat cta_reduce(OnlineStat st, OnlineStat* sh) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    OnlineStat o;
    o.m = __shfl_down_sync(0xffffffffu, st.m, off);
    o.s = __shfl_down_sync(0xffffffffu, st.s, off);
    o.u = __shfl_down_sync(0xffffffffu, st.u, off);
    o.q = kQ ? __shfl_down_sync(0xffffffffu, st.q, off) : 0.f;
    if (lane + off < 32) stat_merge<kQ>(st, o);
  }
  if (lane == 0) sh[warp] = st;
  __syncthreads();
  OnlineStat r = stat_empty();
  if (threadIdx.x == 0) {
    r = sh[0];
    for (int w = 1; w < kRowWarps; ++w) stat_merge<kQ>(r, sh[w]);
  }
  __syncthreads();
  return r;
}

__device__ __forceinline__ void write_row_outputs(int64_t row, const OnlineStat& st, float y_label,
                                                  bool label_ok, float* out_lp, float* out_ent,
                                                  float* out_lse, float* out_sum_p2) {
  const float l2s = log2f(st.s);
  const float lse2 = __fadd_rn(st.m, l2s);
  out_lp[row] = label_ok ? __fmul_rn(kLn2, __fsub_rn(y_label, lse2)) : 0.f;
  if (out_ent) out_ent[row] = __fmul_rn(kLn2, __fsub_rn(l2s, __fdiv_rn(st.u, st.s)));
  if (out_lse) out_lse[row] = __fmul_rn(kLn2, lse2);
  if (out_sum_p2) out_sum_p2[row] = __fdiv_rn(st.q, __fmul_rn(st.s, st.s));
}

// V % 8 == 0: each thread owns the 16-byte vectors tid, tid + 512, ... of its
// row, folded kVecPerIter vectors (32 values) at a time. kQ adds sum p^2.
template <bool kQ>
__global__ void __launch_bounds__(kRowThreads)
    logits_logprob_vec_kernel(const uint16_t* __restrict__ logits, const int32_t* __restrict__ labels,
                              int64_t T, int64_t V, float scale2, float* __restrict__ out_lp,
                              float* __restrict__ out_ent, float* __restrict__ out_lse,
                              float* __restrict__ out_sum_p2) {
  __shared__ OnlineStat sh[kRowWarps];
  const int64_t nvec = V >> 3;
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const uint4* rp = reinterpret_cast<const uint4*>(logits + row * V);
    OnlineStat st = stat_empty();
    for (int64_t base = threadIdx.x; base < nvec; base += (int64_t)kVecPerIter * kRowThreads) {
      uint4 w[kVecPerIter];
      int nv = 0;
#pragma unroll
      for (int k = 0; k < kVecPerIter; ++k) {
        const int64_t idx = base + (int64_t)k * kRowThreads;
        if (idx < nvec) {
          w[k] = ld_stream(rp + idx);
          nv = k + 1;
        } else {
          w[k] = make_uint4(0, 0, 0, 0);
        }
      }
      float y[8 * kVecPerIter];
#pragma unroll
      for (int k = 0; k < kVecPerIter; ++k) {
        y[8 * k + 0] = __fmul_rn(bf16_lo(w[k].x), scale2);
        y[8 * k + 1] = __fmul_rn(bf16_hi(w[k].x), scale2);
        y[8 * k + 2] = __fmul_rn(bf16_lo(w[k].y), scale2);
        y[8 * k + 3] = __fmul_rn(bf16_hi(w[k].y), scale2);
        y[8 * k + 4] = __fmul_rn(bf16_lo(w[k].z), scale2);
        y[8 * k + 5] = __fmul_rn(bf16_hi(w[k].z), scale2);
        y[8 * k + 6] = __fmul_rn(bf16_lo(w[k].w), scale2);
        y[8 * k + 7] = __fmul_rn(bf16_hi(w[k].w), scale2);
      }
      if (nv == kVecPerIter)
        stat_fold<8 * kVecPerIter, kQ>(st, y);
      else
        stat_fold<8 * kVecPerIter, kQ>(st, y, 8 * nv);
    }
    const OnlineStat r = cta_reduce<kQ>(st, sh);
    if (threadIdx.x == 0) {
      const int lab = labels[row];
      const bool ok = lab >= 0 && (int64_t)lab < V;
      float yl = 0.f;
      if (ok) {
        const uint16_t b = logits[row * V + lab];
        yl = __fmul_rn(__uint_as_float(static_cast<uint32_t>(b) << 16), scale2);
      }
      write_row_outputs(row, r, yl, ok, out_lp, out_ent, out_lse, out_sum_p2);
    }
  }
}

// Any V: element-wise loads, 8 values per fold.
template <bool kQ>
__global__ void __launch_bounds__(kRowThreads)
    logits_logprob_scalar_kernel(const uint16_t* __restrict__ logits,
                                 const int32_t* __restrict__ labels, int64_t T, int64_t V,
                                 float scale2, float* __restrict__ out_lp,
                                 float* __restrict__ out_ent, float* __restrict__ out_lse,
                                 float* __restrict__ out_sum_p2) {
  __shared__ OnlineStat sh[kRowWarps];
  constexpr int kGroup = 8;
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const uint16_t* rp = logits + row * V;
    OnlineStat st = stat_empty();
    for (int64_t base = threadIdx.x; base < V; base += (int64_t)kGroup * kRowThreads) {
      float y[kGroup];
      int n = 0;
#pragma unroll
      for (int k = 0; k < kGroup; ++k) {
        const int64_t idx = base + (int64_t)k * kRowThreads;
        if (idx < V) {
          y[k] = __fmul_rn(__uint_as_float(static_cast<uint32_t>(rp[idx]) << 16), scale2);
          n = k + 1;
        } else {
          y[k] = 0.f;
        }
      }
      stat_fold<kGroup, kQ>(st, y, n);
    }
    const OnlineStat r = cta_reduce<kQ>(st, sh);
    if (threadIdx.x == 0) {
      const int lab = labels[row];
      const bool ok = lab >= 0 && (int64_t)lab < V;
      float yl = 0.f;
      if (ok) yl = __fmul_rn(__uint_as_float(static_cast<uint32_t>(rp[lab]) << 16), scale2);
      write_row_outputs(row, r, yl, ok, out_lp, out_ent, out_lse, out_sum_p2);
    }
  }
}

// One thread per row: fold the per-chunk partials in ascending chunk order.
template <bool kQ>
__global__ void fwd_merge_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                                 const float* __restrict__ pu, const float* __restrict__ pq,
                                 const float* __restrict__ pzl, const int32_t* __restrict__ labels,
                                 int64_t T, int n_vunits, int64_t V, float* __restrict__ out_lp,
                                 float* __restrict__ out_ent, float* __restrict__ out_lse,
                                 float* __restrict__ out_sum_p2) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= T) return;
  OnlineStat st = stat_empty();
  for (int c = 0; c < n_vunits; ++c) {
    const int64_t o = (int64_t)c * T + row;
    stat_merge<kQ>(st, OnlineStat{pm[o], ps[o], pu[o], kQ ? pq[o] : 0.f});
  }
  const int lab = labels[row];
  const bool ok = lab >= 0 && (int64_t)lab < V;
  write_row_outputs(row, st, ok ? pzl[row] : 0.f, ok, out_lp, out_ent, out_lse,
                    kQ ? out_sum_p2 : nullptr);
}

// Waits on an mbarrier that nothing will complete; the bounded wait must give
// up after limit_ns, record the timeout in *status and let the kernel return.
__global__ void wait_selftest_kernel(unsigned* status, unsigned long long limit_ns, int* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
    *result = ok ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_logits_logprob(const uint16_t* logits, const int32_t* labels, int64_t T,
                                  int64_t V, float inv_temperature, float* out_lp, float* out_ent,
                                  float* out_lse, float* out_sum_p2, int num_sms,
                                  cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const float scale2 = inv_temperature * kLog2e;
  const int64_t max_grid = (int64_t)num_sms * 4;
  const int grid = (int)(T < max_grid ? T : max_grid);
  const bool vec = (V & 7) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  if (vec && out_sum_p2)
    logits_logprob_vec_kernel<true><<<grid, kRowThreads, 0, stream>>>(
        logits, labels, T, V, scale2, out_lp, out_ent, out_lse, out_sum_p2);
  else if (vec)
    logits_logprob_vec_kernel<false><<<grid, kRowThreads, 0, stream>>>(
        logits, labels, T, V, scale2, out_lp, out_ent, out_lse, nullptr);
  else if (out_sum_p2)
    logits_logprob_scalar_kernel<true><<<grid, kRowThreads, 0, stream>>>(
        logits, labels, T, V, scale2, out_lp, out_ent, out_lse, out_sum_p2);
  else
    logits_logprob_scalar_kernel<false><<<grid, kRowThreads, 0, stream>>>(
        logits, labels, T, V, scale2, out_lp, out_ent, out_lse, nullptr);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_fwd_merge(const float* pm, const float* ps, const float* pu, const float* pq,
                             const float* pzl, const int32_t* labels, int64_t T, int n_vunits,
                             int64_t V, float* out_lp, float* out_ent, float* out_lse,
                             float* out_sum_p2, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int threads = 128;
  const int64_t blocks = (T + threads - 1) / threads;
  if (pq && out_sum_p2)
    fwd_merge_kernel<true><<<(unsigned)blocks, threads, 0, stream>>>(
        pm, ps, pu, pq, pzl, labels, T, n_vunits, V, out_lp, out_ent, out_lse, out_sum_p2);
  else
    fwd_merge_kernel<false><<<(unsigned)blocks, threads, 0, stream>>>(
        pm, ps, pu, nullptr, pzl, labels, T, n_vunits, V, out_lp, out_ent, out_lse, nullptr);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_wait_selftest(unsigned* status, unsigned long long limit_ns, int* result,
                                 cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns, result);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace lmh

// Memory-bound kernels of the LM-head library (sm_103a):
//   * the sampler formula on materialised bf16 logits (one streaming pass per
//     row: fp32 scale by the inverse temperature, or fp32 division by a
//     scalar or per-row temperature; online max / sum-exp / entropy
//     accumulator, optionally sum p^2; label gather),
//   * the fixed-order merge of the fused forward's per-vocab-chunk partials,
//   * the transpose of a row chunk of hidden (grad_weight's K-major operand),
//   * ordered sums of fp32 partials (grad_hidden's two K halves; a
//     vocab-parallel head's per-rank shares),
//   * self-tests of the bounded wait (a barrier that nothing completes) and
//     of the division.
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

// The temperature map of one row: ScaleMul from the folded factor, ScaleDiv
// from the row's own temperature when a per-row array is given. A row
// temperature that is not finite and > 0 becomes NaN, so that row's outputs
// are NaN and no other row is affected.
template <class S>
__device__ __forceinline__ S row_scale(float tparam, const float* row_t, int64_t row);
template <>
__device__ __forceinline__ ScaleMul row_scale<ScaleMul>(float tparam, const float*, int64_t) {
  return ScaleMul{tparam};
}
template <>
__device__ __forceinline__ ScaleDiv row_scale<ScaleDiv>(float tparam, const float* row_t,
                                                        int64_t row) {
  float t = row_t ? row_t[row] : tparam;
  if (!(t > 0.f && t <= 3.402823466e38f)) t = __int_as_float(0x7fffffff);
  return ScaleDiv::make(t);
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

// V % 8 == 0, streamed through shared memory. Warp 0 (one thread) copies each
// row in 16 KB chunks into a kLStages-deep ring with untiled bulk copies, so
// the next chunks (and the next row) are in flight while 8 consumer warps
// fold the current one. Consumer thread t owns the 16-byte vectors t, t+256,
// t+512, t+768 of every chunk, so a row's fold order depends only on V.
// Every wait is bounded; after a timeout the loops still run to the end
// (skipping work) so all consumers reach the same named barriers.
// Three CTAs per SM with a 4-deep ring (measured against two with a 6-deep
// ring: multiply form 0.374 -> 0.361 ms, division form 0.591 -> 0.580 ms on
// [8192, 152064], same bits; four CTAs made the division form spill).
constexpr int kLConsumers = 256;
constexpr int kLThreads = 32 + kLConsumers;
constexpr int kLChunkBytes = 16384;
constexpr int kLVecPerThread = kLChunkBytes / 16 / kLConsumers;  // 4
static_assert(kLVecPerThread == 4, "stat_fold_bf16x32 folds four 16-byte words per thread");
constexpr int kLStages = 4;
constexpr int kLBlocksPerSm = 3;
constexpr int kLSmemBytes = kLStages * kLChunkBytes + 1024;

template <bool kQ, class S>
__global__ void __launch_bounds__(kLThreads, kLBlocksPerSm)
    logits_logprob_tma_kernel(const uint16_t* __restrict__ logits,
                              const int32_t* __restrict__ labels, int64_t T, int64_t V,
                              float tparam, const float* __restrict__ row_t,
                              float* __restrict__ out_lp,
                              float* __restrict__ out_ent, float* __restrict__ out_lse,
                              float* __restrict__ out_sum_p2, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  __shared__ __align__(8) uint64_t bars[2 * kLStages];
  __shared__ OnlineStat sh[2][kLConsumers / 32];
  __shared__ int abort_word;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (kLStages + st); };
  volatile int* abort_flag = &abort_word;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < kLStages; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), kLConsumers / 32);
    }
    abort_word = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int64_t row_bytes = V * 2;
  const int64_t n_chunks = (row_bytes + kLChunkBytes - 1) / kLChunkBytes;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int64_t row = blockIdx.x; ok && row < T; row += gridDim.x) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(logits + row * V);
        for (int64_t c = 0; c < n_chunks; ++c) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          const int64_t off = c * kLChunkBytes;
          const uint32_t bytes = static_cast<uint32_t>(
              row_bytes - off < kLChunkBytes ? row_bytes - off : kLChunkBytes);
          mbar_arrive_expect_tx(full_bar(stage), bytes);
          bulk_load_1d(ring + stage * kLChunkBytes, src + off, bytes, full_bar(stage));
          ++issued;
          if (++stage == kLStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // drain this thread's copies (bounded) before the CTA can exit
        volatile int no_abort = 0;
        const long long n = issued < kLStages ? issued : kLStages;
        uint32_t st = stage, ph = phase;
        for (long long i = 0; i < n; ++i) {
          if (st == 0) {
            st = kLStages - 1;
            ph ^= 1u;
          } else {
            --st;
          }
          mbar_wait(full_bar(st), ph, &no_abort, status);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int ct = threadIdx.x - 32;
    const int cw = warp - 1;
    uint32_t stage = 0, phase = 0, parity = 0;
    bool ok = true;
    for (int64_t row = blockIdx.x; row < T; row += gridDim.x, parity ^= 1u) {
      const S sc = row_scale<S>(tparam, row_t, row);
      OnlineStat st = stat_empty();
      for (int64_t c = 0; c < n_chunks; ++c) {
        if (ok) ok = mbar_wait(full_bar(stage), phase, abort_flag, status);
        if (ok) {
          const int64_t off = c * kLChunkBytes;
          const int64_t bytes = row_bytes - off < kLChunkBytes ? row_bytes - off : kLChunkBytes;
          const int nvec = static_cast<int>(bytes >> 4);
          const uint32_t base = ring + stage * kLChunkBytes;
          uint4 w[kLVecPerThread];
          int nv = 0;
#pragma unroll
          for (int k = 0; k < kLVecPerThread; ++k) {
            const int idx = ct + k * kLConsumers;
            if (idx < nvec) {
              w[k] = ld_shared_v4(base + (static_cast<uint32_t>(idx) << 4));
              nv = k + 1;
            } else {
              w[k] = make_uint4(0, 0, 0, 0);
            }
          }
          if (nv > 0) stat_fold_bf16x32<kQ>(st, w, nv, sc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(stage));  // this warp is done with the chunk
        if (++stage == kLStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // fixed-order reduction: shuffle-down tree, then warp order
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        OnlineStat o;
        o.m = __shfl_down_sync(0xffffffffu, st.m, off);
        o.s = __shfl_down_sync(0xffffffffu, st.s, off);
        o.u = __shfl_down_sync(0xffffffffu, st.u, off);
        o.q = kQ ? __shfl_down_sync(0xffffffffu, st.q, off) : 0.f;
        if (lane + off < 32) stat_merge<kQ>(st, o);
      }
      if (lane == 0) sh[parity][cw] = st;
      named_barrier(1, kLConsumers);
      if (ct == 0 && ok) {
        OnlineStat r = sh[parity][0];
        for (int k = 1; k < kLConsumers / 32; ++k) stat_merge<kQ>(r, sh[parity][k]);
        const int lab = labels[row];
        const bool lab_ok = lab >= 0 && (int64_t)lab < V;
        float yl = 0.f;
        if (lab_ok) yl = sc.y(__uint_as_float(static_cast<uint32_t>(logits[row * V + lab]) << 16));
        write_row_outputs(row, r, yl, lab_ok, out_lp, out_ent, out_lse, out_sum_p2);
      }
    }
  }
}

// Any V: element-wise loads, 8 values per fold.
template <bool kQ, class S>
__global__ void __launch_bounds__(kRowThreads)
    logits_logprob_scalar_kernel(const uint16_t* __restrict__ logits,
                                 const int32_t* __restrict__ labels, int64_t T, int64_t V,
                                 float tparam, const float* __restrict__ row_t,
                                 float* __restrict__ out_lp,
                                 float* __restrict__ out_ent, float* __restrict__ out_lse,
                                 float* __restrict__ out_sum_p2) {
  __shared__ OnlineStat sh[kRowWarps];
  constexpr int kGroup = 8;
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const uint16_t* rp = logits + row * V;
    const S sc = row_scale<S>(tparam, row_t, row);
    OnlineStat st = stat_empty();
    for (int64_t base = threadIdx.x; base < V; base += (int64_t)kGroup * kRowThreads) {
      float y[kGroup];
      int n = 0;
#pragma unroll
      for (int k = 0; k < kGroup; ++k) {
        const int64_t idx = base + (int64_t)k * kRowThreads;
        if (idx < V) {
          y[k] = sc.y(__uint_as_float(static_cast<uint32_t>(rp[idx]) << 16));
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
      if (ok) yl = sc.y(__uint_as_float(static_cast<uint32_t>(rp[lab]) << 16));
      write_row_outputs(row, r, yl, ok, out_lp, out_ent, out_lse, out_sum_p2);
    }
  }
}

// The fixed merge order of a row's per-chunk partials: the n chunks form
// kMergeGroups consecutive groups of ceil(n / kMergeGroups) chunks (the last
// ones shorter or empty); each group is folded in ascending chunk order, then
// the group results in ascending group order. It depends on n (that is, on V)
// alone, and it shortens a row's chain of dependent merges from n to about
// n / 8 + 8.
constexpr int kMergeGroups = 8;

// kMergeGroups threads per row (consecutive lanes), one per group; the
// group's first lane then folds the groups' results in order.
template <bool kQ>
__global__ void __launch_bounds__(256)
    fwd_merge_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                     const float* __restrict__ pu, const float* __restrict__ pq,
                     const float* __restrict__ pzl, const int32_t* __restrict__ labels, int64_t T,
                     int n_vunits, int64_t V, float* __restrict__ out_lp,
                     float* __restrict__ out_ent, float* __restrict__ out_lse,
                     float* __restrict__ out_sum_p2) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = gid / kMergeGroups;
  const int grp = static_cast<int>(gid % kMergeGroups);
  const bool live = row < T;  // whole rows per warp: 32 / kMergeGroups rows
  const int per = (n_vunits + kMergeGroups - 1) / kMergeGroups;
  const int c_begin = grp * per;
  const int c_end = min(n_vunits, c_begin + per);
  OnlineStat st = stat_empty();
  if (live) {
    // Loads of kBatch chunks are issued before their merges, so a thread
    // keeps several loads in flight; the merge order stays ascending.
    constexpr int kBatch = 8;
    for (int c0 = c_begin; c0 < c_end; c0 += kBatch) {
      OnlineStat b[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (c0 + j < c_end) {
          const int64_t o = (int64_t)(c0 + j) * T + row;
          b[j] = OnlineStat{pm[o], ps[o], pu[o], kQ ? pq[o] : 0.f};
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (c0 + j < c_end) stat_merge<kQ>(st, b[j]);
    }
  }
  // the row's groups, in ascending order, into the first lane of the row
  const unsigned lane = threadIdx.x & 31u;
  const unsigned first = lane - lane % kMergeGroups;
  OnlineStat r = st;
#pragma unroll
  for (int g = 1; g < kMergeGroups; ++g) {
    OnlineStat o;
    o.m = __shfl_sync(0xffffffffu, st.m, first + g);
    o.s = __shfl_sync(0xffffffffu, st.s, first + g);
    o.u = __shfl_sync(0xffffffffu, st.u, first + g);
    o.q = kQ ? __shfl_sync(0xffffffffu, st.q, first + g) : 0.f;
    if (grp == 0) stat_merge<kQ>(r, o);
  }
  if (!live || grp != 0) return;
  const int lab = labels[row];
  const bool ok = lab >= 0 && (int64_t)lab < V;
  write_row_outputs(row, r, ok ? pzl[row] : 0.f, ok, out_lp, out_ent, out_lse,
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

// out[c][r] = in[r][c] for a rows x cols bf16 matrix (cols % 8 == 0, rows of
// `in` 16-byte aligned): 64 x 64 tiles through shared memory, 16-byte loads,
// and 16-byte stores where the output row allows them. Each warp stores
// 4 output rows x 128 contiguous bytes.
__global__ void __launch_bounds__(256)
    transpose_bf16_kernel(const uint16_t* __restrict__ in, int64_t rows, int64_t cols,
                          int64_t in_ld, uint16_t* __restrict__ out, int64_t out_ld) {
  __shared__ uint16_t tile[64][64 + 2];
  const int64_t r0 = (int64_t)blockIdx.y * 64;
  const int64_t c0 = (int64_t)blockIdx.x * 64;
  for (int i = threadIdx.x; i < 512; i += 256) {
    const int r = i >> 3, cw = i & 7;
    const int64_t gr = r0 + r, gc = c0 + cw * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (gr < rows && gc < cols) v = *reinterpret_cast<const uint4*>(in + gr * in_ld + gc);
    const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      tile[r][cw * 8 + 2 * j] = static_cast<uint16_t>(ws[j] & 0xffffu);
      tile[r][cw * 8 + 2 * j + 1] = static_cast<uint16_t>(ws[j] >> 16);
    }
  }
  __syncthreads();
  const bool vec_out = (out_ld & 7) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  for (int i = threadIdx.x; i < 512; i += 256) {
    const int c = i >> 3, rw = i & 7;
    const int64_t gc = c0 + c, gr = r0 + rw * 8;
    if (gc >= cols || gr >= rows) continue;
    uint32_t ws[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      ws[j] = static_cast<uint32_t>(tile[rw * 8 + 2 * j][c]) |
              (static_cast<uint32_t>(tile[rw * 8 + 2 * j + 1][c]) << 16);
    uint16_t* dst = out + gc * out_ld + gr;
    if (vec_out && gr + 8 <= rows) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    } else {
      for (int j = 0; j < 8 && gr + j < rows; ++j)
        dst[j] = static_cast<uint16_t>(ws[j >> 1] >> (16 * (j & 1)));
    }
  }
}

// out[i] = ((parts[0][i] + parts[1][i]) + parts[2][i]) + ..., in that order,
// rounded once at the end to bf16 (kBf16) or kept in fp32; part r starts at
// parts + r * stride. It adds the two K segments' partials of grad_hidden, and
// the ranks' grad_hidden partials of a vocab-parallel head, so that every
// caller gets the same bits. Four elements per thread and step when the
// buffers allow 16-byte loads.
template <bool kBf16>
__global__ void __launch_bounds__(256)
    sum_parts_kernel(const float* __restrict__ parts, int n_parts, int64_t stride, int64_t count,
                     void* __restrict__ out) {
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool vec = (count & 3) == 0 && (stride & 3) == 0 &&
                   (reinterpret_cast<uintptr_t>(parts) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & (kBf16 ? 7 : 15)) == 0;
  if (vec) {
    const int64_t n4 = count >> 2;
    for (int64_t i = tid; i < n4; i += step) {
      float4 acc = reinterpret_cast<const float4*>(parts)[i];
      for (int r = 1; r < n_parts; ++r) {
        const float4 v = reinterpret_cast<const float4*>(parts + static_cast<int64_t>(r) * stride)[i];
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
      }
      if constexpr (kBf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t*>(&lo);
        w.y = *reinterpret_cast<const uint32_t*>(&hi);
        reinterpret_cast<uint2*>(out)[i] = w;
      } else {
        reinterpret_cast<float4*>(out)[i] = acc;
      }
    }
  } else {
    for (int64_t i = tid; i < count; i += step) {
      float acc = parts[i];
      for (int r = 1; r < n_parts; ++r) acc = __fadd_rn(acc, parts[static_cast<int64_t>(r) * stride + i]);
      if constexpr (kBf16) {
        const __nv_bfloat16 b = __float2bfloat16_rn(acc);
        static_cast<uint16_t*>(out)[i] = *reinterpret_cast<const uint16_t*>(&b);
      } else {
        static_cast<float*>(out)[i] = acc;
      }
    }
  }
}

// Every bf16 bit pattern x: the library's quotient x / t against IEEE fp32
// division; counts the inputs whose result bits differ (NaN equals NaN).
__global__ void division_selftest_kernel(float t, int* mismatches) {
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 65536u) return;
  const float x = __uint_as_float(i << 16);
  const float a = ScaleDiv::make(t).quotient(x);
  const float b = __fdiv_rn(x, t);
  const bool same = (__float_as_uint(a) == __float_as_uint(b)) || (a != a && b != b);
  if (!same) atomicAdd(mismatches, 1);
}

template <bool kQ, class S>
cudaError_t launch_logits_t(const uint16_t* logits, const int32_t* labels, int64_t T, int64_t V,
                            float tparam, const float* row_t, float* out_lp, float* out_ent,
                            float* out_lse, float* out_sum_p2, int num_sms, unsigned* status,
                            cudaStream_t stream) {
  const bool vec = (V & 7) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  if (vec) {
    const int64_t tgrid = (int64_t)num_sms * kLBlocksPerSm;
    const int grid = (int)(T < tgrid ? T : tgrid);
    const cudaError_t e = cudaFuncSetAttribute(logits_logprob_tma_kernel<kQ, S>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kLSmemBytes);
    if (e != cudaSuccess) return e;
    logits_logprob_tma_kernel<kQ, S><<<grid, kLThreads, kLSmemBytes, stream>>>(
        logits, labels, T, V, tparam, row_t, out_lp, out_ent, out_lse, out_sum_p2, status);
  } else {
    const int64_t max_grid = (int64_t)num_sms * 4;
    const int grid = (int)(T < max_grid ? T : max_grid);
    logits_logprob_scalar_kernel<kQ, S><<<grid, kRowThreads, 0, stream>>>(
        logits, labels, T, V, tparam, row_t, out_lp, out_ent, out_lse, out_sum_p2);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_logits_logprob(const uint16_t* logits, const int32_t* labels, int64_t T,
                                  int64_t V, float temp_value, bool divide,
                                  const float* row_temperature, float* out_lp, float* out_ent,
                                  float* out_lse, float* out_sum_p2, int num_sms, unsigned* status,
                                  cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  cudaError_t e;
  if (divide) {
    e = out_sum_p2 ? launch_logits_t<true, ScaleDiv>(logits, labels, T, V, temp_value,
                                                     row_temperature, out_lp, out_ent, out_lse,
                                                     out_sum_p2, num_sms, status, stream)
                   : launch_logits_t<false, ScaleDiv>(logits, labels, T, V, temp_value,
                                                      row_temperature, out_lp, out_ent, out_lse,
                                                      nullptr, num_sms, status, stream);
  } else {
    const float scale2 = temp_value * kLog2e;  // inverse temperature folded with log2(e)
    e = out_sum_p2 ? launch_logits_t<true, ScaleMul>(logits, labels, T, V, scale2, nullptr,
                                                     out_lp, out_ent, out_lse, out_sum_p2,
                                                     num_sms, status, stream)
                   : launch_logits_t<false, ScaleMul>(logits, labels, T, V, scale2, nullptr,
                                                      out_lp, out_ent, out_lse, nullptr, num_sms,
                                                      status, stream);
  }
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_fwd_merge(const float* pm, const float* ps, const float* pu, const float* pq,
                             const float* pzl, const int32_t* labels, int64_t T, int n_vunits,
                             int64_t V, float* out_lp, float* out_ent, float* out_lse,
                             float* out_sum_p2, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int threads = 64;  // 8 rows per block: a 128-row batch still spreads over 16 SMs
  const int64_t blocks = (T * kMergeGroups + threads - 1) / threads;
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

cudaError_t launch_division_selftest(float t, int* mismatches, cudaStream_t stream) {
  division_selftest_kernel<<<256, 256, 0, stream>>>(t, mismatches);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_transpose_bf16(const uint16_t* in, int64_t rows, int64_t cols, int64_t in_ld,
                                  uint16_t* out, int64_t out_ld, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
  transpose_bf16_kernel<<<grid, 256, 0, stream>>>(in, rows, cols, in_ld, out, out_ld);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_sum_parts(const float* parts, int n_parts, int64_t stride, int64_t count,
                             void* out, bool out_bf16, int num_sms, cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  const int64_t work = (count + 3) / 4;
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  const unsigned g = static_cast<unsigned>(blocks);
  if (out_bf16)
    sum_parts_kernel<true><<<g, 256, 0, stream>>>(parts, n_parts, stride, count, out);
  else
    sum_parts_kernel<false><<<g, 256, 0, stream>>>(parts, n_parts, stride, count, out);
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

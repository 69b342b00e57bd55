// Online (streaming) softmax statistics in base 2.
//
// For the values y of one row (y = z * log2(e), z the temperature-scaled
// logit) the state holds
//   m = max y,   s = sum 2^(y - m),   u = sum 2^(y - m) * (y - m),
//   q = sum 2^(2 (y - m)).
// From it: lse = ln2 * (m + log2 s), entropy = ln2 * (log2 s - u / s),
// because -sum p ln p = ln2 * (log2 s - sum p (y - m)) with p = 2^(y-m) / s,
// and sum p^2 = q / s^2 (kept only when kQ is set).
//
// The flash-style streaming form follows the fused kernel described in the
// SkyRL pull request "Triton backend for fused LM-head log-prob" (an online
// max / sum-exp over vocab tiles); the entropy accumulator u is the same
// streaming idea applied to sum p * log p.
//
// Every function folds its inputs in one fixed order, so a row's state depends
// only on the row's own values and on how the vocabulary is split, never on
// the batch it arrives in. Each operation is an explicit round-to-nearest
// intrinsic, so the compiler cannot contract or reorder any of them: every
// kernel that folds the same values gets the same bits.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace lmh {

struct OnlineStat {
  float m, s, u, q;
};

__device__ __forceinline__ OnlineStat stat_empty() { return OnlineStat{-INFINITY, 0.f, 0.f, 0.f}; }

// a <- a (+) b, a first. An empty side (s == 0) leaves the other unchanged.
template <bool kQ = false>
__device__ __forceinline__ void stat_merge(OnlineStat& a, const OnlineStat& b) {
  if (b.s == 0.f) return;
  if (a.s == 0.f) {
    a = b;
    return;
  }
  const float m = fmaxf(a.m, b.m);
  const float da = __fsub_rn(a.m, m);
  const float db = __fsub_rn(b.m, m);
  const float ea = ex2(da);
  const float eb = ex2(db);
  a.u = __fadd_rn(__fmul_rn(ea, __fmaf_rn(a.s, da, a.u)), __fmul_rn(eb, __fmaf_rn(b.s, db, b.u)));
  a.s = __fadd_rn(__fmul_rn(a.s, ea), __fmul_rn(b.s, eb));
  if (kQ)
    a.q = __fadd_rn(__fmul_rn(a.q, __fmul_rn(ea, ea)), __fmul_rn(b.q, __fmul_rn(eb, eb)));
  a.m = m;
}

// Fold the first n of N values (n <= N, n >= 1) into the state, in index order
// split over two interleaved partial sums.
template <int N, bool kQ = false>
__device__ __forceinline__ void stat_fold(OnlineStat& st, const float (&y)[N], int n = N) {
  float gmax = y[0];
#pragma unroll
  for (int j = 1; j < N; ++j) gmax = (j < n) ? fmaxf(gmax, y[j]) : gmax;
  const float mn = fmaxf(st.m, gmax);
  const float d0 = __fsub_rn(st.m, mn);
  const float a = ex2(d0);
  const float u = (st.s > 0.f) ? __fmul_rn(a, __fmaf_rn(st.s, d0, st.u)) : 0.f;
  const float s = __fmul_rn(st.s, a);
  float s0 = 0.f, s1 = 0.f, u0 = 0.f, u1 = 0.f, q0 = 0.f, q1 = 0.f;
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const float da = (j < n) ? __fsub_rn(y[j], mn) : 0.f;
    const float ea = (j < n) ? ex2(da) : 0.f;
    s0 = __fadd_rn(s0, ea);
    u0 = __fmaf_rn(ea, da, u0);
    if (kQ) q0 = __fmaf_rn(ea, ea, q0);
    if (j + 1 < N) {
      const float db = (j + 1 < n) ? __fsub_rn(y[j + 1], mn) : 0.f;
      const float eb = (j + 1 < n) ? ex2(db) : 0.f;
      s1 = __fadd_rn(s1, eb);
      u1 = __fmaf_rn(eb, db, u1);
      if (kQ) q1 = __fmaf_rn(eb, eb, q1);
    }
  }
  if (kQ) st.q = __fmaf_rn(st.q, __fmul_rn(a, a), __fadd_rn(q0, q1));
  st.s = __fadd_rn(s, __fadd_rn(s0, s1));
  st.u = __fadd_rn(u, __fadd_rn(u0, u1));
  st.m = mn;
}

// Fold 32 bf16 values, given as 4 x 16-byte words (8 values each, of which
// the first nv words are valid), scaled by c > 0, into the state. Same
// statistics as stat_fold on y = x * c, in fewer instructions: the max is taken
// on the raw bf16 pairs (exact, and max commutes with the positive scale), and
// the scale and the max shift are one FMA, d = x * c - m. Every operation is
// still an explicit round-to-nearest intrinsic in a fixed order.
__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <bool kQ>
__device__ __forceinline__ void stat_fold_bf16x32(OnlineStat& st, const uint4 (&w)[4], int nv,
                                                  float c) {
  __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162*>(&w[0].x);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < nv) {
      const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (k > 0 || q > 0) m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&ws[q]));
    }
  }
  const float gmax = fmaxf(__low2float(m2), __high2float(m2));
  const float mn = fmaxf(st.m, __fmul_rn(gmax, c));
  const float d0 = __fsub_rn(st.m, mn);
  const float a = ex2(d0);
  const float u = (st.s > 0.f) ? __fmul_rn(a, __fmaf_rn(st.s, d0, st.u)) : 0.f;
  const float s = __fmul_rn(st.s, a);
  const float nmn = -mn;
  float s0 = 0.f, s1 = 0.f, u0 = 0.f, u1 = 0.f, q0 = 0.f, q1 = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < nv) {
      const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float da = __fmaf_rn(bf16_lo_f(ws[q]), c, nmn);
        const float ea = ex2(da);
        s0 = __fadd_rn(s0, ea);
        u0 = __fmaf_rn(ea, da, u0);
        if (kQ) q0 = __fmaf_rn(ea, ea, q0);
        const float db = __fmaf_rn(bf16_hi_f(ws[q]), c, nmn);
        const float eb = ex2(db);
        s1 = __fadd_rn(s1, eb);
        u1 = __fmaf_rn(eb, db, u1);
        if (kQ) q1 = __fmaf_rn(eb, eb, q1);
      }
    }
  }
  if (kQ) st.q = __fmaf_rn(st.q, __fmul_rn(a, a), __fadd_rn(q0, q1));
  st.s = __fadd_rn(s, __fadd_rn(s0, s1));
  st.u = __fadd_rn(u, __fadd_rn(u0, u1));
  st.m = mn;
}

}  // namespace lmh

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

}  // namespace lmh

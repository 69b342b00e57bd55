// Online (streaming) softmax statistics in base 2.
//
// For the values y of one row (y = z * log2(e), z the temperature-scaled
// logit) the state holds
//   m = max y,   s = sum 2^(y - m),   u = sum 2^(y - m) * (y - m).
// From it: lse = ln2 * (m + log2 s) and entropy = ln2 * (log2 s - u / s),
// because -sum p ln p = ln2 * (log2 s - sum p (y - m)) with p = 2^(y-m) / s.
//
// The flash-style streaming form follows the fused kernel described in the
// SkyRL pull request "Triton backend for fused LM-head log-prob" (an online
// max / sum-exp over vocab tiles); the entropy accumulator u is the same
// streaming idea applied to sum p * log p.
//
// Every function folds its inputs in one fixed order, so a row's state depends
// only on the row's own values and on how the vocabulary is split, never on
// the batch it arrives in.
#pragma once

#include "ptx.cuh"

namespace lmh {

struct OnlineStat {
  float m, s, u;
};

__device__ __forceinline__ OnlineStat stat_empty() { return OnlineStat{-INFINITY, 0.f, 0.f}; }

// a <- a (+) b, a first. An empty side (s == 0) leaves the other unchanged.
__device__ __forceinline__ void stat_merge(OnlineStat& a, const OnlineStat& b) {
  if (b.s == 0.f) return;
  if (a.s == 0.f) {
    a = b;
    return;
  }
  const float m = fmaxf(a.m, b.m);
  const float da = a.m - m;
  const float db = b.m - m;
  const float ea = ex2(da);
  const float eb = ex2(db);
  a.u = ea * (a.u + a.s * da) + eb * (b.u + b.s * db);
  a.s = a.s * ea + b.s * eb;
  a.m = m;
}

// Fold the first n of N values (n <= N, n >= 1) into the state, in index order
// split over two interleaved partial sums.
template <int N>
__device__ __forceinline__ void stat_fold(OnlineStat& st, const float (&y)[N], int n = N) {
  float gmax = y[0];
#pragma unroll
  for (int j = 1; j < N; ++j) gmax = (j < n) ? fmaxf(gmax, y[j]) : gmax;
  const float mn = fmaxf(st.m, gmax);
  const float d0 = st.m - mn;
  const float a = ex2(d0);
  float u = (st.s > 0.f) ? a * (st.u + st.s * d0) : 0.f;
  float s = st.s * a;
  float s0 = 0.f, s1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const float da = y[j] - mn;
    const float ea = (j < n) ? ex2(da) : 0.f;
    s0 += ea;
    u0 = fmaf(ea, (j < n) ? da : 0.f, u0);
    if (j + 1 < N) {
      const float db = y[j + 1] - mn;
      const float eb = (j + 1 < n) ? ex2(db) : 0.f;
      s1 += eb;
      u1 = fmaf(eb, (j + 1 < n) ? db : 0.f, u1);
    }
  }
  st.s = s + (s0 + s1);
  st.u = u + (u0 + u1);
  st.m = mn;
}

}  // namespace lmh

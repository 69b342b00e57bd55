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
  if (n == N && N % 2 == 1) {
#pragma unroll
    for (int j = 1; j + 1 < N; j += 2) gmax = fmax3(gmax, y[j], y[j + 1]);
  } else if (n == N) {
#pragma unroll
    for (int j = 1; j + 1 < N; j += 2) gmax = fmax3(gmax, y[j], y[j + 1]);
    gmax = fmaxf(gmax, y[N - 1]);
  } else {
#pragma unroll
    for (int j = 1; j < N; ++j) gmax = (j < n) ? fmaxf(gmax, y[j]) : gmax;
  }
  const float mn = fmaxf(st.m, gmax);
  const float d0 = __fsub_rn(st.m, mn);
  const float a = ex2(d0);
  const float u = (st.s > 0.f) ? __fmul_rn(a, __fmaf_rn(st.s, d0, st.u)) : 0.f;
  const float s = __fmul_rn(st.s, a);
  float s0 = 0.f, s1 = 0.f, u0 = 0.f, u1 = 0.f, q0 = 0.f, q1 = 0.f;
  if constexpr (N % 2 == 0) {
    // the two partial sums as one packed pair: even values in the low half,
    // odd values in the high half (y - m is y + (-m) exactly)
    const f32x2 nm2 = f2_pack(-mn, -mn);
    f32x2 s2 = f2_pack(0.f, 0.f), u2 = s2, q2 = s2;
#pragma unroll
    for (int j = 0; j < N; j += 2) {
      float da, db;
      f2_unpack(f2_add(f2_pack(y[j], y[j + 1]), nm2), da, db);
      da = (j < n) ? da : 0.f;
      db = (j + 1 < n) ? db : 0.f;
      const f32x2 e2 = f2_pack((j < n) ? ex2(da) : 0.f, (j + 1 < n) ? ex2(db) : 0.f);
      s2 = f2_add(s2, e2);
      u2 = f2_fma(e2, f2_pack(da, db), u2);
      if (kQ) q2 = f2_fma(e2, e2, q2);
    }
    f2_unpack(s2, s0, s1);
    f2_unpack(u2, u0, u1);
    f2_unpack(q2, q0, q1);
  } else {
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
  }
  if (kQ) st.q = __fmaf_rn(st.q, __fmul_rn(a, a), __fadd_rn(q0, q1));
  st.s = __fadd_rn(s, __fadd_rn(s0, s1));
  st.u = __fadd_rn(u, __fadd_rn(u0, u1));
  st.m = mn;
}

// As stat_fold on y = x * c (c > 0), with the scale folded into the shift:
// the max is taken on the raw values (max commutes with the positive scale),
// m = max y is that max times c, and each d = x * c - m is one FMA. The values
// go through the fp32 steps as packed pairs, even indices in the low half.
template <int N, bool kQ = false>
__device__ __forceinline__ void stat_fold_scaled(OnlineStat& st, const float (&x)[N], float c,
                                                 int n = N) {
  static_assert(N % 2 == 0, "pairs of values");
  float gmax = x[0];
  if (n == N) {
#pragma unroll
    for (int j = 1; j + 1 < N; j += 2) gmax = fmax3(gmax, x[j], x[j + 1]);
    gmax = fmaxf(gmax, x[N - 1]);
  } else {
#pragma unroll
    for (int j = 1; j < N; ++j) gmax = (j < n) ? fmaxf(gmax, x[j]) : gmax;
  }
  const float mn = fmaxf(st.m, __fmul_rn(gmax, c));
  const float d0 = __fsub_rn(st.m, mn);
  const float a = ex2(d0);
  const float u = (st.s > 0.f) ? __fmul_rn(a, __fmaf_rn(st.s, d0, st.u)) : 0.f;
  const float s = __fmul_rn(st.s, a);
  const f32x2 c2 = f2_pack(c, c), nm2 = f2_pack(-mn, -mn);
  f32x2 s2 = f2_pack(0.f, 0.f), u2 = s2, q2 = s2;
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    float da, db;
    f2_unpack(f2_fma(f2_pack(x[j], x[j + 1]), c2, nm2), da, db);
    da = (j < n) ? da : 0.f;
    db = (j + 1 < n) ? db : 0.f;
    const f32x2 e2 = f2_pack((j < n) ? ex2(da) : 0.f, (j + 1 < n) ? ex2(db) : 0.f);
    s2 = f2_add(s2, e2);
    u2 = f2_fma(e2, f2_pack(da, db), u2);
    if (kQ) q2 = f2_fma(e2, e2, q2);
  }
  float s0, s1, u0, u1, q0, q1;
  f2_unpack(s2, s0, s1);
  f2_unpack(u2, u0, u1);
  f2_unpack(q2, q0, q1);
  if (kQ) st.q = __fmaf_rn(st.q, __fmul_rn(a, a), __fadd_rn(q0, q1));
  st.s = __fadd_rn(s, __fadd_rn(s0, s1));
  st.u = __fadd_rn(u, __fadd_rn(u0, u1));
  st.m = mn;
}

// How a bf16 logit x becomes y = z * log2(e), z the temperature-scaled logit.
// ScaleMul multiplies by the inverse temperature s, folded with log2(e) into one
// factor c = s * log2(e): y = x * c, and the shifted value y - m is one FMA.
// ScaleDiv divides by the temperature t, z = x / t rounded to nearest exactly
// as IEEE fp32 division rounds it, then y = z * log2(e): the fp32 logits
// divided by an fp32 temperature, as the verl page's temperature-order table
// requires and as a sampler that divides by a per-request temperature tensor
// computes it. Both maps are non-decreasing in x (t, c > 0), so the maximum of
// y is the map of the maximum of x.
__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// The two bf16 of a 32-bit word as an fp32 pair (low half first).
__device__ __forceinline__ f32x2 bf16x2_f2(uint32_t w) { return f2_pack(bf16_lo_f(w), bf16_hi_f(w)); }

struct ScaleMul {
  static constexpr bool kNeedsMin = false;  // group_fast ignores the group's minimum
  float c;
  __device__ __forceinline__ float y(float x) const { return __fmul_rn(x, c); }
  // Every group takes the one-FMA path.
  __device__ __forceinline__ bool group_fast(const uint4 (&)[4], int, float, float, float) const {
    return true;
  }
  // d[i] = the shifted pair y - m of the two bf16 of word i (words of w in
  // order, 4 per 16-byte vector).
  __device__ __forceinline__ void shift_fast(const uint4 (&w)[4], float neg_m,
                                             f32x2 (&d)[16]) const {
    const f32x2 c2 = f2_pack(c, c), nm2 = f2_pack(neg_m, neg_m);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) d[4 * k + q] = f2_fma(bf16x2_f2(ws[q]), c2, nm2);
    }
  }
  __device__ __forceinline__ void shift_exact(const uint4 (&w)[4], int, float neg_m,
                                              f32x2 (&d)[16]) const {
    shift_fast(w, neg_m, d);
  }
  // The shifted pair of one 32-bit word, on either path.
  __device__ __forceinline__ f32x2 shift1_fast(uint32_t w, f32x2 nm2) const {
    return f2_fma(bf16x2_f2(w), f2_pack(c, c), nm2);
  }
  __device__ __forceinline__ f32x2 shift1_exact(uint32_t w, f32x2 nm2) const {
    return shift1_fast(w, nm2);
  }
};

// IEEE fp32 division, kept out of line so the rare callers add no code to the
// unrolled folds.
static __device__ __noinline__ float div_ieee(float x, float t) { return __fdiv_rn(x, t); }

// The quotient uses Markstein's correction of a reciprocal product (P.
// Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): with r = 1/t rounded to nearest,
// q0 = x * r rounded, the remainder x - q0 * t is exact in one FMA, and
// q0 + rem * r rounded once is the correctly rounded quotient. The fast path
// holds for t in [2^-20, 2^20] and |x| in [2^-100, 2^100], where every
// intermediate is exact or a normal fp32 number, so the result scales exactly
// with the exponents of x and t. It was checked by exact arithmetic for every
// bf16 significand against every fp32 temperature significand and for every
// bf16 input in that range at 2000 temperatures, and on the GPU against IEEE
// division for every bf16 input (the library's lmhead_selftest_division,
// which runs this same packed routine). Other inputs (zero, tiny or huge |x|,
// inf, extreme t) take the IEEE division.
struct ScaleDiv {
  static constexpr bool kNeedsMin = true;
  float t;
  float r;  // 1/t rounded to nearest, or 0 when t is outside [2^-20, 2^20]
  __device__ __forceinline__ static ScaleDiv make(float temperature) {
    ScaleDiv d;
    d.t = temperature;
    d.r = (temperature >= 0x1p-20f && temperature <= 0x1p20f) ? __frcp_rn(temperature) : 0.f;
    return d;
  }
  // Both halves of x2 through the fast path (no range check).
  __device__ __forceinline__ f32x2 fast_quotient2(f32x2 x2) const {
    const f32x2 r2 = f2_pack(r, r);
    const f32x2 q0 = f2_mul(x2, r2);
    const f32x2 rem = f2_fma(q0, f2_pack(-t, -t), x2);
    return f2_fma(rem, r2, q0);
  }
  __device__ __forceinline__ static bool in_fast_range(float ax) {
    return ax >= 0x1p-100f && ax <= 0x1p100f;
  }
  __device__ __forceinline__ float quotient(float x) const {
    if (r != 0.f && in_fast_range(fabsf(x))) {
      float lo, hi;
      f2_unpack(fast_quotient2(f2_pack(x, x)), lo, hi);
      return lo;
    }
    return div_ieee(x, t);
  }
  __device__ __forceinline__ float y(float x) const { return __fmul_rn(quotient(x), kLog2e); }
  // True when the fast path gives every shifted value of the group's first nv
  // vectors exactly: gmax and gmin are the group's largest and smallest raw
  // values, mn the running maximum of y after the group. Huge values (|x| >
  // 2^100, inf) need the IEEE division. Tiny ones (|x| < 2^-100, zero
  // included) are outside the fast path's proven range, but once |mn| >=
  // 2^-40 they cannot change a shifted value: |z log2(e)| < 2^-79 is below
  // half an ulp of mn, so d = z log2(e) - m rounds to -m whatever the last
  // bits of z. Only then is the group's smallest magnitude checked.
  __device__ __forceinline__ bool group_fast(const uint4 (&w)[4], int nv, float gmax, float gmin,
                                             float mn) const {
    if (r == 0.f) return false;
    if (!(gmax <= 0x1p100f && gmin >= -0x1p100f)) return false;
    if (fabsf(mn) >= 0x1p-40f) return true;
    __nv_bfloat162 amax = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[0].x));
    __nv_bfloat162 amin = amax;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k < nv) {
        const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __nv_bfloat162 a = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&ws[q]));
          amax = __hmax2(amax, a);
          amin = __hmin2(amin, a);
        }
      }
    }
    return in_fast_range(fminf(__low2float(amin), __high2float(amin))) &&
           in_fast_range(fmaxf(__low2float(amax), __high2float(amax)));
  }
  // d = z * log2(e) - m in one FMA, z = x / t.
  __device__ __forceinline__ void shift_fast(const uint4 (&w)[4], float neg_m,
                                             f32x2 (&d)[16]) const {
    const f32x2 l2 = f2_pack(kLog2e, kLog2e), nm2 = f2_pack(neg_m, neg_m);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) d[4 * k + q] = f2_fma(fast_quotient2(bf16x2_f2(ws[q])), l2, nm2);
    }
  }
  __device__ __forceinline__ void shift_exact(const uint4 (&w)[4], int nv, float neg_m,
                                              f32x2 (&d)[16]) const {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k < nv) {
        const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          d[4 * k + q] = f2_pack(__fmaf_rn(quotient(bf16_lo_f(ws[q])), kLog2e, neg_m),
                                 __fmaf_rn(quotient(bf16_hi_f(ws[q])), kLog2e, neg_m));
      }
    }
  }
  // The shifted pair of one 32-bit word, on either path (same operations as
  // shift_fast / shift_exact).
  __device__ __forceinline__ f32x2 shift1_fast(uint32_t w, f32x2 nm2) const {
    return f2_fma(fast_quotient2(bf16x2_f2(w)), f2_pack(kLog2e, kLog2e), nm2);
  }
  __device__ __forceinline__ f32x2 shift1_exact(uint32_t w, f32x2 nm2) const {
    float lo, hi;
    f2_unpack(nm2, lo, hi);
    return f2_pack(__fmaf_rn(quotient(bf16_lo_f(w)), kLog2e, lo),
                   __fmaf_rn(quotient(bf16_hi_f(w)), kLog2e, hi));
  }
};

// Fold 32 bf16 values, given as 4 x 16-byte words (8 values each, of which
// the first nv words are valid), into the state; sc maps a value to y. Same
// statistics as stat_fold on the mapped values, in fewer instructions: the max
// is taken on the raw bf16 pairs (exact, and max commutes with the
// non-decreasing map); the final scale and the max shift are one FMA,
// d = x * c - m (ScaleMul) or d = z * log2(e) - m (ScaleDiv); and the two bf16
// of each 32-bit word go through every fp32 step as one packed pair, the low
// halves feeding one partial sum and the high halves the other. Every
// operation is still an explicit round-to-nearest operation in a fixed order.
template <bool kQ, class S>
__device__ __forceinline__ void stat_fold_bf16x32(OnlineStat& st, const uint4 (&w)[4], int nv,
                                                  const S& sc) {
  __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162*>(&w[0].x);
  __nv_bfloat162 n2 = m2;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < nv) {
      const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (k > 0 || q > 0) {
          const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&ws[q]);
          m2 = __hmax2(m2, v);
          if (S::kNeedsMin) n2 = __hmin2(n2, v);
        }
    }
  }
  const float gmax = fmaxf(__low2float(m2), __high2float(m2));
  const float gmin = fminf(__low2float(n2), __high2float(n2));
  const float mn = fmaxf(st.m, sc.y(gmax));
  const float d0 = __fsub_rn(st.m, mn);
  const float a = ex2(d0);
  const float u = (st.s > 0.f) ? __fmul_rn(a, __fmaf_rn(st.s, d0, st.u)) : 0.f;
  const float s = __fmul_rn(st.s, a);
  // Each word's shifted pair is formed inside the fold (fewer live
  // registers than forming all 16 first); the fast and exact paths are two
  // copies of the same loop.
  const f32x2 nm2 = f2_pack(-mn, -mn);
  f32x2 s2 = f2_pack(0.f, 0.f), u2 = s2, q2 = s2;
  auto fold_pair = [&](const f32x2 d) {
    float da, db;
    f2_unpack(d, da, db);
    const f32x2 e2 = f2_pack(ex2(da), ex2(db));
    s2 = f2_add(s2, e2);
    u2 = f2_fma(e2, d, u2);
    if (kQ) q2 = f2_fma(e2, e2, q2);
  };
  if (sc.group_fast(w, nv, gmax, gmin, mn)) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k < nv) {
        const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) fold_pair(sc.shift1_fast(ws[q], nm2));
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k < nv) {
        const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) fold_pair(sc.shift1_exact(ws[q], nm2));
      }
    }
  }
  float s0, s1, u0, u1, q0, q1;
  f2_unpack(s2, s0, s1);
  f2_unpack(u2, u0, u1);
  f2_unpack(q2, q0, q1);
  if (kQ) st.q = __fmaf_rn(st.q, __fmul_rn(a, a), __fadd_rn(q0, q1));
  st.s = __fadd_rn(s, __fadd_rn(s0, s1));
  st.u = __fadd_rn(u, __fadd_rn(u0, u1));
  st.m = mn;
}

}  // namespace lmh

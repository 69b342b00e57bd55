// Tensor-core engine for every contraction of the LM head (sm_103a).
//
//   D[M, N] = sum_k A[m, k] * B[n, k]    A, B bf16; D fp32 in TMEM
//
// Each operand is either K-major (stored [rows][K]) or MN-major (stored
// [K][rows]); TMA brings it into shared memory with 128-byte swizzle and the
// MMA's instruction descriptor carries the matching major bit, so no operand
// is ever transposed in memory.
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: a 128x64 A tile and a 256x64 B tile per stage
//               (128-row boxes when K-major, 64-wide boxes when MN-major), 4 stages
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma
//               (M=128, N=256, K=16, four per 64-wide stage) into one of two
//               256-column accumulators, and tcgen05.commit frees the stage
//   warps 2..5  epilogue: each thread owns one accumulator row (its TMEM
//               lane) and reads it 32 columns at a time with tcgen05.ld; a
//               second group (warps 6..9) shares the drain of the forward's
//               and dlogits' wide tiles
// On 256-column tiles the epilogue of tile i overlaps the MMAs of tile i+1
// (double-buffered TMEM), and in the forward and dlogits (K = H) consecutive
// tiles also overlap in K: a tile's last K blocks alternate with the next
// tile's first ones in the operand ring, so two independent accumulator
// chains feed the tensor pipe while each tile keeps a few blocks to itself
// for the other accumulator's drain. A wide tile's one 512-column
// accumulator goes back to the MMA issuer in two halves (below).
//
// Schedule: the output is cut into units (a row tile, or a pair's two, by one
// or more column tiles), rastered in groups of row units so that concurrent
// units share operand tiles in L2. A short launch walks them with a fixed
// stride per CTA. A launch of several waves claims them from a counter in the
// workspace in ascending order: one thread per CTA (per pair) claims and
// passes each unit index to the CTA's other roles, and to the peer CTA,
// through a 16-slot ring of shared-memory words and mbarriers. The claimed
// order keeps concurrent units within about a wave of each other, which a
// fixed stride does not (CTA pairs drifted apart by several units over a
// 125-wave launch and lost the shared W tiles in L2), and it balances the
// tail. Which CTA runs a unit changes none of its arithmetic.
//
// CTA pairs: a cluster of two CTAs owns a 256x256 tile. Each CTA stages its
// own 128 A rows and one 128-row half of B (6 stages of 32 KB); CTA 0 issues
// tcgen05.mma.cta_group::2 (M=256), and each CTA's TMEM receives its 128
// accumulator rows, so the epilogue is the same. Wide pairs own 256x512
// tiles: two N=256 pair MMAs per K step into one 512-column accumulator per
// CTA, two independent chains that share each A stage, so a CTA stages a
// quarter fewer operand bytes per flop and an operand is re-read half as
// often. The accumulator goes back to the MMA issuer in two 256-column
// halves: the next tile's first N block starts once half 0 has been read
// (holding its stages for the second block until half 1 is free), and for
// the forward and dlogits two epilogue groups read half 0 first. The halves
// also reach the epilogue one after the other: a tile's last few K blocks run
// N block 0 first, so half 0 drains while block 1 finishes. A long K
// (grad_hidden, grad_weight) hides the rest of the drain; for the forward and
// dlogits (K = H) the saved operand traffic outweighs it. Every engine walks
// K in the same MMA order for the forward, dlogits and grad_hidden, so their
// bits do not depend on the engine.
//
// Narrow tiles: single CTAs and pairs also take tiles of fewer columns (64,
// 128 or 192 alone, 128 in a pair; MN-major B only), so a short grad_hidden
// (K = V, few row tiles) spreads over more SMs. Their ring is cut into more,
// smaller stages (up to 8) of the same bytes. The column split changes no
// element's K walk, so no bit.
//
// Epilogues (one per contraction of the method):
//   FwdStats   the fused forward of the SkyRL pull request "Triton backend for
//              fused LM-head log-prob" (vocab projection folded into an online
//              softmax over vocab tiles): per row and per 1024-column vocab
//              chunk, the base-2 online statistics (m, s, u, q) and the label
//              logit; no logit ever reaches HBM.
//   DLogits    the recomputed-logits backward: dl = s*(g*onehot - p*(g +
//              gH*(z - lse + H))) with p = exp(z - lse); the gH term is the
//              entropy gradient (dH/dz = -p (z - lse + H)); no one-hot term
//              for an out-of-vocab label (same page, out-of-vocab gradient
//              fix); written as bf16 dl [rows][V].
//   StoreBf16  grad_hidden = dl * W (B = W read MN-major), rounded once to bf16.
//   StoreF32T  grad_weight^T = hidden^T * dl (A = the chunk's hidden^T read
//              K-major, B = dl read MN-major), written transposed as
//              grad_weight [V][H] in fp32, accumulated over row chunks in
//              ascending order. Taking the small hidden operand as A keeps it
//              close to L2 while dl streams through once.
//   StoreF32   D = A * B^T in fp32, row-major (the bare engine GEMM).
//
// Batch invariance: the work split depends only on N (vocab) and never on M
// (rows); a row's forward statistics over a 1024-column unit are folded as two
// streams (its even and odd 256-column blocks, each in column order) merged
// in that order, the same on every engine; there are no atomics; and the
// forward, dlogits and grad_hidden contractions walk K in ascending order for
// every tile. Which engine runs depends on M (a pair
// needs two m tiles), and changes none of their bits. grad_weight, a sum over rows that no row's
// output depends on, walks K downwards on a CTA's odd waves for L2 reuse; its
// bits are fixed by the inputs, the row chunking, the SM count and the engine.
#include <atomic>
#include <cfloat>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda_bf16.h>

#include "internal.h"
#include "online_softmax.cuh"
#include "ptx.cuh"

namespace lmh {

namespace {

constexpr int kABytes = kBM * kBK * 2;           // one 128-row x 64-K A box
constexpr int kBHalfBytes = kBBoxRows * kBK * 2;  // one 128-row x 64-K B box
constexpr int kMnBoxBytes = 64 * kBK * 2;         // one 64(MN) x 64(K) bf16 box
constexpr int kTmemCols = 512;
constexpr int kBarrierBytes = 512;
// Slots of the ring through which a dynamic schedule's claimed unit indices
// reach the CTA's other roles (and the peer CTA of a pair). Unit j + 1 is
// published when the producer starts unit j, after it has issued every stage
// of the units before; a role can trail it by at most the operand ring's
// stages plus the two accumulators (every unit has at least one stage), about
// 11 units, so 16 slots never lap.
constexpr int kUnitSlots = 16;
// Staging for the TMA-store epilogues, 32 KB: two 16 KB buffers of a 128 x 32
// fp32 chunk, or per epilogue warp a share of 2 KB buffers of its 32 x 32 bf16
// boxes.
constexpr int kStagingBytes = kBM * 128;
constexpr uint32_t kStagingTotal = 2 * kStagingBytes;

// Engine modes: one CTA per 128 x 256 tile; a CTA pair per 256 x 256 tile;
// a CTA pair per 256 x 512 tile ("wide": two N=256 pair MMAs per K step into
// one 512-column accumulator per CTA, not double-buffered, for contractions
// whose K is long enough to hide nothing behind the epilogue).
constexpr int kSingle = 0, kPairMode = 1, kWideMode = 2;
// Most stages a ring is cut into (narrow tiles have smaller stages).
constexpr int kMaxStages = 8;

// The operand ring of one CTA. Alone, a CTA stages the whole 256-row B tile
// (48 KB a stage, 4 stages); in a CTA pair it stages half of it (32 KB a
// stage, 6 stages), since the peer holds the other half; in a wide pair it
// stages half of each of the two 256-column B blocks (48 KB, 4 stages).
template <int kMode>
struct Ring {
  static constexpr int kStages = kMode == kPairMode ? 6 : 4;
  static constexpr int kBBytes = kMode == kPairMode ? kBHalfBytes : 2 * kBHalfBytes;
  static constexpr int kNBlocks = kMode == kWideMode ? 2 : 1;  // N=256 MMAs per K step
  static constexpr int kTileN = kNBlocks * kBN;                // accumulator columns
  static constexpr int kAccs = kMode == kWideMode ? 1 : 2;     // accumulators in TMEM
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes + 2 * kStagingBytes + kBarrierBytes + 1024;
  static_assert(kSmemBytes <= 232448, "exceeds the 227 KB shared-memory limit per CTA");
  // full and empty per stage, two accumulator pairs, final, the unit ring's
  // slots, the forward's two exchange buffers' full and empty; then the TMEM
  // address, the abort flag, the peer's load count, two go flags and two unit
  // words per epilogue group, two exchange go flags, the unit ring and two
  // second-half go flags per epilogue group
  static_assert(8 * (2 * kMaxStages + 5 + kUnitSlots + 4) + 4 * (13 + kUnitSlots + 4) <=
                    kBarrierBytes,
                "barrier area too small");
};
constexpr uint32_t kEpiBarrier = 1;  // named barriers 1 and 2: one per epilogue group of 128

// Two epilogue groups share the drain of a wide tile for the forward and the
// bf16 stores: both read half 0 first, so it is handed back after half the
// drain. The fp32 stores keep one group (their long K
// leaves little to overlap, and a 320-thread CTA measured 2.5 % slower for
// grad_hidden and grad_weight even with the second group idle).
template <int E, int kMode>
constexpr bool kSplitHalvesFor =
    kMode == kWideMode &&
    (E == (int)Epi::FwdStats || E == (int)Epi::DLogits || E == (int)Epi::StoreBf16);
template <int E, int kMode>
constexpr int kThreadsFor = kSplitHalvesFor<E, kMode> ? kGemmThreadsTwoGroups : kGemmThreadsOneGroup;

// Unit u -> (m unit, N tiles). Units enumerate (m unit, vocab unit) pairs in
// groups of group_m m units, unit-major inside a group, so concurrently
// running CTAs share B tiles in L2. An m unit is one 128-row m tile, or two
// for a CTA pair. The order changes no value.
// Dynamic schedule: the next unit of the launch, -1 once all are claimed.
__device__ __forceinline__ int claim_unit(const GemmParams& p) {
  const unsigned v = atomicAdd(p.sched, 1u);
  return v < static_cast<unsigned>(p.n_units) ? static_cast<int>(v) : -1;
}

__device__ __forceinline__ void unit_coords(const GemmParams& p, int u, int& m_tile, int& n_first,
                                            int& n_count, int& vunit, int& seg) {
  // with a K split, the second K segment's units follow all of the first's
  seg = 0;
  if (p.k_split > 0) {
    const int per_seg = p.n_units >> 1;
    seg = u >= per_seg ? 1 : 0;
    u -= seg * per_seg;
  }
  const int per_group = p.group_m * p.n_vunits;
  const int g = u / per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.group_m, p.n_m_tiles - first_m);
  const int r = u - g * per_group;
  const int vu = r / gm;
  m_tile = first_m + (r - vu * gm);
  vunit = p.vunit_begin + vu;
  n_first = vunit * p.tiles_per_unit;
  n_count = min(p.tiles_per_unit, p.n_n_tiles - n_first);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// One row's 32 columns into a staging buffer laid out as the TMA store reads
// it (128 rows for fp32, a warp's 32 rows for bf16). fp32: 128-byte rows with
// 128-byte swizzle (16-byte chunk j of row r at chunk j ^ (r % 8)). bf16:
// 64-byte rows with 64-byte swizzle (chunk j at j ^ ((r / 2) % 4)). Either
// way a warp's 32 rows spread evenly over the banks.
__device__ __forceinline__ void stage_row_f32(uint32_t buf, int r, const float (&v)[32]) {
  const uint32_t row = buf + static_cast<uint32_t>(r) * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_shared_v4(row + ((static_cast<uint32_t>(j) ^ (r & 7)) << 4), __float_as_uint(v[4 * j]),
                 __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                 __float_as_uint(v[4 * j + 3]));
}
// Transposed staging for StoreF32T: value i of row r goes to [i][r] of a
// 32 x 128 fp32 box (512-byte rows, no swizzle); for a fixed i the 32 lanes of
// a warp write 32 consecutive words, one per bank.
__device__ __forceinline__ void stage_col_f32(uint32_t buf, int r, const float (&v)[32]) {
  const uint32_t col = buf + static_cast<uint32_t>(r) * 4u;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(col + static_cast<uint32_t>(i) * 512u),
                 "r"(__float_as_uint(v[i]))
                 : "memory");
}
__device__ __forceinline__ void stage_row_bf16(uint32_t buf, int r, const float (&v)[32]) {
  const uint32_t row = buf + static_cast<uint32_t>(r) * 64u;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_v4(row + ((static_cast<uint32_t>(j) ^ ((r >> 1) & 3)) << 4),
                 pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                 pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
}

// One CTA's share of the engine. In the pair modes the CTA is one of a
// cluster pair that shares every MMA (tcgen05 cta_group::2): the pair owns a
// 256 x 256 tile (256 x 512 when wide), each CTA stages the A rows of its own
// 128-row half and its 128-row half of each 256-column B block, and each
// CTA's TMEM receives its 128 rows of the accumulator. CTA 0 issues the MMAs;
// both CTAs' copies of a stage complete on CTA 0's full barrier, and CTA 0's
// commits free the stage and hand over the accumulators in both CTAs.
template <int E, int kMode>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                          const CUtensorMap& tmC, const GemmParams& p) {
  constexpr bool kPair = kMode != kSingle;
  using R = Ring<kMode>;
  constexpr int kS = kMaxStages;  // barrier slots
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  constexpr uint32_t kRingBytes = R::kStages * R::kStageBytes;
  const uint32_t staging = smem_base + kRingBytes;  // 2 x kStagingBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRingBytes + 2 * kStagingBytes);
  // barrier layout: full[kS], empty[kS], tfull[2], tempty[2], final, ufull[kUnitSlots]
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kS + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kS + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kS + 2 + a); };
  const uint32_t final_bar = bar0 + 8u * (2 * kS + 4);
  // the unit ring: slot j % kUnitSlots holds the j-th unit of this CTA's walk
  auto ufull_bar = [&](int j) {
    return bar0 + 8u * static_cast<uint32_t>(2 * kS + 5 + (j & (kUnitSlots - 1)));
  };
  // the forward's group exchange: buffer b's full (group 1 wrote) and empty
  // (group 0 read) barriers
  auto xfull_bar = [&](int b) { return bar0 + 8u * static_cast<uint32_t>(2 * kS + 5 + kUnitSlots + b); };
  auto xempty_bar = [&](int b) {
    return bar0 + 8u * static_cast<uint32_t>(2 * kS + 7 + kUnitSlots + b);
  };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(bars) +
                                                    8 * (2 * kS + 9 + kUnitSlots));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // pair: the number of stage loads CTA 1 issued, published to CTA 0 at the end
  volatile uint32_t* peer_issued = tmem_slot + 2;
  volatile int* epi_go = reinterpret_cast<volatile int*>(tmem_slot + 3);     // [group][2]
  volatile int* epi_unit = reinterpret_cast<volatile int*>(tmem_slot + 7);   // [group][2]
  volatile int* x_go = reinterpret_cast<volatile int*>(tmem_slot + 11);      // [group]
  volatile int* uring = reinterpret_cast<volatile int*>(tmem_slot + 13);     // [kUnitSlots]
  volatile int* epi_go1 = reinterpret_cast<volatile int*>(tmem_slot + 13 + kUnitSlots);  // [group][2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Position in the persistent schedule: a CTA pair walks the units as one.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int first_unit = kPair ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int unit_stride = kPair ? static_cast<int>(cluster_nid_x()) : static_cast<int>(gridDim.x);
  auto cta_m_tile = [&](int m_unit) { return kPair ? 2 * m_unit + static_cast<int>(rank) : m_unit; };

  // The j-th unit of this CTA's walk (-1 past the end). Static: a fixed
  // stride over the units. Dynamic: one thread (CTA 0's producer in a pair)
  // claims units from the launch's counter in ascending order and publishes
  // each in slot j of the unit ring (and of the peer's ring), where every
  // other role reads it; -1 ends the walk. Either way a unit's arithmetic is
  // the same, so the schedule changes no bit.
  const bool dyn = p.dynamic != 0;
  auto static_unit = [&](int j) {
    const long long u = first_unit + static_cast<long long>(j) * unit_stride;
    return u < p.n_units ? static_cast<int>(u) : -1;
  };
  auto ring_unit = [&](int j, int& u) -> bool {  // bounded wait for slot j
    if (!mbar_wait<kPair>(ufull_bar(j), static_cast<uint32_t>(j / kUnitSlots) & 1u, abort_flag,
                          p.status))
      return false;
    u = uring[j & (kUnitSlots - 1)];
    return true;
  };

  // The order in which the operand ring carries K blocks, which the producers
  // and the MMA issuer follow alike. Tiles come in the walk's order (a unit's
  // tiles, then the next unit's); tile t's blocks are issued in its own K
  // order. With p.interleave = X > 0 (same K everywhere, two accumulators),
  // tile t runs its blocks [lead, K - X) alone and then its last X blocks
  // one-to-one with the next tile's first X: the two accumulators' MMA chains
  // then overlap, while during a tile's solo blocks the epilogue drains the
  // other accumulator. X = 0 runs the tiles one after another. The order of
  // each tile's own MMAs, and so every bit, is the same either way.
  const int kb_total = (p.K + kBK - 1) / kBK;
  struct WalkTile {
    int u, idx, m_unit, n_first, n_count, j, vunit, seg, kb0, kb_n;
    bool k_down;
  };
  auto walk = [&](auto&& next_unit, auto&& on_stage) -> bool {
    int uj = 0;
    auto enter_unit = [&](WalkTile& t, int idx) -> bool {
      int u = -1;
      if (!next_unit(uj, u)) return false;
      ++uj;
      t.u = u;
      t.idx = idx;
      if (u < 0) return true;
      unit_coords(p, u, t.m_unit, t.n_first, t.n_count, t.vunit, t.seg);
      t.j = 0;
      t.kb0 = t.seg ? p.k_split : 0;
      t.kb_n = (p.k_split > 0 ? (t.seg ? kb_total : p.k_split) : kb_total) - t.kb0;
      // grad_weight walks K (the rows) downwards on odd waves (a wave: one
      // unit per CTA or pair of the grid), so a wave starts on the operand
      // rows the previous wave touched last, while they are still in L2.
      t.k_down = (E == (int)Epi::StoreF32T) && ((u / unit_stride) & 1);
      return true;
    };
    auto next_tile = [&](const WalkTile& t, WalkTile& n) -> bool {
      if (t.j + 1 < t.n_count) {
        n = t;
        ++n.j;
        ++n.idx;
        return true;
      }
      return enter_unit(n, t.idx + 1);
    };
    WalkTile a{}, b{};
    if (!enter_unit(a, 0)) return false;
    int lead = 0;  // blocks of tile a already issued beside its predecessor
    const int X = p.interleave;
    while (a.u >= 0) {
      for (int i = lead; i < a.kb_n - X; ++i)
        if (!on_stage(a, i)) return false;
      if (!next_tile(a, b)) return false;
      if (X > 0 && b.u >= 0) {
        for (int i = 0; i < X; ++i) {
          if (!on_stage(a, a.kb_n - X + i)) return false;
          if (!on_stage(b, i)) return false;
        }
        lead = X;
      } else {
        for (int i = a.kb_n - X; i < a.kb_n; ++i)
          if (!on_stage(a, i)) return false;
        lead = 0;
      }
      a = b;
    }
    return true;
  };

  // Output columns of a tile, and the B rows (of 64 K elements) this CTA
  // stages per stage: a wide pair's two 128-row halves, a pair's half of its
  // tile, or a single CTA's whole tile. A stage's bytes follow from them, and
  // the ring holds as many stages as fit (up to kMaxStages), so a narrow
  // tile keeps as many bytes in flight as a full one: its loads are
  // latency-bound, not MMA-bound.
  const int tile_n = kMode == kWideMode ? R::kTileN : p.tile_n;
  const int b_rows = kMode == kWideMode ? 2 * kBBoxRows : (kPair ? tile_n / 2 : tile_n);
  const uint32_t stage_tx = static_cast<uint32_t>(kABytes + b_rows * kBK * 2);
  const uint32_t stage_stride = (stage_tx + 1023u) & ~1023u;  // 1024-byte swizzle atoms
  const uint32_t n_st = min(static_cast<uint32_t>(kMaxStages), kRingBytes / stage_stride);

  // A short batch's A boxes fill only the first a_rows rows of each A tile
  // (single CTAs only): the rest is zeroed once, before any MMA reads it.
  const int a_rows = (!kPair && p.a_rows > 0) ? p.a_rows : kBM;
  if constexpr (!kPair) {
    if (a_rows < kBM) {
      const uint32_t n16 = static_cast<uint32_t>((kBM - a_rows) * 128 / 16);
      for (uint32_t i = threadIdx.x; i < n_st * n16; i += blockDim.x) {
        const uint32_t st = i / n16, j = i - st * n16;
        st_shared_v4(
            smem_base + st * stage_stride + static_cast<uint32_t>(a_rows) * 128u + 16u * j, 0u,
            0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(full_bar(s), 1);  // in a pair, only CTA 0's is used: one arrive, both CTAs' bytes
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      // every epilogue thread of the pair releases the accumulator to CTA 0
      // every epilogue thread of the pair (of each group) releases it
      mbar_init(tempty_bar(a), (kPair ? 256 : 128) * (kSplitHalvesFor<E, kMode> ? 2 : 1));
    }
    mbar_init(final_bar, 1);
    for (int j = 0; j < kUnitSlots; ++j) mbar_init(ufull_bar(j), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(xfull_bar(b), 128);
      mbar_init(xempty_bar(b), 128);
    }
    *abort_flag = 0;
    *peer_issued = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (E != (int)Epi::FwdStats) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (kPair) {
    __syncwarp();
    cluster_sync();  // the peer's barriers are initialised before any arrive on them
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  long long issued = 0;  // stage loads issued by this CTA's producer

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      const bool claims = dyn && (!kPair || rank == 0);
      // Slot j of the ring (and of the peer's) gets unit u.
      auto publish = [&](int j, int u) {
        const int s = j & (kUnitSlots - 1);
        uring[s] = u;
        mbar_arrive(ufull_bar(j));  // release: the slot's store before the phase
        if constexpr (kPair) {
          st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(uring + s)), 1),
                                static_cast<uint32_t>(u));
          mbar_arrive_remote_release(mapa_shared(ufull_bar(j), 1));
        }
      };
      // Each unit is published when the one before it starts, so the peer
      // CTA's producer knows it a whole unit before its first load (publishing
      // it at its own start cost short units, e.g. grad_weight at K = 512, a
      // fifth of their time), and claimed one unit earlier still, so the
      // atomic's latency hides behind the loads.
      int cur = -1, nxt = -1;
      if (claims) {
        cur = claim_unit(p);
        publish(0, cur);
        nxt = cur >= 0 ? claim_unit(p) : -1;
      }
      auto next_unit = [&](int uj, int& u) -> bool {
        if (!dyn) {
          u = static_unit(uj);
          return true;
        }
        if (!claims) return ring_unit(uj, u);
        u = cur;
        if (u >= 0) {
          publish(uj + 1, nxt);
          cur = nxt;
          nxt = cur >= 0 ? claim_unit(p) : -1;
        }
        return true;
      };
      auto load_stage = [&](const WalkTile& t, int i) -> bool {
        const int m_tile = cta_m_tile(t.m_unit);
        const int n_tile = t.n_first + t.j;
        const int kb = t.kb0 + (t.k_down ? t.kb_n - 1 - i : i);
        // first B row this CTA stages in each 256-column block: the whole
        // block alone, its half in a pair
        const int b_row0 =
            n_tile * tile_n + (kPair ? static_cast<int>(rank) * (b_rows / R::kNBlocks) : 0);
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) return false;
        const uint32_t sA = smem_base + stage * stage_stride;
        const uint32_t sB = sA + kABytes;
        // One arrive per stage, by CTA 0, expecting both CTAs' bytes; both
        // CTAs' boxes complete on CTA 0's barrier, issued in the pair form
        // (measured: CTA 0 issuing the plain form made the pair 10 % slower).
        if (rank == 0)
          mbar_arrive_expect_tx(full_bar(stage),
                                (kPair ? 2u : 1u) * stage_tx - (kBM - a_rows) * 128);
        const uint32_t fbar = kPair ? mapa_shared(full_bar(stage), 0) : full_bar(stage);
        auto load = [&](uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y) {
          if constexpr (kPair)
            tma_load_2d_pair(dst, map, fbar, x, y);
          else
            tma_load_2d(dst, map, fbar, x, y);
        };
        auto load_a = [&]() {
          if (p.a_mn) {  // [K][M]: two 64(M) x 64(K) boxes
#pragma unroll
            for (int q = 0; q < kBM / 64; ++q)
              load(sA + q * kMnBoxBytes, &tmA, m_tile * kBM + 64 * q, kb * kBK);
          } else {
            load(sA, &tmA, kb * kBK, m_tile * kBM);
          }
        };
        auto load_b = [&]() {
          constexpr int kBlockBytes = R::kBBytes / R::kNBlocks;
          // B rows of one N block this CTA stages (a multiple of 64, and
          // of 128 when B is K-major)
          const int block_rows = b_rows / R::kNBlocks;
#pragma unroll
          for (int nb = 0; nb < R::kNBlocks; ++nb) {
            const uint32_t dst = sB + nb * kBlockBytes;
            const int row = b_row0 + nb * kBN;
            if (p.b_mn) {  // [K][N]: 64(N) x 64(K) boxes
              for (int q = 0; q < block_rows / 64; ++q)
                load(dst + q * kMnBoxBytes, &tmB, row + 64 * q, kb * kBK);
            } else {  // [N][K]: 128-row boxes
              for (int q = 0; q < block_rows / kBBoxRows; ++q)
                load(dst + q * kBHalfBytes, &tmB, kb * kBK, row + kBBoxRows * q);
            }
          }
        };
        // The forward and dlogits stream W as B: B first, so the DRAM
        // loads start before A's (small, L2-resident, or for short batches
        // mostly out-of-bounds zero fill). The other contractions stream
        // A and measured faster with A first.
        if (E == (int)Epi::FwdStats || E == (int)Epi::DLogits) {
          load_b();
          load_a();
        } else {
          load_a();
          load_b();
        }
        ++issued;
        if (++stage == n_st) {
          stage = 0;
          phase ^= 1u;
        }
        return true;
      };
      ok = walk(next_unit, load_stage);
      if (kPair && rank != 0) {
        // CTA 0 drains this CTA's copies at the end; it needs their count
        st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(peer_issued)), 0),
                              static_cast<uint32_t>(issued));
      }
      if (!ok && !kPair) {
        // Drain: wait (bounded, ignoring the abort flag) for the copies this
        // thread issued, so none lands in shared memory after the CTA exits.
        volatile int no_abort = 0;
        const long long n = issued < n_st ? issued : n_st;
        uint32_t s = stage, ph = phase;
        for (long long i = 0; i < n; ++i) {
          if (s == 0) {
            s = n_st - 1;
            ph ^= 1u;
          } else {
            --s;
          }
          mbar_wait(full_bar(s), ph, &no_abort, p.status);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && (!kPair || rank == 0)) {
      // ------------------------------------------------------------ MMA issuer
      // one MMA covers the whole tile, or one 256-column block of a wide tile
      const uint32_t idesc = idesc_bf16_f32(kPair ? 2 * kBM : kBM,
                                            static_cast<uint32_t>(kMode == kWideMode ? kBN : tile_n),
                                            p.a_mn != 0, p.b_mn != 0);
      uint32_t stage = 0, phase = 0;
      auto next_unit = [&](int uj, int& u) -> bool {
        if (!dyn) {
          u = static_unit(uj);
          return true;
        }
        return ring_unit(uj, u);
      };
      // The MMAs of N block nb (one 256-column chain, into TMEM columns from
      // d_tmem) over the K block in stage st, block i of its tile.
      auto issue_chain = [&](uint32_t st, int i, int nb, uint32_t d_tmem) {
        const uint32_t sA = smem_base + st * stage_stride;
        const uint64_t adesc = p.a_mn ? sw128_mnmajor_desc(sA) : sw128_kmajor_desc(sA);
        const uint64_t bdesc =
            p.b_mn ? sw128_mnmajor_desc(sA + kABytes) : sw128_kmajor_desc(sA + kABytes);
        // One K=16 step: +32 bytes inside a K-major 128-byte row, or +16
        // rows of 128 bytes (two 8-row atoms) in an MN-major tile; in the
        // descriptor's 16-byte address units that is +2 or +128.
        const uint64_t astep = p.a_mn ? 128ull : 2ull;
        const uint64_t bstep = p.b_mn ? 128ull : 2ull;
        // a wide pair's second N block: its B half is the next kBlockBytes
        // of the stage (>> 4 in descriptor units), its columns the next 256
        constexpr uint64_t kBlockStep = (R::kBBytes / R::kNBlocks) >> 4;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint32_t accumulate = (i > 0 || k > 0) ? 1u : 0u;
          const uint64_t bd = bdesc + kBlockStep * nb + bstep * k;
          if constexpr (kPair)
            tc_mma_bf16_pair(d_tmem, adesc + astep * k, bd, idesc, accumulate);
          else
            tc_mma_bf16(d_tmem, adesc + astep * k, bd, idesc, accumulate);
        }
      };
      // Both N blocks of a wide tile over the K block in stage st, the two
      // chains alternating at every K step so that each MMA's predecessor in
      // its chain was issued two MMAs earlier.
      auto issue_both = [&](uint32_t st, int i) {
        const uint32_t sA = smem_base + st * stage_stride;
        const uint64_t adesc = p.a_mn ? sw128_mnmajor_desc(sA) : sw128_kmajor_desc(sA);
        const uint64_t bdesc =
            p.b_mn ? sw128_mnmajor_desc(sA + kABytes) : sw128_kmajor_desc(sA + kABytes);
        const uint64_t astep = p.a_mn ? 128ull : 2ull;
        const uint64_t bstep = p.b_mn ? 128ull : 2ull;
        constexpr uint64_t kBlockStep = (R::kBBytes / R::kNBlocks) >> 4;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint32_t accumulate = (i > 0 || k > 0) ? 1u : 0u;
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            const uint64_t bd = bdesc + kBlockStep * nb + bstep * k;
            if constexpr (kPair)
              tc_mma_bf16_pair(tmem_base + nb * kBN, adesc + astep * k, bd, idesc, accumulate);
            else
              tc_mma_bf16(tmem_base + nb * kBN, adesc + astep * k, bd, idesc, accumulate);
          }
        }
      };
      auto free_stage = [&](uint32_t st) {  // free in both CTAs once its MMAs have read it
        if constexpr (kPair)
          tc_commit_pair(empty_bar(st), 0x3);
        else
          tc_commit(empty_bar(st));
      };
      // Wide tiles: the epilogue releases the accumulator's two 256-column
      // halves one after the other (tempty 0, then 1), and each half is handed
      // to it on its own (tfull 0, then 1). A tile's N block 0 starts as soon
      // as half 0 is free; while half 1 is still being drained, its stages
      // are held after block 0's MMAs (at most the whole ring) and block 1
      // catches up on them once half 1 is free. A tile's last `skew` K blocks
      // also run block 0 first, their stages held: half 0 is handed over while
      // block 1's last MMAs run, so its drain overlaps them. Each chain keeps
      // its K order, so no value depends on it.
      const int skew = min(p.wide_skew, static_cast<int>(n_st) - 1);
      bool half1_free = false;
      int n_held = 0;
      uint32_t held_stage[kMaxStages];
      int held_block[kMaxStages];
      auto commit_half = [&](int h) {
        if constexpr (kPair)
          tc_commit_pair(tfull_bar(h), 0x3);
        else
          tc_commit(tfull_bar(h));
      };
      auto wide_stage = [&](const WalkTile& t, int i) -> bool {
        const uint32_t aph = static_cast<uint32_t>(t.idx) & 1u;
        if (i == 0) {
          if (!mbar_wait(tempty_bar(0), aph ^ 1u, abort_flag, p.status)) return false;
          half1_free = mbar_try_wait(tempty_bar(1), aph ^ 1u);
          tc_fence_after();
          n_held = 0;
        }
        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status)) return false;
        tc_fence_after();
        const bool last = i == t.kb_n - 1;
        const bool tail = i >= t.kb_n - skew;
        if (half1_free && !tail) {  // steady state: both chains, interleaved
          issue_both(stage, i);
          free_stage(stage);
          if (++stage == n_st) {
            stage = 0;
            phase ^= 1u;
          }
          if (last) {
            commit_half(0);
            commit_half(1);
          }
          return true;
        }
        // N block 0 alone, the stage held for block 1
        issue_chain(stage, i, 0, tmem_base);
        held_stage[n_held] = stage;
        held_block[n_held] = i;
        ++n_held;
        if (++stage == n_st) {
          stage = 0;
          phase ^= 1u;
        }
        if (last) commit_half(0);
        // block 1 must catch up at the tile's end, or when every stage is held
        const bool must = last || n_held >= static_cast<int>(n_st);
        if (!half1_free) {
          if (mbar_try_wait(tempty_bar(1), aph ^ 1u)) {
            half1_free = true;
          } else if (must) {
            if (!mbar_wait(tempty_bar(1), aph ^ 1u, abort_flag, p.status)) return false;
            half1_free = true;
          }
          if (half1_free) tc_fence_after();
        }
        if (half1_free && (!tail || must)) {
          for (int h = 0; h < n_held; ++h) {
            issue_chain(held_stage[h], held_block[h], 1, tmem_base + kBN);
            free_stage(held_stage[h]);
          }
          n_held = 0;
        }
        if (last) commit_half(1);
        return true;
      };
      // One K block of tile t: its accumulator is t.idx % kAccs; the first
      // block waits until the epilogue has released that accumulator, and
      // the last hands it to the epilogue.
      auto mma_stage = [&](const WalkTile& t, int i) -> bool {
        if constexpr (kMode == kWideMode) return wide_stage(t, i);
        const uint32_t acc = static_cast<uint32_t>(t.idx) % R::kAccs;
        if (i == 0) {
          const uint32_t aph = (static_cast<uint32_t>(t.idx) / R::kAccs) & 1u;
          if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, p.status)) return false;
          tc_fence_after();
        }
        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status)) return false;
        tc_fence_after();
        issue_chain(stage, i, 0, tmem_base + acc * kBN);
        free_stage(stage);
        if (++stage == n_st) {
          stage = 0;
          phase ^= 1u;
        }
        if (i == t.kb_n - 1) {
          if constexpr (kPair)
            tc_commit_pair(tfull_bar(acc), 0x3);
          else
            tc_commit(tfull_bar(acc));
        }
        return true;
      };
      walk(next_unit, mma_stage);
      // All MMAs issued by this thread must finish before TMEM is released
      // (in both CTAs of a pair).
      volatile int no_abort = 0;
      if constexpr (kPair)
        tc_commit_pair(final_bar, 0x3);
      else
        tc_commit(final_bar);
      mbar_wait(final_bar, 0, &no_abort, p.status);
    } else if (kPair && lane == 0) {
      // CTA 0's MMAs read this CTA's shared memory and write its TMEM: wait
      // for their final commit before either is released.
      volatile int no_abort = 0;
      mbar_wait(final_bar, 0, &no_abort, p.status);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // Two groups of four warps (threads 64-191 and 192-319). On a wide tile
    // of the forward or a bf16 store, group g drains the accumulator's
    // 256-column half g and hands it back to the MMA issuer on its own, so
    // the halves drain at the same time. Otherwise group 0 drains every tile
    // (on a wide tile, half 0 first, handed back as soon as it is read) and
    // group 1 has no work: the fp32 stores keep two staging buffers per warp
    // that way, and their long K leaves little to overlap.
    // Control flow is uniform within a group: the group's thread 0 does the
    // bounded wait for each accumulator and publishes the outcome, so no
    // thread can be left waiting at a named barrier the others skipped.
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    const int grp = (warp - 2) >> 2;
    const int gtid = (threadIdx.x - 64) & 127;  // thread within the group
    const uint32_t grp_bar = kEpiBarrier + static_cast<uint32_t>(grp);
    constexpr bool kSplitHalves = kSplitHalvesFor<E, kMode>;
    constexpr int kGroups = kSplitHalves ? 2 : 1;
    // each warp's staging: a quarter of a group's share of the 32 KB
    const uint32_t warp_staging =
        staging + static_cast<uint32_t>(grp * 4 + q) * (kStagingTotal / (4 * kGroups));
    uint32_t it = 0, chunk_ctr = 0;
    bool ok = grp < kGroups;
    for (int uj = 0; ok; ++uj) {
      int u;
      if (!dyn) {
        u = static_unit(uj);
      } else {
        // the group's thread 0 reads the slot (bounded) and shares it: -2 = gave up
        if (gtid == 0) {
          int v = -1;
          epi_unit[grp * 2 + (uj & 1)] = ring_unit(uj, v) ? v : -2;
        }
        named_barrier(grp_bar, 128);
        u = epi_unit[grp * 2 + (uj & 1)];
        if (u == -2) {
          ok = false;
          break;
        }
      }
      if (u < 0) break;
      int m_unit, n_first, n_count, vunit, seg;
      unit_coords(p, u, m_unit, n_first, n_count, vunit, seg);
      const int m_tile = cta_m_tile(m_unit);
      const int row = m_tile * kBM + row_in_tile;
      const bool row_ok = row < p.M;
      // a pair's second half can lie wholly past the last row: nothing to store
      const bool tile_live = m_tile * kBM < p.M;

      // per-row constants
      int lab = -1;
      float lse2 = 0.f, gs = 0.f, c0 = 0.f, c1 = 0.f;
      if constexpr (E == (int)Epi::FwdStats || E == (int)Epi::DLogits) {
        if (row_ok) {
          // the label as a column of this launch (a vocab shard starts at
          // label_base); anything outside [0, N) is out of vocabulary here
          const int64_t l = static_cast<int64_t>(p.labels[row]) - p.label_base;
          lab = (l >= 0 && l < p.N) ? static_cast<int>(l) : -1;
        }
      }
      if constexpr (E == (int)Epi::DLogits) {
        if (row_ok) {
          // dl = s * (g * onehot - p * (g + gH * (z - lse + H))), z - lse = ln2 * t
          // with t = y - lse2: the coefficient of p is c0 + c1 * t.
          const float g = p.grad ? p.grad[row] : 0.f;
          const float ge = p.grad_ent ? p.grad_ent[row] : 0.f;
          lse2 = __fmul_rn(p.lse[row], kLog2e);
          gs = __fmul_rn(g, p.inv_temp);
          c0 = __fmul_rn(p.inv_temp, p.grad_ent ? __fmaf_rn(ge, p.ent[row], g) : g);
          c1 = __fmul_rn(__fmul_rn(p.inv_temp, ge), kLn2);
        }
      }
      // The forward folds a row's vocabulary unit as two streams, the even
      // and the odd 128-column blocks, and merges them at the unit's end: the
      // same on every engine. sb is the stream being folded (parity cur_par);
      // a single group swaps the two as the parity changes (register moves,
      // so neither lives in local memory).
      OnlineStat sb = stat_empty(), sb_other = stat_empty();
      int cur_par = 0;
      float zl = __int_as_float(0x7fc00000);  // NaN until the label column is seen

      for (int j = 0; j < n_count; ++j, ++it) {
        const int n_tile = n_first + j;
        const uint32_t acc = it % R::kAccs;
        const uint32_t aph = (it / R::kAccs) & 1u;
        volatile int* go = epi_go + grp * 2;
        if (gtid == 0) go[it & 1u] = mbar_wait(tfull_bar(acc), aph, abort_flag, p.status) ? 1 : 0;
        named_barrier(grp_bar, 128);
        if (!go[it & 1u]) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN;
        // This group's 32-column chunks, in order: on a wide tile split
        // between two groups, four of half 0 (group g: chunks 4g..4g+3) and
        // then the matching four of half 1, so that half 0 is read, and
        // handed back, after half the drain; otherwise every chunk.
        const int n_iter = kSplitHalves ? 8 : tile_n / 32;
        // hand columns back to the MMA issuer (CTA 0 of a pair): the
        // accumulator, or one 256-column half of a wide one
        auto release = [&](uint32_t bar) {
          tc_fence_before();
          if constexpr (kPair)
            mbar_arrive_remote(mapa_shared(tempty_bar(bar), 0));
          else
            mbar_arrive(tempty_bar(bar));
        };
        bool half0_released = false;
        bool half1_handed = false;  // this tile's tfull(1) has been waited for
        // wait (the group's thread 0, bounded) for half 1's hand-over
        auto wait_half1 = [&]() -> bool {
          volatile int* go1 = epi_go1 + grp * 2;
          if (gtid == 0) go1[it & 1u] = mbar_wait(tfull_bar(1), aph, abort_flag, p.status) ? 1 : 0;
          named_barrier(grp_bar, 128);
          half1_handed = true;
          if (!go1[it & 1u]) return false;
          tc_fence_after();
          return true;
        };
        // the forward's stream: on 256-column tiles the tile's block parity
        // in the unit (a unit starts on a block), on a wide tile the group's
        // own (half g of tile j is block 2j + g)
#pragma unroll 1
        for (int ci = 0; ci < n_iter; ++ci) {
          const int c = kSplitHalves ? (ci >> 2) * (kBN / 32) + 4 * grp + (ci & 3) : ci;
          const int col0 = n_tile * tile_n + c * 32;
          if (col0 >= p.N) break;  // uniform over the CTA
          // A store epilogue stages nothing for a tile wholly past the last
          // row (a pair's second half): every staged chunk is then a
          // committed store, which the staging buffers' reuse wait counts on.
          // (Staging such a tile without storing it let its chunks overwrite
          // a buffer that the last live store was still reading.)
          if (E != (int)Epi::FwdStats && !tile_live) break;
          if constexpr (kMode == kWideMode) {
            // half 1 is handed over on its own, after half 0
            if ((kSplitHalves ? ci == 4 : c == kBN / 32) && !wait_half1()) {
              ok = false;
              break;
            }
          }
          const int nvalid = min(32, p.N - col0);
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          if constexpr (kMode == kWideMode) {
            // the first half has been read (by this group)
            if (kSplitHalves ? ci == 3 : c == kBN / 32 - 1) {
              release(0);
              half0_released = true;
            }
          }

          if constexpr (E == (int)Epi::FwdStats) {
            // The stream of this chunk: its 128-column block's parity in the
            // unit. A group of a split wide tile sees one parity only.
            if constexpr (!kSplitHalves) {
              const int par = ((col0 - n_first * tile_n) >> 7) & 1;
              if (par != cur_par) {
                const OnlineStat t = sb;
                sb = sb_other;
                sb_other = t;
                cur_par = par;
              }
            }
            // y = acc * scale2 (the temperature and log2(e)), folded into
            // the statistics' shift; the label's y is formed on its own. The
            // sum of p^2 is accumulated only when a plane for it was given
            // (m, s and u do not depend on it).
            if (p.part_q) {
              if (nvalid == 32)
                stat_fold_scaled<32, true>(sb, v, p.scale2);
              else
                stat_fold_scaled<32, true>(sb, v, p.scale2, nvalid);
            } else {
              if (nvalid == 32)
                stat_fold_scaled<32, false>(sb, v, p.scale2);
              else
                stat_fold_scaled<32, false>(sb, v, p.scale2, nvalid);
            }
            const int rel = lab - col0;
            if (__any_sync(0xffffffffu, rel >= 0 && rel < nvalid)) {
#pragma unroll
              for (int i = 0; i < 32; ++i) zl = (i == rel) ? __fmul_rn(v[i], p.scale2) : zl;
            }
          } else {
            if constexpr (E == (int)Epi::DLogits) {
              // per value: t = y - lse2, p = 2^t, dl = -p * (c1 * t + c0) (+ gs
              // at the label); pairs of values share each packed operation,
              // and -(p * coef) is p * (-c1 * t - c0) exactly.
              const int rel = lab - col0;
              const f32x2 sc2 = f2_pack(p.scale2, p.scale2), nl2 = f2_pack(-lse2, -lse2);
              const f32x2 nc1 = f2_pack(-c1, -c1), nc0 = f2_pack(-c0, -c0);
              if (p.grad_ent) {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                  const f32x2 t2 = f2_fma(f2_pack(v[i], v[i + 1]), sc2, nl2);
                  float ta, tb;
                  f2_unpack(t2, ta, tb);
                  const f32x2 d2 = f2_mul(f2_pack(ex2(ta), ex2(tb)), f2_fma(nc1, t2, nc0));
                  f2_unpack(d2, v[i], v[i + 1]);
                }
              } else {
                // no entropy term: the coefficient is the constant -c0
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                  float ta, tb;
                  f2_unpack(f2_fma(f2_pack(v[i], v[i + 1]), sc2, nl2), ta, tb);
                  const f32x2 d2 = f2_mul(f2_pack(ex2(ta), ex2(tb)), nc0);
                  f2_unpack(d2, v[i], v[i + 1]);
                }
              }
              // the one-hot term, in the rare chunks that hold some row's label
              if (__any_sync(0xffffffffu, static_cast<unsigned>(rel) < 32u)) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (i == rel) v[i] = __fadd_rn(v[i], gs);
              }
            }
            // Each warp stages its 32 rows of the chunk and its lane 0 stores
            // them with one TMA bulk store (or reduce-add) of a 32 x 32 box;
            // rows and columns outside the output are clipped. No barrier
            // across the warps: a warp reuses a buffer once its own store from
            // that buffer (kBufs chunks back) has read it.
            // bf16: each warp stages its 32 rows of the chunk and its lane 0
            // stores them with one TMA bulk store of a 32 x 32 box, with no
            // barrier across the warps (a warp reuses a buffer once its own
            // store from it, kBufs chunks back, has read it). fp32: the group
            // stages the whole 128 x 32 chunk in one of two buffers and its
            // thread 0 stores (or reduce-adds) it, which measured 5 % faster
            // than 32-row boxes for a short grad_weight. Rows and columns
            // outside the output are clipped.
            constexpr bool kBf16Out = E == (int)Epi::DLogits || E == (int)Epi::StoreBf16;
            if constexpr (kBf16Out) {
              constexpr uint32_t kBufBytes = 32 * 64;
              constexpr uint32_t kBufs = kStagingTotal / (4 * kGroups) / kBufBytes;
              const uint32_t buf = warp_staging + (chunk_ctr % kBufs) * kBufBytes;
              if (lane == 0) bulk_wait_group_read<kBufs - 1>();
              __syncwarp();
              stage_row_bf16(buf, lane, v);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                const int r0 = m_tile * kBM + q * 32;
                tma_store_2d(&tmC, buf, col0, r0 + seg * p.seg_rows);
                bulk_commit_group();
              }
            } else {
              const uint32_t buf = staging + (chunk_ctr & 1u) * kStagingBytes;
              if (gtid == 0) bulk_wait_group_read<1>();  // this buffer's last store has read it
              named_barrier(grp_bar, 128);
              if constexpr (E == (int)Epi::StoreF32)
                stage_row_f32(buf, row_in_tile, v);
              else
                stage_col_f32(buf, row_in_tile, v);
              fence_proxy_async_smem();
              named_barrier(grp_bar, 128);
              if (gtid == 0) {
                // (x, y) of the box in the output: transposed for StoreF32T
                const int ox = E == (int)Epi::StoreF32T ? m_tile * kBM : col0;
                const int oy = E == (int)Epi::StoreF32T ? col0 : m_tile * kBM + seg * p.seg_rows;
                if (p.accumulate)
                  tma_reduce_add_2d(&tmC, buf, ox, oy);
                else
                  tma_store_2d(&tmC, buf, ox, oy);
                bulk_commit_group();
              }
            }
            ++chunk_ctr;
          }
        }
        if constexpr (kMode == kWideMode) {
          // Half 1 goes back only after its own hand-over, read or not. A
          // group that read none of it (a pair half past the last row, or
          // columns past N) could otherwise reach the next tile, whose half 0
          // may be handed over before this tile's half 1 is free, and arrive
          // on tempty 1 again before its peer CTA arrived for this tile: the
          // two arrivals would complete the phase while the peer still reads.
          if (ok && !half1_handed && !wait_half1()) ok = false;
          if (!half0_released) release(0);
          release(1);
        } else {
          release(acc);
        }
        if (!ok) break;
      }
      if (!ok) break;

      if constexpr (E == (int)Epi::FwdStats) {
        // a single group: sb holds the stream of parity cur_par
        OnlineStat all = cur_par ? sb_other : sb;
        OnlineStat odd = cur_par ? sb : sb_other;
        if constexpr (kSplitHalves) {
          // Group 1 (the odd blocks) hands its stream to group 0 through one
          // of two shared-memory buffers (in the staging area, which the
          // forward does not store through). Each buffer has a full and an
          // empty barrier; a group's thread 0 waits on it (bounded) and
          // shares the outcome over the group's named barrier.
          const int b = uj & 1;
          const uint32_t xph = static_cast<uint32_t>(uj >> 1) & 1u;
          float* xrow = reinterpret_cast<float*>(smem + kRingBytes) + b * (kBM * 5) + row_in_tile * 5;
          if (grp == 1) {
            if (gtid == 0) x_go[1] = mbar_wait(xempty_bar(b), xph ^ 1u, abort_flag, p.status) ? 1 : 0;
            named_barrier(grp_bar, 128);
            if (!x_go[1]) break;
            xrow[0] = sb.m;
            xrow[1] = sb.s;
            xrow[2] = sb.u;
            xrow[3] = sb.q;
            xrow[4] = zl;
            mbar_arrive(xfull_bar(b));  // release: this thread's row is written
            continue;
          }
          if (gtid == 0) x_go[0] = mbar_wait(xfull_bar(b), xph, abort_flag, p.status) ? 1 : 0;
          named_barrier(grp_bar, 128);
          if (!x_go[0]) break;
          odd = OnlineStat{xrow[0], xrow[1], xrow[2], xrow[3]};
          const float zl_odd = xrow[4];
          mbar_arrive(xempty_bar(b));  // this thread has read its row
          // the label's 128-column block decides whose capture holds its logit
          if (lab >= 0 && ((lab >> 7) & 1)) zl = zl_odd;
        }
        if (p.part_q)
          stat_merge<true>(all, odd);
        else
          stat_merge<false>(all, odd);
        if (row_ok) {
          const int64_t o = static_cast<int64_t>(vunit) * p.part_ld + row;
          p.part_m[o] = all.m;
          p.part_s[o] = all.s;
          p.part_u[o] = all.u;
          if (p.part_q) p.part_q[o] = all.q;
          const int c0 = n_first * tile_n;
          const int c1 = min(p.N, (n_first + n_count) * tile_n);
          if (lab >= c0 && lab < c1) p.part_zl[row] = zl;
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();  // every output store of this warp has completed
  }

  tc_fence_before();
  if constexpr (kPair) {
    // Neither CTA leaves (or frees TMEM) while the other may still touch its
    // barriers, shared memory or TMEM. Between the two cluster barriers CTA 0
    // waits for every stage load still in flight in either CTA: all loads
    // before the last n_st of the further-ahead producer were consumed by MMAs,
    // so their phases completed. A phase one CTA never loaded gets that
    // CTA's share settled here (CTA 0's arrive, or CTA 1's bytes as done),
    // so it completes when the other's bytes land. Each wait is bounded.
    __syncwarp();
    cluster_sync();
    if (rank == 0 && warp == 0 && lane == 0) {
      const long long n0 = issued, n1 = static_cast<long long>(*peer_issued);
      const long long hi = n0 > n1 ? n0 : n1;
      volatile int no_abort = 0;
      for (long long i = hi > n_st ? hi - n_st : 0; i < hi; ++i) {
        const int s = static_cast<int>(i % n_st);
        const uint32_t par = static_cast<uint32_t>((i / n_st) & 1);
        if (i < n0 && i >= n1)
          mbar_complete_tx(full_bar(s), stage_tx);
        else if (i >= n0 && i < n1)
          mbar_arrive_expect_tx(full_bar(s), stage_tx);
        mbar_wait(full_bar(s), par, &no_abort, p.status);
      }
    }
    __syncwarp();
    cluster_sync();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int E>
__global__ void __launch_bounds__(kGemmThreadsOneGroup, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  gemm_body<E, kSingle>(tmA, tmB, tmC, p);
}

// kMode: kPairMode or kWideMode
template <int E, int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsFor<E, kMode>, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  gemm_body<E, kMode>(tmA, tmB, tmC, p);
}

// Clusters of two that fit on the device at once (one CTA per SM), per
// device; 0 when none does (the caller then runs single CTAs). The cache is
// shared by host threads: any of them may fill a slot, with the same value.
template <int E, int kMode>
int pair_slots(int num_sms) {
  static std::atomic<int> cached[16];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 16) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  if (cudaFuncSetAttribute(gemm_tc_pair_kernel<E, kMode>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Ring<kMode>::kSmemBytes) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
  cfg.blockDim = dim3(kThreadsFor<E, kMode>);
  cfg.dynamicSmemBytes = Ring<kMode>::kSmemBytes;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_pair_kernel<E, kMode>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  n = n < num_sms / 2 ? n : num_sms / 2;
  if (dev >= 0 && dev < 16) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// `lanes`: the most CTAs (single) or CTA pairs of the persistent grid.
template <int E, int kMode>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                       const GemmParams& p, int lanes, cudaStream_t stream) {
  cudaError_t e;
  if constexpr (kMode != kSingle) {
    // Set on every launch: the attribute belongs to the current device's context.
    e = cudaFuncSetAttribute(gemm_tc_pair_kernel<E, kMode>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Ring<kMode>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (lanes <= 0) return cudaErrorInvalidConfiguration;  // launch_gemm checked it first
    const int clusters = p.n_units < lanes ? p.n_units : lanes;  // persistent
    gemm_tc_pair_kernel<E, kMode>
        <<<2 * clusters, kThreadsFor<E, kMode>, Ring<kMode>::kSmemBytes, stream>>>(a, b, c, p);
  } else {
    e = cudaFuncSetAttribute(gemm_tc_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Ring<kSingle>::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = p.n_units < lanes ? p.n_units : lanes;  // persistent: <= one CTA per SM
    gemm_tc_kernel<E><<<grid, kGemmThreadsOneGroup, Ring<kSingle>::kSmemBytes, stream>>>(a, b, c, p);
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

// The store epilogues (grad_hidden, grad_weight, the bare engine GEMM), whose
// engine and tile width are chosen by cost and can be forced.
template <int E>
constexpr bool kStoreEpi = !(E == (int)Epi::FwdStats || E == (int)Epi::DLogits);

template <int E>
int slots_for(int mode, int num_sms) {
  if (mode == kPairMode) return pair_slots<E, kPairMode>(num_sms);
  if (mode == kWideMode) return pair_slots<E, kWideMode>(num_sms);
  return 0;
}

template <int E>
cudaError_t launch_mode(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                        const GemmParams& p, int mode, int lanes, cudaStream_t stream) {
  if (mode == kPairMode) return launch_one<E, kPairMode>(a, b, c, p, lanes, stream);
  if (mode == kWideMode) return launch_one<E, kWideMode>(a, b, c, p, lanes, stream);
  return launch_one<E, kSingle>(a, b, c, p, lanes, stream);
}

// An engine and tile width for one launch.
struct Engine {
  int mode, tile_n;
};

// Estimated time of a launch on engine `g` whose K loop dominates (grad_hidden,
// K = V): waves of units over the SMs (or cluster slots), times the time of one
// wave. The wave times are measured, not modelled: alone on a GB300, one wave
// of grad_hidden at H = 3584, V = 152064 took (ms) single CTAs 0.653 (64
// columns), 0.686 (128), 0.80 (192), 0.88 (256); pairs 0.697 (128), 0.72
// (256); wide pairs 1.258 (512). A narrow tile does a quarter of a full one's
// work in three quarters of its time: its K steps are bound by operand
// delivery, not by the MMAs. The costs below are those times over 0.88.
// With a K split, every tile is two units of half the K loop each.
double engine_cost(const Engine& g, long long m_tiles, long long n, int num_sms, int slots,
                   int segs = 1) {
  const long long rows = g.mode == kSingle ? 1 : 2;
  const long long m_units = (m_tiles + rows - 1) / rows;
  const long long units = m_units * ((n + g.tile_n - 1) / g.tile_n) * segs;
  const long long lanes = g.mode == kSingle ? num_sms : slots;
  if (lanes <= 0) return 1e30;
  const long long waves = (units + lanes - 1) / lanes;
  double wave;
  if (g.mode == kWideMode)
    wave = 1.43;
  else if (g.mode == kPairMode)
    wave = g.tile_n == 128 ? 0.79 : 0.82;
  else
    wave = g.tile_n == 64 ? 0.74 : g.tile_n == 128 ? 0.78 : g.tile_n == 192 ? 0.91 : 1.0;
  return static_cast<double>(waves) * wave / segs;
}

// CTAs that a launch of engine g keeps busy: one per unit (two per pair
// unit), at most one wave.
long long engine_ctas(const Engine& g, long long m_tiles, long long n, int num_sms, int slots,
                      int segs = 1) {
  const long long rows = g.mode == kSingle ? 1 : 2;
  const long long m_units = (m_tiles + rows - 1) / rows;
  const long long units = m_units * ((n + g.tile_n - 1) / g.tile_n) * segs;
  const long long lanes = g.mode == kSingle ? num_sms : slots;
  return (units < lanes ? units : lanes) * rows;
}

template <int E>
cudaError_t launch_gemm_e(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                          GemmParams p, int tiles_per_unit, int num_sms, cudaStream_t stream) {
  // Engine per contraction. The forward and dlogits (K = H) run on CTA
  // pairs for an even number of m tiles (alone at H = 3584, V = 152064,
  // 256-wide pairs against single CTAs, forward: -8.5 % at 129 rows, -2 % at
  // 2048; dlogits: -11 % at 512 rows, -3.5 % at 4096), and for an odd number
  // above 32, where the pair half past the last row costs little (forward on
  // 3 m tiles: +14 %, on 9: +4.5 %). Among pairs they take wide ones: a wide
  // pair stages a quarter fewer operand bytes per flop, which the 256-wide
  // pairs' tensor pipe was waiting on (76-79 % busy at V = 32000 against 87 %
  // wide), and that outweighs its epilogue no longer overlapping the next
  // tile. Alone, 256-wide / wide (ms): forward 0.335 / 0.315 at 512 rows,
  // 1.237 / 1.147 at 2048, 2.434 / 2.247 at 4096, 9.86-10.03 / 9.24-9.30 at
  // 16384, 0.618 / 0.571 at 4096 x 4096 x 32000, even at 256 rows; dlogits
  // 0.347 / 0.343 at 512, 1.242 / 1.220 at 2048, 2.59 / 2.52 at 4096,
  // 10.97-11.09 / 10.63-10.75 at 16384; the short step 396-402k / 408-417k
  // tokens/s.
  // grad_weight and grad_hidden take the engines below; at the 16384 x 3584 x
  // 152064 step, which runs at the power cap, both are on wide pairs (kernels
  // -6 % and -13 %, step -1.4 % and -1.8 %). A pair needs two m tiles: a
  // launch with a single 128-row m tile runs on single CTAs, which keep every
  // SM busy instead of leaving half of each pair idle.
  const int m_tiles = (p.M + kBM - 1) / kBM;
  const int env = gemm_pair_mode();
  Engine g{kSingle, kBN};
  if (env == 1 && m_tiles >= 2) {
    g = Engine{kWideMode, 2 * kBN};
  } else if (env == 2 && m_tiles >= 2) {
    g = Engine{kPairMode, kBN};
  } else if (env < 0 && E == (int)Epi::StoreF32T) {
    // grad_weight (K = the chunk's rows): 256-wide pairs, whose epilogue
    // overlaps the next tile's MMAs, while K is short enough for the fp32
    // output's stores to matter; wide pairs from 2048 rows. Alone at H =
    // 3584, V = 152064 (ms, pairs / wide): 0.34 / 0.36 at 128 rows, 0.44 /
    // 0.54 at 512, 0.69 / 0.79 at 1024, 1.29 / 1.28 at 2048, 2.62 / 2.50 at
    // 4096, 5.47 / 5.01 at 8192. Beside grad_hidden (corun) wide pairs
    // again: whole backward 0.741 / 0.737 ms at 128 rows, 1.154 / 1.131 at
    // 512, 1.960 / 1.931 at 1024.
    if (m_tiles >= 2)
      g = (p.K < 2048 && !p.corun) ? Engine{kPairMode, kBN} : Engine{kWideMode, 2 * kBN};
  } else if (env < 0 && kStoreEpi<E>) {
    // grad_hidden and the bare engine GEMM: the cheapest engine by
    // engine_cost (pairs only over two or more m tiles). Narrower tiles need
    // an MN-major B (64-column boxes); each output element's K walk is the
    // same on all of them.
    const int wide_slots = m_tiles >= 2 ? slots_for<E>(kWideMode, num_sms) : 0;
    const int pair_slots_n = m_tiles >= 2 ? slots_for<E>(kPairMode, num_sms) : 0;
    const Engine cand[7] = {{kWideMode, 2 * kBN}, {kPairMode, kBN}, {kSingle, kBN},
                            {kPairMode, 128},     {kSingle, 192},  {kSingle, 128},
                            {kSingle, 64}};
    const int n_cand = p.b_mn ? 7 : 3;
    const int segs = p.k_split > 0 ? 2 : 1;
    double best = 1e30, best_half = 1e30;
    Engine half = g;
    for (int i = 0; i < n_cand; ++i) {
      const int slots = cand[i].mode == kWideMode ? wide_slots : pair_slots_n;
      const double cost = engine_cost(cand[i], m_tiles, p.N, num_sms, slots, segs);
      if (cost < best * 0.999) {
        best = cost;
        g = cand[i];
      }
      if (cost < best_half * 0.999 &&
          2 * engine_ctas(cand[i], m_tiles, p.N, num_sms, slots, segs) <= num_sms) {
        best_half = cost;
        half = cand[i];
      }
    }
    // Beside grad_weight (corun), grad_hidden of a short batch gives up some
    // speed for SMs: alone at H = 3584, V = 152064, whole backward with the
    // two side by side (ms): 128 rows, 64-column tiles on 112 CTAs 0.826,
    // 128-column on 56 CTAs 0.766; 512 rows, 256-wide pairs on 112 SMs 1.185,
    // wide pairs on 56 SMs 1.101 (alone the wide pairs take 0.644 ms against
    // 0.418).
    if (p.corun && best_half <= 2.0 * best) g = half;
  } else if (env < 0 && (E == (int)Epi::FwdStats || E == (int)Epi::DLogits) && m_tiles >= 2 &&
             (m_tiles % 2 == 0 || m_tiles > 32)) {
    g = Engine{kWideMode, 2 * kBN};
  }
  // LMH_GEMM_STORE_ENGINE forces the store contractions' engine and width
  if constexpr (kStoreEpi<E>) {
    int fm = -1, fn = 0;
    gemm_store_engine(&fm, &fn);
    if (fm == kSingle || (fm >= 0 && m_tiles >= 2)) {
      g = Engine{fm, fn};
      if (!p.b_mn && fm != kWideMode) g.tile_n = kBN;  // narrow tiles need an MN-major B
    }
  }
  // no room for a cluster of two (a partitioned GPU, say): single CTAs, which
  // give the same bits
  if (g.mode != kSingle && slots_for<E>(g.mode, num_sms) <= 0) g = Engine{kSingle, kBN};
  if (g.mode == kWideMode) g.tile_n = 2 * kBN;
  if (E == (int)Epi::FwdStats && g.tile_n != kBN && !(g.mode == kWideMode && g.tile_n == 2 * kBN))
    return cudaErrorInvalidValue;  // chunk grid: 1024-column chunks of whole tiles
  const int kb_total = (p.K + kBK - 1) / kBK;
  if (p.k_split != 0 && (!(E == (int)Epi::StoreF32 || E == (int)Epi::StoreBf16) || p.k_split < 0 ||
                         p.k_split >= kb_total || p.seg_rows < (p.M + kBM - 1) / kBM * kBM))
    return cudaErrorInvalidValue;  // a K split: two non-empty segments, partials apart
  if (g.mode != kWideMode && g.tile_n != kBN &&
      (!p.b_mn || g.tile_n % 64 != 0 || (g.mode == kPairMode && g.tile_n != 128)))
    return cudaErrorInvalidValue;  // narrow tiles need 64-column MN-major B boxes
  const int m_rows = g.mode != kSingle ? 2 * kBM : kBM;
  p.tile_n = g.mode == kWideMode ? 0 : g.tile_n;
  p.n_m_tiles = (p.M + m_rows - 1) / m_rows;
  p.n_n_tiles = (p.N + g.tile_n - 1) / g.tile_n;
  // a vocab unit keeps its columns on wider tiles (the forward's 1024-column
  // chunk is two 512-column wide tiles)
  if (tiles_per_unit * kBN % g.tile_n == 0 && g.tile_n > kBN)
    tiles_per_unit = tiles_per_unit * kBN / g.tile_n;
  p.tiles_per_unit = tiles_per_unit;
  const int all_vunits = (p.n_n_tiles + tiles_per_unit - 1) / tiles_per_unit;
  const int vu_end = (p.vunit_end > 0 && p.vunit_end < all_vunits) ? p.vunit_end : all_vunits;
  if (p.vunit_begin < 0 || p.vunit_begin > vu_end) return cudaErrorInvalidValue;
  p.n_vunits = vu_end - p.vunit_begin;
  // Unit indices are int on the device; sizes whose unit count does not fit
  // are refused (they would need terabytes of workspace anyway).
  const long long units =
      static_cast<long long>(p.n_m_tiles) * p.n_vunits * (p.k_split > 0 ? 2 : 1);
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.n_units = static_cast<int>(units);
  // Rows per raster group, per contraction (same-session sweep of 4/8/16/32
  // 128-row m tiles on the Qwen-like step; 1, 2 and 4 again for grad_hidden):
  // the N = V contractions (forward, dlogits) share W tiles across more m
  // tiles, the K = V grad_hidden (bf16 out, or its K halves in fp32) prefers
  // small groups. A pair's m unit is two m tiles.
  const int group_tiles = (E == (int)Epi::FwdStats || E == (int)Epi::DLogits ||
                           E == (int)Epi::StoreF32T)
                              ? 32
                              : ((E == (int)Epi::StoreBf16 || p.k_split > 0) ? 4 : 8);
  p.group_m = g.mode != kSingle ? group_tiles / 2 : group_tiles;
  if (p.n_units <= 0) return cudaSuccess;
  // Schedule. A static stride lets CTA pairs drift apart: at 16384 x 3584 x
  // 152064 the pairs sharing a W tile started 13-35 us apart in the first
  // quarter of the forward and 140-300 us (2-4 units) apart in the last,
  // where single CTAs stayed within 15 us; the forward read W about 12 times
  // instead of once per raster group, and the slowest pair set the end. A
  // launch of several waves therefore claims units from a counter in
  // ascending order, which keeps concurrent units together and balances the
  // tail.
  // grad_weight keeps the fixed stride while K (the chunk's rows) is short:
  // its units are then a few microseconds of MMAs behind a long fp32 store,
  // and claimed units measured slower (alone at H = 3584, V = 152064, ms,
  // fixed / claimed: 0.446 / 0.540 at 512 rows, 0.689 / 0.774 at 1024, 1.279 /
  // 1.290 at 2048; 9.60-9.65 / 9.19-9.26 at 16384).
  int sched_mode = -1, grid_cap = 0;
  gemm_schedule(&sched_mode, &grid_cap);
  int lanes = g.mode == kSingle ? num_sms : slots_for<E>(g.mode, num_sms);
  if (grid_cap > 0 && grid_cap < lanes) lanes = grid_cap;
  const bool claim_by_default =
      p.claim != 0 || (p.n_units >= static_cast<long long>(kDynamicMinWaves) * lanes &&
                       !(E == (int)Epi::StoreF32T && p.K < kDynamicMinGradWeightK));
  p.dynamic =
      (p.sched != nullptr && (sched_mode == 1 || (sched_mode < 0 && claim_by_default))) ? 1 : 0;
  if (p.dynamic) {
    const cudaError_t e = cudaMemsetAsync(p.sched, 0, sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
  }
  // The forward and dlogits (K = H, two accumulators) overlap consecutive
  // tiles: each tile runs kSoloBlocks of its K blocks alone, while the
  // epilogue drains the other accumulator, and the rest one-to-one with its
  // neighbours. Alone at 16384 x 3584 x 152064, two runs each (ms, forward /
  // dlogits): not overlapped 10.32, 10.22 / 11.29, 11.39; 4 solo blocks 10.15,
  // 10.11 / 11.26, 11.19; 8: 9.90, 10.14 / 10.99, 11.11; 12: 10.25, 10.13 /
  // 10.95, 11.00; 16: 10.21, 10.04 / 11.03, 11.11; 24: 10.30, 10.23 / 11.16,
  // 11.04. At V = 32000 the tensor pipe went from 76 % to 78-79 % busy.
  p.wide_skew = g.mode == kWideMode ? gemm_wide_skew() : 0;
  p.interleave = 0;
  if ((E == (int)Epi::FwdStats || E == (int)Epi::DLogits) && g.mode != kWideMode &&
      p.k_split == 0 && gemm_interleave_enabled()) {
    const int kb = (p.K + kBK - 1) / kBK;
    if (kb >= kSoloBlocks + 2) p.interleave = (kb - kSoloBlocks) / 2;
  }
  return launch_mode<E>(a, b, c, p, g.mode, lanes, stream);
}

}  // namespace

cudaError_t launch_gemm(Epi e, const CUtensorMap& a, const CUtensorMap& b, GemmParams p,
                        int tiles_per_unit, int num_sms, cudaStream_t stream,
                        const CUtensorMap* c) {
  if (e != Epi::FwdStats && !c) return cudaErrorInvalidValue;  // output map required
  if (p.a_rows != 0 &&
      (p.a_rows < 8 || p.a_rows > kBM || p.a_rows % 8 != 0 || p.a_mn || p.M > p.a_rows))
    return cudaErrorInvalidValue;  // a short A box covers every row of a K-major A
  CUtensorMap none{};
  const CUtensorMap& c_map = c ? *c : none;
  switch (e) {
    case Epi::FwdStats:
      return launch_gemm_e<(int)Epi::FwdStats>(a, b, c_map, p, tiles_per_unit, num_sms, stream);
    case Epi::DLogits:
      return launch_gemm_e<(int)Epi::DLogits>(a, b, c_map, p, tiles_per_unit, num_sms, stream);
    case Epi::StoreBf16:
      return launch_gemm_e<(int)Epi::StoreBf16>(a, b, c_map, p, tiles_per_unit, num_sms, stream);
    case Epi::StoreF32:
      return launch_gemm_e<(int)Epi::StoreF32>(a, b, c_map, p, tiles_per_unit, num_sms, stream);
    case Epi::StoreF32T:
      return launch_gemm_e<(int)Epi::StoreF32T>(a, b, c_map, p, tiles_per_unit, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

void gemm_store_engine(int* mode, int* tile_n) {
  static const Engine forced = [] {
    const char* v = std::getenv("LMH_GEMM_STORE_ENGINE");
    if (!v || !v[0]) return Engine{-1, 0};
    if (v[0] == 'w' && v[1] == 0) return Engine{kWideMode, 2 * kBN};
    const int n = std::atoi(v + 1);
    if (v[0] == 'p' && (n == 128 || n == 256)) return Engine{kPairMode, n};
    if (v[0] == 's' && (n == 64 || n == 128 || n == 192 || n == 256)) return Engine{kSingle, n};
    return Engine{-1, 0};
  }();
  *mode = forced.mode;
  *tile_n = forced.tile_n;
}

void gemm_schedule(int* schedule, int* grid_cap) {
  static const int forced = [] {
    const char* v = std::getenv("LMH_GEMM_SCHEDULE");
    if (v && std::strcmp(v, "static") == 0) return 0;
    if (v && std::strcmp(v, "dynamic") == 0) return 1;
    return -1;
  }();
  static const int cap = [] {
    const char* v = std::getenv("LMH_GEMM_GRID_CAP");
    const int n = v ? std::atoi(v) : 0;
    return n > 0 ? n : 0;
  }();
  *schedule = forced;
  *grid_cap = cap;
}

int gemm_wide_skew() {
  static const int skew = [] {
    const char* v = std::getenv("LMH_GEMM_WIDE_SKEW");
    if (!v || !*v) return kWideSkewBlocks;
    const int n = std::atoi(v);
    return n < 0 ? 0 : (n > kMaxStages ? kMaxStages : n);
  }();
  return skew;
}

bool gemm_interleave_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("LMH_GEMM_INTERLEAVE");
    return !(v && v[0] == '0');
  }();
  return on;
}

int gemm_pair_mode() {
  static const int mode = [] {
    const char* v = std::getenv("LMH_GEMM_CTA_PAIRS");
    if (v && v[0] == '0') return 0;
    if (v && v[0] == '1') return 1;
    if (v && v[0] == '2') return 2;
    return -1;
  }();
  return mode;
}

}  // namespace lmh

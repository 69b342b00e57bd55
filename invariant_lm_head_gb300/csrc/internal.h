// Host-side declarations shared by the translation units of liblmhead.so.
// Nothing here is part of the public C ABI (see include/lmhead.h).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lmh {

// Tile shape of the tensor-core engine: one CTA owns a 128 x 256 fp32
// accumulator in TMEM (double-buffered: 2 x 256 of the 512 columns) and walks
// K in 64-element steps through a TMA ring. CTA pairs share each MMA of a
// 256 x 256 tile, each CTA staging half of the B tile. K-major B operands
// are read in 128-row boxes (two per tile alone, one per CTA of a pair).
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kBBoxRows = kBN / 2;
// Engine CTA: warp 0 TMA, warp 1 MMA, then one or two epilogue groups of four
// warps (two only where a wide tile's halves drain in parallel).
constexpr int kGemmThreadsOneGroup = 192;
constexpr int kGemmThreadsTwoGroups = 320;

// Forward: a vocab chunk is kFwdTilesPerChunk N-tiles (1024 columns). The
// chunk grid depends only on V, so per-row partials and their merge order
// never depend on the number of rows.
constexpr int kFwdTilesPerChunk = 4;
constexpr int kFwdChunkCols = kFwdTilesPerChunk * kBN;

// The A box rows for a forward of M rows: M rounded up to 8 when M < kBM,
// else 0 (the full kBM-row box).
inline int short_a_rows(int64_t M) {
  return M < kBM ? static_cast<int>(M < 8 ? 8 : (M + 7) / 8 * 8) : 0;
}

// Backward: rows are processed in fixed chunks of kBwdRowChunk (or of a
// caller's multiple of kBM up to kBwdMaxRowChunk).
constexpr int64_t kBwdRowChunk = 16384;
constexpr int64_t kBwdMaxRowChunk = 1 << 20;

// StoreF32T stores the transpose: D[m][n] goes to out[n][m].
enum class Epi : int { FwdStats = 0, DLogits = 1, StoreBf16 = 2, StoreF32 = 3, StoreF32T = 4 };

// Operand layouts. K-major: the operand is stored [rows][K] (K contiguous);
// MN-major: stored [K][rows] (rows contiguous). Both are read by TMA with
// 128-byte swizzle and described to tcgen05.mma with the matching major bit.
struct GemmParams {
  int M, N, K;  // D[M, N] = sum_k A[m, k] * B[n, k]
  int a_mn, b_mn;  // 1 = operand stored MN-major ([K][M] / [K][N])
  int n_m_tiles, n_n_tiles, tiles_per_unit, n_vunits, n_units, group_m;
  // Vocab units [vunit_begin, vunit_end) of N taken by this launch (vunit_end
  // 0 = to the end); launch_gemm turns them into n_vunits, and a unit's vocab
  // unit index stays global, so partials land in their usual planes.
  int vunit_begin, vunit_end;
  // Rows of each A box (K-major A, single-CTA launches with M <= a_rows): 0
  // means kBM. A short batch then loads M rounded up to 8 rows instead of a
  // 128-row box that is almost all out-of-bounds fill; the rest of the A tile
  // is zero in shared memory, and the valid rows' products are unchanged.
  int a_rows;
  // Columns of each tile on single CTAs and CTA pairs (set by launch_gemm):
  // 256, or 64, 128 or 192 for an MN-major B (a pair: 128 or 256), so that a
  // short launch spreads over more SMs. Each output element's K walk is the
  // same for every width, so the width changes no bit.
  int tile_n;
  // Store contractions: a K split fixed by K alone. When k_split > 0, every
  // output tile is two units, one per K segment ([0, k_split) and [k_split,
  // end) in 64-wide K blocks); segment s writes its fp32 partial at output
  // row offset s * seg_rows, and a separate kernel adds the two in order.
  int k_split;
  int seg_rows;
  // Dynamic schedule: a 32-bit unit counter in the caller's workspace (NULL =
  // none). launch_gemm zeroes it and sets `dynamic` for launches of several
  // waves; the CTAs (or CTA pairs) then claim units in ascending order instead
  // of walking a fixed stride. A unit's arithmetic is the same either way.
  unsigned* sched;
  int dynamic;
  // Host hints for a launch that shares the GPU with another. claim: claim
  // units whatever the wave count (its CTAs start as SMs come free). corun:
  // grad_hidden (and the bare engine GEMM) leaves at least half the SMs to
  // the other launch when an engine that does so costs at most twice the
  // cheapest; grad_weight takes wide pairs whatever its K.
  int claim;
  int corun;
  // K blocks by which consecutive tiles overlap (set by launch_gemm; 0 = none):
  // a tile's last `interleave` blocks alternate with the next tile's first.
  int interleave;
  // Wide tiles: K blocks at a tile's end that run N block 0 before block 1
  // (set by launch_gemm; capped by the ring), so that half 0 drains early.
  int wide_skew;
  unsigned* status;
  // FwdStats / DLogits
  float scale2;    // inv_temperature * log2(e)
  float inv_temp;  // inv_temperature
  const int32_t* labels;
  int64_t label_base;      // FwdStats / DLogits: labels are global, columns start here
  const float* grad;       // DLogits: upstream grad of logprob [M] (may be NULL = 0)
  const float* grad_ent;   // DLogits: upstream grad of entropy [M] (NULL = none)
  const float* lse;        // DLogits: natural-log lse [M]
  const float* ent;        // DLogits: entropy [M] (read only with grad_ent)
  // FwdStats partials: planes [n_vunits][part_ld] for m, s, u (and q when
  // part_q is not NULL); zl [M]
  float* part_m;
  float* part_s;
  float* part_u;
  float* part_q;
  float* part_zl;
  int64_t part_ld;
  // StoreF32(T): D += result (TMA reduce-add) instead of D = result. The output
  // of every store epilogue is described by the C tensor map of launch_gemm.
  int accumulate;
};

// Counts every kernel this library launches (reported by lmhead_kernel_launches).
void note_launch();

// Kinds of launch that the opt-in per-launch timing records (their names,
// reported by lmhead_timing_kind_name, are in api.cu).
enum KernelKind : int {
  K_FWD_GEMM = 0,
  K_FWD_MERGE,
  K_DLOGITS_GEMM,
  K_DHIDDEN_GEMM,
  K_DWEIGHT_GEMM,
  K_LOGITS_ROWWISE,
  K_ENGINE_GEMM,
  K_SELFTEST,
  K_LOGITS_ROWWISE_DIV,
  K_HIDDEN_TRANSPOSE,
  K_SUM_PARTS,
  K_DHIDDEN_SUM,
  K_COUNT
};

// Brackets the launches made during its lifetime with two CUDA events on
// `st` while timing is enabled (lmhead_timing_enable), recording `kind`;
// does nothing otherwise. Defined in api.cu.
class KernelTimer {
 public:
  KernelTimer(int kind, cudaStream_t st);
  ~KernelTimer();
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  int kind_;
  cudaStream_t st_;
  cudaEvent_t b_ = nullptr;
};

// Shared host helpers of the C ABI (defined in api.cu): record the calling
// thread's error message, query the current device (sm_103 check, SM count,
// status word) and encode a 2-D bf16 TMA descriptor. Each returns an LMH_* code.
int api_set_error(int code, const char* msg);
int api_device(int* sms, unsigned** status);
// The device address of the no-allocation forward's scratch array on the
// current device, from the same per-device record as the status word.
int api_noalloc_scratch(void** scratch);
// Looks up that address with the current device's context (defined in
// noalloc.cu, the file that holds the array); called once per device.
int noalloc_scratch_lookup(void** scratch);
int api_make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

size_t gemm_smem_bytes();
// Which contractions run on CTA pairs (launches with two or more 128-row m
// tiles only), from LMH_GEMM_CTA_PAIRS, read once: "0" none (0), "1" all on
// wide pairs (1), "2" all on 256-wide pairs (2), unset the per-contraction
// default (-1: grad_hidden and grad_weight by their measured engine choice;
// the forward and dlogits on wide pairs over an even number of m tiles or an
// odd number above 32). The forward, dlogits and grad_hidden give the same
// bits on every engine; grad_weight's summation order follows the engine's
// waves.
int gemm_pair_mode();
// From LMH_GEMM_STORE_ENGINE, read once (a diagnostic, for tests and
// measurements): the engine and tile width forced on the store contractions
// (grad_hidden, grad_weight and the bare engine GEMM): "w" wide pairs,
// "p256" / "p128" pairs, "s256" / "s192" / "s128" / "s64" single CTAs. Pairs
// need two m tiles, and widths below 256 an MN-major B; *mode is -1 when
// unset or not one of these (the cost model then decides).
void gemm_store_engine(int* mode, int* tile_n);
// From LMH_GEMM_SCHEDULE and LMH_GEMM_GRID_CAP, read once (diagnostics, for
// tests and measurements): *schedule is 0 for "static" (every launch walks a
// fixed stride), 1 for "dynamic" (every launch with a unit counter claims
// units), -1 unset (dynamic from kDynamicMinWaves waves); *grid_cap is the
// most CTAs (single) or CTA pairs a launch uses, 0 when unset (all SMs).
void gemm_schedule(int* schedule, int* grid_cap);
// Whether the forward and dlogits overlap consecutive tiles' K loops
// (LMH_GEMM_INTERLEAVE, read once: "0" off, a diagnostic; on by default), and
// how many K blocks each tile then runs alone.
bool gemm_interleave_enabled();
constexpr int kSoloBlocks = 10;
// K blocks at a wide tile's end that run N block 0 first (LMH_GEMM_WIDE_SKEW,
// read once, overrides it: a diagnostic; 0 runs both blocks to the end).
constexpr int kWideSkewBlocks = 3;
int gemm_wide_skew();
// A launch of at least this many waves of units claims them dynamically
// (grad_weight only from this many rows of K).
constexpr int kDynamicMinWaves = 4;
constexpr int kDynamicMinGradWeightK = 8192;

// a / b: operand maps with boxes of 64(K) x 128 rows (A, and B in kBBoxRows-row
// boxes) when K-major, 64(MN) x 64(K) when MN-major. c is the output tensor map
// of the store epilogues (NULL for FwdStats): fp32 [M][N] with a 32 x 128 box
// and 128-byte swizzle for StoreF32, fp32 [N][M] with a 128 x 32 box and no
// swizzle for StoreF32T, bf16 [M][N] with a 32 x 128 box and
// 64-byte swizzle for StoreBf16 and DLogits.
cudaError_t launch_gemm(Epi e, const CUtensorMap& a, const CUtensorMap& b, GemmParams p,
                        int tiles_per_unit, int num_sms, cudaStream_t stream,
                        const CUtensorMap* c = nullptr);

// out_sum_p2 may be NULL; when it is not, sum_v p^2 is accumulated too.
// temp_value is the inverse temperature (divide == false: z = x * s) or the
// temperature (divide == true: z = x / t, IEEE fp32 division); with divide,
// row_temperature (f32 [T] or NULL) gives each row its own t.
cudaError_t launch_logits_logprob(const uint16_t* logits, const int32_t* labels, int64_t T,
                                  int64_t V, float temp_value, bool divide,
                                  const float* row_temperature, float* out_logprob,
                                  float* out_entropy, float* out_lse, float* out_sum_p2,
                                  int num_sms, unsigned* status, cudaStream_t stream);

// pq and out_sum_p2 may be NULL (both or neither).
// Counts (into *mismatches, which the caller zeroes) the bf16 inputs x whose
// quotient x / t in the logits path differs from IEEE fp32 division.
cudaError_t launch_division_selftest(float t, int* mismatches, cudaStream_t stream);

// out[c][r] = in[r][c] for a rows x cols bf16 matrix; cols % 8 == 0 and
// `in` rows 16-byte aligned (in_ld % 8 == 0).
cudaError_t launch_transpose_bf16(const uint16_t* in, int64_t rows, int64_t cols, int64_t in_ld,
                                  uint16_t* out, int64_t out_ld, cudaStream_t stream);

cudaError_t launch_fwd_merge(const float* pm, const float* ps, const float* pu, const float* pq,
                             const float* pzl, const int32_t* labels, int64_t T, int n_vunits,
                             int64_t V, float* out_logprob, float* out_entropy, float* out_lse,
                             float* out_sum_p2, cudaStream_t stream);

// out[i] = sum_r parts[r * stride + i], r ascending (n_parts >= 1), for
// i < count; bf16 (rounded once) when out_bf16, else fp32.
cudaError_t launch_sum_parts(const float* parts, int n_parts, int64_t stride, int64_t count,
                             void* out, bool out_bf16, int num_sms, cudaStream_t stream);

cudaError_t launch_wait_selftest(unsigned* status, unsigned long long limit_ns, int* result,
                                 cudaStream_t stream);

}  // namespace lmh

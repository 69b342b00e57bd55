/*
 * lmhead.h - batch-invariant LM-head token log-probabilities for one GB300
 * GPU (sm_103a). C ABI of liblmhead.so.
 *
 * What is computed (the "sampler formula"): for each token row t,
 *   z[t, v]     = s * logits[t, v]                 (s = inv_temperature, fp32;
 *                 logprob_from_logits_div: logits[t, v] / t, fp32 division)
 *   logprob[t]  = z[t, label[t]] - logsumexp_v z[t, v]
 *   entropy[t]  = -sum_v p[t, v] * log p[t, v],     p = softmax(z[t, :])
 * i.e. an fp32 log_softmax over the full vocabulary followed by a gather of
 * the label, as defined in the verl pull request "batch-invariant actor
 * forward and sampler log-prob formula" (the logprobs_from_logits_sampler
 * diff), with the temperature applied as an fp32 factor to the fp32 logits
 * (same page, the temperature-order comment: never round the temperature to
 * bf16). In the fused entry points logits = hidden * weight^T is never
 * materialised (SkyRL pull request "Triton backend for fused LM-head
 * log-prob", summary: the vocab projection folded into a chunked log-prob).
 *
 * Batch invariance: every reduction runs in an order fixed by V and H alone.
 * A row's logprob, entropy, lse and grad_hidden row are bit-identical whatever
 * batch, chunk, offset or packing the row arrives in. grad_weight sums over
 * rows: it is deterministic run to run for identical inputs on the same GPU
 * model (its summation order also depends on the SM count and the engine
 * chosen below), not invariant to the order of rows.
 *
 * Conventions shared by all entry points
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major, device memory.
 *  - Labels are int32. A label outside [0, V) (for example -100) gives
 *    logprob 0; entropy and lse are still those of the full row, and the
 *    backward keeps the -softmax * g term and drops the one-hot term (SkyRL
 *    page, out-of-vocab gradient fix). To ignore a padding row entirely, pass
 *    g = 0 for it.
 *  - All pointers are device pointers owned by the caller, except the host
 *    buffers of lmhead_logprob_fwd_host. The library never allocates device
 *    memory, and outside the diagnostics that say so it never synchronises or
 *    reads results back: everything is enqueued on `stream` (NULL = legacy
 *    default stream) of the current device, or on a stream of the library's
 *    own that forks from `stream` and joins back into it within the call. A
 *    whole step can therefore be captured into a CUDA graph once a first call
 *    has set up the device.
 *  - Return value: LMH_OK, or an error code with nothing launched (argument
 *    errors) or with the launch failing (LMH_ERR_LAUNCH). The message of the
 *    last error of the calling thread is lmhead_last_error_string().
 *  - The current device must be sm_103 (GB300); any other device returns
 *    LMH_ERR_UNSUPPORTED_DEVICE. There is no fallback path.
 *  - Range: the statistics fold the temperature into the max shift (one FMA,
 *    d = x * c - m with m the rounded maximum), so the maximum's own shifted
 *    value is the rounding residual of its product, up to half an ulp of it.
 *    Outputs stay finite for temperature-scaled logits |z| < 2^30 (the
 *    residual is below 2^-3 for |z| < 2^20); beyond that they may be inf or
 *    NaN. A logit of -inf (a masked vocabulary entry) contributes nothing to
 *    logprob and lse; entropy then comes out NaN (p log p = 0 * -inf), as
 *    it does in an fp32 entropy of such logits.
 *  - Every wait inside the kernels is bounded; a wait that runs out sets a
 *    device status bit that lmhead_device_status() reports.
 *  - The environment variable LMH_GEMM_CTA_PAIRS, read once per process,
 *    picks the tensor-core engine: "0" single CTAs for every contraction,
 *    "1" wide CTA pairs (two SMs per pair of MMAs, 256 x 512 tiles) wherever
 *    a launch has more than 128 rows, "2" 256 x 256 pairs there, unset the
 *    default (wide pairs for the forward and dlogits over an even number of
 *    128-row tiles, or an odd number above 32; for grad_weight and
 *    grad_hidden the engine that needs the fewest waves by measured cost).
 *    log-prob, entropy, lse, sum_p2 and grad_hidden are bit-identical
 *    whichever engine runs. grad_weight is deterministic for a given engine
 *    and SM count; its summation order follows the engine's waves.
 *  - By default a short grad_hidden (few 128-row tiles) also runs on
 *    narrower tiles (64, 128 or 192 columns, or 128-column pairs) so that it
 *    spreads over more SMs; each output element's K walk, and so its bits,
 *    stay the same. LMH_GEMM_STORE_ENGINE (a diagnostic, read once per
 *    process) forces the engine of grad_hidden and grad_weight: "w" wide
 *    pairs, "p256" / "p128" pairs, "s256" / "s192" / "s128" / "s64" single
 *    CTAs; it overrides LMH_GEMM_CTA_PAIRS for them.
 *  - A contraction of several waves of output tiles (four or more; for
 *    grad_weight, a row chunk of 8192 rows or more as well) hands its tiles
 *    to the SMs in ascending order from a counter kept in the workspace
 *    (zeroed in stream order before each launch), so tiles that share
 *    operands run together; shorter ones, and calls without a workspace,
 *    walk a fixed stride. No output bit depends on it. Two
 *    diagnostics, read once per process: LMH_GEMM_SCHEDULE ("static" or
 *    "dynamic") forces either order wherever a workspace is given, and
 *    LMH_GEMM_GRID_CAP=n runs every contraction on at most n CTAs (or CTA
 *    pairs). LMH_GEMM_INTERLEAVE=0 (a diagnostic) stops the forward and
 *    dlogits from overlapping consecutive tiles' K loops; bits are the same.
 *    LMH_GEMM_WIDE_SKEW=n (a diagnostic) sets how many K blocks at the end of
 *    a wide tile run its first 256 columns ahead of the second (default 3,
 *    at most the operand ring less one; 0 runs the two together to the
 *    end); bits are the same.
 *  - The backward of a row chunk of up to 1024 rows runs grad_hidden beside
 *    grad_weight: grad_hidden on a second stream that the library keeps per
 *    device, forked from `stream` after dlogits and joined back before the
 *    call returns (an event record and a stream wait each way, so the call
 *    stays ordered on `stream` as a whole, and stream capture records the
 *    two as parallel branches). grad_hidden then takes an engine that leaves
 *    at least half the SMs free when one costs at most twice the fastest
 *    (its bits do not change), and grad_weight runs on wide pairs whose CTAs
 *    claim their tiles as SMs come free (deterministic; its summation order
 *    is that of the wide pairs, not of the 256-wide pairs it takes alone).
 *    Concurrent backward calls from several host threads on one device take
 *    turns while enqueuing. LMH_BWD_OVERLAP (a diagnostic, read once per
 *    process) forces it off ("0") or on for every chunk ("1").
 */
#ifndef LMHEAD_H
#define LMHEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

#define LMH_OK 0
#define LMH_ERR_INVALID_ARG 1        /* null pointer, bad size or temperature   */
#define LMH_ERR_ALIGNMENT 2          /* pointer or leading dimension misaligned */
#define LMH_ERR_WORKSPACE 3          /* workspace missing or too small          */
#define LMH_ERR_UNSUPPORTED_DEVICE 4 /* current device is not sm_103            */
#define LMH_ERR_LAUNCH 5             /* CUDA runtime error while launching      */
#define LMH_ERR_DEVICE_TIMEOUT 6     /* a bounded device wait ran out           */

#define LMH_OP_FWD 0
#define LMH_OP_BWD 1
#define LMH_OP_LOGITS 2

/* Largest T, H and V accepted (row and column indices stay within int32). */
#define LMH_MAX_DIM 2147483392LL

/*
 * Bytes of workspace that `op` needs for these sizes (0 for LMH_OP_LOGITS).
 * Returns SIZE_MAX for invalid arguments. The forward needs 16 bytes per row
 * per 1024 vocabulary columns (+4 per row, and a 4-byte tile counter); the
 * backward adds 12 bytes per
 * row, a bf16 dlogits buffer of min(T, 16384) x V, a bf16 transpose of one
 * 16384-row chunk of hidden (H x min(T, 16384)) and the fp32 partials of one
 * chunk's grad_hidden, one per half of the vocabulary (2 x min(T, 16384) x H,
 * rows rounded up to 128), and a second 4-byte tile counter.
 */
size_t lmhead_workspace_size(int op, int64_t T, int64_t H, int64_t V);

/*
 * Fused forward: the vocab projection folded into the log-prob pass (SkyRL
 * page, summary) computing the sampler formula (verl page).
 *   hidden   bf16 [T, H], 16-byte aligned, H % 8 == 0
 *   weight   bf16 [V, H] (nn.Linear layout), 16-byte aligned
 *   labels   int32 [T]
 *   inv_temperature  finite, > 0 (1.0 gives the plain formula)
 *   out_logprob  f32 [T], required
 *   out_entropy  f32 [T] or NULL
 *   out_lse      f32 [T] or NULL (natural-log logsumexp of z; feed it to the
 *                backward to skip its recompute of the statistics)
 *   workspace    >= lmhead_workspace_size(LMH_OP_FWD, T, H, V) bytes,
 *                16-byte aligned; contents need not be initialised
 * T == 0 is a no-op (then every pointer may be NULL).
 */
int lmhead_logprob_fwd(const uint16_t* hidden, const uint16_t* weight, const int32_t* labels,
                       int64_t T, int64_t H, int64_t V, float inv_temperature,
                       float* out_logprob, float* out_entropy, float* out_lse, void* workspace,
                       size_t workspace_bytes, struct CUstream_st* stream);

/*
 * lmhead_logprob_fwd plus sum_pi_squared: out_sum_p2[t] = sum_v p[t, v]^2 of
 * the same distribution (verl page, the review note that lists entropy and
 * sum_pi_squared as the per-token statistics still taken from the logits).
 * Same pass, one more accumulator; out_sum_p2 f32 [T] or NULL. Same
 * workspace as lmhead_logprob_fwd. logprob, entropy and lse are bit-identical
 * to those of lmhead_logprob_fwd.
 */
int lmhead_logprob_fwd_stats(const uint16_t* hidden, const uint16_t* weight, const int32_t* labels,
                             int64_t T, int64_t H, int64_t V, float inv_temperature,
                             float* out_logprob, float* out_entropy, float* out_lse,
                             float* out_sum_p2, void* workspace, size_t workspace_bytes,
                             struct CUstream_st* stream);

/*
 * Fused backward of sum_t grad_logprob[t] * logprob[t] (SkyRL page: logits
 * recomputed per chunk in backward; verl page: the per-chunk recompute that
 * keeps no [rows, V] fp32 activation alive).
 *   dlogits[t, v] = g[t] * s * (onehot(label[t])[v] - softmax(z[t])[v])
 *   grad_hidden   bf16 [T, H], overwritten: dlogits * weight (rounded once)
 *   grad_weight   f32  [V, H], overwritten: dlogits^T * hidden
 *   grad_logprob  f32 [T]
 *   lse           f32 [T] from lmhead_logprob_fwd, or NULL to recompute it
 *   workspace     >= lmhead_workspace_size(LMH_OP_BWD, T, H, V) bytes
 * Rows are processed in fixed chunks of 16384; dlogits of a chunk are rounded
 * to bf16 before both contractions; grad_weight sums the chunks in ascending
 * order. grad_hidden sums over the vocabulary in two fixed halves (the first
 * ceil(nk / 2) of the nk 64-column blocks, then the rest), each in order, and
 * rounds their fp32 sum once; the halves depend on V alone, so every row gets
 * the same association in any batch. T == 0 zeroes grad_weight (then only
 * grad_weight has to be a valid pointer).
 */
int lmhead_logprob_bwd(const uint16_t* hidden, const uint16_t* weight, const int32_t* labels,
                       const float* grad_logprob, const float* lse, int64_t T, int64_t H,
                       int64_t V, float inv_temperature, uint16_t* grad_hidden,
                       float* grad_weight, void* workspace, size_t workspace_bytes,
                       struct CUstream_st* stream);

/*
 * Fused backward with an entropy term: differentiates
 *   sum_t grad_logprob[t] * logprob[t] + grad_entropy[t] * entropy[t].
 * The SkyRL page leaves entropy under the fused head metric-only ("until
 * entropy gradients are wired"); this wires it. With p = softmax(z[t]),
 *   d entropy[t] / d z[t, v] = -p[v] * (z[t, v] - lse[t] + entropy[t]),
 * so dlogits[t, v] = s * (g[t] * onehot[v] - p[v] * (g[t] + gH[t] *
 * (z[t, v] - lse[t] + entropy[t]))).
 *   grad_logprob, grad_entropy  f32 [T] or NULL (= zero); not both NULL
 *   lse, entropy  f32 [T] from lmhead_logprob_fwd, or NULL to recompute both
 * Everything else as lmhead_logprob_bwd (same workspace size).
 */
int lmhead_logprob_entropy_bwd(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* labels, const float* grad_logprob,
                               const float* grad_entropy, const float* lse, const float* entropy,
                               int64_t T, int64_t H, int64_t V, float inv_temperature,
                               uint16_t* grad_hidden, float* grad_weight, void* workspace,
                               size_t workspace_bytes, struct CUstream_st* stream);

/*
 * lmhead_logprob_entropy_bwd with a caller-chosen row chunk, to bound the
 * backward's memory. The verl page recomputes the logits chunk by chunk in
 * its checkpointed backward so that no [rows, V] activation stays alive; here
 * the workspace holds one chunk's bf16 dlogits [row_chunk, V] and its
 * transposed hidden [H, row_chunk], so a smaller chunk shrinks it (at
 * H = 3584, V = 152064: about 5.1 GB at 16384 rows, 1.3 GB at 4096).
 *   row_chunk  a multiple of 128 in [128, 1048576]; LMH_ERR_INVALID_ARG else
 *   workspace  >= lmhead_workspace_size_bwd(T, H, V, row_chunk) bytes
 * Everything else as lmhead_logprob_entropy_bwd (grad_entropy may be NULL,
 * then the plain backward). grad_hidden does not depend on row_chunk, bit for
 * bit: each row's dlogits and its K = V walk are the same. grad_weight sums
 * the chunks in ascending order, so its rounding depends on row_chunk
 * (deterministically). lmhead_logprob_bwd uses row_chunk = 16384.
 */
int lmhead_logprob_bwd_chunked(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* labels, const float* grad_logprob,
                               const float* grad_entropy, const float* lse, const float* entropy,
                               int64_t T, int64_t H, int64_t V, float inv_temperature,
                               int64_t row_chunk, uint16_t* grad_hidden, float* grad_weight,
                               void* workspace, size_t workspace_bytes,
                               struct CUstream_st* stream);
/* Workspace bytes of lmhead_logprob_bwd_chunked (SIZE_MAX for bad arguments). */
size_t lmhead_workspace_size_bwd(int64_t T, int64_t H, int64_t V, int64_t row_chunk);

/*
 * Sampler formula on materialised logits (verl page, the
 * logprobs_from_logits_sampler diff): fp32 log_softmax of s * logits over the
 * full row, then gather. One streaming pass over the logits.
 *   logits  bf16 [T, V]; 16-byte aligned when V % 8 == 0, else 2-byte aligned
 *   out_logprob f32 [T] required; out_entropy, out_lse f32 [T] or NULL
 */
int logprob_from_logits(const uint16_t* logits, const int32_t* labels, int64_t T, int64_t V,
                        float inv_temperature, float* out_logprob, float* out_entropy,
                        float* out_lse, struct CUstream_st* stream);

/*
 * logprob_from_logits plus sum_pi_squared (out_sum_p2 f32 [T] or NULL), in the
 * same single pass over the logits; the other outputs are bit-identical to
 * those of logprob_from_logits.
 */
int logprob_from_logits_stats(const uint16_t* logits, const int32_t* labels, int64_t T, int64_t V,
                              float inv_temperature, float* out_logprob, float* out_entropy,
                              float* out_lse, float* out_sum_p2, struct CUstream_st* stream);

/*
 * Sampler-parity form of the sampler formula: the temperature is applied as
 * an fp32 division of the fp32 logits, z = fp32(logits) / t, rounded to
 * nearest as IEEE division is (verl page, temperature-order table: cast to
 * fp32 first, then divide by the fp32 temperature), which is what an inference
 * sampler computes when it divides the logits by a per-request temperature
 * tensor. logprob_from_logits instead multiplies by an inverse temperature,
 * which can differ from the division in the last bit of z.
 *   temperature      t for every row (finite, > 0) when row_temperature is NULL
 *   row_temperature  f32 [T] device array of per-row temperatures, or NULL;
 *                    a row whose value is not finite and > 0 gets NaN outputs
 *                    (the host cannot check device values)
 *   out_sum_p2       f32 [T] or NULL, as in logprob_from_logits_stats
 * Everything else (layouts, labels outside [0, V), errors, batch invariance)
 * as logprob_from_logits.
 */
int logprob_from_logits_div(const uint16_t* logits, const int32_t* labels, int64_t T, int64_t V,
                            float temperature, const float* row_temperature, float* out_logprob,
                            float* out_entropy, float* out_lse, float* out_sum_p2,
                            struct CUstream_st* stream);

/*
 * Forward from host memory: copies hidden, weight and labels from host
 * buffers into the caller's device buffers and runs lmhead_logprob_fwd on
 * them, with the host-to-device copies overlapped with the tensor-core work.
 * The weight is copied in vocabulary slices (whole 1024-column chunks; the
 * first small, later ones up to a quarter of V) on a copy stream, and the
 * forward GEMM runs as one launch per slice, each after its slice has landed,
 * so only the copy of hidden and of the first slice is exposed. An addition of
 * this library for callers whose inputs live in host memory (an offloaded LM
 * head, a host-side data loader); the pages have no counterpart.
 *   hidden_host  bf16 [T, H], weight_host bf16 [V, H], labels_host int32 [T]:
 *                host memory, page-locked for the copies to overlap (pageable
 *                memory works but is copied synchronously by the driver)
 *   hidden, weight, labels  device buffers of the same shapes, written by the
 *                call (the backward can then run on them)
 *   out_logprob_host, out_entropy_host  f32 [T] host buffers or NULL: filled
 *                after the forward, in `stream` order (out_entropy_host needs
 *                out_entropy)
 *   copy_stream  stream for the host-to-device copies, or NULL for one the
 *                library creates per device on first use
 * Results are bit-identical to lmhead_logprob_fwd on the same data: every tile
 * is computed as in the single launch. Ordering: the copies start after the
 * work already enqueued on `stream` (an event recorded on `stream` at entry),
 * and `stream` waits for every copy before the kernels that read it, so all of
 * the call is ordered on `stream` as if it ran there. Nothing is allocated on
 * the device; the library keeps a copy stream and a few events per device,
 * created by this entry point's first call (which therefore comes before any
 * stream capture of it).
 * Everything else (workspace, sizes, errors) as lmhead_logprob_fwd.
 */
int lmhead_logprob_fwd_host(const uint16_t* hidden_host, const uint16_t* weight_host,
                            const int32_t* labels_host, int64_t T, int64_t H, int64_t V,
                            float inv_temperature, uint16_t* hidden, uint16_t* weight,
                            int32_t* labels, float* out_logprob, float* out_entropy,
                            float* out_lse, float* out_logprob_host, float* out_entropy_host,
                            void* workspace, size_t workspace_bytes, struct CUstream_st* stream,
                            struct CUstream_st* copy_stream);

/*
 * The forward split by vocabulary shards, for a vocab-parallel (tensor-
 * parallel) LM head whose ranks each hold rows [v_offset, v_offset + V) of
 * the weight. The pages' vocab-parallel log-softmax (SkyRL page, the chunked
 * distributed log-prob) exchanges per-row max / sum-exp / label-logit
 * statistics between ranks; here the statistics are the forward's own
 * per-1024-column partials, so the merged result is bit-identical to
 * lmhead_logprob_fwd on the whole weight, whatever the number of shards.
 *
 * lmhead_logprob_fwd_partials: this shard's statistics.
 *   hidden bf16 [T, H], weight bf16 [V, H] (the shard), labels int32 [T] as
 *   indices into the whole vocabulary.
 *   v_offset  the shard's first row, a multiple of 1024 (LMH_ERR_ALIGNMENT
 *             otherwise); every shard but the last should hold a multiple
 *             of 1024 rows so that the shards' chunks tile the vocabulary
 *   part_m, part_s, part_u  f32 planes [ceil(V / 1024)][T] receiving the
 *             chunks' base-2 max, sum and entropy accumulators. Point them at
 *             chunk v_offset / 1024 of the whole-vocabulary planes
 *             [ceil(V_total / 1024)][T].
 *   label_logit f32 [T]: the scaled label logit (base 2) of rows whose label
 *             is in this shard, 0 for every other row. Summing the shards'
 *             buffers gives every row its value: exactly one term is nonzero.
 * lmhead_logprob_merge: the fixed-order merge of the whole-vocabulary planes
 *   (V = V_total) and the summed label_logit, into logprob, entropy and lse
 *   as lmhead_logprob_fwd returns them.
 * The exchange between ranks is the caller's: all-gather each plane's slice
 * in rank order, and sum label_logit. On one GPU, several shards of one weight
 * write into one set of planes directly.
 */
int lmhead_logprob_fwd_partials(const uint16_t* hidden, const uint16_t* weight,
                                const int32_t* labels, int64_t T, int64_t H, int64_t V,
                                int64_t v_offset, float inv_temperature, float* part_m,
                                float* part_s, float* part_u, float* label_logit,
                                struct CUstream_st* stream);
int lmhead_logprob_merge(const float* part_m, const float* part_s, const float* part_u,
                         const float* label_logit, const int32_t* labels, int64_t T, int64_t V,
                         float* out_logprob, float* out_entropy, float* out_lse,
                         struct CUstream_st* stream);

/*
 * The backward of one vocab shard (the SkyRL page's chunked distributed
 * log-prob, whose tensor-parallel ranks each hold a slice of the vocabulary).
 * The shard holds rows [v_offset, v_offset + V) of the weight; labels index
 * the whole vocabulary, and a label outside the shard gets no one-hot term
 * here (its shard adds it), so no caller shifts labels.
 *   lse          f32 [T], required: the whole vocabulary's lse, as
 *                lmhead_logprob_merge returns it (a shard cannot recompute it)
 *   grad_logprob, grad_entropy, entropy  as lmhead_logprob_entropy_bwd;
 *                entropy (the whole distribution's) is required with
 *                grad_entropy
 *   v_offset     >= 0 (no alignment needed in the backward)
 *   grad_hidden_part  f32 [T, H], overwritten with this shard's dlogits * W,
 *                16-byte aligned. The whole grad_hidden is the sum over the
 *                shards: lmhead_sum_ranks_bf16 adds the ranks' parts in rank
 *                order and rounds once, so every rank gets the same bits.
 *   grad_weight  f32 [V, H], overwritten: this shard's rows (no exchange)
 *   workspace    >= lmhead_workspace_size(LMH_OP_BWD, T, H, V) (V = the shard's)
 */
int lmhead_logprob_bwd_shard(const uint16_t* hidden, const uint16_t* weight,
                             const int32_t* labels, const float* grad_logprob,
                             const float* grad_entropy, const float* lse, const float* entropy,
                             int64_t T, int64_t H, int64_t V, int64_t v_offset,
                             float inv_temperature, float* grad_hidden_part, float* grad_weight,
                             void* workspace, size_t workspace_bytes,
                             struct CUstream_st* stream);

/*
 * out[i] = bf16(((parts[0][i] + parts[1][i]) + ...) + parts[n_parts - 1][i]),
 * round to nearest once at the end: a fixed, rank-ordered sum of the shards'
 * grad_hidden partials after they are all-gathered (parts f32
 * [n_parts][count], contiguous; out bf16 [count]). n_parts in [1, 65536].
 */
int lmhead_sum_ranks_bf16(const float* parts, int64_t n_parts, int64_t count, uint16_t* out,
                          struct CUstream_st* stream);

/*
 * Forward without a workspace, for callers that cannot allocate device memory
 * (a plugin whose host framework owns all device memory and hands out no
 * workspace, or code that must not call cudaMalloc because it can block and
 * synchronise the device). The pages have no counterpart: this is an addition
 * of this library.
 *
 * Same arguments, results and rules as lmhead_logprob_fwd minus the
 * workspace. The forward's partials go to a fixed scratch array compiled into
 * the library (LMH_NOALLOC_SCRATCH_BYTES, 16 MiB, held on every GPU where the
 * library's device code is loaded until the process exits); nothing is
 * allocated. The partials need 12 * ceil(V / 1024) * T + 4 * T bytes (each
 * part rounded up to 256); larger calls return LMH_ERR_WORKSPACE with nothing
 * launched (for V = 152064 that is T up to about 9300 rows).
 * The library's first call on a device (of any entry point) looks up the
 * scratch array's device address (cudaGetSymbolAddress); make it before any
 * stream capture. All calls share
 * the one array, which keeps the previous call's contents (nothing in it needs
 * to start at zero). Calls that overlap on the GPU (other streams, or
 * unordered host threads) race on it: serialise them.
 */
#define LMH_NOALLOC_SCRATCH_BYTES (16u << 20)
int lmhead_logprob_fwd_noalloc(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* labels, int64_t T, int64_t H, int64_t V,
                               float inv_temperature, float* out_logprob, float* out_entropy,
                               float* out_lse, struct CUstream_st* stream);

/* ---------------------------------------------------------------- diagnostics */

/* Message of the calling thread's last error ("" if none). */
const char* lmhead_last_error_string(void);

/* ABI version of this header (incremented on incompatible changes). */
int lmhead_abi_version(void);

/* Number of CUDA kernels this library has launched in this process so far. */
unsigned long long lmhead_kernel_launches(void);

/*
 * Per-launch timing (diagnostics, off by default). While enabled, every kernel
 * launch of the library is bracketed by two CUDA events recorded on the
 * launching stream. lmhead_timing_enable(1) starts recording and discards old
 * records; lmhead_timing_enable(0) stops. lmhead_timing_read() waits for the
 * recorded events, writes up to `capacity` (kind, milliseconds) pairs, sets
 * *count and discards the records. lmhead_timing_kind_name() names a kind
 * (for example "fused_fwd_gemm"), "" for an unknown one.
 */
int lmhead_timing_enable(int on);
int lmhead_timing_read(int* kinds, float* ms, int capacity, int* count);
const char* lmhead_timing_kind_name(int kind);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word. Returns LMH_ERR_DEVICE_TIMEOUT if a bounded wait ran out since the
 * last call, LMH_ERR_LAUNCH if the stream reports a CUDA error, else LMH_OK.
 * *bits (may be NULL) receives the raw word.
 */
int lmhead_device_status(struct CUstream_st* stream, unsigned* bits);

/*
 * Self-test of the bounded wait: launches one thread that waits on a barrier
 * nothing completes, with a limit of limit_ns nanoseconds (1e3..1e10), and
 * synchronises `stream`. Expected result: LMH_ERR_DEVICE_TIMEOUT, with the
 * timeout bit left set in the status word (lmhead_device_status clears it).
 * No fault, trap or hang is involved.
 */
int lmhead_selftest_wait_timeout(uint64_t limit_ns, struct CUstream_st* stream);

/*
 * Self-test of the division that logprob_from_logits_div applies: for every
 * one of the 65536 bf16 bit patterns x, compares its quotient x / temperature
 * with IEEE fp32 division (round to nearest) and stores in *mismatches the
 * number of inputs whose result bits differ (NaN counts as equal to NaN);
 * 0 means the division form is bit-exact for this temperature. Synchronises
 * `stream`. Any temperature may be given, including 0, negative, inf or NaN.
 */
int lmhead_selftest_division(float temperature, int* mismatches, struct CUstream_st* stream);

/*
 * The tensor-core engine alone, for engine tests: D[M, N] = sum_k A[m, k] B[n, k]
 * with bf16 operands and an f32 row-major D (N % 8 == 0, 16-byte aligned),
 * fp32 accumulation in K order. layout bit 0: A is stored [K][M] (else
 * [M][K]); bit 1: B is stored [K][N] (else [N][K]). Leading dimensions equal
 * the stored row length, which must be a multiple of 8.
 */
int lmhead_engine_gemm(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                       int layout, float* D, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* LMHEAD_H */

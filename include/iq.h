/*
 * iq.h — C ABI of the B300 (sm_103a) IQ codebook library: the importance-weighted encoder for the
 * GGML IQ formats (IQ2_XXS, IQ2_XS, IQ2_S, IQ1_S, IQ1_M), its decoder, and the per-expert imatrix
 * statistic that supplies the encoder's importance weights.
 *
 * Conventions for every call
 *  - Pointers named as device pointers are CUDA global-memory addresses on the current device;
 *    the caller allocates and owns every buffer.  The library keeps no state and allocates nothing;
 *    calls that need scratch take a caller-provided `workspace` of at least the size reported by
 *    the matching *_workspace_size call (device memory, 256-byte aligned, contents ignored).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *  - Return value: IQ_OK (0) or a negative IQ_ERR_* code.  Argument checks run on the host before
 *    anything is launched or written (a refused call changes no buffer).
 *  - Data-dependent problems are never trapped and never synchronise the host: the kernels OR an
 *    IQ_STATUS_* bit into `*status` (a device int32, may be NULL) and skip the offending unit.
 *  - Matrices are row-major and contiguous.  A weight [rows, cols] has cols % 256 == 0 and is cut
 *    into B = rows * cols / 256 blocks of 256 consecutive values of a row; block b covers row
 *    b / (cols/256), columns 256 * (b % (cols/256)) ...; a block has 32 vectors of 8 values.
 *
 * Sources (web pages, cited by title and section):
 *  [imatrix]  "Add imatrix calibration for the GGML formats and use it for fused MoE experts"
 *             (PR #2735), "What imatrix does" and its unit-test list.
 *  [coverage] "MoE expert coverage in imatrix calibration", Facts.
 *  [formats]  PR #2513: the IQ2_XXS, IQ2_S and IQ1_M commit texts and the IQ1_M description.
 *  [choices]  PR #3157 "[1/5] Let the GGML IQ encoders take fixed per-group choices", PR #3159
 *             "one-pass every-choice encode" and PR #3158 "local_hessian for GGML IQ" (same
 *             page).
 *  [iq1m-cuda] the IQ1_M CUDA-encoder commit message on the recipes-folder page.
 */
#ifndef IQ_B300_IQ_H
#define IQ_B300_IQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define IQ_API __attribute__((visibility("default")))
#else
#define IQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { IQ2_XXS = 0, IQ2_XS = 1, IQ2_S = 2, IQ1_S = 3, IQ1_M = 4 } iq_format;
typedef enum { IQ_F32 = 0, IQ_BF16 = 1 } iq_dtype;

enum {
  IQ_OK = 0,
  IQ_ERR_ARG = -1,       /* null / misaligned pointer, bad size or enum, cols % 256 != 0, ... */
  IQ_ERR_CUDA = -2,      /* a CUDA call or launch failed */
  IQ_ERR_WORKSPACE = -3, /* workspace missing or smaller than the reported size */
  IQ_ERR_TOO_LARGE = -4  /* the problem needs more scratch than the fixed static array holds */
};

/* Bits OR-ed into *status by the kernels. */
#define IQ_STATUS_BAD_CHOICE 1        /* a fixed choice >= num_choices: that block is all zero */
#define IQ_STATUS_BAD_EXPERT_ID 2     /* an expert id outside [0, num_experts): that slot ignored */
#define IQ_STATUS_NONFINITE_SUM2 4    /* a non-finite in_sum2 value of an expert this call touched */
#define IQ_STATUS_DUP_EXPERT_ID 8     /* an id repeated within one token's top-k: counted once */
#define IQ_STATUS_BAD_INPUT 16        /* a non-finite weight value: that block is all zero */
#define IQ_STATUS_BAD_IMPORTANCE 32   /* a negative or non-finite importance: that block is all zero */
#define IQ_STATUS_BAD_SCALE 64        /* a negative / inf / nan fp16 scale: that block is all zero */
#define IQ_STATUS_BAD_GRID 128        /* codebook values outside the format's set: all blocks zero */
#define IQ_STATUS_TIMEOUT 256         /* an internal bounded wait gave up: results unspecified */

typedef struct {
  int block_bytes;        /* payload bytes per 256-value block */
  int choice_groups;      /* groups per block that each store one choice */
  int num_choices;        /* choices per group: valid choice values are [0, num_choices) */
  int grid_entries;       /* codebook rows (each 8 fp32 values) */
  int vectors_per_group;  /* 8-value vectors per choice group */
  int index_bits;         /* bits of a stored codebook index */
} iq_format_info_t;

/* Per-format constants [formats]: bits per weight 2.0625 / 2.3125 / 2.5625 / 1.5625 / 1.75 give
 * 66 / 74 / 82 / 50 / 56 bytes per block.  Returns IQ_ERR_ARG for an unknown format. */
IQ_API int iq_format_info(iq_format f, iq_format_info_t *out);

/*
 * Block layouts (bit p of a block is bit p % 8 of byte p / 8; multi-byte fields little-endian).
 * g = vector (8 values) 0..31, s = sub-block of 32 values 0..7, cg = choice group.
 *  IQ2_XXS (66 B): d fp16 @0; per s: 4 index bytes @2+8s (vectors 4s..4s+3), then a u32 @6+8s with
 *           four 7-bit sign indices (bits 7k..7k+6, vector 4s+k) and the 4-bit scale (bits 28..31).
 *           cg = s (32 values, 8 per block).
 *  IQ2_XS  (74 B): d @0; per g a u16 @2+2g = 9-bit index | 7-bit sign index << 9; byte 66+s holds
 *           the scales of cg 2s (low nibble) and 2s+1 (high).  cg = g/2 (16 values, 16 per block).
 *  IQ2_S   (82 B): d @0; index low bytes @2+g; 8-bit sign masks @34+g; byte 66+s holds the index
 *           high 2 bits of vector 4s+k at bits 2k; byte 74+s the scales of cg 2s, 2s+1.  cg = g/2.
 *  IQ1_S   (50 B): d @0; index low bytes @2+g; per s a u16 @34+2s: index high 3 bits of vector
 *           4s+k at bits 3k, scale at bits 12..14, delta bit at 15.  cg = s; choice = scale + 8*delta.
 *  IQ1_M   (56 B): index low bytes @g; byte 32+g/2, nibble g%2: index high 3 bits | delta bit << 3;
 *           u16 @48+2k: scales of cg 4k..4k+3 at bits 3j, and d's fp16 bits 4k..4k+3 at 12..15.
 *           cg = g/2; choice = scale (the delta is per vector, free in the entry search).
 * Values: IQ2 q = d * (2s+1)/8 * g[i], negated where sign bit i is set; IQ2_XXS/XS store bits 0..6
 * and bit 7 is the parity of bits 0..6 (even parity).  IQ1 q = d * (2s+1) * (g[i] + delta), delta
 * = +1/8 for delta bit 0 and -1/8 for 1.  Codebooks: IQ2 values must be integers in [1, 127], IQ1
 * values in {-1, 0, 1}; every decoded value is then exact in fp32.
 */

/* ---- imatrix ([imatrix] "What imatrix does", Bounded memory; [coverage] Facts) ----------------
 * For each chunk of `rows_per_chunk` consecutive tokens (1,024 on the pages) and each expert e the
 * chunk routes tokens to: partial[e][j] starts at +0 and, over the chunk's tokens whose top-k ids
 * contain e in ascending token order, becomes fl(partial + fl(x[t][j]*x[t][j])) -- the square
 * rounded to fp32 (exact for bf16 activations), then added with one more rounding (no fused
 * multiply-add for fp32 activations); then in_sum2[e][j] = fl(in_sum2[e][j] +
 * partial[e][j]) (chunk order) and counts[e] += tokens routed to e.  A token's ids are a set (a
 * repeated id counts once and sets IQ_STATUS_DUP_EXPERT_ID; an id outside [0, num_experts) is
 * skipped and sets IQ_STATUS_BAD_EXPERT_ID).  After the call, a non-finite in_sum2 value of an
 * expert this call touched sets IQ_STATUS_NONFINITE_SUM2.
 *   x            device, [tokens, cols] of dtype dt (IQ_F32 or IQ_BF16), 16-byte aligned
 *   expert_ids   device, [tokens, top_k] int32
 *   in_sum2      device, [num_experts, cols] fp32, accumulated in place (16-byte aligned)
 *   counts       device, [num_experts] int64, accumulated in place
 *   workspace    device scratch of iq_imatrix_workspace_size bytes (256-byte aligned)
 *   requires cols % 64 == 0, 1 <= top_k <= min(num_experts, 64), num_experts <= 1024,
 *   1 <= rows_per_chunk <= 4096, tokens < 2^31 and at most 65535 chunks.
 * Results are bit-identical to the sequential definition above, whatever the launch layout. */
IQ_API int iq_imatrix_workspace_size(int64_t tokens, int64_t cols, iq_dtype dt, int num_experts, int top_k,
                              int64_t rows_per_chunk, size_t *bytes);
IQ_API int iq_imatrix_accumulate(const void *x, iq_dtype dt, int64_t tokens, int64_t cols,
                          const int32_t *expert_ids, int top_k, int num_experts, int64_t rows_per_chunk,
                          float *in_sum2, int64_t *counts, int32_t *status, void *workspace,
                          size_t workspace_bytes, void *stream);

/* Importance weights ([imatrix] "Why the square root"; [coverage] Facts: count 0 -> weight 1):
 * w[e][j] = sqrt(m) with m = in_sum2[e][j] / (float)counts[e] (IEEE fp32 division and square root),
 * m raised to `floor` first when floor > 0 and m < floor; w = 1 for every channel of an expert
 * with counts[e] == 0.  All pointers device; w may not alias in_sum2. */
IQ_API int iq_imatrix_weights(const float *in_sum2, const int64_t *counts, int num_experts, int64_t cols,
                       float floor, float *w, void *stream);

/* ---- merging, neutral entries, coverage ([coverage] Facts) --------------------------------------
 * iq_imatrix_merge: in_sum2 += src_in_sum2 (fp32, one rounding per value) and counts += src_counts,
 *   the merge of two statistics of the same tensor (GGUF imatrix files keep in_sum2 and counts so
 *   that they can be merged).  Sums that become non-finite set IQ_STATUS_NONFINITE_SUM2.  Sources
 *   must not alias the destinations.  All device pointers, [num_experts, cols] and [num_experts].
 * iq_imatrix_neutral_entries: every expert whose count is 0 gets in_sum2 = 1 on every channel and
 *   count 1, the legacy writer's neutral entry (its weight stays 1).
 * iq_imatrix_coverage: out (device int64 [4]) = experts with at least one token, tokens over all
 *   experts, least count, largest count; out[0] / num_experts is the "partial data" share of the
 *   saving log, out[0] == 0 its "no data". */
IQ_API int iq_imatrix_merge(float *in_sum2, int64_t *counts, const float *src_in_sum2, const int64_t *src_counts,
                            int num_experts, int64_t cols, int32_t *status, void *stream);
IQ_API int iq_imatrix_neutral_entries(float *in_sum2, int64_t *counts, int num_experts, int64_t cols, void *stream);
IQ_API int iq_imatrix_coverage(const int64_t *counts, int num_experts, int64_t *out, void *stream);

/* ---- super-block scale anchor ([formats]: "single-pass grid search at a fixed anchored
 * super-block scale"; IQ1_S flat 0.61; IQ1_M clamp(0.58 + 0.035 * peak_to_rms, 0.65, 0.95)) -----
 * d16[b] = fp16 (round to nearest even, saturated at 65504) of (ratio * amax) / K, amax = max |x|
 * over the block, K = 166.625 (IQ2: 43 * 31/8) or 15 (IQ1), ratio = 1 for IQ2, 0.61 for IQ1_S and
 * the clamp above for IQ1_M with rms = sqrt(s/256), s = sum of x^2 summed as 32 sequential partial
 * sums of 8 consecutive squares, then pairwise (l, l+16), (l, l+8), (l, l+4), (l, l+2), (l, l+1).
 * Blocks with a non-finite value get d16 = 0 and IQ_STATUS_BAD_INPUT.  W device [rows, cols]. */
IQ_API int iq_anchor_scales(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols, uint16_t *d16,
                     int32_t *status, void *stream);

/* ---- encoder ([formats]; [choices]; [iq1m-cuda]) --------------------------------------------
 * For every choice group: for every allowed choice c, each vector takes the candidate (entry, plus
 * the delta for IQ1_M) with the least weighted squared error sum_i w_i (x_i - q_i)^2; the group
 * takes the choice with the least sum over its vectors (lowest c on equal error), and each vector
 * its best candidate under it (lowest (delta bit, entry) on equal error).  IQ2_XXS/XS first flip
 * the sign of argmin_i w_i x_i^2 when an odd number of x_i are negative (even parity); IQ2_S keeps
 * the input signs.  Decisions equal those of an exact evaluation: candidates the fp32 sweep cannot
 * separate from the best within its rounding bound are rescored in fp64 (the bound is proven for
 * the rescoring's fp32 FMA chains; for the sweep's tensor-core sums it rests on the measured
 * accumulation error of the MMAs, about a third of what it allows).
 *   W            device [rows, cols], dtype dt; 16-byte aligned
 *   importance   device fp32, NULL (w = 1), [cols] (rows_per_expert == 0) or [E, cols] with row r
 *                using expert r / rows_per_expert ([coverage]: global row / rows per expert)
 *   grid         device fp32 [grid_entries, 8] codebook
 *   d16          device fp16 bits [B], or NULL to compute the anchor above inside the call
 *   choices      device uint8 [B, choice_groups] fixed choices, or NULL to search; a value >=
 *                num_choices sets IQ_STATUS_BAD_CHOICE and zeroes that block
 *   payload      device uint8 [B, block_bytes] output
 *   group_errors device fp32 [B, choice_groups, num_choices] or NULL: with choices == NULL, the
 *                weighted squared error of every (group, choice) pair from the same sweep (the
 *                every-choice mode); each value is within 2^-17 * (4 * sum_g w x^2 + 2 * E) of exact
 *   workspace    device scratch of iq_encode_workspace_size bytes
 * A block whose scale is 0 encodes to all-zero bytes ([choices] review: zero blocks). */
IQ_API int iq_encode_workspace_size(iq_format f, int64_t rows, int64_t cols, size_t *bytes);
IQ_API int iq_encode(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols, const float *importance,
              int64_t rows_per_expert, const float *grid, const uint16_t *d16, const uint8_t *choices,
              uint8_t *payload, float *group_errors, int32_t *status, void *workspace,
              size_t workspace_bytes, void *stream);

/* Encode and write back ([imatrix] What imatrix does: the encoder encodes each weight with its
 * statistic, writes the decoded weight back and pins the payload): iq_encode (no table), then W is
 * overwritten in place with the decoded payload in its own dtype (bf16: rounded to nearest even;
 * fp32: exact).  Blocks the encoder rejected decode to zeros.  Arguments as in iq_encode. */
IQ_API int iq_encode_write_back(iq_format f, void *W, iq_dtype dt, int64_t rows, int64_t cols,
                                const float *importance, int64_t rows_per_expert, const float *grid,
                                const uint16_t *d16, const uint8_t *choices, uint8_t *payload, int32_t *status,
                                void *workspace, size_t workspace_bytes, void *stream);

/* Every-choice error table only (same sweep, no payload): group_errors as in iq_encode. */
IQ_API int iq_group_errors(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols,
                    const float *importance, int64_t rows_per_expert, const float *grid, const uint16_t *d16,
                    float *group_errors, int32_t *status, void *workspace, size_t workspace_bytes,
                    void *stream);

/* Every-choice payloads ([choices] PR #3159, What does this PR do? and Usage): payloads[c] is the
 * payload of the forced encode with every group at choice c, byte-identical to iq_encode with
 * choices = c everywhere.
 * One pass: the first sweep gives every (vector, choice) minimum, the second the entry attaining
 * it under every choice, and near ties are rescored exactly per (block, choice).
 *   payloads   device uint8 [num_choices, B, block_bytes] output (any alignment)
 *   workspace  device scratch of iq_encode_workspace_size(f, rows * num_choices, cols) bytes
 *   other arguments as in iq_encode; a zero-scale block is all zero under every choice.
 * IQ_ERR_TOO_LARGE for B >= 2^27 blocks. */
IQ_API int iq_encode_every_choice(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols,
                                  const float *importance, int64_t rows_per_expert, const float *grid,
                                  const uint16_t *d16, uint8_t *payloads, int32_t *status, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* ---- local-Hessian choice search ([choices] PR #3158, What does this PR do?) -------------------
 * Picks every group's choice by the layer-output error dw H' dw^T over the block's 256-column
 * diagonal block of the input Hessian, given the every-choice payloads:
 *   H' = H_bb + perc_damp * mean(diag(H_bb)) * I            (damped as GPTQ damps; pages: 0.3)
 *   dw_c = x - q_c, q_c the decoded block of payloads[c]
 *   1. each group takes argmin_c dw_g(c)^T H'_gg dw_g(c)      (lowest c on equal values)
 *   2. two passes over the groups in ascending order: a group moves to the choice that minimises
 *      the block error with the other groups held, if that is strictly lower than with its current
 *      choice (lowest c among equal minima).
 * The payload under the searched choices is iq_encode(..., choices).  The pages use
 * importance = sqrt(diag(H)) for the every-choice encode.  Arithmetic is fp32; a pick can differ
 * from an exact evaluation only where two choices' errors are within fp32 rounding of each other.
 *   W          device [rows, cols] of dtype dt, 16-byte aligned (the weight being encoded)
 *   grid       device fp32 [grid_entries, 8], 16-byte aligned
 *   payloads   device uint8 [num_choices, B, block_bytes] (iq_encode_every_choice), 2-byte
 *              aligned (read as 16-bit words; every block_bytes is even)
 *   hessian    device fp32 [cols / 256, 256, 256]: the diagonal blocks of the symmetric input
 *              Hessian, block j for columns 256 j ... 256 j + 255; 16-byte aligned
 *   perc_damp  finite, >= 0
 *   choices    device uint8 [B, choice_groups] output
 *   status     IQ_STATUS_BAD_INPUT when a block's damping term is not finite
 *   workspace  unused (iq_local_hessian_workspace_size reports 0 bytes; may be NULL): the search
 *              decodes the payloads itself, block by block in shared memory */
IQ_API int iq_local_hessian_workspace_size(iq_format f, int64_t rows, int64_t cols, size_t *bytes);
IQ_API int iq_local_hessian_choices(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols,
                                    const float *grid, const uint8_t *payloads, const float *hessian,
                                    float perc_damp, uint8_t *choices, int32_t *status, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* ---- encoder without caller-provided scratch --------------------------------------------------
 * No counterpart on the pages: this is an addition for callers that cannot allocate device memory
 * (code running under CUDA-graph stream capture in the global mode, where cudaMalloc is refused;
 * plug-ins inside a framework that owns all device memory through its own pool; serving loops that
 * may not block on an allocation).  Same arguments and results as iq_encode, minus the workspace:
 * the scratch is one file-scope 1 MiB device array per GPU, kept until the process exits.
 *  - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *  - Size limit: a problem whose iq_encode_workspace_size exceeds 1 MiB returns IQ_ERR_TOO_LARGE
 *    before anything is launched; iq_encode_static_scratch_capacity gives the largest block count
 *    per format (114,656 blocks of 256 values for IQ1_S / IQ1_M, 128,992 for IQ2_XXS).
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress); make
 *    that first call before any stream capture.
 *  - Calls on one device share the array: each call clears what must start at zero, and calls
 *    whose kernels overlap on the GPU (e.g. on two streams) race, so keep them in order on one
 *    stream. */
IQ_API int iq_encode_static_scratch_capacity(iq_format f, int64_t *max_blocks);
IQ_API int iq_encode_static_scratch(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols,
                             const float *importance, int64_t rows_per_expert, const float *grid,
                             const uint16_t *d16, const uint8_t *choices, uint8_t *payload, float *group_errors,
                             int32_t *status, void *stream);

/* ---- decoder ([formats]: the value rule above) ------------------------------------------------
 * out[rows, cols] (device; IQ_F32, or IQ_BF16 rounded to nearest even) from payload [B,
 * block_bytes].  fp32 output is exact.  payload may have any alignment inside an allocation whose
 * start is 4-byte aligned (any cudaMalloc buffer); grid and out must be 16-byte aligned. */
IQ_API int iq_decode(iq_format f, const uint8_t *payload, int64_t rows, int64_t cols, const float *grid, void *out,
              iq_dtype out_dtype, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* IQ_B300_IQ_H */

/*
 * gg.h — C ABI of the GB300 (sm_103) grouped expert MLP.
 *
 * One Mixture-of-Experts expert layer over frozen, bias-free BF16 expert
 * weights with ragged per-expert token counts (experts with zero tokens are
 * legal): the routed-token permute, grouped FC1 with a fused SwiGLU, grouped
 * FC2, the probability-weighted unpermute/combine, and the input gradient
 * (dgrad) through the same frozen weights. Each grouped GEMM is one persistent
 * kernel launch over all experts that reads the per-expert row offsets from
 * device memory, so no call synchronises with the host.
 *
 * Sources, by page title and section:
 *  [P1] "perf(moe): add frozen grouped GEMM for adapter training"
 *       (AlignmentResearch/Megatron-LM PR #3) — "Why this change": the frozen
 *       base weights of all local experts go through one grouped kernel
 *       instead of one small GEMM per expert; "Why existing behavior remains
 *       safe": only grouped, frozen, bias-free BF16 expert weights are
 *       accepted, everything else fails during preparation; each expert
 *       parameter is a view into one contiguous buffer; forward output and
 *       input gradient, empty batches and zero-token experts are covered.
 *  [P2] "feat(moe+ssm): expert-LoRA GEMM stack and hybrid-recompute guard on
 *       the d12f6c8c base" (AlignmentResearch/Megatron-LM issue #1) — "What's
 *       in it": the grouped-offsets dtype and zero-token grouped-split
 *       contracts.
 *  [P3] NVIDIA/Megatron-LM PR #7333 — "Summary": device-metadata grouped GEMM
 *       (per-expert sizes stay on the device), 256-row expert padding,
 *       separate workspace per forward/dgrad layout, unsupported GPU/library
 *       pairs fail explicitly, batch-invariant results.
 *  [P4] "[Main] Support paged stash with device-initiated GroupedLinear"
 *       (NVIDIA/Megatron-LM PR #6828) — "What does this PR do?": grouped FC1,
 *       fused SwiGLU with GLU interleaving disabled, grouped FC2; the routing
 *       probability is applied at the fused-activation boundary; unsupported
 *       combinations are rejected instead of falling back.
 *
 * Notation: T tokens, k routed slots per token, E experts, H hidden size,
 * F expert FFN width (FC1 has 2F outputs: gate = first F, up = last F),
 * P per-expert row padding multiple, R_cap = T*k + E*(P-1) rows of every
 * permuted buffer. All matrices are row-major. Weights use the nn.Linear
 * [out, in] layout per expert and are packed contiguously over experts:
 * W1[E][2F][H], W2[E][H][F].
 *
 * Conventions common to every call:
 *  - All data pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing and keeps no state besides cached device attributes and
 *    the driver entry point used to encode TMA tensor maps. Tensor maps are
 *    encoded per call, so rewriting an expert's weights needs no invalidation.
 *  - BF16 tensors are passed as gg_bf16 (the 16-bit pattern). Every BF16
 *    matrix pointer must be 16-byte aligned; H and F must be multiples of 64.
 *  - Calls only enqueue work on `stream` (a cudaStream_t); none synchronises
 *    and none allocates. gg_read_status() is the only call that waits.
 *  - Arguments the host can check are checked before anything is launched;
 *    a failing check returns its gg_status and enqueues nothing.
 *  - Data errors only the device can see (an expert id outside [0, E),
 *    offsets that are not a valid padded prefix sum, a bounded wait inside a
 *    kernel that ran out) are written as a gg_status code into the status
 *    word at the start of the workspace `ws` (first error wins); the kernels
 *    skip the offending work and never trap. Read it with gg_read_status()
 *    and clear it with gg_clear_status().
 *  - The device must have compute capability 10.3 (GB300, sm_103); any other
 *    device gets GG_ERR_UNSUPPORTED_DEVICE. There is no fallback path.
 */
#ifndef GG_H_
#define GG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gg_bf16;                 /* BF16 bit pattern */
typedef struct CUstream_st* gg_stream_t;  /* same handle as cudaStream_t */

typedef enum gg_status {
  GG_OK = 0,
  GG_ERR_INVALID_ARG = 1,          /* null pointer, negative size, k > 32, ... */
  GG_ERR_UNSUPPORTED_SHAPE = 2,    /* H or F not a multiple of 64, E > 1024, ... */
  GG_ERR_MISALIGNED = 3,           /* a matrix pointer is not 16-byte aligned */
  GG_ERR_WORKSPACE_TOO_SMALL = 4,
  GG_ERR_UNSUPPORTED_DEVICE = 5,   /* not compute capability 10.3 */
  GG_ERR_CUDA = 6,                 /* a CUDA runtime or driver call failed */
  /* codes written by kernels into the workspace status word */
  GG_ERR_DEVICE_BAD_EXPERT_ID = 16,  /* idx[t][j] outside [0, E): pair skipped */
  GG_ERR_DEVICE_BAD_OFFSETS = 17,    /* offsets not monotone / offsets[E] > R_cap */
  GG_ERR_DEVICE_BAD_ROW = 18,        /* a row map entry outside [-1, R_cap) */
  GG_ERR_DEVICE_TIMEOUT = 19         /* a bounded in-kernel wait gave up */
} gg_status;

/* Epilogues. The gated activations ([P4] "What does this PR do?": fused
 * SwiGLU or QuickGeGLU, GLU interleaving disabled) are act(g) * u with
 * act(g) = g * sigmoid(alpha * g): alpha = 1 (SwiGLU) or 1.702 (QuickGeGLU,
 * the QuickGELU gate; the page names it without a formula). */
typedef enum gg_epilogue {
  GG_EPI_NONE = 0,        /* store the BF16-rounded accumulator */
  GG_EPI_SWIGLU = 1,      /* gg_grouped_fwd only: fused SwiGLU, see below */
  GG_EPI_SWIGLU_BWD = 2,  /* gg_grouped_dgrad only: fused SwiGLU backward */
  GG_EPI_QGEGLU = 3,      /* gg_grouped_fwd only: fused QuickGeGLU */
  GG_EPI_QGEGLU_BWD = 4   /* gg_grouped_dgrad only: fused QuickGeGLU backward */
} gg_epilogue;

/* Human-readable name of a status code (static string, never NULL). */
const char* gg_status_string(int status);

/* Library version string, e.g. "gg 0.1 sm_103a". */
const char* gg_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads). Lets a caller count the launches inside a timed region. */
uint64_t gg_launch_count(void);

/* Bytes of workspace every call below needs for a batch of T tokens with
 * top-k routing over E experts. The first 256 bytes hold the status word;
 * the rest is scratch for the permute's per-block expert histograms (one
 * int32 per expert and block; at most 128 blocks, each of a multiple of
 * 1024 pairs, at least 1024). */
size_t gg_workspace_size(int T, int k, int E);

/* Zero the status word at the start of `ws` (stream-ordered). */
gg_status gg_clear_status(void* ws, gg_stream_t stream);

/* Copy the status word to *host_status after all work queued on `stream`
 * so far has finished. The only call that waits for the device. */
gg_status gg_read_status(const void* ws, gg_stream_t stream, int32_t* host_status);

/* ---------------------------------------------------------------------------
 * gg_permute — routed-token permute ([P1] "B200 throughput evidence": ordinary
 * all-to-all dispatch groups tokens by expert before the grouped GEMM; [P2]
 * zero-token grouped-split contracts; [P3] 256-row expert padding).
 *
 * Stable counting sort of the T*k (token, slot) pairs by expert id: expert
 * e's rows are its pairs in ascending (t, j) order, then zero rows up to a
 * multiple of `pad_multiple` (P >= 1). Outputs:
 *   offsets[E+1]      int32, offsets[0] = 0, offsets[e+1] - offsets[e] = the
 *                     padded row count of expert e (0 for an empty expert);
 *   row_of_slot[T*k]  int32, row of pair t*k+j (-1 if its id was invalid);
 *   slot_of_row[R_cap] int32, pair id t*k+j of a row, -1 on padding rows and
 *                     on rows >= offsets[E];
 *   prob_of_row[R_cap] fp32, prob[t][j] of the row's pair, 0 on padding and
 *                     on rows >= offsets[E];
 *   Xp[R_cap][H]      BF16, Xp[row] = x[t]; zero on padding rows; rows
 *                     >= offsets[E] are left untouched. Xp may be NULL:
 *                     then only the row maps and offsets are produced (the
 *                     gathered GEMMs below read the token rows themselves).
 * Inputs: x[T][H] BF16, idx[T][k] int32 expert ids, prob[T][k] fp32; k <= 32.
 * Indices are bit-exact and independent of scheduling. T = 0 only writes
 * offsets (all zero). An id outside [0, E) sets GG_ERR_DEVICE_BAD_EXPERT_ID
 * and that pair is dropped. Workspace: gg_workspace_size(T, k, E) bytes.
 * ------------------------------------------------------------------------- */
gg_status gg_permute(const gg_bf16* x, const int32_t* idx, const float* prob,
                     int T, int H, int k, int E, int pad_multiple,
                     gg_bf16* Xp, int32_t* offsets, int32_t* row_of_slot,
                     int32_t* slot_of_row, float* prob_of_row,
                     void* ws, size_t ws_bytes, gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * gg_permute_noalloc — gg_permute for callers that cannot allocate device
 * memory (the pages have no counterpart: this is a service of this library).
 *
 * Some callers cannot provide a workspace: runtimes whose memory pool owns
 * the whole GPU after start-up and forbid cudaMalloc on the hot path, plugins
 * that receive only pre-sized input and output buffers from their host, C
 * callers without a device allocator. This entry point computes exactly what
 * gg_permute computes (same arguments, same outputs, bit-identical results)
 * but takes no `ws`: its scratch (status word + per-block expert histograms)
 * lives in a fixed 256 KiB (+ 256 bytes) array in the library's device
 * image, which every GPU that loads the library keeps until the process
 * exits. It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - Limit: gg_workspace_size(T, k, E) <= 256 KiB + 256 bytes: any batch for
 *     E <= 512; for larger E, T*k <= 1024 * floor(65536 / E) pairs (65,536
 *     at E = 1024). Larger batches are rejected with
 *     GG_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - Xp may be NULL (row maps, offsets and per-row probabilities only), and
 *     x is then not read, exactly as for gg_permute.
 *   - Set-up: the first call on a device (made with that device current)
 *     looks up the array's device address; make that first call before any
 *     stream capture. Only a successful lookup is kept: if it fails the call
 *     returns GG_ERR_CUDA and the next call on that device tries again.
 *   - Device ordinals of 64 and above are refused with
 *     GG_ERR_UNSUPPORTED_DEVICE.
 *   - Every call on a device shares the one array and it keeps the previous
 *     call's contents; each call clears the status word itself. Calls whose
 *     work overlaps on the GPU (different streams without ordering between
 *     them) race on the array and must not be issued.
 *   - There is no readable status word: an expert id outside [0, E) is
 *     visible in the outputs as row_of_slot == -1 and offsets[E] < T*k.
 * ------------------------------------------------------------------------- */
gg_status gg_permute_noalloc(const gg_bf16* x, const int32_t* idx, const float* prob,
                             int T, int H, int k, int E, int pad_multiple,
                             gg_bf16* Xp, int32_t* offsets, int32_t* row_of_slot,
                             int32_t* slot_of_row, float* prob_of_row,
                             gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * gg_permute_rows — gather of a token-major tensor into the permuted row
 * order of an earlier gg_permute (the combine's backward: the output
 * gradient dOut[T][H] is routed to the rows its token was sent to), using
 * that permute's row maps and padding multiple:
 *   dst[row_of_slot[t*k+j]] = src[t] for every pair with a row, and (when
 *   pad_multiple > 1) zero on the padding rows below offsets[E] (slot -1);
 *   rows >= offsets[E] are left untouched.
 * src[T][H], dst[R_cap][H] BF16; k <= 32. With prob NULL the probability
 * is not applied (the dgrad FC2 epilogue applies it, FC2 being linear); with
 * prob[T][k] fp32 each copy is scaled, dst[row] = bf16(prob[t][j] * src[t])
 * in fp32 — the optional pre-FC1 probability multiply ([P4] "What does this
 * PR do?"). A row map entry outside [-1, R_cap) sets GG_ERR_DEVICE_BAD_ROW.
 * ------------------------------------------------------------------------- */
gg_status gg_permute_rows(const gg_bf16* src, const int32_t* row_of_slot,
                          const int32_t* slot_of_row, const int32_t* offsets,
                          int T, int H, int k, int E, int pad_multiple, int R_cap,
                          const float* prob, gg_bf16* dst, void* ws, size_t ws_bytes,
                          gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * gg_grouped_fwd — grouped GEMM over all experts in one persistent launch
 * ([P1] "Why this change": one grouped kernel instead of one small GEMM per
 * expert; [P3] "Summary": per-expert sizes read from device metadata).
 *
 * For every expert e and every row r in [offsets[e], offsets[e+1]):
 *   acc[r][n] = sum_c A[r][c] * B[e][n][c]     (fp32 accumulation, n < N)
 * A[R_cap][K] BF16 row-major, B[E][N][K] BF16 (nn.Linear weight per expert),
 * offsets[E+1] int32 on the device. K and N must be multiples of 64.
 *   GG_EPI_NONE:   C[R_cap][N]   = bf16(acc). H1_save must be NULL.
 *   GG_EPI_SWIGLU: N = 2F; with g = bf16(acc[:, :F]) and u = bf16(acc[:, F:])
 *                  ([P4] "What does this PR do?": fused SwiGLU, gate and up
 *                  halves not interleaved), C[R_cap][F] = bf16(silu(g) * u)
 *                  computed in fp32 from the rounded g and u, and, when
 *                  H1_save is not NULL, H1_save[R_cap][2F] = [g, u] (kept
 *                  for the backward pass).
 *   GG_EPI_QGEGLU: the same with g * sigmoid(1.702 g) in place of silu(g).
 *   prob_of_row (nullable, gated epilogues only): the weighted activation
 *                  ([P4]: the probability at the fused-activation boundary),
 *                  C[r][j] = bf16(prob_of_row[r] * act(g) * u) in fp32.
 * Rows outside [0, offsets[E]) are never written. Results of a row depend
 * only on that row and its expert's weights (bitwise batch invariance).
 * Offsets that are not monotone, do not start at 0 or end past R_cap set
 * GG_ERR_DEVICE_BAD_OFFSETS and nothing is computed.
 * ------------------------------------------------------------------------- */
gg_status gg_grouped_fwd(const gg_bf16* A, const gg_bf16* B, const int32_t* offsets,
                         int E, int R_cap, int K, int N, gg_epilogue epi,
                         gg_bf16* C, gg_bf16* H1_save, const float* prob_of_row,
                         void* ws, size_t ws_bytes, gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * gg_swiglu — the unfused SwiGLU ([P4] "What does this PR do?") on a stored
 * FC1 output, bitwise identical to the GG_EPI_SWIGLU epilogue:
 *   A[r][j] = bf16(silu(H1[r][j]) * H1[r][F + j]) in fp32, r < offsets[E].
 * H1[R_cap][2F], A[R_cap][F] BF16; F a multiple of 64.
 * ------------------------------------------------------------------------- */
gg_status gg_swiglu(const gg_bf16* H1, const int32_t* offsets, int E, int R_cap,
                    int F, gg_bf16* A, gg_stream_t stream);

/* gg_glu — the unfused gated activation of either kind (epi = GG_EPI_SWIGLU
 * or GG_EPI_QGEGLU), optionally weighted by prob_of_row (nullable), bitwise
 * identical to the matching gg_grouped_fwd epilogue:
 *   A[r][j] = bf16([prob_of_row[r] *] act(H1[r][j]) * H1[r][F + j]). */
gg_status gg_glu(const gg_bf16* H1, const int32_t* offsets, int E, int R_cap, int F,
                 gg_epilogue epi, const float* prob_of_row, gg_bf16* A, gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * gg_grouped_dgrad — input gradient of gg_grouped_fwd through the same
 * frozen weights ([P1] "Why existing behavior remains safe": input-gradient
 * parity; the weights get no gradient). B is the FORWARD weight B[E][N][K];
 * the kernel reads it transposed (N-contiguous) straight from that layout:
 *   acc[r][c] = sum_n dC[r][n] * B[e][n][c]    (fp32, c < K)
 * dC[R_cap][N] BF16. K and N multiples of 64.
 *   prob_of_row (nullable): acc[r][:] *= prob_of_row[r] in fp32 first
 *                  ([P4]: the routing probability at the activation boundary).
 *   GG_EPI_NONE:   dA[R_cap][K] = bf16(acc). H1 must be NULL.
 *   GG_EPI_SWIGLU_BWD: the SwiGLU backward with K = F, using the saved
 *                  H1[R_cap][2F] = [g, u] (BF16) and s = sigmoid(g):
 *                    dA[r][j]     = bf16(acc * u * s * (1 + g * (1 - s)))
 *                    dA[r][F + j] = bf16(acc * g * s)
 *                  so dA is [R_cap][2F] (the gradient w.r.t. FC1's output).
 *   GG_EPI_QGEGLU_BWD: the same with s = sigmoid(1.702 g) and the gate
 *                  derivative s * (1 + 1.702 * g * (1 - s)).
 *   rowdot (nullable, gated backward epilogues only): partial sums for the routing-
 *                  probability gradient ([P4] "What does this PR do?": the
 *                  probability multiplies the expert output at the combine,
 *                  so its gradient is <dOut_t, Yp[r]> = <dC[r] * W_e, A[r]>
 *                  for the FC2 weight W_e and activation output A). With
 *                  a[r][j] = bf16(act(g) * u) (the forward's unweighted A,
 *                  same arithmetic; also right when the forward weighted the
 *                  activation, whose output is linear in the probability) and
 *                  the accumulator taken BEFORE the prob_of_row scale:
 *                    rowdot[r][b] = sum_{128b <= j < min(128b + 128, F)} acc[r][j] * a[r][j]
 *                  in fp32 (any order), for b < gg_rowdot_blocks(K); layout
 *                  [R_cap][gg_rowdot_stride(K)] fp32 (one 32-byte-aligned
 *                  group per row; entries b >= gg_rowdot_blocks(K) are not
 *                  written), 32-byte aligned. The blocks' sum
 *                  (gg_unpermute_combine's dprob) is the gradient.
 * Rows outside [0, offsets[E]) are never written.
 * ------------------------------------------------------------------------- */
gg_status gg_grouped_dgrad(const gg_bf16* dC, const gg_bf16* B, const int32_t* offsets,
                           int E, int R_cap, int K, int N, gg_epilogue epi,
                           const gg_bf16* H1, const float* prob_of_row, gg_bf16* dA,
                           float* rowdot, void* ws, size_t ws_bytes, gg_stream_t stream);

/* Number of fp32 partial sums per permuted row written to `rowdot` by the
 * SwiGLU-backward dgrad with F = K: 2 * ceil(F / 256) (0 if F <= 0), and the
 * row stride of `rowdot` in floats: gg_rowdot_blocks(F) rounded up to a
 * multiple of 8. */
int gg_rowdot_blocks(int F);
int gg_rowdot_stride(int F);

/* ---------------------------------------------------------------------------
 * gg_grouped_fwd_gather / gg_grouped_dgrad_gather — the same GEMMs with the
 * permuted operand gathered on the fly instead of read from a materialised
 * buffer ([P3] "Summary": per-expert metadata on the device; the permute
 * only has to produce row maps):
 *   A[r] = src[slot_of_row[r] / k] for slot_of_row[r] >= 0, zero otherwise,
 * with src token-major [T][K] (fwd: x; dgrad: dOut, then [T][N]) and
 * slot_of_row / k from gg_permute. Every other argument, output and error is
 * as in gg_grouped_fwd / gg_grouped_dgrad, and the results are bitwise equal
 * to running them on the gathered buffer (gg_permute's Xp, or
 * gg_permute_rows' output). The tensor core's A tiles are loaded by TMA
 * four-row gathers, so the permuted copy never exists: this saves its
 * R_cap x K x 2 bytes of memory, at a throughput cost (each A row is gathered
 * once per 256-column block, and many small TMA requests run well below the
 * tile-load rate), so the whole-layer calls use the materialised path.
 * ------------------------------------------------------------------------- */
gg_status gg_grouped_fwd_gather(const gg_bf16* src, int T, const int32_t* slot_of_row, int k,
                                const gg_bf16* B, const int32_t* offsets,
                                int E, int R_cap, int K, int N, gg_epilogue epi,
                                gg_bf16* C, gg_bf16* H1_save, const float* prob_of_row,
                                void* ws, size_t ws_bytes, gg_stream_t stream);

gg_status gg_grouped_dgrad_gather(const gg_bf16* src, int T, const int32_t* slot_of_row, int k,
                                  const gg_bf16* B, const int32_t* offsets,
                                  int E, int R_cap, int K, int N, gg_epilogue epi,
                                  const gg_bf16* H1, const float* prob_of_row, gg_bf16* dA,
                                  float* rowdot, void* ws, size_t ws_bytes,
                                  gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * gg_unpermute_combine — probability-weighted combine ([P4] "What does this
 * PR do?": the probability boundary; [P1]: the all-to-all combine side):
 *   out[t] = bf16( sum_{j<k} prob[t][j] * Yp[row_of_slot[t*k+j]] )
 * accumulated in fp32 in slot order j = 0..k-1 and rounded once. prob NULL
 * gives the unweighted sum (the input-gradient combine). Pairs whose row is
 * -1 contribute nothing. Yp[R_cap][H], out[T][H] BF16; k <= 32. A row outside
 * [-1, R_cap) sets GG_ERR_DEVICE_BAD_ROW and is skipped.
 * dprob (nullable): the routing-probability gradient, from exactly one of
 *   rowdot (the partial sums of gg_grouped_dgrad's `rowdot`, [R_cap][stride]
 *     fp32 with stride = n_rowdot rounded up to a multiple of 8,
 *     n_rowdot >= 1, 32-byte aligned):
 *       dprob[t*k+j] = sum_{b < n_rowdot} rowdot[row_of_slot[t*k+j]][b]
 *     in fp32, b ascending;
 *   dot_src (token-major [T][H] BF16, the pre-FC1 form: Xp = prob * x):
 *       dprob[t*k+j] = <dot_src[t], Yp[row_of_slot[t*k+j]]>
 *     in fp32 (fixed order);
 * and 0 for a pair without a row. dprob NULL requires rowdot and dot_src
 * NULL (n_rowdot ignored).
 * ------------------------------------------------------------------------- */
gg_status gg_unpermute_combine(const gg_bf16* Yp, const int32_t* row_of_slot,
                               const float* prob, int T, int k, int H, int R_cap,
                               gg_bf16* out, const float* rowdot, int n_rowdot,
                               const gg_bf16* dot_src, float* dprob, void* ws,
                               size_t ws_bytes, gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * gg_unpermute_combine_dot — the combine of gg_unpermute_combine together
 * with a routing-probability gradient that is a dot product of a token row
 * with a second permuted tensor ([P4] "What does this PR do?": the
 * probability boundary; with the probability applied at the combine,
 * out_t = sum_j p_tj * Yp[row(t, j)], so d out / d p_tj = Yp[row(t, j)]):
 *   out[t]       = bf16( sum_{j<k} [prob[t][j] *] Sp[row_of_slot[t*k+j]] )
 *                  fp32 in slot order, one rounding (prob NULL: plain sum);
 *   dprob[t*k+j] = <dot_src[t], dot_rows[row_of_slot[t*k+j]]>
 *                  fp32, fixed order; 0 for a pair without a row.
 * The MXFP8 layer's backward calls it with Sp = dXp (out = dX), dot_src =
 * dOut and dot_rows = the forward's Yp, so that its probability gradient is
 * formed from its definition rather than from the quantised input-gradient
 * GEMM. Sp, dot_rows [R_cap][H]; dot_src, out [T][H] BF16 (16-byte
 * aligned); dprob [T][k] fp32; k <= 32. All pointers are required when
 * T > 0 (GG_ERR_INVALID_ARG). A row outside [-1, R_cap) sets
 * GG_ERR_DEVICE_BAD_ROW in the status word of `ws` and is skipped.
 * ------------------------------------------------------------------------- */
gg_status gg_unpermute_combine_dot(const gg_bf16* Sp, const int32_t* row_of_slot,
                                   const float* prob, int T, int k, int H, int R_cap,
                                   gg_bf16* out, const gg_bf16* dot_src,
                                   const gg_bf16* dot_rows, float* dprob, void* ws,
                                   size_t ws_bytes, gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * Helpers of expert parallelism: the all-to-all dispatch around the local
 * grouped GEMM ([P1] "B200 throughput evidence": ordinary all-to-all
 * dispatch; each of n_ranks ranks owns El consecutive experts).
 *
 * gg_ep_split_ids — for every pair i < n of the global expert ids idx[n]:
 *   dest[i] = idx[i] / El (the owning rank), local_eid[i] = idx[i] % El (the
 *   expert on that rank), for ids in [0, El * n_ranks). Any other id gives
 *   dest = local_eid = -1 and sets GG_ERR_DEVICE_BAD_EXPERT_ID (a permute by
 *   dest then leaves the pair without a row). idx, dest, local_eid int32 on
 *   the device, owned by the caller; El * n_ranks must fit an int.
 *
 * gg_gather_rows32 — out[i][c] = src[index[i]][c] for i < n, c < width, on
 *   32-bit elements (int32 or fp32 bits): src[src_rows][width],
 *   index[n] int32, out[n][width], all on the device and owned by the
 *   caller. index -1 gives a zero row; an index outside [-1, src_rows) gives
 *   a zero row and sets GG_ERR_DEVICE_BAD_ROW. Used to carry each pair's
 *   local expert id into send order and to bring the probability gradients
 *   of the returned rows back into token order.
 *
 * Both write only their outputs and the status word at the start of ws
 * (>= gg_workspace_size(1, 1, 1) bytes), and enqueue nothing when n == 0.
 * ------------------------------------------------------------------------- */
gg_status gg_ep_split_ids(const int32_t* idx, int n, int El, int n_ranks, int32_t* dest,
                          int32_t* local_eid, void* ws, size_t ws_bytes, gg_stream_t stream);
gg_status gg_gather_rows32(const void* src, int src_rows, int width, const int32_t* index,
                           int n, void* out, void* ws, size_t ws_bytes, gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * Whole expert layer. The caller owns one device buffer that holds every
 * intermediate; gg_moe_buffers_bind() carves it (256-byte aligned pieces).
 * ------------------------------------------------------------------------- */
typedef struct gg_moe_buffers {
  gg_bf16* Xp;          /* [R_cap][H]  permuted input                     */
  gg_bf16* H1;          /* [R_cap][2F] FC1 output (BF16), kept for dgrad  */
  gg_bf16* A;           /* [R_cap][F]  SwiGLU output                      */
  gg_bf16* Yp;          /* [R_cap][H]  FC2 output                         */
  gg_bf16* dYp;         /* [R_cap][H]  permuted output gradient           */
  gg_bf16* dH;          /* [R_cap][2F] gradient w.r.t. FC1 output         */
  gg_bf16* dXp;         /* [R_cap][H]  gradient w.r.t. permuted input     */
  int32_t* offsets;     /* [E+1]                                          */
  int32_t* row_of_slot; /* [T*k]                                          */
  int32_t* slot_of_row; /* [R_cap]                                        */
  float* prob_of_row;   /* [R_cap]                                        */
  float* rowdot;        /* [R_cap][gg_rowdot_stride(F)] dprob partial sums */
  void* ws;             /* gg_workspace_size(T, k, E) bytes, status first */
  size_t ws_bytes;
} gg_moe_buffers;

/* Bytes of the single buffer gg_moe_buffers_bind() carves. */
size_t gg_moe_buffers_size(int T, int H, int F, int k, int E, int pad_multiple);

/* Fill *out with pointers into `base` (device memory, 256-byte aligned,
 * `bytes` >= gg_moe_buffers_size(...)). Host-only; enqueues nothing. */
gg_status gg_moe_buffers_bind(void* base, size_t bytes, int T, int H, int F, int k,
                              int E, int pad_multiple, gg_moe_buffers* out);

/* Forward: permute -> grouped FC1 + fused SwiGLU (H1 kept) -> grouped FC2
 * -> probability-weighted combine into out[T][H]. All on `stream`, no host
 * synchronisation. */
gg_status gg_moe_mlp_fwd(const gg_bf16* x, const int32_t* idx, const float* prob,
                         const gg_bf16* W1, const gg_bf16* W2,
                         int T, int H, int F, int k, int E, int pad_multiple,
                         gg_bf16* out, const gg_moe_buffers* buf, gg_stream_t stream);

/* Input gradient of gg_moe_mlp_fwd (same buffers, after the forward):
 * permute dOut -> dgrad FC2 with probability scale and fused SwiGLU
 * backward -> dgrad FC1 -> unweighted combine into dX[T][H]. With dprob
 * (nullable) also the routing-probability gradient dprob[T][k] fp32,
 * dprob[t][j] = <dOut[t], FC2 output of pair (t, j)>, from partial sums the
 * SwiGLU-backward epilogue accumulates and the dX combine adds up. */
gg_status gg_moe_mlp_bwd(const gg_bf16* dOut, const gg_bf16* W1, const gg_bf16* W2,
                         int T, int H, int F, int k, int E, int pad_multiple,
                         gg_bf16* dX, float* dprob, const gg_moe_buffers* buf,
                         gg_stream_t stream);

/* Layer options ([P4] "What does this PR do?"): the gated activation and the
 * place where the routing probability p of a (token, slot) pair is applied. */
typedef enum gg_activation {
  GG_ACT_SWIGLU = 0,      /* silu(g) * u                                   */
  GG_ACT_QGEGLU = 1       /* g * sigmoid(1.702 g) * u                      */
} gg_activation;
typedef enum gg_prob_mode {
  GG_PROB_COMBINE = 0,    /* out_t = sum_j p * FC2(act): gg_moe_mlp_fwd     */
  GG_PROB_ACTIVATION = 1, /* A = p * act (weighted activation), out_t =
                             sum_j FC2(A): the same function, rounded once
                             more inside FC2's input                       */
  GG_PROB_PRE_FC1 = 2     /* Xp = p * x before FC1, out_t = sum_j FC2(act):
                             a different function                          */
} gg_prob_mode;
typedef struct gg_moe_options {
  int activation;         /* gg_activation */
  int prob_mode;          /* gg_prob_mode  */
  int recompute_h1;       /* 0: the forward stores FC1's output H1 for the
                             backward; 1: the forward does not store it and
                             the backward recomputes it (a plain grouped FC1
                             on the kept Xp, same bits: "save vs recompute"
                             of [P1] "Scope deliberately omitted" /
                             expert_fc1_act). The H1 region of the buffers is
                             then scratch of the backward call only, free for
                             the caller between forward and backward. */
} gg_moe_options;

/* gg_moe_mlp_fwd / gg_moe_mlp_bwd with options (NULL = SwiGLU, probability
 * at the combine: the calls above). The backward needs the forward's x and
 * prob for GG_PROB_PRE_FC1 (dX_t = sum_j p * dXp[row], dprob = <x_t,
 * dXp[row]>); they are ignored (may be NULL) otherwise. Returns
 * GG_ERR_INVALID_ARG for an unknown activation or mode. */
gg_status gg_moe_mlp_fwd_ex(const gg_bf16* x, const int32_t* idx, const float* prob,
                            const gg_bf16* W1, const gg_bf16* W2,
                            int T, int H, int F, int k, int E, int pad_multiple,
                            const gg_moe_options* opt, gg_bf16* out,
                            const gg_moe_buffers* buf, gg_stream_t stream);
gg_status gg_moe_mlp_bwd_ex(const gg_bf16* dOut, const gg_bf16* x, const float* prob,
                            const gg_bf16* W1, const gg_bf16* W2,
                            int T, int H, int F, int k, int E, int pad_multiple,
                            const gg_moe_options* opt, gg_bf16* dX, float* dprob,
                            const gg_moe_buffers* buf, gg_stream_t stream);

/* -------------------------------------------------------------------------
 * MXFP8 expert layer. [P3] "Validation": routed expert projections only in
 * MXFP8, other modules BF16; [P4] "End-to-end GB300 validation": MXFP8 on
 * GB300. The pages do not define the encoding; it is read as the OCP
 * microscaling format with E4M3 elements: one E8M0 scale 2^e per 32
 * consecutive elements along each GEMM's reduction dimension, e the smallest
 * exponent with max|v| / 2^e <= 448 (clamped to [-127, 127]; -127 for an
 * all-zero block), elements v * 2^-e rounded to nearest-even E4M3. Both
 * operands of every GEMM are MXFP8 (block-scaled tcgen05 MMAs, FP32
 * accumulation). Results pass between GEMMs as BF16 values that the next
 * GEMM's quantiser reads: H1 (kept for the backward) and the activation
 * bf16(act(H1)) before it is quantised for FC2, and likewise dH1 before the
 * second input-gradient GEMM.
 *
 * Shapes: H and F multiples of 128, E <= 1024. The weights are quantised once
 * (gg_mx_prepare_weights): along their input dimension for the forward and,
 * transposed, along their output dimension for the input gradient.
 *
 * Scale tiles (bytes holding E8M0 codes e + 127):
 *  - activation operands: per expert-local 128-row tile t of expert e, tile
 *    index tiles_before[e] + t (tiles_before = exclusive prefix sum of
 *    ceil(rows_e / 128)); for K = 128 * KG columns a tile holds KG blocks of
 *    512 bytes, byte (r % 32) * 16 + (r / 32) * 4 + b of block kg holding the
 *    scale of row r of the tile, 32-column block 4 * kg + b. Rows of a tile
 *    past the expert's end hold code 0. Every activation scale buffer holds
 *    gg_mx_row_tiles() tiles.
 *  - weight operands: per expert and 256-column tile of the GEMM that reads
 *    them (FC1: 128 gate rows followed by the 128 matching up rows, FC1 tile
 *    j covering gate rows 128j..), KG blocks of 1024 bytes, byte
 *    (n / 128) * 512 + ((n % 128) % 32) * 16 + ((n % 128) / 32) * 4 + b for
 *    column n of the tile; columns past the weight's rows hold code 0.
 * ------------------------------------------------------------------------- */

/* Row-scale tiles of one activation operand: ceil(R_cap / 128) + E. */
int gg_mx_row_tiles(int T, int k, int E, int pad_multiple);

/* Byte offsets of the prepared weights inside the buffer of
 * gg_mx_prepare_weights (each piece 256-byte aligned). */
typedef struct gg_mx_weights_layout {
  size_t w1, w1_scales;   /* FC1: E4M3 [E][2F][H], along H; scale tiles
                             [E][F/128][H/128]                             */
  size_t w2, w2_scales;   /* FC2: E4M3 [E][H][F], along F;
                             [E][ceil(H/256)][F/128]                       */
  size_t w2t, w2t_scales; /* input gradient of FC2: E4M3 [E][F][H] = W2
                             transposed, along H; [E][ceil(F/256)][H/128]  */
  size_t w1t, w1t_scales; /* input gradient of FC1: E4M3 [E][H][2F] = W1
                             transposed, along 2F; [E][ceil(H/256)][2F/128] */
  size_t bytes;           /* total                                         */
} gg_mx_weights_layout;

/* Host only. GG_ERR_UNSUPPORTED_SHAPE unless H % 128 == 0, F % 128 == 0 and
 * 0 < E <= 1024. */
gg_status gg_mx_weights_layout_of(int E, int H, int F, gg_mx_weights_layout* out);

/* Quantise the frozen BF16 weights W1 [E][2F][H] and W2 [E][H][F] into the
 * four MXFP8 operands at `mxw` (device, 256-byte aligned, `bytes` >= the
 * layout's total). Run once per weight set; the layer calls read `mxw` only. */
gg_status gg_mx_prepare_weights(const gg_bf16* W1, const gg_bf16* W2, int E, int H, int F,
                                void* mxw, size_t bytes, gg_stream_t stream);

/* Permuted MXFP8 activation operand, from the permute's maps. Writes
 * tiles_before[E+1] from offsets, then for every (token t, slot j) with a
 * row r = row_of_slot[t*k+j]: Q[r] = the E4M3 codes of src[t] (times
 * prob[t*k+j], rounded to BF16, when prob is not NULL) and its scales into
 * the tiles of the expert whose rows contain r. Every other scale byte of S
 * (n_tiles tiles of K/128 blocks) is set to code 0: rows that no pair
 * reaches, padding rows and the tiles past the last expert's; padding rows
 * (pad_multiple > 1, slot -1) of Q are zeroed. src [T][K] BF16,
 * Q [R_cap][K], K a multiple of 128. A row outside [0, R_cap) is skipped
 * and reported as GG_ERR_DEVICE_BAD_ROW. */
gg_status gg_mx_quantize_rows(const gg_bf16* src, int T, int K, int k,
                              const int32_t* row_of_slot, const int32_t* slot_of_row,
                              const int32_t* offsets, const float* prob, int E,
                              int pad_multiple, int n_tiles, int32_t* tiles_before, uint8_t* Q,
                              uint8_t* S, void* ws, size_t ws_bytes, gg_stream_t stream);

/* The four MXFP8 grouped GEMMs of the layer, with the weights of `mxw`:
 *  GG_MX_FC1        A = Xq [R_cap][H]: H1 = bf16(A W1^T) stored to H1 (may
 *                   be NULL), a = bf16(act(H1) [* row_scale]) quantised to
 *                   Cq [R_cap][F] + Cs;
 *  GG_MX_FC2        A = Aq [R_cap][F]: C = bf16(A W2^T) [R_cap][H];
 *  GG_MX_DGRAD_FC2  A = dYq [R_cap][H]: dA = (A W2) [* row_scale], dH1 =
 *                   bf16(act'(H1) applied to dA) quantised to Cq [R_cap][2F]
 *                   + Cs; rowdot (may be NULL) gets per-row partial sums of
 *                   <A W2, act(H1)>, gg_mx_rowdot_blocks(F) of them
 *                   (2 * ceil(F / 128): one per 64 columns),
 *                   gg_mx_rowdot_stride(F) floats apart;
 *  GG_MX_DGRAD_FC1  A = dHq [R_cap][2F]: C = bf16(A W1) [R_cap][H].
 * `activation` is a gg_activation; As, Cs hold n_tiles row-scale tiles. */
typedef enum gg_mx_gemm {
  GG_MX_FC1 = 0,
  GG_MX_FC2 = 1,
  GG_MX_DGRAD_FC2 = 2,
  GG_MX_DGRAD_FC1 = 3
} gg_mx_gemm;
int gg_mx_rowdot_blocks(int F);
int gg_mx_rowdot_stride(int F);
gg_status gg_mx_grouped_gemm(int which, int activation, const uint8_t* Aq, const uint8_t* As,
                             const void* mxw, const int32_t* offsets, int E, int R_cap, int H,
                             int F, int n_tiles, gg_bf16* C, uint8_t* Cq, uint8_t* Cs,
                             gg_bf16* H1, const float* row_scale, float* rowdot, void* ws,
                             size_t ws_bytes, gg_stream_t stream);

/* Buffers of the MXFP8 layer, carved by gg_mx_buffers_bind(). */
typedef struct gg_mx_buffers {
  uint8_t* Xq;          /* [R_cap][H]  permuted input, E4M3               */
  uint8_t* Xs;          /* its row-scale tiles                            */
  gg_bf16* H1;          /* [R_cap][2F] FC1 output, kept for the backward  */
  uint8_t* Aq;          /* [R_cap][F]  activation, E4M3                   */
  uint8_t* As;
  gg_bf16* Yp;          /* [R_cap][H]  FC2 output                         */
  uint8_t* dYq;         /* [R_cap][H]  permuted output gradient, E4M3     */
  uint8_t* dYs;
  uint8_t* dHq;         /* [R_cap][2F] gradient of H1, E4M3               */
  uint8_t* dHs;
  gg_bf16* dXp;         /* [R_cap][H]  gradient of the permuted input     */
  int32_t* offsets;     /* [E+1]                                          */
  int32_t* row_of_slot; /* [T*k]                                          */
  int32_t* slot_of_row; /* [R_cap]                                        */
  float* prob_of_row;   /* [R_cap]                                        */
  int32_t* tiles_before;/* [E+1]                                          */
  float* rowdot;        /* [R_cap][gg_mx_rowdot_stride(F)]                */
  int n_tiles;          /* gg_mx_row_tiles(T, k, E, pad_multiple)         */
  void* ws;             /* gg_workspace_size(T, k, E) bytes, status first */
  size_t ws_bytes;
} gg_mx_buffers;

size_t gg_mx_buffers_size(int T, int H, int F, int k, int E, int pad_multiple);
gg_status gg_mx_buffers_bind(void* base, size_t bytes, int T, int H, int F, int k, int E,
                             int pad_multiple, gg_mx_buffers* out);

/* The MXFP8 layer: forward (permute -> quantise rows -> FC1 + activation +
 * quantise -> FC2 -> combine into out[T][H]) and backward (quantise dOut
 * rows -> input gradient of FC2 + activation backward + quantise -> input
 * gradient of FC1 -> combine into dX[T][H], dprob[T][k] when not NULL).
 * Options as gg_moe_mlp_fwd_ex except recompute_h1, which must be 0
 * (GG_ERR_INVALID_ARG). dprob is the gradient where the probability enters
 * the forward: <dOut_t, Yp[row]> on the forward's kept Yp when it is applied
 * at the combine (formed by gg_unpermute_combine_dot; no quantiser lies
 * between p and out), the row sum of dA0 * act(H1) with the weighted
 * activation (dA0 the input gradient of FC2, before the probability scale;
 * the probability sits inside FC2's quantised operand), <x_t, dXp[row]> for
 * the pre-FC1 mode. The forward's Yp must therefore still hold its values
 * when the combine-mode backward runs with dprob. */
gg_status gg_moe_mlp_fwd_mx(const gg_bf16* x, const int32_t* idx, const float* prob,
                            const void* mxw, int T, int H, int F, int k, int E,
                            int pad_multiple, const gg_moe_options* opt, gg_bf16* out,
                            const gg_mx_buffers* buf, gg_stream_t stream);
gg_status gg_moe_mlp_bwd_mx(const gg_bf16* dOut, const gg_bf16* x, const float* prob,
                            const void* mxw, int T, int H, int F, int k, int E,
                            int pad_multiple, const gg_moe_options* opt, gg_bf16* dX,
                            float* dprob, const gg_mx_buffers* buf, gg_stream_t stream);

/* Test hook for the bounded waits: one CTA waits on a barrier that nothing
 * completes, gives up after `limit_ns` nanoseconds (clamped to 1 s), writes
 * GG_ERR_DEVICE_TIMEOUT into the status word and returns normally. */
gg_status gg_selftest_bounded_wait(void* ws, size_t ws_bytes, uint64_t limit_ns,
                                   gg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GG_H_ */

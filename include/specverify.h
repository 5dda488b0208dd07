/*
 * specverify.h -- C ABI of libspecverify, the verify-and-sample step of
 * speculative decoding on one NVIDIA GB300 (sm_103a).
 *
 * The operation (one call = one round, for a batch of B independent rows):
 *   "Fast Inference from Transformers via Speculative Decoding"
 *   (intuitivepapers.ai), section "The loop: draft, verify in one pass, keep a
 *   prefix", Algorithm 1 steps 3-4, and the course notes "Speculative Decoding",
 *   section "The algorithm":
 *     - p_i = softmax(target_logits[b][i] / T), q_i = softmax(draft_logits[b][i] / T)
 *       (temperature applied to both, "already adjusted" distributions);
 *     - walk i = 0..gamma-1, accept draft x_i iff u_i <= min(1, p_i(x_i)/q_i(x_i)),
 *       stop at the first rejection; n = number accepted;
 *     - if n < gamma emit one token from max(0, p_n - q_n) (normalised), else one
 *       token from p_gamma (the bonus token);
 *     - output x_0..x_{n-1}, then that token.
 *   Greedy mode (lihaoran.work essay, "What does unchanged output mean?"): keep
 *   the longest prefix where the draft equals the target argmax, then append the
 *   target argmax at the stop position.
 *
 * Randomness (no state): Philox4x32-10 (Salmon et al., SC'11), key = (lo32(seed),
 * hi32(seed)), counter = (c0, (tag<<24)|position, b, lo32(round)).  Tag 0 is the
 * acceptance uniform (c0 = 0, lane 0; u = (2*(x>>9)+1)*2^-24 in (0,1)).  Tag 1 at
 * the draw position n draws the target's own token by Gumbel-max: entry v gets
 * u_v from counter (v>>2, (1<<24)|n, b, lo32(round)), lane v&3 (same mapping to
 * (0,1)), g_v = -ln(-ln u_v), and the token is the argmax over the entries of
 * positive weight w_v (max(0, p_n - q_n), or p_n) of ln w_v + g_v, ties to the
 * lowest index.  On the GPU the race runs in fp32 on w_v / (-log2 u_v) (the same
 * argmax); when its two best keys lie within 2^-10 of each other they are
 * re-decided in double from the logits, so the token can differ from an exact
 * evaluation only where the two best exact keys are within the rounding of the
 * row sums.  sv_options.sampler selects the inverse transform instead (see
 * there).  Outputs depend only on the values, the shapes and (seed, round): not
 * on the stream, the launch shape or where the arrays sit in memory (every row
 * is cut into pieces counted from the row's own start).
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers, row-major and contiguous; the caller
 *     owns every buffer.  The library never allocates or frees device memory and
 *     keeps no state between calls except per-device caches of launch facts (SM
 *     count, resident CTAs per SM, resident CTA clusters per cluster size) and, for
 *     spec_verify_noalloc only, its one
 *     static scratch array and that array's cached device address (see there).
 *   - Work is queued on `cuda_stream` (a cudaStream_t; NULL = legacy default stream)
 *     and the call returns at once.  The return value reports only errors the host
 *     can see: bad arguments, misalignment, a too-small workspace, a launch failure.
 *     Data-dependent conditions are reported per batch row in `out_flags`.
 *   - Logit pointers must be 16-byte aligned; int32/float outputs 4-byte aligned;
 *     the workspace 256-byte aligned.
 *   - Workspace: at least sv_workspace_bytes(...) bytes of device memory owned by
 *     the caller; no initial contents are needed (each call zeroes the counters it
 *     uses before using them).  Calls that may run concurrently on the GPU need
 *     separate workspaces; calls queued one after another may share one.
 *   - Limits: 1 <= gamma <= 32, 1 <= V < 2^31, B >= 0 (B == 0 is a no-op).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_ARG = -1,         /* null required pointer, size out of range, temperature <= 0 */
  SV_ERR_DTYPE = -2,       /* dtype not SV_F32 / SV_BF16                                  */
  SV_ERR_ALIGN = -3,       /* pointer misaligned (see conventions)                       */
  SV_ERR_WORKSPACE = -4,   /* workspace null or smaller than sv_workspace_bytes()        */
  SV_ERR_CUDA = -5,        /* a CUDA runtime call or kernel launch failed                */
  SV_ERR_UNSUPPORTED = -6  /* device is not sm_103, or a size an entry point does not
                              support (stated at that entry point)                     */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Per-batch-row flags written to out_flags[b] (bitwise OR). */
enum {
  SV_FLAG_ZERO_MASS = 1,         /* a logit row of this batch row has no finite entry; an
                                    empty draw emits token 0                              */
  SV_FLAG_NONFINITE = 2,         /* a softmax normaliser is NaN/inf (NaN or +inf logits, bad
                                    per-row temperature) or q(x_i) == 0 at a tested i;
                                    outputs of the row are then in range but unspecified  */
  SV_FLAG_RESIDUAL_FALLBACK = 4, /* max(0, p_n - q_n) had no positive entry in floating
                                    point; the token was drawn from p_n                   */
  SV_FLAG_TIMEOUT = 8,           /* a bounded device-side wait of the fused LM head gave up
                                    (a tile that never arrived); the row's outputs are then
                                    unspecified                                          */
  SV_FLAG_BAD_TOKEN = 16         /* a draft token outside [0, V): treated as p = q = 0    */
};

enum { SV_MODE_SAMPLE = 0, SV_MODE_GREEDY = 1, SV_MODE_LMHEAD = 2, SV_MODE_DRAFT = 3 };

/* Bytes of workspace a call with these sizes needs (0 for B == 0).  `mode` is one
 * of SV_MODE_*.  For SV_MODE_LMHEAD, V and the hidden sizes of spec_lmhead_verify
 * do not change the answer beyond V. */
size_t sv_workspace_bytes(int B, int gamma, int64_t V, int mode);

/* Zero `bytes` of workspace on `cuda_stream` (a cudaMemsetAsync).  Not required
 * by the entry points; provided for callers that want a known initial state. */
int sv_workspace_init(void* workspace, size_t bytes, void* cuda_stream);

/*
 * spec_verify -- sampling verify (Algorithm 1, steps 3-4).
 *   target_logits   [B][gamma+1][V]  dtype (fp32, or bf16 bit patterns)
 *   draft_logits    [B][gamma][V]    dtype
 *   draft_tokens    [B][gamma]       int32; a token outside [0,V) counts as p=q=0
 *   temperature     used when row_temperature == NULL; must be > 0 and finite
 *   row_temperature [B] float or NULL; applies to all 2*gamma+1 rows of batch row b
 *   seed, round     RNG key and round number (see header comment)
 * Outputs (device):
 *   out_tokens      [B][gamma+1] int32: x_0..x_{n-1}, the emitted token, then -1
 *   out_counts      [B] int32: n, accepted drafts, 0..gamma
 *   out_p_at_draft  [B][gamma] float or NULL: p_i(x_i) for every i (not only tested)
 *   out_q_at_draft  [B][gamma] float or NULL: q_i(x_i)
 *   out_alpha       [B] float or NULL: (1/gamma) sum_i sum_v min(p_i, q_i) -- the
 *                   overlap of "Fast Inference ...", section "The acceptance rate is
 *                   the overlap of p and q"; costs one extra pass over 2*gamma rows
 *   out_flags       [B] uint8 or NULL: SV_FLAG_* bits
 *   workspace       >= sv_workspace_bytes(B, gamma, V, SV_MODE_SAMPLE), see conventions
 */
int spec_verify(const void* target_logits, const void* draft_logits,
                const int32_t* draft_tokens, int B, int gamma, int64_t V, int dtype,
                float temperature, const float* row_temperature, uint64_t seed,
                uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                float* out_p_at_draft, float* out_q_at_draft, float* out_alpha,
                uint8_t* out_flags, void* workspace, size_t workspace_bytes,
                void* cuda_stream);

/* How the target's own token (the residual after a rejection, or the bonus
 * token) is drawn; see the header comment.  SV_SAMPLER_GUMBEL is the round's
 * contract; SV_SAMPLER_INVERSE is an opt-in alternative with its own stream. */
enum { SV_SAMPLER_GUMBEL = 0, SV_SAMPLER_INVERSE = 1 };

/*
 * Variants of the round for spec_verify_opts.
 *   lenience  l in (0, 1]; 1 is the exact round.  q(x) is multiplied by l before
 *             the comparison, so draft i is accepted iff u_i <= p_i(x_i) /
 *             (l q_i(x_i)).  This accepts more and gives up exactness: no token
 *             is then emitted more than 1/l times as often as the target would
 *             emit it ("Fast Inference from Transformers via Speculative
 *             Decoding", the paragraph on sharper distributions, Appendix A.5 as
 *             summarised there).  The page changes only the comparison, so the
 *             token drawn after a rejection still comes from max(0, p_n - q_n).
 *   top_k     0: off.  k > 0: every target and draft row is adjusted before the
 *             round: entries whose logit is below the row's k-th largest
 *             (repeats counted, NaN not ranked) get probability 0 and the rest
 *             are renormalised; ties at the boundary are all kept (same page,
 *             section "The loop": top-k zeroes the tail and renormalises, and
 *             the round runs on the adjusted p and q).  k >= V changes nothing.
 *             Costs one radix-select pass over every row before the sweep.
 *   top_p     in (0, 1]; 1: off.  After top-k, every row keeps the smallest set
 *             of its largest-logit entries whose probability reaches top_p,
 *             every entry equal to the last one kept as well (same passage:
 *             nucleus zeroes the tail and renormalises).  The cut depends on the
 *             temperature.  Costs a sweep for the row maxima and a radix-select
 *             pass with exact fixed-point mass sums before the round's sweep;
 *             where top_p lies within about 1e-6 of a cumulative probability at
 *             the cut, the cut may differ from one taken in exact arithmetic by
 *             that boundary group.  top_p < 1 needs V <= 2^21
 *             (SV_ERR_UNSUPPORTED otherwise).
 *   sampler   SV_SAMPLER_GUMBEL (default) or SV_SAMPLER_INVERSE: the inverse
 *             transform with one 53-bit uniform per draw (tag 1 at the draw
 *             position, counter word 0 = 0; U = k 2^-53, k = (x0>>11) 2^32 +
 *             x1): the smallest v, in vocabulary order, whose cumulative weight
 *             exceeds U times the total weight, the weights summed in fp32 runs
 *             of 8 and exactly above them, so an interval end is exact up to
 *             about 1e-6 of the total.
 */
typedef struct {
  float lenience;
  int32_t top_k;
  float top_p;
  int32_t sampler;  /* SV_SAMPLER_GUMBEL (0, the default) or SV_SAMPLER_INVERSE */
} sv_options;

/*
 * spec_verify_opts -- spec_verify with sv_options (NULL: the exact round, the
 * same results as spec_verify).  A lenience or top_p outside (0, 1] (or NaN)
 * or a negative top_k returns SV_ERR_ARG.  The other arguments, outputs and
 * errors are those of spec_verify.  With top_k or top_p, p_at_draft /
 * q_at_draft and alpha are those of the adjusted rows.
 */
int spec_verify_opts(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, int B, int gamma, int64_t V, int dtype,
                     float temperature, const float* row_temperature, uint64_t seed,
                     uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                     float* out_p_at_draft, float* out_q_at_draft, float* out_alpha,
                     uint8_t* out_flags, const sv_options* options, void* workspace,
                     size_t workspace_bytes, void* cuda_stream);

/*
 * spec_verify_noalloc -- spec_verify for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for the deployment.
 * Some callers are handed only their input and output buffers (a plugin inside
 * another runtime, code that must not call into an allocator on the hot path, a
 * pool that may not grow).  This call takes the same arguments as spec_verify minus
 * the workspace and gives the same results.  Its scratch memory is one static 4 MiB
 * device array inside the library, held by every GPU that loads the library until
 * the process exits.
 *   - Sizes with sv_workspace_bytes(B, gamma, V, SV_MODE_SAMPLE) > 4 MiB (4194304
 *     bytes) are rejected with SV_ERR_WORKSPACE before anything is queued.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device (with that device current) looks up the array's
 *     device address and caches it; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents; each
 *     call first resets, on its stream, the counters and markers it relies on.
 *     Calls that overlap on the GPU (different streams or host threads) race on
 *     it: serialise them.
 *   - The cached address belongs to the CUDA context current at the first call.
 *     Calling spec_verify_noalloc after that context was destroyed
 *     (cudaDeviceReset, or a primary context released and re-created) is not
 *     supported: the cache is not refreshed.
 */
int spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, int B, int gamma, int64_t V, int dtype,
                        float temperature, const float* row_temperature, uint64_t seed,
                        uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                        float* out_p_at_draft, float* out_q_at_draft, float* out_alpha,
                        uint8_t* out_flags, void* cuda_stream);

/*
 * spec_verify_greedy -- greedy verify.  Reads only the target logits.
 *   t_i = argmax_v target_logits[b][i][v] on the raw values (exact comparison; NaN
 *   counts as -inf; ties, including an all -inf row, go to the lowest index);
 *   n = first i with draft_tokens[b][i] != t_i, else gamma;
 *   out_tokens[b] = x_0..x_{n-1}, t_n, -1...; out_counts[b] = n.
 *   workspace >= sv_workspace_bytes(B, gamma, V, SV_MODE_GREEDY).
 */
int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B,
                       int gamma, int64_t V, int dtype, int32_t* out_tokens,
                       int32_t* out_counts, void* workspace, size_t workspace_bytes,
                       void* cuda_stream);

/*
 * spec_lmhead_verify -- fused target/draft LM heads + sampling verify.  The logits
 * are the final projection of the two models' passes ("Fast Inference ...",
 * section "The loop ...", steps 1-2: one target pass over gamma+1 positions, the
 * draft distributions q_i), computed on the tensor cores and consumed by the
 * verify sweep without being written to HBM.
 *   h_target  [B*(gamma+1)][Ht] bf16 (row b*(gamma+1)+i = position i of batch row b)
 *   W_target  [Ht][V]           bf16
 *   h_draft   [B*gamma][Hd]     bf16
 *   W_draft   [Hd][V]           bf16
 *   then as spec_verify (temperature scalar only).
 *   debug_logits: NULL in production; else [B*(2*gamma+1)][V] float receives the
 *   logits the kernel used (target rows of batch row b first, then its draft rows),
 *   so that decisions can be checked on identical logits.
 * Returns SV_ERR_UNSUPPORTED for hidden sizes that are not multiples of 64 or
 * B*(gamma+1) > 256.
 */
int spec_lmhead_verify(const void* h_target, const void* W_target, int Ht,
                       const void* h_draft, const void* W_draft, int Hd,
                       const int32_t* draft_tokens, int B, int gamma, int64_t V,
                       float temperature, uint64_t seed, uint64_t round,
                       int32_t* out_tokens, int32_t* out_counts, float* out_p_at_draft,
                       float* out_q_at_draft, uint8_t* out_flags, float* debug_logits,
                       void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * spec_lmhead_draft -- the draft side of a round for one position: the draft
 * model's LM head and the draw of its token ("Fast Inference ...", section "The
 * loop", step 1: run M_q gamma times, drawing x_i ~ q_i; the course notes' "The
 * algorithm": x_{t+i} ~ q(. | prefix)).  The draft model's forward pass that
 * gives h_draft is the caller's.
 *   h_draft  [B][Hd] bf16: the draft's last hidden state of each batch row
 *   W_draft  [Hd][V] bf16
 *   pos      the position i of the tokens drawn (0..gamma-1), part of the RNG counter
 * q = softmax(z / T) with z = h_draft W_draft (bf16 operands, fp32 accumulation
 * on the tensor cores) and the scale fl32(1/T) as for the verify step; the token
 * is argmax_v z_v/T + g_v, ties to the lowest v, with g_v Gumbel noise from
 * Philox tag 2 at position pos (counter (v>>2, (2<<24)|pos, b, lo32(round)),
 * lane v&3).  The logits are not written to HBM.
 * Outputs (device):
 *   out_tokens   [B] int32, the drafted tokens x_i (0 for an empty row)
 *   out_q        [B] float or NULL: q_i(x_i)
 *   out_lse      [B] float or NULL: log sum_v exp(z_v / T)
 *   out_logit    [B] float or NULL: z at the drafted token (-inf for an empty row)
 *   debug_logits NULL in production; else [B][V] float receives the logits used
 *   workspace    >= sv_workspace_bytes(B, 1, V, SV_MODE_DRAFT)
 * Returns SV_ERR_UNSUPPORTED for Hd not a multiple of 64 (or above 16384),
 * B > 128 or V not a multiple of 8; SV_ERR_ARG for pos outside [0, 2^24).
 */
int spec_lmhead_draft(const void* h_draft, const void* W_draft, int Hd, int B, int64_t V,
                      float temperature, uint64_t seed, uint64_t round, int pos,
                      int32_t* out_tokens, float* out_q, float* out_lse, float* out_logit,
                      float* debug_logits, void* workspace, size_t workspace_bytes,
                      void* cuda_stream);

/*
 * spec_lmhead_verify_drafted -- spec_lmhead_verify for a round whose drafts came
 * from spec_lmhead_draft: the draft step already knows each draft row's
 * log-normaliser and the logit at its token, so the first GEMM pass computes
 * the target rows only (W_target alone streams once; W_draft is read only by
 * the pass that redraws a rejected row).
 *   draft_lse    [B][gamma] float: out_lse of the draft step at each position
 *   draft_logit  [B][gamma] float: out_logit of the draft step at each position
 *   other arguments as spec_lmhead_verify (the same temperature as the draft
 *   step); debug_logits receives the target rows only.
 * q_i(x_i) is exp(draft_logit / T - draft_lse); the draft rows' flags follow
 * from draft_lse (-inf: no mass; NaN or +inf: not finite).
 */
int spec_lmhead_verify_drafted(const void* h_target, const void* W_target, int Ht,
                               const void* h_draft, const void* W_draft, int Hd,
                               const int32_t* draft_tokens, const float* draft_lse,
                               const float* draft_logit, int B, int gamma, int64_t V,
                               float temperature, uint64_t seed, uint64_t round,
                               int32_t* out_tokens, int32_t* out_counts, float* out_p_at_draft,
                               float* out_q_at_draft, uint8_t* out_flags, float* debug_logits,
                               void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Profiling aid (not thread-safe): when `events` is non-NULL, following calls
 * record events on their stream: for spec_verify events[0] before the first
 * kernel, events[1] after the softmax sweep (and the top-k / top-p kernels
 * before it) and events[2] after the draw kernel (which takes the decision at
 * its start and merges at its end; n >= 3); for spec_lmhead_verify events[0]
 * first and events[k] after the first GEMM pass, the decision, the recompute
 * pass and the merge (n >= 5).  Only events[0..n-1] are recorded (n >= 1; at
 * most 8).  NULL switches recording off.  The events are cudaEvent_t created by
 * the caller; they change no result. */
int sv_set_timing_events(void* const* events, int n);

/* Test only: failure detection without a GPU fault.  The next spec_lmhead_verify
 * and spec_lmhead_verify_drafted calls withhold, in the first CTA of the first
 * GEMM pass, the hand-over of accumulator `job` to the epilogue (job < 0: none),
 * so that the epilogue's bounded wait runs out; and every bounded wait of the
 * fused LM head gives up after `wait_limit` tries (0: the default limit).  A wait
 * that gives up ends the CTA's other roles, lets the copies it issued land (a
 * bounded wait again), frees its tensor memory and returns; the call still
 * returns SV_OK and the batch rows carry SV_FLAG_TIMEOUT.  The setting stays
 * until changed; not thread-safe.  Returns 0. */
int sv_test_lmhead_stall(int job, uint32_t wait_limit);

/* Human-readable name of a status code. */
const char* sv_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int sv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */

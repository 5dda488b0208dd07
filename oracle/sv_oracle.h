/*
 * sv_oracle.h -- CPU oracle for the speculative-decoding verify-and-sample step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check in
 * __graft_entry__.py and the cpu_baseline / reference leg of bench.py load
 * this library.  It shares no source with the CUDA path: its Philox, its
 * softmax and its samplers are written here from the method's definition.
 *
 * Everything is single-threaded, double precision, and follows the pages'
 * order of steps (Algorithm 1 of "Fast Inference from Transformers via
 * Speculative Decoding", section "The loop: draft, verify in one pass, keep a
 * prefix"; the algorithm box "Speculative sampling, one round" of the course
 * notes "Speculative Decoding").
 *
 * Layouts (row-major, contiguous):
 *   zt [B][gamma+1][V]  target logits   (f32 or bf16 bits)
 *   zd [B][gamma][V]    draft logits    (same dtype)
 *   xt [B][gamma]       draft tokens    (int32)
 *   tokens [B][gamma+1] emitted tokens, -1 padded; counts [B] accepted drafts.
 */
#ifndef SV_ORACLE_H
#define SV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { SVO_F32 = 0, SVO_BF16 = 1 };

/* Per batch-row flags (same bit values as the product's documented flags). */
enum {
  SVO_FLAG_ZERO_MASS = 1,         /* a logit row used by the step has no finite entry   */
  SVO_FLAG_NONFINITE = 2,         /* a normaliser is NaN/inf, or q(x~)=0 at a tested i  */
  SVO_FLAG_RESIDUAL_FALLBACK = 4, /* residual max(0,p-q) had no positive entry          */
  SVO_FLAG_BAD_TOKEN = 16         /* a draft token outside [0, V)                       */
};

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11), one block. */
void svo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Uniform in (0,1) from the verify step's counter layout:
 * counter = (c0, (tag<<24)|pos, b, lo32(round)), key = (lo32(seed), hi32(seed)),
 * lane in 0..3; u = (2*(x>>9)+1) * 2^-24. */
double svo_uniform(uint64_t seed, uint32_t tag, uint32_t pos, uint32_t b,
                   uint64_t round, uint32_t c0, int lane);

/* svo_uniform for vocabulary entries v0..v0+n-1 (c0 = v>>2, lane = v&3). */
void svo_uniform_row(uint64_t seed, uint32_t tag, uint32_t pos, uint32_t b, uint64_t round,
                     int64_t v0, int64_t n, double* out);

/* Samplers of the target's own token (the residual after a rejection, or the
 * bonus token): Gumbel-max over per-entry noise of Philox tag 1 at the draw
 * position (default), or the inverse transform with one 53-bit uniform. */
enum { SVO_SAMPLER_GUMBEL = 0, SVO_SAMPLER_INVERSE = 1 };

/* Uniform in [0,1) of the inverse-transform draw at position pos: counter
 * (0, (1<<24)|pos, b, lo32(round)); U = k 2^-53 with
 * k = (out[0] >> 11) * 2^32 + out[1]. */
double svo_draw_uniform(uint64_t seed, uint32_t pos, uint32_t b, uint64_t round);

/* Probability-level pieces of the accept/reject rule (double in, double out). */
double svo_accept_mass(const double* p, const double* q, int64_t V, double* out_min);
double svo_residual(const double* p, const double* q, int64_t V, double* out_resid);

/* Softmax of s (double) into p; returns S = sum exp(s - max). */
double svo_softmax(const double* s, int64_t V, double* p);

/* Full sampling verify.  Optional outputs may be NULL.
 *   p_at, q_at, ratio, u_acc : [B][gamma]  p(x~), q(x~), p/q, acceptance uniform
 *   beta                     : [B][gamma]  sum_v min(p_i, q_i)   (diagnostic)
 *   draw_gap                 : [B]         the margin of the target's own draw:
 *                                          Gumbel-max (default): top-1 minus top-2
 *                                          key, log w + g in natural-log units;
 *                                          inverse transform: distance of U W from
 *                                          the nearer end of the drawn token's
 *                                          cumulative interval (probability units)
 *   resid_mass               : [B]         sum_v max(0, p_n - q_n) (NaN if n == gamma)
 * Returns 0, or -1 on bad arguments. */
int svo_spec_verify(const void* zt, const void* zd, const int32_t* xt,
                    int B, int gamma, int64_t V, int dtype,
                    float temperature, const float* row_temperature,
                    uint64_t seed, uint64_t round,
                    int32_t* tokens, int32_t* counts,
                    double* p_at, double* q_at, double* ratio, double* u_acc,
                    double* beta, double* draw_gap, double* resid_mass,
                    uint8_t* flags);

/* Same, for batch rows [b_begin, b_end) only (rows keep their global index b in
 * the RNG counters; other rows of the outputs are left untouched). */
int svo_spec_verify_rows(const void* zt, const void* zd, const int32_t* xt,
                         int B, int gamma, int64_t V, int dtype,
                         float temperature, const float* row_temperature,
                         uint64_t seed, uint64_t round,
                         int32_t* tokens, int32_t* counts,
                         double* p_at, double* q_at, double* ratio, double* u_acc,
                         double* beta, double* draw_gap, double* resid_mass,
                         uint8_t* flags, int b_begin, int b_end);

/* Variants of the round.  lenience l ("Fast Inference from Transformers via
 * Speculative Decoding", the paragraph on sharper distributions, Appendix A.5
 * as summarised there): q(x) is multiplied by l before the comparison, so a
 * draft is accepted iff u <= p/(l q); l = 1 is the exact round.  The
 * correction after a rejection is the residual of Algorithm 1, unchanged (the
 * page changes only the comparison).
 * top_k (same page, "already adjusted" distributions: top-k zeroes the tail and
 * renormalises): with top_k > 0 every target and draft row keeps the entries
 * whose scaled logit is at least its k-th largest (ties at the boundary kept,
 * NaN left in place), the rest get probability 0; 0 is off.
 * top_p (nucleus, same passage), after top-k: every row keeps the smallest set
 * of largest-logit entries whose probability reaches top_p (entries equal to
 * the last one kept too); 1 is off.  nucleus_gap (optional output, [B]): per
 * batch row the smallest distance of top_p from the cumulative probabilities
 * just before and at a row's cut (inf without a cut).  sampler: SVO_SAMPLER_*
 * for the target's own token. */
typedef struct {
  double lenience;     /* in (0, 1] */
  int top_k;           /* >= 0 */
  double top_p;        /* in (0, 1] */
  double* nucleus_gap; /* [B] or NULL */
  int sampler;         /* SVO_SAMPLER_GUMBEL (default) or SVO_SAMPLER_INVERSE */
} svo_options;

/* svo_spec_verify_rows with options (NULL: the exact round). */
int svo_spec_verify_ex(const void* zt, const void* zd, const int32_t* xt,
                       int B, int gamma, int64_t V, int dtype,
                       float temperature, const float* row_temperature,
                       uint64_t seed, uint64_t round,
                       int32_t* tokens, int32_t* counts,
                       double* p_at, double* q_at, double* ratio, double* u_acc,
                       double* beta, double* draw_gap, double* resid_mass,
                       uint8_t* flags, int b_begin, int b_end, const svo_options* opt);

/* Greedy verify on raw target logits. */
int svo_spec_verify_greedy(const void* zt, const int32_t* xt, int B, int gamma,
                           int64_t V, int dtype, int32_t* tokens, int32_t* counts);

/* Draft sampling of one position from given logits [B][V] (float): with
 * s = z * fl32(1/T), x = argmax_v s_v + g_v over finite s_v (ties to the lowest
 * v), g_v Gumbel from Philox with tag 2 at position pos (counter (v>>2,
 * (2<<24)|pos, b, round), lane v&3).  Outputs tokens [B] (0 for an empty row),
 * q_at [B] = q(x), lse [B] = log sum_v exp(s_v), gumbel_gap [B] = top-1 minus
 * top-2 key; the last three may be NULL.  Returns 0, or -1 on bad arguments. */
int svo_draft_sample(const float* logits, int B, int64_t V, float temperature, uint64_t seed,
                     uint64_t round, int pos, int32_t* tokens, double* q_at, double* lse,
                     double* gumbel_gap);

/* Plain matmul reference for the fused LM head: logits[M][V] = h[M][H] * W[H][V]
 * with bf16 inputs, accumulated in double, written as float. */
void svo_lmhead_logits(const uint16_t* h, const uint16_t* W, int M, int H, int64_t V,
                       const int64_t* cols, int64_t ncols, float* out);

#ifdef __cplusplus
}
#endif
#endif

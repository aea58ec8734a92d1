/*
 * qspec.h -- C ABI of the QSPEC hot-path library (libqspec.so, sm_103a).
 *
 * QSPEC (speculative decoding with complementary quantisation schemes) drafts
 * tokens with a W4A4 pass and verifies them with a W4A16 pass over ONE shared
 * set of 4-bit weights, then overwrites the draft KV-cache entries of accepted
 * tokens with the verify pass's.  This library holds the data-parallel steps of
 * one such round.
 *
 * Sources, cited by page title and section:
 *   [QS-bg]     "QSPEC: Speculative Decoding with Complementary Quantization
 *               Schemes" summary page (molayo1419.me), background terms.
 *   [QS-design] same page, "QSPEC structure".
 *   [SQ]        "SpecQuant: Speculative Decoding with Multi-Parent
 *               Quantization for Adaptive LLM Inference" summary page.
 *
 * Conventions for every call
 *   - Every pointer argument is a DEVICE pointer, owned by the caller, unless
 *     stated otherwise.  The library allocates no device memory and keeps no
 *     state between calls, with one exception: the fixed scratch array of
 *     qspec_verify_sample_noalloc (below), which lives in the library image
 *     and keeps its contents from one call of that entry point to the next.
 *     Outputs are written in place.
 *   - bf16 and fp16 values travel as uint16_t bit patterns.
 *   - Calls are enqueued on `stream` and return right after launch; results
 *     and *dev_status are valid once the stream has synchronised.
 *   - The return value reports what the host can check before launch
 *     (QSPEC_ERR_NULL, _SHAPE, _ALIGN, _WORKSPACE, _UNSUPPORTED) and launch
 *     failures (QSPEC_ERR_LAUNCH; see qspec_last_cuda_error()).  Nothing is
 *     launched when it is not QSPEC_OK.
 *   - dev_status (nullable) is a device int32 the caller zeroes.  Kernels that
 *     detect a data error (QSPEC_ERR_RANGE, _ZERO_POINT, _NONFINITE) store its
 *     code there if it still holds 0 (first error wins) and carry on; the
 *     outputs that depend on the bad data are then unspecified.  No kernel
 *     traps or spins without a bound.
 *   - K is a multiple of the quantisation group, 128.  G = K / 128.
 */
#ifndef QSPEC_H
#define QSPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so this header needs no CUDA
 * header.  NULL is the legacy default stream. */
typedef struct CUstream_st *qspec_stream_t;

enum qspec_status {
    QSPEC_OK = 0,
    QSPEC_ERR_NULL = 1,        /* a required pointer is NULL */
    QSPEC_ERR_SHAPE = 2,       /* a size is out of range (K % 128, gamma, ...) */
    QSPEC_ERR_ALIGN = 3,       /* a pointer or leading dimension is misaligned */
    QSPEC_ERR_LAUNCH = 4,      /* the CUDA launch failed */
    QSPEC_ERR_WORKSPACE = 5,   /* the workspace is smaller than required */
    QSPEC_ERR_RANGE = 6,       /* device: an index or code is out of range */
    QSPEC_ERR_ZERO_POINT = 7,  /* device: a zero point is not an integer 0..15 */
    QSPEC_ERR_NONFINITE = 8,   /* device: NaN / +inf input, or a row with no mass */
    QSPEC_ERR_TIMEOUT = 9,     /* device: a bounded wait expired */
    QSPEC_ERR_UNSUPPORTED = 10 /* the current device is not sm_103 */
};

#define QSPEC_GROUP 128
#define QSPEC_MAX_GAMMA 16

/* Library version as major*10000 + minor*100 + patch. */
int qspec_version(void);

/* Static string naming a status code. */
const char *qspec_status_string(int status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char *qspec_last_cuda_error(void);

/* Number of kernel launches this library has issued since it was loaded,
 * all threads together, counting a launch recorded into a CUDA graph once
 * (at capture).  Host only; never fails. */
unsigned long long qspec_kernel_launches(void);

/*
 * a1. Pack INT4 weights.  [QS-bg] dequantisation W^ = s (W_INT4 - z);
 * [QS-design] one 4-bit weight set serves both the W4A4 draft and the W4A16
 * verify kernels, so this is the only weight format either reads.
 *
 *   codes  uint8  [N][K]   values 0..15 (output channel n, input index k)
 *   s_fp16 uint16 [N][G]   fp16 scale of group g = k / 128 of row n
 *   z_fp16 uint16 [N][G]   fp16 zero point; must be an integer 0..15
 *   packed uint8  [N][K/2] out: byte j = code[2j] | code[2j+1] << 4
 *   sz     uint32 [N][G]   out: fp16 bits of s | fp16 bits of z << 16
 * Device errors: QSPEC_ERR_RANGE (a code > 15), QSPEC_ERR_ZERO_POINT,
 * QSPEC_ERR_NONFINITE (a scale is inf/NaN).  codes, packed: 16-byte aligned.
 */
int qspec_pack_weights(const uint8_t *codes, const uint16_t *s_fp16, const uint16_t *z_fp16,
                       int N, int K, uint8_t *packed, uint32_t *sz, int32_t *dev_status,
                       qspec_stream_t stream);

/*
 * a2. Quantise activations to symmetric INT4 per token and 128-group.
 * [QS-bg] W4A4 quantises activations as well as weights to 4 bits.
 * Per row m and group g: amax = max |x|, sx = amax / 7 (fp32, IEEE
 * division), q = clamp(rint(x / sx), -7, 7) (q = 0 when sx == 0), qs = sum q.
 *
 *   x_bf16 uint16 [M][ldx]  input rows (ldx >= K, ldx % 8 == 0, 16-byte aligned)
 *   xq     uint8  [M][K/2]  out: two's-complement nibbles, byte j = q[2j] | q[2j+1] << 4
 *                           (8-byte aligned)
 *   sx     float  [M][G]    out: scales
 *   qs     int32  [M][G]    out: group sums of q
 * Device errors: QSPEC_ERR_NONFINITE (a NaN or inf input).
 */
int qspec_quant_act_int4(const uint16_t *x_bf16, int M, int K, int ldx, uint8_t *xq, float *sx,
                         int32_t *qs, int32_t *dev_status, qspec_stream_t stream);

/*
 * a3. W4A4 linear (draft).  [QS-bg] 4-bit activations times 4-bit weights,
 * products accumulated in INT32, then scaled to 16 bits; [QS-design] the
 * draft pass.  Bit-exact definition:
 *   I[m][n][g] = sum_{k in g} q[m][k] * (W[n][k] - z[n][g])        (exact int)
 *   acc = 0; for g = 0..G-1: acc = fmaf((float)I, sx[m][g] * s[n][g], acc)
 *   y[m][n] = bf16 round-to-nearest-even(acc)
 *
 *   xq, sx, qs      from qspec_quant_act_int4 (qs must be its output)
 *   packed, sz      from qspec_pack_weights, N rows
 *   y_bf16 uint16 [M][ldy]  out (ldy >= N)
 *   dbg_I  int32 [M][N][G]  nullable: out, the group integers I
 * Any M >= 1; large M runs on the tensor cores (FP8 E4M3 operands holding the
 * small integers exactly, fp32 accumulation of integer partial sums below 2^24
 * -- exact -- drained per group).
 */
int qspec_linear_w4a4(const uint8_t *xq, const float *sx, const int32_t *qs,
                      const uint8_t *packed, const uint32_t *sz, int M, int N, int K,
                      uint16_t *y_bf16, int ldy, int32_t *dbg_I, int32_t *dev_status,
                      qspec_stream_t stream);

/*
 * a2 + a3 in one call: the draft-pass linear on bf16 activations.  The
 * activations are quantised exactly as qspec_quant_act_int4 does it and the
 * product is exactly qspec_linear_w4a4's; [QS-design] the draft pass runs
 * the quantiser in front of every W4A4 linear, and at decode sizes one launch
 * instead of two removes the second launch's latency from the critical path
 * (every CTA quantises the tokens it needs; CTA column 0 stores them).
 *
 *   x_bf16 uint16 [M][ldx]  (ldx >= K, ldx % 8 == 0, 16-byte aligned)
 *   packed, sz              from qspec_pack_weights, N rows
 *   y_bf16 uint16 [M][ldy]  out (ldy >= N)
 *   xq, sx, qs              out: the quantised activations, as from
 *                           qspec_quant_act_int4 (xq 16-byte aligned)
 *   dbg_I  int32 [M][N][G]  nullable: out, the group integers I
 * Device errors: QSPEC_ERR_NONFINITE (a NaN or inf input).
 */
int qspec_linear_w4a4_bf16(const uint16_t *x_bf16, int ldx, const uint8_t *packed,
                           const uint32_t *sz, int M, int N, int K, uint16_t *y_bf16, int ldy,
                           uint8_t *xq, float *sx, int32_t *qs, int32_t *dbg_I,
                           int32_t *dev_status, qspec_stream_t stream);

/*
 * a4. W4A16 linear (verify).  [QS-bg] Y = X W^, W^ = s (W_INT4 - z),
 * 16-bit activations; [QS-design] the verify pass over the gamma+1 rows of
 * every sequence (M = B (gamma + 1)).  fp32 accumulation, bf16 output,
 * within 1e-2 (1 + |ref|) of the fp64 value of the same definition.
 *
 *   x_bf16 uint16 [M][ldx]  (ldx >= K, ldx % 8 == 0, 16-byte aligned)
 *   packed, sz              from qspec_pack_weights, N rows
 *   y_bf16 uint16 [M][ldy]  out (ldy >= N)
 */
int qspec_linear_w4a16(const uint16_t *x_bf16, int ldx, const uint8_t *packed, const uint32_t *sz,
                       int M, int N, int K, uint16_t *y_bf16, int ldy, int32_t *dev_status,
                       qspec_stream_t stream);

/*
 * a4 + a7 in one call: the verify pass's k / v projection, writing its
 * outputs into the KV caches from the epilogue.  [QS-design] for accepted
 * tokens the W4A4 cache entries are replaced by the W4A16 ones; doing it in
 * the projection that produces those entries removes the separate copy
 * (qspec_kv_overwrite) and its second read.
 *
 * Computes y exactly as qspec_linear_w4a16 (M = B (gamma + 1) verify rows,
 * row m = b (gamma + 1) + r) and also stores every output of columns
 *   [kv_col0, kv_col0 + H D)          into k_cache[b][h][base_pos[b] + r][d]
 *   [kv_col0 + H D, kv_col0 + 2 H D)  into v_cache[b][h][base_pos[b] + r][d]
 * (column kv_col0 + h D + d), for r = 0 .. n_acc[b] -- or, with n_acc NULL,
 * for every r = 0 .. gamma: the verify pass runs before acceptance is known,
 * and the rows past the accepted ones lie beyond the cache length the caller
 * keeps (base_pos[b] + n_acc[b] + 1), so the cache read afterwards is the
 * same as with qspec_kv_overwrite.
 *
 *   x_bf16 .. ldy                     as in qspec_linear_w4a16
 *   kv_col0, H, D                     the K columns' offset in y, heads, head dim
 *   T                                 cache capacity (positions)
 *   k_cache, v_cache uint16 [B][H][T][D]  one layer's caches, bf16 (either may be
 *                                     NULL; with v_cache NULL only H D columns
 *                                     are needed)
 *   base_pos int32 [B], n_acc int32 [B] (nullable)
 * Device errors: QSPEC_ERR_RANGE when base_pos < 0, n_acc outside [0, gamma]
 * or base_pos + (the last row written) >= T (that sequence's cache is left
 * untouched; y is still written).
 */
int qspec_linear_w4a16_kv(const uint16_t *x_bf16, int ldx, const uint8_t *packed, const uint32_t *sz, int M,
                          int N, int K, uint16_t *y_bf16, int ldy, int kv_col0, int H, int D, int T, int gamma,
                          uint16_t *k_cache, uint16_t *v_cache, const int32_t *base_pos, const int32_t *n_acc,
                          int32_t *dev_status, qspec_stream_t stream);

/* Bytes of workspace the verification calls need for (B, gamma, V). */
size_t qspec_verify_workspace_bytes(int B, int gamma, int V);

/*
 * a5. Greedy verification.  [QS-bg] under greedy decoding a draft token is
 * accepted when it is the target's top-1 token; nothing after the first
 * rejection is kept; the target supplies one more token (the correction at
 * the first mismatch, or a bonus token when all gamma drafts are accepted).
 *
 *   p_logits uint16 [B][gamma+1][V]  target (W4A16) logits, bf16
 *   draft    int32  [B][gamma]       draft tokens
 *   n_acc    int32  [B]              out: accepted drafts A_b (0..gamma)
 *   out      int32  [B][gamma+1]     out: drafts 1..A_b, then the target's
 *                                    argmax of row A_b (lowest id on ties);
 *                                    entries after A_b are -1
 *   workspace, ws_bytes              device scratch of
 *                                    qspec_verify_workspace_bytes(B, gamma, V)
 * 1 <= gamma <= 16.  Device errors: QSPEC_ERR_NONFINITE (NaN logit),
 * QSPEC_ERR_RANGE (draft id outside [0, V)).
 */
int qspec_verify_greedy(const uint16_t *p_logits, const int32_t *draft, int B, int gamma, int V,
                        int32_t *n_acc, int32_t *out, void *workspace, size_t ws_bytes,
                        int32_t *dev_status, qspec_stream_t stream);

/*
 * a6. Sampled verification (speculative sampling).  [QS-bg] accept draft x
 * with probability min(1, p(x|h) / q(x|h)); stop at the first rejection;
 * replace it with a token drawn from the normalised residual max(0, p - q),
 * or draw a bonus token from the last target row when all are accepted.
 * Every decision is made in integers so that it is reproducible bit for bit:
 *   E_v = rint(qexp(l_v - max_row) * 2^32) (own exp: Cody-Waite reduction and
 *   a degree-7 Taylor polynomial in fp32), S = sum_v E_v;
 *   accept iff U_i * Eq_t * Sp < 2^24 * Ep_t * Sq, U_i a 24-bit uniform;
 *   residual R_v = max(0, Ep_v * Sq - Eq_v * Sp) (the target row if all zero);
 *   draw v* = min{v : sum_{u<=v} w_u > floor(U' * sum w / 2^24)}.
 * Uniforms: Philox4x32-10 (Salmon et al., SC'11), key = seed, counter =
 * (slot, b, round lo, round hi), U = word0 >> 8; slot i-1 for draft i, slot
 * gamma for the correction / bonus draw.
 *
 *   p_logits uint16 [B][gamma+1][V], q_logits uint16 [B][gamma][V] (bf16)
 *   draft, n_acc, out, workspace: as in qspec_verify_greedy
 * Device errors: QSPEC_ERR_NONFINITE (NaN or +inf logit, or a row that is all
 * -inf), QSPEC_ERR_RANGE (draft id outside [0, V)).
 */
int qspec_verify_sample(const uint16_t *p_logits, const uint16_t *q_logits, const int32_t *draft,
                        int B, int gamma, int V, uint64_t seed, uint64_t round, int32_t *n_acc,
                        int32_t *out, void *workspace, size_t ws_bytes, int32_t *dev_status,
                        qspec_stream_t stream);

/*
 * Sampled verification for callers that cannot allocate device memory (for
 * example code that runs while a CUDA graph is being captured, or a plugin
 * with no allocator of its own).  Same inputs, outputs, decisions and device
 * errors as qspec_verify_sample, bit for bit; the pages have no counterpart,
 * this is an interface convenience.
 *
 * The scratch is a fixed array inside the library, QSPEC_VERIFY_NOALLOC_-
 * SCRATCH_BYTES (1 MiB) on every GPU that loads the library, held until the
 * process exits.  Sizes whose workspace (qspec_verify_workspace_bytes) would
 * not fit return QSPEC_ERR_WORKSPACE before any launch -- e.g. B = 256,
 * gamma = 4, V = 128256 needs about 0.4 MiB.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  The address is remembered per CUDA context:
 * after a cudaDeviceReset, or in a new context on the same device, the next
 * call looks it up again, so that call too must come before any capture.
 * Every call shares the one array and leaves its
 * contents behind (the parts that must start at zero are cleared on the
 * stream by each call): calls that may overlap on the GPU -- on different
 * streams, or from different threads -- race and must not be issued.
 */
#define QSPEC_VERIFY_NOALLOC_SCRATCH_BYTES (1 << 20)
int qspec_verify_sample_noalloc(const uint16_t *p_logits, const uint16_t *q_logits,
                                const int32_t *draft, int B, int gamma, int V, uint64_t seed,
                                uint64_t round, int32_t *n_acc, int32_t *out, int32_t *dev_status,
                                qspec_stream_t stream);

/* Bytes of workspace qspec_draft_sample needs for (B, V). */
size_t qspec_draft_workspace_bytes(int B, int V);

/*
 * Draft-side sampling with the draft statistics.  [QS-bg] the draft model
 * proposes x ~ q(x|h), the distribution the acceptance test of
 * qspec_verify_sample divides by.  SpecKV blog ("SpecKV: compression-aware
 * gamma selection"), architecture section, feature extraction: a gamma
 * controller reads the confidence (the largest probability) and the entropy
 * -sum_v p_v log(p_v + 1e-9) of the draft model's softmax.  Per row b, with
 * the fixed-point weights of qspec_verify_sample (E_v, S = sum_v E_v):
 *   token[b]      = min{v : sum_{u<=v} E_u > floor(U * S / 2^24)}, U the
 *                   24-bit Philox uniform of slot 16 + step (slots 0..16 are
 *                   the verification's), so a draft drawn here is
 *                   distributed as the q' the acceptance test uses;
 *   confidence[b] = max_v E_v / S, the fp64 quotient rounded to fp32
 *                   (bit-exact);
 *   entropy[b]    = -sum_v p_v log(p_v + 1e-9), p_v = E_v / S, summed in
 *                   fp32 (within 1e-4 (1 + H) of the fp64 value).
 *
 *   q_logits   uint16 [B][V]   draft logits of one draft position, bf16
 *   step       1..16           the draft position (selects the uniform)
 *   token      int32  [B]      out
 *   confidence float  [B]      out
 *   entropy    float  [B]      out
 *   workspace, ws_bytes        device scratch of qspec_draft_workspace_bytes(B, V)
 * Device errors: QSPEC_ERR_NONFINITE (NaN or +inf logit, or a row that is
 * all -inf; that row's outputs are unspecified).
 */
int qspec_draft_sample(const uint16_t *q_logits, int B, int V, uint64_t seed, uint64_t round, int step,
                       int32_t *token, float *confidence, float *entropy, void *workspace, size_t ws_bytes,
                       int32_t *dev_status, qspec_stream_t stream);

/*
 * a7. KV overwrite.  [QS-design] for accepted tokens the low-precision (W4A4)
 * KV-cache entries are replaced with the W4A16 ones, so later steps read the
 * high-precision context from the one shared cache.  For each sequence b and
 * r = 0..n_acc[b] (the last confirmed token and the accepted drafts):
 *   cache[l][b][h][base_pos[b] + r][:] = new[l][b][r][h][:]   (K and V)
 *
 *   k_cache, v_cache uint16 [L][B][H][T][D]         bf16, updated in place
 *   k_new, v_new     uint16 [L][B][gamma+1][H][D]   bf16 verify-pass rows
 *   base_pos, n_acc  int32  [B]
 * D % 8 == 0, all four tensors 16-byte aligned.  Device errors:
 * QSPEC_ERR_RANGE when base_pos < 0, n_acc outside [0, gamma] or
 * base_pos + n_acc >= T (that sequence is left untouched).
 */
int qspec_kv_overwrite(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                       const uint16_t *v_new, const int32_t *base_pos, const int32_t *n_acc,
                       int L, int B, int H, int T, int D, int gamma, int32_t *dev_status,
                       qspec_stream_t stream);

/*
 * SpecQuant Q8 variant.  [SQ] "SpecQuant: Speculative Decoding with
 * Multi-Parent Quantization for Adaptive LLM Inference" summary page,
 * contributions and approach: INT4 (Q4), FP8 (Q8) and FP16 (Q16) variants are
 * derived post-training from one FP16 parent with shared base weights, and
 * the chosen parent verifies the draft.  FP8 is E4M3 (1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits, largest finite 448); a conversion rounds
 * to nearest even and saturates at +-448.
 *
 * qspec_quant_weights_fp8: per output channel n of the parent weights,
 *   s8[n] = amax_k |W[n][k]| / 448 (fp32, IEEE division),
 *   w8[n][k] = E4M3(W[n][k] / s8[n]) (fp32 IEEE quotient); a zero row gives
 *   s8 = 0 and codes 0.
 *   w_fp16 uint16 [N][K] fp16 bits (16-byte aligned), w8 uint8 [N][K] out
 *   (8-byte aligned), s8 float [N] out.
 * qspec_quant_act_fp8: the same per token m of bf16 activations.
 *   x_bf16 uint16 [M][ldx] (ldx >= K, ldx % 8 == 0, 16-byte aligned),
 *   xq uint8 [M][K] out, sa float [M] out.
 * qspec_linear_fp8: the Q8 linear on the tensor cores (E4M3 x E4M3, fp32
 *   accumulation): y[m][n] = bf16(sum_k E4M3(xq) E4M3(w8) * sa[m] * s8[n]),
 *   within 1e-2 (1 + |ref|) of the fp64 value of the same sum.
 *   xq, w8 16-byte aligned; y_bf16 uint16 [M][ldy] out (ldy >= N).
 * K is a multiple of 128.  Device errors: QSPEC_ERR_NONFINITE (a NaN or inf
 * input to a quantiser), QSPEC_ERR_TIMEOUT (a bounded wait expired).
 */
int qspec_quant_weights_fp8(const uint16_t *w_fp16, int N, int K, uint8_t *w8, float *s8,
                            int32_t *dev_status, qspec_stream_t stream);
int qspec_quant_act_fp8(const uint16_t *x_bf16, int M, int K, int ldx, uint8_t *xq, float *sa,
                        int32_t *dev_status, qspec_stream_t stream);
int qspec_linear_fp8(const uint8_t *xq, const float *sa, const uint8_t *w8, const float *s8, int M, int N,
                     int K, uint16_t *y_bf16, int ldy, int32_t *dev_status, qspec_stream_t stream);

/*
 * Diagnostic for tests of the bounded waits; the pages have no counterpart.
 * Runs one of the library's tensor-core linear kernels on the same arguments
 * as qspec_linear_w4a16 / qspec_linear_w4a4 would, with every barrier wait of
 * that kernel bounded by `wait_limit` polls instead of the library's default
 * (2^22; each poll suspends for a hardware-chosen time), and, when `stall` is
 * non-zero, with the kernel's MMA issuer first waiting on a barrier that
 * nothing ever arrives at, so that this wait runs out.  The kernel then leaves
 * its loops, lets its copies and MMAs in flight finish (bounded waits of the
 * default length), frees its tensor memory, stores QSPEC_ERR_TIMEOUT in
 * *dev_status and returns; its outputs are unspecified.  With stall == 0 and
 * a long enough wait_limit the outputs are those of the regular call.
 *
 *   kernel  QSPEC_KERNEL_W4A16_TC       the W4A16 kernel for M > 16 (any M here); reads x_bf16
 *           QSPEC_KERNEL_W4A4_GEMV_TC   the decode-sized W4A4 kernel (3 <= M <= 16); reads xq, sx, qs
 *           QSPEC_KERNEL_W4A4_TC        the W4A4 kernel for larger M (any M here); reads xq, sx, qs
 *   the other pointers and sizes as in qspec_linear_w4a16 / qspec_linear_w4a4
 *   (x_bf16 rows are K long, ldx = K).
 * Returns QSPEC_ERR_SHAPE, before any launch, when the shape does not suit
 * the kernel; wait_limit must be at least 1.
 */
#define QSPEC_KERNEL_W4A16_TC 0
#define QSPEC_KERNEL_W4A4_GEMV_TC 1
#define QSPEC_KERNEL_W4A4_TC 2
int qspec_debug_linear_bounded(int kernel, const uint16_t *x_bf16, const uint8_t *xq, const float *sx,
                               const int32_t *qs, const uint8_t *packed, const uint32_t *sz, int M, int N,
                               int K, uint16_t *y_bf16, int ldy, uint32_t wait_limit, int stall,
                               int32_t *dev_status, qspec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QSPEC_H */

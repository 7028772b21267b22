/*
 * alibi.h - C ABI of the GB300 (sm_103a) ALiBi causal attention library.
 *
 * Operation (all entry points):
 *   O = softmax( Q K^T / sqrt(d) - m_h * (i - j), causal mask ) V
 * with the per-head slope m_h of the ALiBi schedule. Sources (page title,
 * then section / equation):
 *   - "When Attention Goes Blind: Numerical Failure in ALiBi Positional
 *     Encodings" (arXiv 2608.03994), sec. 3.1 eq. 1-3: A = QK^T / sqrt(d_k),
 *     B = -m D, D = i - j.
 *   - "ALiBi: Attention with Linear Biases" (abhik.ai): "From distance to a
 *     normalized weight" (keys j <= i allowed, future keys masked);
 *     "Different heads, different distance penalties" (slope schedule); the
 *     KV-cache paragraph after the full-sequence example (true positions).
 *
 * Conventions shared by every call:
 *   - Tensors are dense, row-major and contiguous. Prefill: q, k, v, out are
 *     [B, H, N, d]; lse is [B, H, N]. Decode: q and out are [B, H, d]; the
 *     caches are [B, H, L, d].
 *   - bf16 means IEEE-style bfloat16 (1-8-7), stored as 16-bit words.
 *   - Device pointers must be CUDA device (or managed) memory of the current
 *     device, 16-byte aligned. The caller owns every buffer; the library never
 *     frees or retains a caller pointer after the call returns.
 *   - stream is a cudaStream_t (NULL = the legacy default stream). Calls are
 *     asynchronous: results are valid once the stream has been synchronised.
 *   - scale is 1/sqrt(d); slopes are always those of alibi_slopes(H).
 *   - The library keeps some state per device for the life of the process:
 *     the device status word, a stream-ordered memory pool, kernel attributes
 *     and the work-order tables of the prefill and backward (see
 *     alibi_attn_fwd_ex). cudaDeviceReset() of a
 *     device destroys that state with the context; do not call the library on
 *     that device again in the same process after a reset.
 *   - Return value: ALIBI_OK, or a negative alibi_status. Argument errors are
 *     detected on the host before anything is launched. No call aborts the
 *     process, traps on the device or waits without bound: every device-side
 *     wait has a time limit, after which the kernel records ALIBI_ERR_TIMEOUT
 *     in a device status word and returns; alibi_check_error() reports it.
 */
#ifndef ALIBI_H
#define ALIBI_H

#if defined(__GNUC__) || defined(__clang__)
#define ALIBI_API __attribute__((visibility("default")))
#else
#define ALIBI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ALIBI_OK = 0,
    ALIBI_ERR_INVALID = -1,     /* null pointer, non-positive size, misaligned pointer */
    ALIBI_ERR_UNSUPPORTED = -2, /* valid request the library does not implement (e.g. d) */
    ALIBI_ERR_CUDA = -3,        /* a CUDA runtime/driver call or kernel launch failed    */
    ALIBI_ERR_TIMEOUT = -4,     /* a bounded device-side wait expired (see alibi_check_error) */
    ALIBI_ERR_CHECK = -5        /* debug-checks build only: a kernel found a bad TMA / TMEM / shared
                                   address, recorded it and skipped the access */
} alibi_status;

/* Library version as an integer (major * 10000 + minor * 100 + patch). */
ALIBI_API int alibi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
ALIBI_API const char *alibi_status_str(int status);

/*
 * ALiBi slopes for H heads, written to HOST memory out_host[0..H-1] as fp32.
 * "ALiBi: Attention with Linear Biases", "Different heads, different distance
 * penalties": for a power-of-two H, m_h = 2^(-8(h+1)/H); otherwise the
 * schedule of the largest power of two c < H followed by every other entry
 * (1st, 3rd, ...) of the 2c schedule, H - c of them. Each value is the exact
 * real rounded once to fp32 (round to nearest even). Host-only; H in [1, 4096].
 */
ALIBI_API int alibi_slopes(int H, float *out_host);

/*
 * Causal prefill, bf16 in / bf16 out, fp32 LSE (natural log).
 * q, k, v: device bf16 [B, H, N, d]; out: device bf16 [B, H, N, d];
 * lse: device fp32 [B, H, N] (may be NULL to skip it);
 * LSE_i = ln sum_{j<=i} exp(q_i.k_j/sqrt(d) - m_h (i - j)).
 * d in {16, 32, 64, 128} (16 and 32 run the d = 64 tiles with zero columns);
 * N >= 1; causal = 1 (0: symmetric bias over all keys, see
 * alibi_attn_fwd_ex).
 * Runs the tcgen05/TMEM/TMA kernel: scores and P.V on the tensor cores with
 * fp32 accumulation; the bias is generated from tile coordinates and never
 * stored; online softmax in fp32; P rounded to bf16 for the P.V product.
 * Large launches take the blocked work order described under
 * alibi_attn_fwd_ex (same results).
 */
ALIBI_API int alibi_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                   int B, int H, int N, int d, int causal, void *stream);

/* Flags of alibi_attn_fwd_ex. */
#define ALIBI_FWD_SKIP_UNDERFLOW 1u /* leave out tiles whose weights flush to zero (exact)   */
#define ALIBI_FWD_CLAMP 2u          /* bias B* = max(B, clamp_min)                          */
#define ALIBI_FWD_LOGDIST 4u        /* distance D* = ln(D + 1)                              */
#define ALIBI_FWD_SOFTCAP 8u        /* content score A* = z tanh(A / z), z = softcap_z      */
#define ALIBI_FWD_NOMINAL_ORDER 16u /* keep the nominal work order (see below)               */

/*
 * Options of alibi_attn_fwd_ex (plain C; pass NULL for the defaults).
 */
typedef struct alibi_fwd_options {
    unsigned int flags;   /* ALIBI_FWD_* bits                                             */
    float clamp_min;      /* ALIBI_FWD_CLAMP: bias floor in natural-log units, < 0         */
    float softcap_z;      /* ALIBI_FWD_SOFTCAP: cap z > 0                                  */
    const float *slopes;  /* optional HOST array of H per-head slopes (natural-log units,
                             finite, >= 0; > 0 with ALIBI_FWD_SKIP_UNDERFLOW); NULL means
                             alibi_slopes(H). alibi_slopes_explicit() builds the paper's
                             robust / explicit schedules.                               */
} alibi_fwd_options;

/*
 * alibi_attn_fwd with options; opt = NULL (or all-zero) is exactly alibi_attn_fwd.
 * causal = 0 selects the symmetric bias -m_h |i - j| over all keys ("ALiBi and
 * Relative Position Bias", "The mechanics"; the encoder models of "When
 * Attention Goes Blind", Table 5).
 *
 * ALIBI_FWD_SKIP_UNDERFLOW (causal only): leave out the KV tiles at the far end
 * of each query block's causal range whose weights provably flush to zero
 * ("When Attention Goes Blind", sec. 3.2-3.3: past the blindness distance the
 * exponent falls below the smallest normal number; sec. 5.2: steep heads act
 * as a sliding window). A pre-pass bounds every score by |q_i| max_j |k_j| and
 * the running max from below by the diagonal score; a tile is left out only if
 * every exponent in it is below -127 (base 2), where the kernel's
 * flush-to-zero exponential returns exactly 0. Output and LSE are therefore
 * bit-identical to the same call without the flag. The pre-pass reads Q and K
 * once and takes a plan buffer (16 bytes per work item and 8 per query row)
 * from the library's stream-ordered pool.
 *
 * ALIBI_FWD_CLAMP / _LOGDIST / _SOFTCAP: the mitigations of "When Attention
 * Goes Blind", sec. 3.4 (the paper trains with clamp_min = -87, sec. 4.3, and
 * z = 50), in any combination. They cannot be combined with
 * ALIBI_FWD_SKIP_UNDERFLOW (clamped or log-scaled biases do not underflow). *
 * Work order: a launch (causal or not) whose K and V (4 B H N d bytes) exceed
 * half the L2 cache and that has at most 16 blocks of 256 rows per head runs
 * its work items head by head in blocks of two rounds of the persistent grid,
 * so each head's K and V are read from DRAM about once. The first such launch
 * of a shape on a device builds a table of B H ceil(N/256) x 8 bytes in device
 * memory, which the library keeps for the life of the process (at most 256
 * shapes and 256 MiB; beyond that, and when the first launch of a shape is
 * made while its stream is being captured, the nominal order runs). Every
 * item computes the same values in either order: output and LSE are
 * bit-identical. ALIBI_FWD_NOMINAL_ORDER keeps the nominal longest-first order
 * (no table). alibi_attn_bwd applies the same rule to its two kernels (dK/dV
 * items stream a head's Q and dO, dQ items its K and V; one table of
 * B H ceil(N/128) x 8 bytes each), without the limit on blocks per head, and
 * honours the same flag; its gradients are bit-identical in either order too.
 */
ALIBI_API int alibi_attn_fwd_ex(const void *q, const void *k, const void *v, void *out, float *lse,
                   int B, int H, int N, int d, int causal, const alibi_fwd_options *opt, void *stream);

/*
 * Explicit ("robust") slopes, "When Attention Goes Blind" sec. 3.4 "Robust
 * Slopes" and sec. 4.3: choose the slopes so the blindness distances
 * delta_h = min{D : -m_h D* <= tau} spread geometrically from delta_first
 * (head 0, steepest) to delta_last (head H-1): delta_h = delta_first
 * (delta_last / delta_first)^(h / (H - 1)), m_h = -tau / delta_h with linear
 * distances, or m_h = -tau / ln(delta_h + 1) with log-scaled distances (the
 * E+L combination). tau < 0 is the underflow threshold in natural-log units
 * (ln 2^-126 = -87.3365 reproduces the paper's tables). Host-only; writes H
 * fp32 values (rounded to nearest) to out_host.
 */
ALIBI_API int alibi_slopes_explicit(int H, double delta_first, double delta_last, double tau, int log_distance,
                   float *out_host);

/*
 * The skip plan alone (analysis and tests): for each work item w = (b*H + h) *
 * ceil(N/256) + blk (query rows [256 blk, 256 blk + 256) of head (b, h)),
 * first_tile[w] is the first 128-key tile the skipping kernel computes; tiles
 * 0 .. first_tile[w]-1 are left out. first_tile: device int32 [B*H*ceil(N/256)].
 * slopes: optional HOST array of H slopes as in alibi_fwd_options (NULL:
 * alibi_slopes(H)). d in {16, 32, 64, 128}.
 */
ALIBI_API int alibi_attn_skip_plan(const void *q, const void *k, int B, int H, int N, int d, const float *slopes,
                   int *first_tile, void *stream);

/*
 * Backward of alibi_attn_fwd / alibi_attn_fwd_ex: the gradients of sum(dout * out)
 * with respect to q, k and v. There is no trainable parameter in the bias; the
 * weights are recomputed from the forward's LSE (P_ij = exp(x_ij - lse_i)), so
 * a weight that underflowed in the forward carries no gradient here either
 * ("When Attention Goes Blind", sec. 5.1).
 *   dV = P^T dO,  dS = P o (dO V^T - rowsum(dO o O)),  dQ = dS K / sqrt(d),
 *   dK = dS^T Q / sqrt(d).
 * q, k, v, out, dout, dq, dk, dv: device bf16 [B, H, N, d] (out is the
 * forward's output); lse: device fp32 [B, H, N] (the forward's natural-log
 * LSE). All device pointers 16-byte aligned. d in {64, 128}; causal and opt
 * exactly as the forward ran (NULL: defaults). With ALIBI_FWD_CLAMP / _LOGDIST
 * the weights are recomputed with that bias; with ALIBI_FWD_SOFTCAP dS is also
 * multiplied by the cap's derivative 1 - tanh^2(A / z) before it meets K or Q.
 * ALIBI_FWD_SKIP_UNDERFLOW has no backward (ALIBI_ERR_UNSUPPORTED).
 * Deterministic (no atomics). Takes B*H*N*4 bytes of scratch from the
 * library's stream-ordered pool for the row sums.
 */
ALIBI_API int alibi_attn_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d, int causal,
                   const alibi_fwd_options *opt, void *stream);

/*
 * alibi_attn_bwd in fp32 at reference precision (CUDA cores, IEEE expf): all
 * tensors device fp32 with the same layouts; lse from alibi_attn_fwd_f32;
 * d in [1, 256]; default slopes.
 */
ALIBI_API int alibi_attn_bwd_f32(const float *q, const float *k, const float *v, const float *out,
                   const float *lse, const float *dout, float *dq, float *dk, float *dv, int B, int H, int N,
                   int d, int causal, void *stream);

/*
 * Causal prefill in fp32 (reference precision): all inputs, outputs and
 * arithmetic in fp32 on the CUDA cores with IEEE expf. Same layouts and
 * semantics as alibi_attn_fwd (causal = 0: symmetric bias); d in [1, 256];
 * lse may be NULL.
 */
ALIBI_API int alibi_attn_fwd_f32(const float *q, const float *k, const float *v, float *out, float *lse,
                       int B, int H, int N, int d, int causal, void *stream);

/*
 * Decode: one new query per (b, h) at its true sequence position L - 1,
 * attending to keys 0..L-1 of the cache ("ALiBi: Attention with Linear
 * Biases", KV-cache paragraph): s_j = q.k_j/sqrt(d) - m_h (L - 1 - j).
 * q: device bf16 [B, H, d]; kcache, vcache: device bf16 [B, H, L, d];
 * out: device bf16 [B, H, d]. d in {16, 32, 64, 128}; L >= 1.
 * Split-K over the cache with an fp32 partial-softmax merge, done in the same
 * kernel by the CTA that finishes each (b, h) last. When it splits, the
 * partials buffer and B*H split counters are taken from a library-owned
 * stream-ordered memory pool (cudaMallocFromPoolAsync / cudaFreeAsync on
 * `stream`) and the counters are zeroed with cudaMemsetAsync on `stream`.
 */
ALIBI_API int alibi_attn_decode(const void *q, const void *kcache, const void *vcache, void *out,
                      int B, int H, int L, int d, void *stream);

/*
 * Per-block maximum key norms for skipping in the decode: knorm[b][h][c] =
 * max over keys j in [64 c, 64 c + 64) of |k_j|_2 (fp32, from the bf16 cache).
 * kcache: device bf16 [B, H, L, d]; knorm: device fp32 [B, H, ceil(L/64)],
 * caller-owned. Only blocks c >= blk_begin are (re)computed, so a serving loop
 * that appends keys refreshes the tail block(s) alone (blk_begin = old L / 64);
 * blk_begin = 0 computes all. d in {16, 32, 64, 128}.
 */
ALIBI_API int alibi_kv_block_norms(const void *kcache, float *knorm, int B, int H, int L, int d, int blk_begin,
                   void *stream);

/*
 * alibi_attn_decode that leaves out the cache rows whose weights are provably
 * below 2^-127 of the row's largest ("When Attention Goes Blind" sec. 3.2-3.3
 * and 5.2: past a head's blindness distance its weights underflow; steep heads
 * act as sliding windows). With the last key's logit x_last as a lower bound of
 * the row max and c1 = log2(e)/sqrt(d), a step of keys is skipped when
 * c1 |q| max|k| - m_h log2(e) (L - 1 - j) <= x_last - 127 for all its keys
 * (with a 2^-10 relative slack on the norms); those K and V rows are never
 * read. The omitted weights are below the fp32 resolution of the normaliser, so
 * the output matches alibi_attn_decode within rounding. knorm from
 * alibi_kv_block_norms for the same cache. Other arguments as alibi_attn_decode.
 */
ALIBI_API int alibi_attn_decode_skip(const void *q, const void *kcache, const void *vcache, const float *knorm,
                   void *out, int B, int H, int L, int d, void *stream);

/*
 * Number of KV-cache splits alibi_attn_decode uses for this shape (host-only,
 * deterministic for a given device). 1 means a single kernel with no partials
 * buffer; S > 1 means one kernel of S CTAs per (b, h) whose last CTA merges,
 * with a partials buffer of B*H*S*(d+4) floats and B*H counters. Returns a
 * negative alibi_status on invalid arguments.
 */
ALIBI_API int alibi_attn_decode_splits(int B, int H, int L, int d);

/*
 * Decode that allocates nothing. The pages have no counterpart to this entry
 * point: it is for callers that cannot let a library allocate device memory
 * (a serving process whose allocator already reserved the whole GPU, a
 * real-time decode loop that cannot absorb allocation latency, a runtime that
 * forbids allocations outside its own arena). Same arguments, layouts, split
 * plan and results as alibi_attn_decode; the caller still passes inputs and
 * outputs. The split-K partials live in a fixed 4 MiB device buffer and the
 * split counters in a fixed 128 KiB one, both compiled into the library (held
 * by every GPU that loads it until process exit); no cudaMalloc, cudaFree, pool
 * allocation or memset happens.
 *   - The first call on each device does a one-time set-up (it looks up the
 *     buffer's device address); make that first call before any stream capture.
 *   - All calls share the buffer and it keeps the last call's contents (each
 *     call overwrites every partial it reads, so nothing needs clearing, and
 *     leaves every counter at zero, as the library loads them). Calls that
 *     overlap on the GPU (e.g. on different streams) race on it: order them.
 *   - Returns ALIBI_ERR_UNSUPPORTED if the split plan needs more than 4 MiB of
 *     partials (B*H*S*(d+4)*4 bytes with S = alibi_attn_decode_splits(...)) or
 *     more than 32768 (b, h) pairs split.
 */
ALIBI_API int alibi_attn_decode_noalloc(const void *q, const void *kcache, const void *vcache, void *out,
                      int B, int H, int L, int d, void *stream);

/*
 * Attention weights of the fp32 path (test and analysis export):
 * P[b,h,i,j] = exp(q_i.k_j/sqrt(d) - m_h (i - j) - lse[b,h,i]) for j <= i,
 * 0 for j > i. q, k: device fp32 [B, H, N, d]; lse: device fp32 [B, H, N]
 * from alibi_attn_fwd_f32; P: device fp32 [B, H, N, N]. d in [1, 256].
 */
ALIBI_API int alibi_attn_probs_f32(const float *q, const float *k, const float *lse, float *P,
                         int B, int H, int N, int d, void *stream);

/* alibi_attn_probs_f32 for either mask: causal = 0 uses exp(x_ij - lse_i) with the
 * symmetric bias -m_h |i - j| for every key. */
ALIBI_API int alibi_attn_probs_f32_ex(const float *q, const float *k, const float *lse, float *P,
                         int B, int H, int N, int d, int causal, void *stream);

/*
 * Underflow count ("When Attention Goes Blind", sec. 3.2-3.3): per head h,
 * the number of causal pairs (b, i, j <= i) whose max-subtracted exponent
 * x_ij - M_i (natural-log units, x_ij = q_i.k_j/sqrt(d) - m_h (i - j),
 * M_i = max_j x_ij) is <= tau. Two passes per row in fp32 (row max, then
 * count). q, k: device bf16 [B, H, N, d]; counts: device uint64 [H],
 * overwritten (zeroed on `stream` first). d in {16, 32, 64, 128}.
 */
ALIBI_API int alibi_attn_underflow_bf16(const void *q, const void *k, int B, int H, int N, int d, float tau,
                              unsigned long long *counts, void *stream);

/*
 * The same count for the decode row ("When Attention Goes Blind", sec. 3.2-3.3,
 * applied to the query at position L-1 of "ALiBi: Attention with Linear Biases",
 * the KV-cache paragraph): per head h, summed over b, the number of cached keys j
 * (0 <= j < L) whose max-subtracted exponent x_j - M is <= tau, with
 * x_j = q.k_j/sqrt(d) - m_h (L-1-j) and M = max_j x_j. Two passes over K in
 * fp32. q: device bf16 [B, H, d]; kcache: device bf16 [B, H, L, d]; counts:
 * device uint64 [H], overwritten (zeroed on `stream` first). d in
 * {16, 32, 64, 128}. Reporting only (it reads K twice).
 */
ALIBI_API int alibi_decode_underflow_bf16(const void *q, const void *kcache, int B, int H, int L, int d, float tau,
                                          unsigned long long *counts, void *stream);

/*
 * Self-test of the failure path; the pages have no counterpart to it. Launches
 * one CTA whose thread waits on a shared-memory barrier that nothing ever
 * arrives on, through the same bounded wait every kernel uses. After about one
 * second the wait gives up, records a timeout in the device status word and the
 * kernel returns normally; alibi_check_error(stream) then returns
 * ALIBI_ERR_TIMEOUT and clears the word. No fault, trap or hang is involved and
 * the CUDA context stays usable.
 */
ALIBI_API int alibi_selftest_timeout(void *stream);

/*
 * Self-test of the failure path through the bf16 prefill kernel itself; the
 * pages have no counterpart to it. Runs the bf16 prefill on the caller's buffers
 * (same arguments, layouts and checks as alibi_attn_fwd; the kernel build that
 * carries the mitigations, none of them enabled) with two changes: each CTA's TMA producer
 * leaves out the loads of its first work item's Q tiles, and every bounded
 * wait gives up after wait_us microseconds (1 <= wait_us <= 1000000). The MMA
 * issuer's wait for that tile runs out; the kernel records ALIBI_ERR_TIMEOUT in
 * the device status word, its other roles stop at their next wait, every load
 * and MMA already issued is waited for, TMEM is freed and the kernel returns.
 * out and lse are left undefined. alibi_check_error(stream) then returns
 * ALIBI_ERR_TIMEOUT and the context stays usable. No fault, trap or hang is
 * involved.
 */
ALIBI_API int alibi_selftest_fwd_timeout(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                                         int H, int N, int d, int wait_us, void *stream);

/*
 * Synchronise `stream`, then read and clear the device status word of the
 * current device. Returns ALIBI_ERR_TIMEOUT if a kernel gave up a bounded
 * wait since the last check, ALIBI_ERR_CUDA if the stream reports an error,
 * ALIBI_ERR_CHECK if a kernel of the debug-checks build (the same library compiled
 * with -DALIBI_CHECKS: every TMA coordinate, TMEM address and shared-memory operand
 * tested before use) found a bad one (the second word of the status records the
 * check and the value), else ALIBI_OK. The word accumulates until it is collected here, but an
 * uncollected error does not affect later calls: a kernel's waits give up early
 * only on a failure inside the same CTA, so calls made after a timeout compute
 * their results normally (the timeout is still reported by the next check).
 */
ALIBI_API int alibi_check_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ALIBI_H */

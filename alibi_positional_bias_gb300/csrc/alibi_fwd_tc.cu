// ALiBi prefill on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, per (b, h) and query row i,
//   x_ij = q_i.k_j / sqrt(d) - m_h (i - j)   for j <= i        (causal: keys j > i masked)
//   x_ij = q_i.k_j / sqrt(d) - m_h |i - j|   for all j < N     (non-causal, symmetric bias
//          of "ALiBi and Relative Position Bias" (quantmemo.com), "The mechanics")
//   O_i  = sum_j softmax_j(x_ij) v_j,   LSE_i = ln sum_j exp(x_ij)
// following "When Attention Goes Blind: Numerical Failure in ALiBi Positional
// Encodings" (arXiv 2608.03994) sec. 3.1 eq. 1-3 and App. B.1 (max-shifted
// softmax), and "ALiBi: Attention with Linear Biases" (abhik.ai), "From
// distance to a normalized weight" and the remark after the full-sequence
// example that a production kernel generates the biases inside its tiles.
//
// Design (one persistent CTA per SM, 384 threads):
//   warp 0      TMA producer: Q tiles once per work item, K/V tiles through a
//               2-stage ring of units, each K(u) with V(u-1) behind one barrier
//               pair (128-byte swizzle, zero fill past N), so the MMA issuer
//               tests one barrier and commits one release per KV tile.
//   warp 1      TMEM allocator and MMA issuer (converged, one elected lane
//               issues):
//                 S_s = Q_s K^T   (128 x 128, fp32 in TMEM, smem x smem)
//                 O_s += P_s V    (128 x d,   fp32 in TMEM, P read from TMEM)
//   warps 4-7   softmax for Q tile slot 0, warps 8-11 for slot 1: each thread
//               owns one query row (tcgen05.ld gives a thread a whole TMEM
//               lane), so the row max and row sum need no shuffles. The bias
//               is generated from the integer tile coordinates; the running
//               max is raised lazily (only when a tile exceeds it by 2^8).
//               The same warps write O / l through per-warp staging boxes and
//               bulk tensor stores.
// A work item is (b*H + h, block of 256 query rows = two 128-row tiles);
// KV tiles are visited from the diagonal downwards. Causal: tiles entirely
// above the diagonal are never loaded. Non-causal: after tile 0 the walk wraps
// to the last tile and comes back down to the diagonal, so every row meets its
// largest biases (the diagonal) first. Items are dealt longest-first in snake
// order.
//
// TMEM columns: S/P slot s at [128 s, 128 s + 128), O slot s at 256 + 128 s.
// P (bf16, two per 32-bit column) overwrites the first 64 columns of S.

#include <cuda.h>

#include <type_traits>

#include "ptx.cuh"

namespace alibi {
namespace {

constexpr int BM = 128;  // query rows per tile (MMA M)
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 384;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Register split: the kernel launches with kLaunchRegs per thread (384 threads,
// one CTA per SM); the producer/MMA warpgroup gives registers back and the two
// softmax warpgroups take them. The shares add up exactly to the launch total.
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kRegsLow = 88;    // warps 0-3
constexpr uint32_t kRegsHigh = 208;  // warps 4-11
static_assert(128 * kRegsLow + 256 * kRegsHigh == kThreads * kLaunchRegs, "register split must match launch");

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms along d
    static constexpr uint32_t kChunkBytes = BM * 128;      // one 64-column box: 16 KB
    static constexpr uint32_t kTileBytes = BM * D * 2;     // one 128 x D bf16 tile
    static constexpr uint32_t kQ = 0;                      // 2 Q tiles
    static constexpr uint32_t kK = 2 * kTileBytes;         // K tiles of the two ring stages
    static constexpr uint32_t kV = kK + kKStages * kTileBytes;  // V tiles of the two ring stages
    // One 128 x 64 swizzle atom of bias operands: ones (K-step 0, the A side), the
    // column bias m log2(e) c / c1 for the two items in flight (K-steps 1, 2, the B
    // side), and minus ones (K-step 3, the A side that turns the same column bias
    // into -m log2(e) c / c1 for keys after the rows, non-causal).
    static constexpr uint32_t kAux = kV + kVStages * kTileBytes;
    // Epilogue staging: 2 KB per softmax warp, one 32 x 32 bf16 box of O at a time.
    static constexpr uint32_t kStage = kAux + kChunkBytes;
    static constexpr uint32_t kBar = kStage + kChunkBytes;
    static constexpr uint32_t kSmem = kBar + 256 + 1024;   // barriers, TMEM slot, alignment slack
};

struct FwdParams {
    CUtensorMap tq, tk, tv;  // [BH, N, d] bf16, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tout;        // [BH, N, d] bf16, box {32, 32, 1}, no swizzle (epilogue stores)
    __nv_bfloat16 *out;
    float *lse;
    uint32_t *err;
    uint64_t wait_ns;  // limit of every bounded wait
    int test_skip_q0;  // failure-path self-test (mitigation kernels only): the producer leaves out the first item's Q tiles
    int N, BH, H, NQB, NQT, num_items;
    FastDiv div_bh, div_h, div_nqb;  // by B*H, H and NQB
    int dr;  // the tensors' head size (<= D: the D = 64 kernel also serves d = 16 and 32)
    int causal;  // 1: keys j <= i only; 0: every key, distance |i - j|
    float c1;  // log2(e) / sqrt(d)
    const int2 *plan;  // optional: work order (item, first KV tile); null = dense, nominal order
    // Mitigations of "When Attention Goes Blind" sec. 3.4 (kFwdClamp / kFwdLogDist /
    // kFwdSoftcap bits; 0 = plain ALiBi). Constants in base-2 exponent units:
    unsigned int variant;
    float clamp2;  // clamp_min log2(e)
    float cap_k;   // 2 log2(e) / (sqrt(d) z): 2^(s cap_k) = e^(2 A / z)
    float cap_zl;  // z log2(e)
    Slopes slopes;
};

enum : uint32_t {
    SITE_PROD_Q = 0x101, SITE_PROD_K = 0x102, SITE_PROD_V = 0x103,
    SITE_MMA_Q = 0x201, SITE_MMA_K = 0x202, SITE_MMA_V = 0x203, SITE_MMA_P = 0x204, SITE_MMA_O = 0x205,
    SITE_MMA_DONE = 0x206, SITE_SM_S = 0x301, SITE_SM_O = 0x302,
};

struct Item {
    int bh, qb;
    int top;  // first KV tile visited (the diagonal of the item's upper Q tile)
    int n;    // KV tiles visited: top, top - 1, ..., then (non-causal) NQT - 1, ..., top + 1
    bool q1valid;
};

__device__ __forceinline__ float lg2_approx(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The plain kernel adds the column part of the bias on the tensor core (the bias
// operands of ptx.cuh): for a KV tile left of a Q tile's diagonal the bias is
// -m (i - k0) + m c and B row c holds m log2(e) c / c1; right of it (non-causal)
// it is -m (k0 - i) - m c and B row c holds -m log2(e) c / c1. S' = q.k + bias / c1
// comes out of the accumulator and the softmax only adds the row part. Diagonal
// tiles of the non-causal kernel (|i - k| is not linear in c) take no bias step.
__device__ __forceinline__ bool use_aux_bias(const FwdParams &p, bool var) { return !var; }

__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Max of 128 values as 8 independent chains of three-input max (short dependency chains).
__device__ __forceinline__ float row_max128(const float (&x)[128])
{
    float m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m[k] = x[k];
#pragma unroll
        for (int t = 1; t + 1 < 16; t += 2) m[k] = max3f(m[k], x[k + 8 * t], x[k + 8 * (t + 1)]);
        m[k] = fmaxf(m[k], x[k + 8 * 15]);
    }
    return fmaxf(max3f(m[0], m[1], m[2]), max3f(max3f(m[3], m[4], m[5]), m[6], m[7]));
}

__device__ __forceinline__ int item_index(int k)
{
    const int G = gridDim.x, c = blockIdx.x;
    return (k & 1) ? (k + 1) * G - 1 - c : k * G + c;
}

// Work item at position idx of the schedule. Without a plan, items are taken
// longest-first: round r holds the 256-row block NQB-1-r of every (b, h). With a
// plan (underflow skipping), the plan gives the item and the first KV tile worth
// computing, already sorted by the tiles the item spans.
__device__ __forceinline__ Item decode_item(const FwdParams &p, int idx, bool causal)
{
    Item it;
    int first = 0;
    if (p.plan) {
        const int2 e = p.plan[idx];
        it.bh = fdiv(e.x, p.div_nqb);
        it.qb = e.x - it.bh * p.NQB;
        first = e.y;
    } else {
        const int round = fdiv(idx, p.div_bh);
        it.bh = idx - round * p.BH;
        it.qb = p.NQB - 1 - round;
    }
    const int qt1 = 2 * it.qb + 1;
    it.q1valid = qt1 < p.NQT;
    it.top = it.q1valid ? qt1 : qt1 - 1;
    it.n = causal ? it.top + 1 - first : p.NQT;
    return it;
}

// KV tile visited at iteration `it` of an item (0 <= it < n).
__device__ __forceinline__ int kv_tile(const FwdParams &p, const Item &t, int it)
{
    const int j = t.top - it;
    return j >= 0 ? j : j + p.NQT;
}

// Is Q slot s active at iteration `it`? Causal: slot 0 skips the first tile (the
// diagonal of slot 1 lies entirely above slot 0's rows). Non-causal: always.
__device__ __forceinline__ bool slot_active(const Item &t, int s, int it, bool causal)
{
    return s == 1 ? t.q1valid : (t.q1valid && causal ? it >= 1 : true);
}

// VAR: compiled with the sec. 3.4 mitigation path (p.variant selects which ones);
// the plain ALiBi kernel (VAR = false) carries none of that code.
template <int D, bool VAR, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ FwdParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBar);
    uint64_t *q_full = bars + 0;    // [1] both Q tiles of the item loaded
    uint64_t *q_empty = bars + 2;   // [1]
    uint64_t *unit_full = bars + 3;    // [2] ring unit of stage s loaded (K(u) and V(u - 1))
    uint64_t *unit_empty = bars + 5;   // [2] ring unit of stage s read by the MMAs
    uint64_t *s_full = bars + 11;   // [2]
    uint64_t *p_full = bars + 13;   // [2]
    uint64_t *o_full = bars + 15;   // [2]
    uint64_t *o_empty = bars + 17;  // [2]
    uint64_t *mma_done = bars + 19; // [1]
    uint64_t *p_hi = bars + 20;     // [2] P of keys 64..127 written (p_full covers keys 0..63)
    uint64_t *bias_full = bars + 22;  // [2] column-bias operand of item k written (buffer k & 1)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 24);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint32_t *err = p.err;

    if (threadIdx.x == 0) {
        cta_err_init(p.wait_ns);
        cta_check_init(p.err, smem_raw, C::kSmem);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&unit_full[s], 1);
            mbar_init(&unit_empty[s], 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 4);   // one arrival per softmax warp
            mbar_init(&p_hi[s], 4);
            mbar_init(&o_full[s], 1);
            mbar_init(&o_empty[s], 4);
        }
        mbar_init(q_empty, 1);
        mbar_init(q_full, 1);
        mbar_init(mma_done, 1);
        mbar_init(&bias_full[0], 4);  // the slot-0 softmax warps
        mbar_init(&bias_full[1], 4);
        fence_mbar_init();
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tk);
        tma_prefetch_desc(&p.tv);
        tma_prefetch_desc(&p.tout);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (use_aux_bias(p, VAR) && threadIdx.x < 2 * BM) {
        // ones in logical 16-byte chunks 0-1 of every row (the A operand of the bias MMA)
        write_ones_chunk(smem + C::kAux, threadIdx.x >> 1, threadIdx.x & 1);
        if (!CAUSAL && (threadIdx.x & 1)) write_neg_ones_step3(smem + C::kAux, threadIdx.x >> 1);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
    // producer / MMA warpgroup: give registers back (all four warps execute this)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t uc = 0;       // ring units issued
            int qk = -1;           // item whose Q tiles were issued last
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int w = item_index(k);
                if (w >= p.num_items) break;
                const Item t = decode_item(p, w, CAUSAL);
                ok = mbar_wait(q_empty, (k & 1) ^ 1, err, SITE_PROD_Q);
                if (!ok) break;
                // both Q tiles of the item behind one barrier (the failure-path self-test
                // leaves out the first item's Q: the issuer's wait for it runs out)
                if (!(VAR && p.test_skip_q0 && k == 0)) {
                    qk = k;
                    mbar_arrive_expect_tx(&q_full[0], 2 * C::kTileBytes);
                    for (int s = 0; s < 2; ++s)
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d(smem + C::kQ + s * C::kTileBytes + c * C::kChunkBytes, &p.tq, 64 * c,
                                        (2 * t.qb + s) * BM, t.bh, &q_full[0]);
                }
                // One ring unit per step u = 0 .. n: K(u) (u < n) and V(u - 1) (u >= 1) into the
                // K and V buffers of stage uc % 2, behind one barrier pair. Unit u is consumed
                // in the MMA issuer's iteration u - 1 (P V of V(u-1), then S of K(u)).
                for (int u = 0; u <= t.n && ok; ++u) {
                    const uint32_t st = uc % 2, ph = (uc / 2) & 1;
                    ok = mbar_wait(&unit_empty[st], ph ^ 1, err, SITE_PROD_K);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&unit_full[st], (u < t.n ? C::kTileBytes : 0u) + (u >= 1 ? C::kTileBytes : 0u));
                    for (int c = 0; c < C::kChunks; ++c) {
                        if (u < t.n)
                            tma_load_3d(smem + C::kK + st * C::kTileBytes + c * C::kChunkBytes, &p.tk, 64 * c,
                                        kv_tile(p, t, u) * BN, t.bh, &unit_full[st]);
                        if (u >= 1)
                            tma_load_3d(smem + C::kV + st * C::kTileBytes + c * C::kChunkBytes, &p.tv, 64 * c,
                                        kv_tile(p, t, u - 1) * BN, t.bh, &unit_full[st]);
                    }
                    ++uc;
                }
            }
            // Drain (also after an error): the last Q load and the last load into each ring stage
            // has landed before the CTA can exit. Earlier loads into a stage were consumed,
            // hence complete, before the stage was reused.
            if (qk >= 0) mbar_wait(&q_full[0], qk & 1, err, SITE_PROD_Q, true);
            for (uint32_t n = uc > 2 ? uc - 2 : 0; n < uc; ++n)
                mbar_wait(&unit_full[n % 2], (n / 2) & 1, err, SITE_PROD_K, true);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        // The whole warp runs this loop (converged, warp-uniform values); one elected
        // lane issues each tcgen05 instruction.
        {
            constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0);
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, 1);
            const uint32_t sQ = smem_u32(smem + C::kQ);
            const uint32_t sK = smem_u32(smem + C::kK);
            const uint32_t sV = smem_u32(smem + C::kV);
            const bool aux = use_aux_bias(p, VAR);
            const uint64_t auxd = smem_desc_sw128(smem_u32(smem + C::kAux), 16, 1024);
            uint32_t uc = 0;  // ring units consumed
            uint32_t p_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int w = item_index(k);
                if (w >= p.num_items) break;
                const Item t = decode_item(p, w, CAUSAL);
                ok = mbar_wait(&q_full[0], k & 1, err, SITE_MMA_Q);
                if (ok && aux) ok = mbar_wait(&bias_full[k & 1], (k >> 1) & 1, err, SITE_MMA_Q);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;

                // S_s = Q_s K^T over d in steps of 16 (K-major operands, 32-byte steps inside a
                // swizzle atom, 16 KB per 64-column atom). Descriptors are built once per tile;
                // each step adds a compile-time offset to the 14-bit address field (smem
                // addresses stay below 256 KB, so the field never carries).
                auto issue_S = [&](int s, uint32_t kst, int jt) {
                    const uint64_t qd = smem_desc_sw128(sQ + s * C::kTileBytes, 16, 1024);
                    const uint64_t kd = smem_desc_sw128(sK + kst * C::kTileBytes, 16, 1024);
                    const uint32_t dst = tmem + s * 128;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t step = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
                        mma_ss_w(dst, qd + step, kd + step, idS, kk > 0);
                    }
                    // column bias: ones (K-step 0 of atom A) x this item's bias rows
                    if (aux) {
                        const int qt = 2 * t.qb + s;
                        if (CAUSAL || jt < qt)
                            mma_ss_w(dst, auxd, auxd + 2 * (1 + (k & 1)), idS, 1u);
                        else if (jt > qt)
                            mma_ss_w(dst, auxd + 6, auxd + 2 * (1 + (k & 1)), idS, 1u);  // minus ones
                    }
                    mma_commit_w(&s_full[s]);
                };
                // O_s += P_s V over the 128 keys in steps of 16 (V is MN-major: d contiguous;
                // 16 keys = 2048 bytes per step)
                // (issued in two halves of 64 keys as the softmax hands P over)
                auto issue_PV_half = [&](int s, uint32_t vst, bool first, int half) {
                    const uint64_t vd = smem_desc_sw128(sV + vst * C::kTileBytes, C::kChunkBytes, 1024);
                    const uint32_t dst = tmem + 256 + s * 128, pa = tmem + s * 128;
#pragma unroll
                    for (int k4 = 0; k4 < BN / 32; ++k4) {
                        const int kk = half * (BN / 32) + k4;
                        mma_ts_w(dst, pa + kk * 8, vd + ((kk * 2048) >> 4), idO, (first && kk == 0) ? 0u : 1u);
                    }
                };

                bool first_pv[2] = {true, true};
                // prologue: K(0) and the S of slots active at it = 0
                {
                    const uint32_t st = uc % 2, ph = (uc / 2) & 1;  // unit 0: K(0)
                    ok = mbar_wait(&unit_full[st], ph, err, SITE_MMA_K);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    for (int s = 0; s < 2; ++s)
                        if (slot_active(t, s, 0, CAUSAL)) issue_S(s, st, kv_tile(p, t, 0));
                    mma_commit_w(&unit_empty[st]);
                    ++uc;
                }
                for (int it = 0; it < t.n && ok; ++it) {
                    // unit it + 1: V(it) and K(it + 1), normally resident long before needed
                    const uint32_t vst = uc % 2, uph = (uc / 2) & 1;
                    ok = mbar_wait(&unit_full[vst], uph, err, SITE_MMA_V);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    for (int s = 0; s < 2 && ok; ++s) {
                        if (slot_active(t, s, it, CAUSAL)) {
                            ok = mbar_wait_spin(&p_full[s], p_cnt[s] & 1, err, SITE_MMA_P);
                            if (ok && first_pv[s]) ok = mbar_wait(&o_empty[s], (o_cnt[s] & 1) ^ 1, err, SITE_MMA_O);
                            ok = __all_sync(0xffffffffu, ok);
                            if (!ok) break;
                            tc_fence_after();
                            issue_PV_half(s, vst, first_pv[s], 0);
                            ok = mbar_wait_spin(&p_hi[s], p_cnt[s] & 1, err, SITE_MMA_P);
                            ++p_cnt[s];
                            ok = __all_sync(0xffffffffu, ok);
                            if (!ok) break;
                            tc_fence_after();
                            issue_PV_half(s, vst, first_pv[s], 1);
                            first_pv[s] = false;
                            if (it == t.n - 1) {
                                mma_commit_w(&o_full[s]);
                                ++o_cnt[s];
                            }
                        }
                        if (it + 1 < t.n && slot_active(t, s, it + 1, CAUSAL))
                            issue_S(s, vst, kv_tile(p, t, it + 1));
                    }
                    mma_commit_w(&unit_empty[vst]);  // the unit's V and K have both been read
                    ++uc;
                }
                mma_commit_w(q_empty);
            }
            // drain: every MMA issued above completes before TMEM is released
            mma_commit_w(mma_done);
            mbar_wait(mma_done, 0, err, SITE_MMA_DONE, true);
        }
    }
    } else {
        // ------------------------------------------------ softmax warpgroups
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        const int s = (warp - 4) >> 2;
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        uint32_t s_cnt = 0, o_cnt = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int w = item_index(k);
            if (w >= p.num_items) break;
            const Item t = decode_item(p, w, CAUSAL);
            if (s == 0 && use_aux_bias(p, VAR)) {
                // Column-bias operand, one row per thread, one item ahead: item 0's at the
                // start, item k+1's at the start of item k (buffer (k+1) & 1; every MMA that
                // read that buffer for item k-1 completed before this warp's epilogue of k-1).
                auto publish = [&](int kk) {
                    const int wn = item_index(kk);
                    if (wn >= p.num_items) return;
                    const Item tn = decode_item(p, wn, CAUSAL);
                    const float bv = p.slopes.log2e[fmod_(tn.bh, p.div_h)] * static_cast<float>(r) / p.c1;
                    write_bias_row(smem + C::kAux, r, kk & 1, bv);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bias_full[kk & 1]);
                };
                if (k == 0) publish(0);
                publish(k + 1);
            }
            if (s == 1 && !t.q1valid) continue;
            const int qt = 2 * t.qb + s;
            const int i = qt * BM + r;
            const float sl2 = p.slopes.log2e[fmod_(t.bh, p.div_h)];
            const int it0 = (s == 0 && t.q1valid && CAUSAL) ? 1 : 0;
            float M = -INFINITY, l = 0.f;
            for (int it = it0; it < t.n; ++it) {
                const int j = kv_tile(p, t, it);
                ok = mbar_wait(&s_full[s], s_cnt & 1, err, SITE_SM_S);
                ++s_cnt;
                ok = __all_sync(0xffffffffu, ok);  // keep the warp converged for tcgen05.ld
                if (!ok) break;
                tc_fence_after();
                uint32_t sraw[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
                    tmem_ld32(lane_addr + s * 128 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sraw[c * 32]));
                tmem_wait_ld();
                // x = s log2(e)/sqrt(d) - m log2(e) (i - j): the bias of key k0 + c is
                // nb + sl2 c with nb = -sl2 (i - k0) from the integer offset, so no large
                // absolute position enters the fp32 arithmetic.
                const float nb = -sl2 * static_cast<float>(i - j * BN);
                const float2 c1v = make_float2(p.c1, p.c1);
                // Non-causal tiles at or right of the diagonal hold keys past the query:
                // there the distance is |i - k| and the bias -|nb + sl2 c| (sl2 >= 0).
                const bool sym = !CAUSAL && j >= qt;
                float x[BN];
                // rel: x holds the exponent relative to the running max M (the row offset and
                // -M folded into one FMA); otherwise the absolute exponent
                bool rel = false;
                if (VAR) {
                    // Mitigation variants, element by element in base-2 units:
                    //   content  A = s / sqrt(d), soft-capped to z tanh(A / z) with
                    //            tanh(y) = 1 - 2 / (e^{2y} + 1);
                    //   distance D = |i - (k0 + c)|, or ln(D + 1); bias -m D (as
                    //            -m log2(D + 1) in base 2), clamped from below.
                    const bool cap = p.variant & kFwdSoftcap, logd = p.variant & kFwdLogDist,
                               clamp = p.variant & kFwdClamp;
                    const float mnat = p.slopes.nat[fmod_(t.bh, p.div_h)];
                    const float di = static_cast<float>(i - j * BN);  // exact: |i - k0| < 2^24
#pragma unroll
                    for (int c = 0; c < BN; ++c) {
                        const float sv = __uint_as_float(sraw[c]);
                        const float a = cap ? fmaf(-2.0f * p.cap_zl, rcp_approx(ex2_approx(sv * p.cap_k) + 1.0f), p.cap_zl)
                                            : sv * p.c1;
                        float b;
                        if (logd) {
                            b = -mnat * lg2_approx(fabsf(di - static_cast<float>(c)) + 1.0f);
                        } else {
                            b = fmaf(sl2, static_cast<float>(c), nb);
                            if (sym) b = -fabsf(b);
                        }
                        if (clamp) b = fmaxf(b, p.clamp2);
                        x[c] = a + b;
                    }
                } else if (CAUSAL || j != qt) {
                    // The column part of the bias is already in S (see use_aux_bias); the row
                    // part is nb for keys before the rows and -nb for keys after them.
                    rel = it != it0;
                    const float rb = ((CAUSAL || j < qt) ? nb : -nb) - (rel ? M : 0.f);
                    const float2 rbv = make_float2(rb, rb);
#pragma unroll
                    for (int u = 0; u < BN / 2; ++u) {
                        const float2 xv = __ffma2_rn(
                            make_float2(__uint_as_float(sraw[2 * u]), __uint_as_float(sraw[2 * u + 1])), c1v, rbv);
                        x[2 * u] = xv.x;
                        x[2 * u + 1] = xv.y;
                    }
                } else {
                    // non-causal diagonal tile (raw S): bias -|nb + sl2 c|
#pragma unroll
                    for (int u = 0; u < BN / 2; ++u) {
                        const float2 b = make_float2(-fabsf(fmaf(sl2, static_cast<float>(2 * u), nb)),
                                                     -fabsf(fmaf(sl2, static_cast<float>(2 * u + 1), nb)));
                        const float2 xv = __ffma2_rn(
                            make_float2(__uint_as_float(sraw[2 * u]), __uint_as_float(sraw[2 * u + 1])), c1v, b);
                        x[2 * u] = xv.x;
                        x[2 * u + 1] = xv.y;
                    }
                }
                if (CAUSAL) {
                    if (j == qt) {  // diagonal tile: keys after the query are masked
#pragma unroll
                        for (int c = 0; c < BN; ++c) x[c] = (c > r) ? -INFINITY : x[c];
                    }
                } else if (j == p.NQT - 1) {
                    // last tile: the keys past N (zero-filled by TMA) are masked; every
                    // tile keeps at least its first key, so the row max stays finite
                    const int kv = p.N - j * BN;
                    if (kv < BN) {
#pragma unroll
                        for (int c = 0; c < BN; ++c) x[c] = (c >= kv) ? -INFINITY : x[c];
                    }
                }
                const float mt = row_max128(x);
                // Raise the running max lazily: only when this tile exceeds it by 2^8. The
                // decision is per row, but tcgen05.ld/st are warp-collective (.sync.aligned),
                // so the warp rescales together when any of its rows needs it and rows that
                // do not use alpha = 1. O_s is quiescent here: S_s(it) completing implies
                // PV_s(it-1), issued before it, has completed.
                const bool need = rel ? mt > kRescaleThreshold : (it != it0) && (mt > M + kRescaleThreshold);
                if (it == it0) M = mt;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? ex2_approx(rel ? -mt : M - mt) : 1.0f;
                    if (need) {
                        M = rel ? M + mt : mt;
                        l *= alpha;
                    }
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(lane_addr + 256 + s * 128 + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
                        tmem_st32(lane_addr + 256 + s * 128 + c * 32, o);
                    }
                }
                // what the exponent still needs subtracted: the new max's rise (relative x), or M
                const float shift = rel ? (need ? mt : 0.f) : M;
                // p = 2^(x - shift), packed to bf16 pairs; four independent pair sums
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                // Two halves of 64 keys: the first half of P is handed to the MMA issuer
                // (p_full) while the second half is still being exponentiated (p_hi).
                uint32_t pk[BN / 2];
                auto exps = [&](auto sub_c) {
                    const float2 negs = make_float2(-shift, -shift);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
#pragma unroll
                        for (int u = half * (BN / 4); u < (half + 1) * (BN / 4); ++u) {
                            float2 dv = make_float2(x[2 * u], x[2 * u + 1]);
                            if (decltype(sub_c)::value) dv = __fadd2_rn(dv, negs);
                            const float2 pv = make_float2(ex2_approx(dv.x), ex2_approx(dv.y));
                            acc[u & 3] = __fadd2_rn(acc[u & 3], pv);
                            pk[u] = pack_bf16x2(pv.x, pv.y);
                        }
                        tmem_st32(lane_addr + s * 128 + half * 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[half * 32]));
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(half == 0 ? &p_full[s] : &p_hi[s]);
                    }
                };
                if (__any_sync(0xffffffffu, shift != 0.f))
                    exps(std::true_type{});
                else
                    exps(std::false_type{});
                const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
                const float2 a = __fadd2_rn(a01, a23);
                l += a.x + a.y;
            }
            if (!ok) break;
            // ------------------------------------------------------ epilogue
            ok = mbar_wait(&o_full[s], o_cnt & 1, err, SITE_SM_O);
            ++o_cnt;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float inv_l = 1.0f / l;
            const bool valid = i < p.N;
            // only the D = 64 kernel serves smaller head sizes; D = 128 keeps a compile-time row size
            const int dr = D == 64 ? p.dr : D;
            // O / l goes out through a per-warp staging box and bulk tensor stores, so the
            // warp does not wait for its global stores before its next tile (rows past N are
            // clipped by the tensor map)
            uint8_t *stg = smem + C::kStage + (warp - 4) * 2048;
            const int row0 = qt * BM + quad * 32;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                if (c * 32 >= dr || row0 >= p.N) break;
                uint32_t o[32];
                tmem_ld32(lane_addr + 256 + s * 128 + c * 32, o);
                tmem_wait_ld();
                uint32_t b[16];
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    b[u] = pack_bf16x2(__uint_as_float(o[2 * u]) * inv_l, __uint_as_float(o[2 * u + 1]) * inv_l);
                if (lane == 0) bulk_wait_read();  // the previous box has left the staging
                __syncwarp();
                uint4 *dst = reinterpret_cast<uint4 *>(stg + lane * 64);
#pragma unroll
                for (int u = 0; u < 4; ++u) dst[u] = make_uint4(b[4 * u], b[4 * u + 1], b[4 * u + 2], b[4 * u + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&p.tout, stg, c * 32, row0, t.bh);
                    bulk_commit();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[s]);
            if (valid && p.lse) p.lse[static_cast<size_t>(t.bh) * p.N + i] = (M + __log2f(l)) * 0.69314718055994531f;
        }
    }

    if (warp >= 4 && lane == 0) bulk_wait_all();  // the epilogue's stores are done
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// dr <= D is the tensors' head size: for dr < 64 the D = 64 kernel runs with a
// 64-column TMA box over dr-column rows, so the columns past dr arrive as zeros
// (they add nothing to S, and the matching columns of O come out zero and are
// not stored).
template <int D, bool VAR>
static cudaError_t launch_fwd_tc_d(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                                   int H, int N, int dr, int causal, const Slopes &slopes, const int2 *plan,
                                   unsigned int variant, float clamp_min, float softcap_z, uint64_t test_wait_ns,
                                   cudaStream_t stream)
{
    using C = Cfg<D>;
    FwdParams p;
    const uint64_t BH = static_cast<uint64_t>(B) * H;
    if (!encode_tmap_bf16_3d(&p.tq, q, dr, N, BH, 64, BM) || !encode_tmap_bf16_3d(&p.tk, k, dr, N, BH, 64, BN) ||
        !encode_tmap_bf16_3d(&p.tv, v, dr, N, BH, 64, BN) ||
        !encode_tmap_bf16_3d(&p.tout, out, dr, N, BH, 32, 32, false))
        return cudaErrorInvalidValue;
    p.dr = dr;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.lse = lse;
    p.err = device_status_word();
    if (!p.err) return cudaErrorInvalidDevice;
    p.wait_ns = test_wait_ns ? test_wait_ns : kWaitLimitNs;
    p.test_skip_q0 = test_wait_ns != 0;
    p.N = N;
    p.BH = static_cast<int>(BH);
    p.H = H;
    p.NQT = (N + BM - 1) / BM;
    p.NQB = (p.NQT + 1) / 2;
    p.num_items = p.NQB * p.BH;
    p.div_bh = make_fastdiv(static_cast<uint32_t>(p.BH));
    p.div_h = make_fastdiv(static_cast<uint32_t>(H));
    p.div_nqb = make_fastdiv(static_cast<uint32_t>(p.NQB));
    p.causal = causal;
    p.c1 = 1.4426950408889634f / sqrtf(static_cast<float>(dr));
    p.slopes = slopes;
    p.plan = plan;
    p.variant = variant & (kFwdClamp | kFwdLogDist | kFwdSoftcap);
    p.clamp2 = clamp_min * 1.4426950408889634f;
    p.cap_k = (variant & kFwdSoftcap) ? 2.0f * 1.4426950408889634f / (sqrtf(static_cast<float>(dr)) * softcap_z) : 0.f;
    p.cap_zl = softcap_z * 1.4426950408889634f;

    // The register split above only balances if the kernel launches with exactly
    // kLaunchRegs per thread; prepare_kernel refuses otherwise (an unbalanced
    // setmaxnreg.inc would wait for registers that never come).
    for (int c = 0; c < 2; ++c) {
        const auto kern = c ? fwd_tc_kernel<D, VAR, true> : fwd_tc_kernel<D, VAR, false>;
        const cudaError_t e = prepare_kernel(reinterpret_cast<const void *>(kern), C::kSmem, kLaunchRegs);
        if (e != cudaSuccess) return e;
    }
    const int grid = p.num_items < num_sms() ? p.num_items : num_sms();
    if (causal)
        fwd_tc_kernel<D, VAR, true><<<grid, kThreads, C::kSmem, stream>>>(p);
    else
        fwd_tc_kernel<D, VAR, false><<<grid, kThreads, C::kSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int N,
                          int d, int causal, unsigned int flags, float clamp_min, float softcap_z, const Slopes &slopes,
                          cudaStream_t stream, uint64_t test_wait_ns)
{
    if (d != 128 && d != 64 && d != 32 && d != 16) return cudaErrorInvalidValue;
    auto run = [&](const int2 *plan) {
        // the failure-path self-test runs the mitigation instantiation (with none enabled),
        // so the plain kernels carry no test hook
        const bool var = (flags & (kFwdClamp | kFwdLogDist | kFwdSoftcap)) != 0 || test_wait_ns != 0;
        if (d == 128)
            return var ? launch_fwd_tc_d<128, true>(q, k, v, out, lse, B, H, N, d, causal, slopes, plan, flags,
                                                    clamp_min, softcap_z, test_wait_ns, stream)
                       : launch_fwd_tc_d<128, false>(q, k, v, out, lse, B, H, N, d, causal, slopes, plan, flags,
                                                     clamp_min, softcap_z, test_wait_ns, stream);
        return var ? launch_fwd_tc_d<64, true>(q, k, v, out, lse, B, H, N, d, causal, slopes, plan, flags, clamp_min,
                                               softcap_z, test_wait_ns, stream)
                   : launch_fwd_tc_d<64, false>(q, k, v, out, lse, B, H, N, d, causal, slopes, plan, flags, clamp_min,
                                                softcap_z, test_wait_ns, stream);
    };
    const int NQT = (N + BM - 1) / BM, NQB = (NQT + 1) / 2;
    if (!(flags & kFwdSkipUnderflow)) {
        // dense: the nominal order, or for launches whose K and V exceed half the L2 the
        // cached blocked order (same items, same results)
        const bool blocked = !(flags & kFwdNominalOrder) && test_wait_ns == 0;
        return run(blocked ? work_order(OrderKind::Prefill, causal, B * H, N, d, stream) : nullptr);
    }
    // underflow skipping: the plan lives in a stream-ordered scratch buffer for this call
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, skip_plan_bytes(B * H, N), decode_pool(), stream);
    if (e != cudaSuccess) return e;
    int2 *plan = nullptr;
    e = launch_skip_plan(q, k, B, H, N, d, slopes, ws, &plan, nullptr, stream);
    if (e == cudaSuccess) e = run(plan);
    const cudaError_t f = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : f;
}

}  // namespace alibi

// ALiBi attention backward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Gradients of sum(dO * O) for O = softmax(x) V with
//   x_ij = q_i.k_j / sqrt(d) - m_h (i - j)   (causal; keys j > i masked)
//   x_ij = q_i.k_j / sqrt(d) - m_h |i - j|   (non-causal)
// the forward of "When Attention Goes Blind: Numerical Failure in ALiBi
// Positional Encodings" (arXiv 2608.03994) sec. 3.1 eq. 1-4 (its sec. 5.1 notes
// that only weights that did not underflow carry gradient: here, as in the
// forward, a weight whose base-2 exponent is below -126 is exactly zero). With
// the forward's LSE the weights are recomputed tile by tile, never stored:
//   P_ij  = exp(x_ij - LSE_i),   dP_ij = dO_i . v_j,   D_i = dO_i . O_i,
//   dS_ij = P_ij (dP_ij - D_i),
//   dV = P^T dO,   dK = dS^T Q / sqrt(d),   dQ = dS K / sqrt(d).
// The bias has no trainable parameter and enters only through P. With the
// mitigations of sec. 3.4 (the VAR instantiations) P is recomputed with the
// clamped / log-distance bias and the soft-capped logit, and the soft cap's
// derivative 1 - tanh^2(A / z) multiplies dS before it meets K or Q.
//
// Three launches, no atomics (the result is deterministic):
//   bwd_prep_kernel   D_i = dO_i . O_i (fp32 from the bf16 tensors)
//   bwd_dkdv_kernel   one work item per (b, h) and 128-key tile: K, V stay in
//                     shared memory, Q / dO tiles stream through 2-stage rings;
//                     S^T = K Q^T and dP^T = V dO^T in TMEM, in two 64-query
//                     halves pipelined against the two elementwise warpgroups,
//                     then dV += P^T dO and dK += dS^T Q with P^T, dS^T read
//                     from TMEM
//   bwd_dq_kernel     one work item per (b, h) and 128-query tile: Q, dO are
//                     copied into TMEM (tcgen05.cp), K / V stream; S = Q K^T,
//                     dP = dO V^T with A from TMEM (two 64-key halves,
//                     pipelined the same way), dQ += dS K
// Roles as in the forward kernel: warp 0 TMA producer, warp 1 TMEM allocator
// and MMA issuer (converged, one elected lane issues), warps 4-7 / 8-11 two
// elementwise warpgroups that split each tile's 128 columns in halves (TMEM
// lane = row of the tile) and write the gradients through per-warp staging
// boxes and bulk tensor stores.

#include <cuda.h>

#include <type_traits>

#include "ptx.cuh"

namespace alibi {
namespace {

constexpr int BT = 128;  // rows / columns of every tile
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kRegsLow = 88;
constexpr uint32_t kRegsHigh = 208;
static_assert(128 * kRegsLow + 256 * kRegsHigh == kThreads * kLaunchRegs, "register split must match launch");
constexpr float kLog2e = 1.4426950408889634f;

// TMEM columns (both main kernels): accumulators at 0 and 128 (dV, dK or dQ),
// S / S^T at 256 (P or dS bf16 written over its halves), dP / dP^T at 384.
constexpr uint32_t kColAcc0 = 0, kColAcc1 = 128, kColS = 256, kColP = 384;
// dQ kernel: the item's Q and dO, copied from shared memory into the columns the
// second accumulator takes in the dK/dV kernel, as the A operands of S and dP
// (bf16 pairs, K-step kk at + 8 kk): 128 x 64 products with A in TMEM read only B
// from shared memory and run at the tensor rate.
constexpr uint32_t kColQ = 128, kColDO = 192;

template <int D>
struct BwdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kChunkBytes = BT * 128;
    static constexpr uint32_t kTileBytes = BT * D * 2;
    // dKdV: K, V resident; Q, dO rings. dQ: Q, dO staged (then copied into TMEM); K, V
    // rings. Same layout:
    static constexpr uint32_t kRes0 = 0;                         // K (dKdV) / Q (dQ)
    static constexpr uint32_t kRes1 = kTileBytes;                // V (dKdV) / dO (dQ)
    static constexpr uint32_t kRing0 = 2 * kTileBytes;           // Q / K, 2 stages
    static constexpr uint32_t kRing1 = 4 * kTileBytes;           // dO / V, 2 stages
    // 2 KB per elementwise warp: dKdV's column statistics (2 x (64 + 64) floats) during
    // the tile loop, then (both kernels) the epilogue's staging box of 32 x 32 bf16
    static constexpr uint32_t kStats = 6 * kTileBytes;
    static constexpr uint32_t kAux = kStats + 8 * 2048;          // bias operands (ptx.cuh), one atom
    static constexpr uint32_t kBar = kAux + kChunkBytes;
    static constexpr uint32_t kSmem = kBar + 256 + 1024;
};

struct BwdParams {
    CUtensorMap tq, tk, tv, tdo;  // [BH, N, d] bf16, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tg0, tg1;         // the gradients g0, g1: box {16, 32, 1}, no swizzle (epilogue stores)
    const float *lse;             // [BH, N] natural log (forward output)
    const float *dsum;            // [BH, N] D_i
    __nv_bfloat16 *g0, *g1;       // dKdV: dk, dv; dQ: dq
    uint32_t *err;
    int N, BH, H, NT, num_items, causal;
    const int2 *order;  // optional work order: entry .x = b h * NT + tile; null = nominal order
    float c1;       // log2(e) / sqrt(d)
    float inv_sqrt_d;
    // mitigations (kFwdClamp / kFwdLogDist / kFwdSoftcap), constants in base-2 units as in the forward
    unsigned int variant;
    float clamp2, cap_k, cap_zl;
    Slopes slopes;
};

__device__ __forceinline__ float lg2_approx_b(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx_b(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One element with the mitigations, base-2 units: raw score sv, distance |i - j|
// (exact integer in fp32), the row / column's -LSE log2(e). Returns P and sets
// *fac to d(capped logit)/d(raw logit).
__device__ __forceinline__ float var_weight(const BwdParams &p, float mnat, float sl2, float sv, float dist,
                                            float nlse2, float *fac)
{
    const bool cap = p.variant & kFwdSoftcap, logd = p.variant & kFwdLogDist, clamp = p.variant & kFwdClamp;
    float a = sv * p.c1, f = 1.0f;
    if (cap) {
        // z tanh(A / z) with tanh(y) = 1 - 2 / (e^{2y} + 1); the derivative is 1 - tanh^2
        const float th = fmaf(-2.0f, rcp_approx_b(ex2_approx(sv * p.cap_k) + 1.0f), 1.0f);
        a = th * p.cap_zl;
        f = (1.0f - th) * (1.0f + th);
    }
    float b = logd ? -mnat * lg2_approx_b(dist + 1.0f) : -sl2 * dist;
    if (clamp) b = fmaxf(b, p.clamp2);
    *fac = f;
    return ex2_approx(a + b + nlse2);
}

// Causal plain kernels add the column part of the bias on the tensor core (the bias
// operands of ptx.cuh): one more K-step after S = Q K^T (dQ; B row = key column c:
// m log2(e) c / c1) or S^T = K Q^T (dK/dV; B row = query column c: -m log2(e) c / c1).
__device__ __forceinline__ bool bwd_aux(bool causal, bool var) { return causal && !var; }

enum : uint32_t {
    SITE_B_PROD_RES = 0x401, SITE_B_PROD_RING = 0x402, SITE_B_MMA_RES = 0x411, SITE_B_MMA_RING = 0x412,
    SITE_B_MMA_P = 0x413, SITE_B_MMA_ACC = 0x414, SITE_B_MMA_DONE = 0x415, SITE_B_EW_S = 0x421,
    SITE_B_EW_ACC = 0x422,
};

__device__ __forceinline__ int item_index(int k)
{
    const int G = gridDim.x, c = blockIdx.x;
    return (k & 1) ? (k + 1) * G - 1 - c : k * G + c;
}

struct BItem {
    int bh, tile, n;
};

// Item at position idx of an order table: (b h, tile).
__device__ __forceinline__ void table_item(const BwdParams &p, int idx, BItem *it)
{
    const int e = p.order[idx].x;
    it->bh = e / p.NT;
    it->tile = e - it->bh * p.NT;
}

// dKdV items: round r of the nominal schedule is KV tile r of every (b, h) (causal:
// the longest first, since tile jt meets NT - jt query tiles); an order table gives
// the blocked order of large causal launches instead.
__device__ __forceinline__ BItem dkdv_item(const BwdParams &p, int idx, bool causal)
{
    BItem it;
    if (p.order) {
        table_item(p, idx, &it);
    } else {
        const int round = idx / p.BH;
        it.bh = idx - round * p.BH;
        it.tile = round;
    }
    it.n = causal ? p.NT - it.tile : p.NT;
    return it;
}

// Query tile visited at iteration `it` of a dKdV item (causal: from the diagonal up).
__device__ __forceinline__ int dkdv_qtile(const BItem &t, int it, bool causal)
{
    return causal ? t.tile + it : it;
}

// dQ items: round r of the nominal schedule is query tile NT - 1 - r of every
// (b, h) (causal: longest first), or the order table's item.
__device__ __forceinline__ BItem dq_item(const BwdParams &p, int idx, bool causal)
{
    BItem it;
    if (p.order) {
        table_item(p, idx, &it);
    } else {
        const int round = idx / p.BH;
        it.bh = idx - round * p.BH;
        it.tile = p.NT - 1 - round;
    }
    it.n = causal ? it.tile + 1 : p.NT;
    return it;
}

// Descriptor helpers (128-byte swizzle, as the TMA writes it).
// K-major operand (the contraction runs along d): 32-byte steps inside a swizzle
// atom, one 16 KB atom per 64 columns of d.
template <int D>
__device__ __forceinline__ uint32_t kmajor_step(int kk)
{
    return ((kk >> 2) * BwdCfg<D>::kChunkBytes + (kk & 3) * 32) >> 4;
}
// MN-major operand (the contraction runs along the tile's rows): 16 rows = 2048 bytes per step.
__device__ __forceinline__ uint32_t mnmajor_step(int kk) { return (kk * 2048) >> 4; }

// A operand read from TMEM: bf16 pairs written by the two warpgroups over the
// first 32 columns of their own 64-column halves of the S / dP region.
__device__ __forceinline__ uint32_t tmem_a_col(uint32_t region, int kk)
{
    return region + 64 * (kk >> 2) + (kk & 3) * 8;
}

// Epilogue of one accumulator: this warpgroup's half of d for the warp's 32 rows
// (row0 ..), as 32 x 16 boxes through the two 1 KB halves of the warp's staging in
// turn and bulk tensor stores (rows past N are clipped by the tensor map), so the
// warp neither waits for its global stores nor for each box to leave before
// writing the next.
template <int D>
__device__ __forceinline__ void store_acc_half(uint32_t lane_addr, uint32_t col0, int s, uint8_t *stg,
                                               const CUtensorMap *tmap, int row0, int bh, float scale)
{
    constexpr int kHalf = D / 2;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + col0 + s * kHalf + c * 32, o);
        tmem_wait_ld();
        uint32_t b[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
            b[u] = pack_bf16x2(__uint_as_float(o[2 * u]) * scale, __uint_as_float(o[2 * u + 1]) * scale);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {  // two 32 x 16 boxes, the staging's two halves in turn
            uint8_t *buf = stg + hb * 1024;
            if (lane == 0) bulk_wait_read1();  // the box before the previous one has left
            __syncwarp();
            uint4 *dst = reinterpret_cast<uint4 *>(buf + lane * 32);
            dst[0] = make_uint4(b[8 * hb], b[8 * hb + 1], b[8 * hb + 2], b[8 * hb + 3]);
            dst[1] = make_uint4(b[8 * hb + 4], b[8 * hb + 5], b[8 * hb + 6], b[8 * hb + 7]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(tmap, buf, s * kHalf + c * 32 + hb * 16, row0, bh);
                bulk_commit();
            }
        }
    }
}

// ------------------------------------------------------------------ dK, dV

template <int D, bool VAR, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBar);
    uint64_t *kv_full = bars + 0;
    uint64_t *kv_empty = bars + 1;
    uint64_t *qo_full = bars + 2;   // [2]
    uint64_t *qo_empty = bars + 4;  // [2]
    uint64_t *s_full = bars + 6;   // [2] S^T and dP^T of query half h in TMEM
    uint64_t *p_full = bars + 11;  // [2] P^T and dS^T of query half h written back
    uint64_t *acc_full = bars + 8;
    uint64_t *acc_empty = bars + 9;
    uint64_t *mma_done = bars + 10;
    uint64_t *bias_full = bars + 13;  // [2] column-bias operand of item k written (buffer k & 1)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *err = p.err;

    if (threadIdx.x == 0) {
        cta_err_init(kWaitLimitNs);
        cta_check_init(p.err, smem_raw, C::kSmem);
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qo_full[s], 1);
            mbar_init(&qo_empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&s_full[h], 1);
            mbar_init(&p_full[h], 4);  // the four warps of the half's warpgroup
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);
        mbar_init(mma_done, 1);
        mbar_init(&bias_full[0], 4);  // the first elementwise warpgroup
        mbar_init(&bias_full[1], 4);
        fence_mbar_init();
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tk);
        tma_prefetch_desc(&p.tv);
        tma_prefetch_desc(&p.tdo);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (bwd_aux(CAUSAL, VAR) && threadIdx.x < 2 * BT) {
        write_ones_chunk(smem + C::kAux, threadIdx.x >> 1, threadIdx.x & 1);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // D from the row-sum pre-pass is complete and visible from here on; the dQ
    // kernel, which reads nothing this kernel writes, may then take each SM this
    // grid's CTAs leave
    griddep_wait();
    griddep_launch_dependents();

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------ TMA producer
            uint32_t qc = 0;
            int kres = -1;  // item whose resident K, V were issued last
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int w = item_index(k);
                if (w >= p.num_items) break;
                const BItem t = dkdv_item(p, w, CAUSAL);
                ok = mbar_wait(kv_empty, (k & 1) ^ 1, err, SITE_B_PROD_RES);
                if (!ok) break;
                kres = k;
                mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(smem + C::kRes0 + c * C::kChunkBytes, &p.tk, 64 * c, t.tile * BT, t.bh, kv_full);
                    tma_load_3d(smem + C::kRes1 + c * C::kChunkBytes, &p.tv, 64 * c, t.tile * BT, t.bh, kv_full);
                }
                for (int it = 0; it < t.n && ok; ++it, ++qc) {
                    const uint32_t st = qc & 1, ph = (qc >> 1) & 1;
                    ok = mbar_wait(&qo_empty[st], ph ^ 1, err, SITE_B_PROD_RING);
                    if (!ok) break;
                    const int qt = dkdv_qtile(t, it, CAUSAL);
                    mbar_arrive_expect_tx(&qo_full[st], 2 * C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_3d(smem + C::kRing0 + st * C::kTileBytes + c * C::kChunkBytes, &p.tq, 64 * c,
                                    qt * BT, t.bh, &qo_full[st]);
                        tma_load_3d(smem + C::kRing1 + st * C::kTileBytes + c * C::kChunkBytes, &p.tdo, 64 * c,
                                    qt * BT, t.bh, &qo_full[st]);
                    }
                }
            }
            // Drain (also after an error): the last resident load and the last load into
            // each ring stage have landed before the CTA can exit.
            if (kres >= 0) mbar_wait(kv_full, kres & 1, err, SITE_B_PROD_RES, true);
            for (uint32_t n = qc > 2 ? qc - 2 : 0; n < qc; ++n)
                mbar_wait(&qo_full[n & 1], (n >> 1) & 1, err, SITE_B_PROD_RING, true);
        } else if (warp == 1) {
            // whole warp, converged; one elected lane issues each tcgen05 instruction
            // -------------------------------------------------------- MMA issuer
            // Each query tile is computed in two halves of 64 queries (the columns of one
            // elementwise warpgroup each): warpgroup 0 starts on its half while the tensor
            // core computes the other, and each half's dV / dK products go out as soon as
            // its P^T and dS^T are back, followed by the next tile's S^T / dP^T for that half.
            constexpr uint32_t idH = idesc_bf16_f32(BT, BT / 2, 0);  // 128 keys x 64 queries
            constexpr uint32_t idG = idesc_bf16_f32(BT, D, 1);
            constexpr uint32_t kHalfOff = (BT / 2) * 128;              // bytes to query row 64 of a chunk
            const uint32_t sK = smem_u32(smem + C::kRes0), sV = smem_u32(smem + C::kRes1);
            const uint32_t sQ = smem_u32(smem + C::kRing0), sO = smem_u32(smem + C::kRing1);
            const uint64_t kd = smem_desc_sw128(sK, 16, 1024), vd = smem_desc_sw128(sV, 16, 1024);
            const bool aux = bwd_aux(CAUSAL, VAR);
            const uint64_t auxd = smem_desc_sw128(smem_u32(smem + C::kAux), 16, 1024);
            uint32_t qc = 0, pc[2] = {0, 0};
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int w = item_index(k);
                if (w >= p.num_items) break;
                const BItem t = dkdv_item(p, w, CAUSAL);
                ok = mbar_wait(kv_full, k & 1, err, SITE_B_MMA_RES);
                if (ok && aux) ok = mbar_wait(&bias_full[k & 1], (k >> 1) & 1, err, SITE_B_MMA_RES);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const uint32_t qb0 = qc;  // ring counter of this item's first query tile
                auto wait_tile = [&](int it) -> bool {
                    const uint32_t c = qb0 + it;
                    bool okw = mbar_wait(&qo_full[c & 1], (c >> 1) & 1, err, SITE_B_MMA_RING);
                    okw = __all_sync(0xffffffffu, okw);
                    if (okw) tc_fence_after();
                    return okw;
                };
                // S^T = K Q^T and dP^T = V dO^T for query half h of tile it (operands K-major along d)
                auto issue_SP = [&](int it, int h) {
                    const uint32_t st = (qb0 + it) & 1;
                    const uint64_t qd = smem_desc_sw128(sQ + st * C::kTileBytes + h * kHalfOff, 16, 1024);
                    const uint64_t od = smem_desc_sw128(sO + st * C::kTileBytes + h * kHalfOff, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss_w(tmem + kColS + 64 * h, kd + kmajor_step<D>(kk), qd + kmajor_step<D>(kk), idH, kk > 0);
                    // column (query) bias: ones x this item's bias rows 64 h ..
                    if (aux)
                        mma_ss_w(tmem + kColS + 64 * h, auxd, auxd + 2 * (1 + (k & 1)) + ((h * kHalfOff) >> 4), idH,
                                 1u);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss_w(tmem + kColP + 64 * h, vd + kmajor_step<D>(kk), od + kmajor_step<D>(kk), idH, kk > 0);
                    mma_commit_w(&s_full[h]);
                };
                // dV += P^T dO and dK += dS^T Q over the 64 queries of half h (B MN-major)
                auto issue_GG = [&](int it, int h) {
                    const uint32_t st = (qb0 + it) & 1;
                    const uint64_t omn = smem_desc_sw128(sO + st * C::kTileBytes, C::kChunkBytes, 1024);
                    const uint64_t qmn = smem_desc_sw128(sQ + st * C::kTileBytes, C::kChunkBytes, 1024);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int kk = 4 * h + k4;
                        mma_ts_w(tmem + kColAcc0, tmem + tmem_a_col(kColS, kk), omn + mnmajor_step(kk), idG,
                                 (it > 0 || kk > 0) ? 1u : 0u);
                    }
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int kk = 4 * h + k4;
                        mma_ts_w(tmem + kColAcc1, tmem + tmem_a_col(kColP, kk), qmn + mnmajor_step(kk), idG,
                                 (it > 0 || kk > 0) ? 1u : 0u);
                    }
                };
                ok = wait_tile(0);
                if (!ok) break;
                issue_SP(0, 0);
                issue_SP(0, 1);
                if (t.n == 1) mma_commit_w(kv_empty);  // K and V read for the last time
                for (int it = 0; it < t.n && ok; ++it) {
                    for (int h = 0; h < 2 && ok; ++h) {
                        // P^T and dS^T of this half written back by its warpgroup
                        ok = mbar_wait(&p_full[h], pc[h] & 1, err, SITE_B_MMA_P);
                        ++pc[h];
                        if (ok && it == 0 && h == 0) ok = mbar_wait(acc_empty, (k & 1) ^ 1, err, SITE_B_MMA_ACC);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        tc_fence_after();
                        issue_GG(it, h);
                        if (h == 1) mma_commit_w(&qo_empty[(qb0 + it) & 1]);  // tile it read for the last time
                        if (it + 1 < t.n) {
                            if (h == 0 && !(ok = wait_tile(it + 1))) break;
                            issue_SP(it + 1, h);  // over the columns whose P^T / dS^T were just consumed
                            if (h == 1 && it + 2 == t.n) mma_commit_w(kv_empty);  // K and V read for the last time
                        }
                    }
                }
                qc += t.n;
                if (!ok) break;
                mma_commit_w(acc_full);
            }
            mma_commit_w(mma_done);
            mbar_wait(mma_done, 0, err, SITE_B_MMA_DONE, true);
        }
    } else {
        // --------------------------------------------------- elementwise warps
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        const int s = (warp - 4) >> 2;  // query columns [64 s, 64 s + 64) of every tile
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // key row of the tile
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        // per-warp double buffer of the 64 columns' -LSE (base 2) and -D
        uint8_t *stg = smem + C::kStats + (warp - 4) * 2048;
        float *stats = reinterpret_cast<float *>(stg);
        uint32_t s_cnt = 0;
        bool ok = true;
        // this lane's share of the column statistics of item ti's iteration `it`
        auto fetch = [&](const BItem &ti, int it, float (&v)[4]) {
            const size_t rb = static_cast<size_t>(ti.bh) * p.N;
            const int q0 = dkdv_qtile(ti, it, CAUSAL) * BT + 64 * s;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = q0 + lane + 32 * h;
                const bool in = i < p.N;
                v[h] = in ? -p.lse[rb + i] * kLog2e : -INFINITY;  // -LSE log2(e); past N: weight 0
                v[2 + h] = in ? -p.dsum[rb + i] : 0.f;              // -D
            }
        };
        float pre[4];  // prefetched one iteration ahead, across items too
        for (int k = 0; ok; ++k) {
            const int w = item_index(k);
            if (w >= p.num_items) break;
            const BItem t = dkdv_item(p, w, CAUSAL);
            const float sl2 = p.slopes.log2e[t.bh % p.H];
            if (k == 0) fetch(t, 0, pre);
            if (s == 0 && bwd_aux(CAUSAL, VAR)) {
                // column-bias rows (query column c: -m log2(e) c / c1), one item ahead
                auto publish = [&](int kk) {
                    const int wn = item_index(kk);
                    if (wn >= p.num_items) return;
                    const BItem tn = dkdv_item(p, wn, CAUSAL);
                    write_bias_row(smem + C::kAux, r, kk & 1, -p.slopes.log2e[tn.bh % p.H] * static_cast<float>(r) / p.c1);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bias_full[kk & 1]);
                };
                if (k == 0) publish(0);
                publish(k + 1);
            }
            if (lane == 0) bulk_wait_read();  // the previous item's epilogue boxes have left the buffer
            __syncwarp();
            for (int it = 0; it < t.n; ++it) {
                const int qt = dkdv_qtile(t, it, CAUSAL);
                float *buf = stats + (it & 1) * 128;
                buf[lane] = pre[0];
                buf[lane + 32] = pre[1];
                buf[64 + lane] = pre[2];
                buf[64 + lane + 32] = pre[3];
                __syncwarp();
                if (it + 1 < t.n) fetch(t, it + 1, pre);
                ok = mbar_wait(&s_full[s], s_cnt & 1, err, SITE_B_EW_S);
                ++s_cnt;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t sraw[64], draw[64];
                tmem_ld32(lane_addr + kColS + 64 * s, *reinterpret_cast<uint32_t(*)[32]>(&sraw[0]));
                tmem_ld32(lane_addr + kColS + 64 * s + 32, *reinterpret_cast<uint32_t(*)[32]>(&sraw[32]));
                tmem_ld32(lane_addr + kColP + 64 * s, *reinterpret_cast<uint32_t(*)[32]>(&draw[0]));
                tmem_ld32(lane_addr + kColP + 64 * s + 32, *reinterpret_cast<uint32_t(*)[32]>(&draw[32]));
                tmem_wait_ld();
                // sl2 (i - j) for query i = qt*128 + 64 s + c and key j = jt*128 + r, from integers
                const float base = sl2 * static_cast<float>((qt - t.tile) * BT + 64 * s - r);
                const bool diag = CAUSAL && qt == t.tile;
                uint32_t pk[32], dk[32];
                if (VAR) {
                    const float mnat = p.slopes.nat[t.bh % p.H];
                    const float di = static_cast<float>((qt - t.tile) * BT + 64 * s - r);  // i - j at c = 0
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        float pv[2], dv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int c = 2 * u + e;
                            float f;
                            float w = var_weight(p, mnat, sl2, __uint_as_float(sraw[c]),
                                                 fabsf(di + static_cast<float>(c)), buf[c], &f);
                            if (diag && 64 * s + c < r) w = 0.f;  // query before key: masked
                            pv[e] = w;
                            dv[e] = w * (__uint_as_float(draw[c]) + buf[64 + c]) * f;
                        }
                        pk[u] = pack_bf16x2(pv[0], pv[1]);
                        dk[u] = pack_bf16x2(dv[0], dv[1]);
                    }
                } else {
                    // causal: the column bias is already in S^T (bwd_aux); what is left per
                    // element is c1 S' + (row part) - LSE_c, the exponential, and P (dP - D)
                    const float rowpart = -sl2 * static_cast<float>((qt - t.tile) * BT - r);
                    auto run_aux = [&](auto diag_c) {
                        const float2 c1v = make_float2(p.c1, p.c1), rp = make_float2(rowpart, rowpart);
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            const float2 nl = *reinterpret_cast<const float2 *>(buf + 2 * u);
                            const float2 nd = *reinterpret_cast<const float2 *>(buf + 64 + 2 * u);
                            float2 xv = __fadd2_rn(
                                __ffma2_rn(make_float2(__uint_as_float(sraw[2 * u]), __uint_as_float(sraw[2 * u + 1])),
                                           c1v, rp),
                                nl);
                            if (decltype(diag_c)::value) {  // query before key: masked
                                if (64 * s + 2 * u < r) xv.x = -INFINITY;
                                if (64 * s + 2 * u + 1 < r) xv.y = -INFINITY;
                            }
                            const float2 pv = make_float2(ex2_approx(xv.x), ex2_approx(xv.y));
                            const float2 dv = __fmul2_rn(
                                pv, __fadd2_rn(make_float2(__uint_as_float(draw[2 * u]), __uint_as_float(draw[2 * u + 1])),
                                               nd));
                            pk[u] = pack_bf16x2(pv.x, pv.y);
                            dk[u] = pack_bf16x2(dv.x, dv.y);
                        }
                    };
                    // one loop per (mask, bias form): the tile-uniform choices stay out of the element loop
                    auto run = [&](auto diag_c, auto sym_c) {
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            float pv[2], dv[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int c = 2 * u + e;
                                const float tt = fmaf(sl2, static_cast<float>(c), base);
                                const float b = decltype(sym_c)::value ? -fabsf(tt) : -tt;
                                float x = fmaf(__uint_as_float(sraw[c]), p.c1, b + buf[c]);
                                if (decltype(diag_c)::value && 64 * s + c < r) x = -INFINITY;  // query before key
                                pv[e] = ex2_approx(x);
                                dv[e] = pv[e] * (__uint_as_float(draw[c]) + buf[64 + c]);
                            }
                            pk[u] = pack_bf16x2(pv[0], pv[1]);
                            dk[u] = pack_bf16x2(dv[0], dv[1]);
                        }
                    };
                    if (!CAUSAL)
                        run(std::false_type{}, std::true_type{});
                    else if (diag)
                        run_aux(std::true_type{});
                    else
                        run_aux(std::false_type{});
                }
                tmem_st32(lane_addr + kColS + 64 * s, pk);
                tmem_st32(lane_addr + kColP + 64 * s, dk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[s]);
            }
            if (!ok) break;
            // ------------------------------------------------------ epilogue
            {  // the next item's first statistics load while this one's gradients go out
                const int wn = item_index(k + 1);
                if (wn < p.num_items) fetch(dkdv_item(p, wn, CAUSAL), 0, pre);
            }
            ok = mbar_wait(acc_full, k & 1, err, SITE_B_EW_ACC);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int row0 = t.tile * BT + quad * 32;
            if (row0 < p.N) {
                store_acc_half<D>(lane_addr, kColAcc0, s, stg, &p.tg1, row0, t.bh, 1.0f);          // dV
                store_acc_half<D>(lane_addr, kColAcc1, s, stg, &p.tg0, row0, t.bh, p.inv_sqrt_d);  // dK
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
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

// ---------------------------------------------------------------------- dQ

template <int D, bool VAR, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBar);
    uint64_t *qd_full = bars + 0;
    uint64_t *qd_empty = bars + 1;
    uint64_t *kv_full = bars + 2;   // [2]
    uint64_t *kv_empty = bars + 4;  // [2]
    uint64_t *s_full = bars + 6;   // [2] S and dP of key half h in TMEM
    uint64_t *p_full = bars + 11;  // [2] dS of key half h written back
    uint64_t *acc_full = bars + 8;
    uint64_t *acc_empty = bars + 9;
    uint64_t *mma_done = bars + 10;
    uint64_t *bias_full = bars + 13;  // [2] column-bias operand of item k written (buffer k & 1)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *err = p.err;

    if (threadIdx.x == 0) {
        cta_err_init(kWaitLimitNs);
        cta_check_init(p.err, smem_raw, C::kSmem);
        mbar_init(qd_full, 1);
        mbar_init(qd_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&s_full[h], 1);
            mbar_init(&p_full[h], 4);  // the four warps of the half's warpgroup
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);
        mbar_init(mma_done, 1);
        mbar_init(&bias_full[0], 4);  // the first elementwise warpgroup
        mbar_init(&bias_full[1], 4);
        fence_mbar_init();
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tk);
        tma_prefetch_desc(&p.tv);
        tma_prefetch_desc(&p.tdo);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (bwd_aux(CAUSAL, VAR) && threadIdx.x < 2 * BT) {
        write_ones_chunk(smem + C::kAux, threadIdx.x >> 1, threadIdx.x & 1);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
        if (warp == 0 && lane == 0) {
            uint32_t kc = 0;
            int kres = -1;  // item whose resident Q, dO were issued last
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int w = item_index(k);
                if (w >= p.num_items) break;
                const BItem t = dq_item(p, w, CAUSAL);
                ok = mbar_wait(qd_empty, (k & 1) ^ 1, err, SITE_B_PROD_RES);
                if (!ok) break;
                kres = k;
                mbar_arrive_expect_tx(qd_full, 2 * C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(smem + C::kRes0 + c * C::kChunkBytes, &p.tq, 64 * c, t.tile * BT, t.bh, qd_full);
                    tma_load_3d(smem + C::kRes1 + c * C::kChunkBytes, &p.tdo, 64 * c, t.tile * BT, t.bh, qd_full);
                }
                for (int it = 0; it < t.n && ok; ++it, ++kc) {
                    const uint32_t st = kc & 1, ph = (kc >> 1) & 1;
                    ok = mbar_wait(&kv_empty[st], ph ^ 1, err, SITE_B_PROD_RING);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&kv_full[st], 2 * C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_3d(smem + C::kRing0 + st * C::kTileBytes + c * C::kChunkBytes, &p.tk, 64 * c,
                                    it * BT, t.bh, &kv_full[st]);
                        tma_load_3d(smem + C::kRing1 + st * C::kTileBytes + c * C::kChunkBytes, &p.tv, 64 * c,
                                    it * BT, t.bh, &kv_full[st]);
                    }
                }
            }
            // Drain (also after an error), as in the dK/dV kernel.
            if (kres >= 0) mbar_wait(qd_full, kres & 1, err, SITE_B_PROD_RES, true);
            for (uint32_t n = kc > 2 ? kc - 2 : 0; n < kc; ++n)
                mbar_wait(&kv_full[n & 1], (n >> 1) & 1, err, SITE_B_PROD_RING, true);
        } else if (warp == 1) {
            // whole warp, converged; one elected lane issues each tcgen05 instruction
            // S and dP in two halves of 64 keys (the columns of one elementwise warpgroup
            // each); each half's dQ product goes out as soon as its dS is back, followed
            // by the next tile's S / dP for that half.
            constexpr uint32_t idH = idesc_bf16_f32(BT, BT / 2, 0);  // 128 queries x 64 keys
            constexpr uint32_t idG = idesc_bf16_f32(BT, D, 1);
            constexpr uint32_t kHalfOff = (BT / 2) * 128;              // bytes to key row 64 of a chunk
            const uint32_t sQ = smem_u32(smem + C::kRes0), sO = smem_u32(smem + C::kRes1);
            const uint32_t sK = smem_u32(smem + C::kRing0), sV = smem_u32(smem + C::kRing1);
            const uint64_t qd = smem_desc_sw128(sQ, 16, 1024), od = smem_desc_sw128(sO, 16, 1024);
            const bool aux = bwd_aux(CAUSAL, VAR);
            const uint64_t auxd = smem_desc_sw128(smem_u32(smem + C::kAux), 16, 1024);
            uint32_t kc = 0, pc[2] = {0, 0};
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int w = item_index(k);
                if (w >= p.num_items) break;
                const BItem t = dq_item(p, w, CAUSAL);
                ok = mbar_wait(qd_full, k & 1, err, SITE_B_MMA_RES);
                if (ok && aux) ok = mbar_wait(&bias_full[k & 1], (k >> 1) & 1, err, SITE_B_MMA_RES);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                // Q and dO into TMEM (after the previous item's MMAs in issue order); the
                // shared-memory copies are free once these complete
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    tmem_cp_w(tmem + kColQ + 8 * kk, qd + kmajor_step<D>(kk));
                    tmem_cp_w(tmem + kColDO + 8 * kk, od + kmajor_step<D>(kk));
                }
                mma_commit_w(qd_empty);
                const uint32_t kb0 = kc;  // ring counter of this item's first key tile
                auto wait_tile = [&](int it) -> bool {
                    const uint32_t c = kb0 + it;
                    bool okw = mbar_wait(&kv_full[c & 1], (c >> 1) & 1, err, SITE_B_MMA_RING);
                    okw = __all_sync(0xffffffffu, okw);
                    if (okw) tc_fence_after();
                    return okw;
                };
                // S = Q K^T and dP = dO V^T for key half h of tile it: A (Q, dO) from TMEM,
                // B (the half's 64 keys) K-major from the ring
                auto issue_SP = [&](int it, int h) {
                    const uint32_t st = (kb0 + it) & 1;
                    const uint64_t kd = smem_desc_sw128(sK + st * C::kTileBytes + h * kHalfOff, 16, 1024);
                    const uint64_t vd = smem_desc_sw128(sV + st * C::kTileBytes + h * kHalfOff, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ts_w(tmem + kColS + 64 * h, tmem + kColQ + 8 * kk, kd + kmajor_step<D>(kk), idH, kk > 0);
                    // column (key) bias: ones x this item's bias rows 64 h ..
                    if (aux)
                        mma_ss_w(tmem + kColS + 64 * h, auxd, auxd + 2 * (1 + (k & 1)) + ((h * kHalfOff) >> 4), idH,
                                 1u);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ts_w(tmem + kColP + 64 * h, tmem + kColDO + 8 * kk, vd + kmajor_step<D>(kk), idH, kk > 0);
                    mma_commit_w(&s_full[h]);
                };
                ok = wait_tile(0);
                if (!ok) break;
                issue_SP(0, 0);
                issue_SP(0, 1);
                for (int it = 0; it < t.n && ok; ++it) {
                    for (int h = 0; h < 2 && ok; ++h) {
                        ok = mbar_wait(&p_full[h], pc[h] & 1, err, SITE_B_MMA_P);
                        ++pc[h];
                        if (ok && it == 0 && h == 0) ok = mbar_wait(acc_empty, (k & 1) ^ 1, err, SITE_B_MMA_ACC);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        tc_fence_after();
                        // dQ += dS K over the 64 keys of half h (K MN-major: the contraction runs over keys)
                        const uint32_t st = (kb0 + it) & 1;
                        const uint64_t kmn = smem_desc_sw128(sK + st * C::kTileBytes, C::kChunkBytes, 1024);
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const int kk = 4 * h + k4;
                            mma_ts_w(tmem + kColAcc0, tmem + tmem_a_col(kColS, kk), kmn + mnmajor_step(kk), idG,
                                     (it > 0 || kk > 0) ? 1u : 0u);
                        }
                        if (h == 1) mma_commit_w(&kv_empty[st]);  // tile it read for the last time
                        if (it + 1 < t.n) {
                            if (h == 0 && !(ok = wait_tile(it + 1))) break;
                            issue_SP(it + 1, h);
                        }
                    }
                }
                kc += t.n;
                if (!ok) break;
                mma_commit_w(acc_full);
            }
            mma_commit_w(mma_done);
            mbar_wait(mma_done, 0, err, SITE_B_MMA_DONE, true);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        const int s = (warp - 4) >> 2;  // key columns [64 s, 64 s + 64) of every tile
        const int quad = warp & 3;
        uint8_t *stg = smem + C::kStats + (warp - 4) * 2048;  // epilogue staging box
        // this thread's row statistics (LSE log2(e), D) of item ti
        auto load_stats = [&](const BItem &ti, float (&v)[2]) {
            const int ii = ti.tile * BT + quad * 32 + lane;
            const bool in = ii < p.N;
            const size_t rb = static_cast<size_t>(ti.bh) * p.N;
            v[0] = in ? p.lse[rb + ii] * kLog2e : 0.f;
            v[1] = in ? p.dsum[rb + ii] : 0.f;
        };
        float nxt[2];  // loaded one item ahead
        const int r = quad * 32 + lane;  // query row of the tile
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        uint32_t s_cnt = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int w = item_index(k);
            if (w >= p.num_items) break;
            const BItem t = dq_item(p, w, CAUSAL);
            const float sl2 = p.slopes.log2e[t.bh % p.H];
            if (s == 0 && bwd_aux(CAUSAL, VAR)) {
                // column-bias rows (key column c: m log2(e) c / c1), one item ahead
                auto publish = [&](int kk) {
                    const int wn = item_index(kk);
                    if (wn >= p.num_items) return;
                    const BItem tn = dq_item(p, wn, CAUSAL);
                    write_bias_row(smem + C::kAux, r, kk & 1, p.slopes.log2e[tn.bh % p.H] * static_cast<float>(r) / p.c1);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bias_full[kk & 1]);
                };
                if (k == 0) publish(0);
                publish(k + 1);
            }
            const int i = t.tile * BT + r;
            if (k == 0) load_stats(t, nxt);
            const float lse2 = nxt[0], Di = nxt[1];
            for (int it = 0; it < t.n; ++it) {
                ok = mbar_wait(&s_full[s], s_cnt & 1, err, SITE_B_EW_S);
                ++s_cnt;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t sraw[64], draw[64];
                tmem_ld32(lane_addr + kColS + 64 * s, *reinterpret_cast<uint32_t(*)[32]>(&sraw[0]));
                tmem_ld32(lane_addr + kColS + 64 * s + 32, *reinterpret_cast<uint32_t(*)[32]>(&sraw[32]));
                tmem_ld32(lane_addr + kColP + 64 * s, *reinterpret_cast<uint32_t(*)[32]>(&draw[0]));
                tmem_ld32(lane_addr + kColP + 64 * s + 32, *reinterpret_cast<uint32_t(*)[32]>(&draw[32]));
                tmem_wait_ld();
                // -sl2 (i - k) for key k = it*128 + 64 s + c, from the integer offset
                const float nb = -sl2 * static_cast<float>(i - it * BT - 64 * s);
                const bool diag = CAUSAL && it == t.tile;
                const float nl = -lse2;
                uint32_t dk[32];
                if (VAR) {
                    const float mnat = p.slopes.nat[t.bh % p.H];
                    const float di = static_cast<float>(i - it * BT - 64 * s);  // i - k at c = 0
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        float dv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int c = 2 * u + e;
                            float f;
                            float w = var_weight(p, mnat, sl2, __uint_as_float(sraw[c]),
                                                 fabsf(di - static_cast<float>(c)), nl, &f);
                            if (diag && 64 * s + c > r) w = 0.f;  // key after the query: masked
                            dv[e] = w * (__uint_as_float(draw[c]) - Di) * f;
                        }
                        dk[u] = pack_bf16x2(dv[0], dv[1]);
                    }
                } else {
                    // causal: the column bias is already in S (bwd_aux): exponent c1 S' + (nb - LSE)
                    const float rowoff = -sl2 * static_cast<float>(i - it * BT) + nl;
                    auto run_aux = [&](auto diag_c) {
                        const float2 c1v = make_float2(p.c1, p.c1), ro = make_float2(rowoff, rowoff);
                        const float2 nD = make_float2(-Di, -Di);
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            float2 xv = __ffma2_rn(
                                make_float2(__uint_as_float(sraw[2 * u]), __uint_as_float(sraw[2 * u + 1])), c1v, ro);
                            if (decltype(diag_c)::value) {  // key after the query: masked
                                if (64 * s + 2 * u > r) xv.x = -INFINITY;
                                if (64 * s + 2 * u + 1 > r) xv.y = -INFINITY;
                            }
                            const float2 pv = make_float2(ex2_approx(xv.x), ex2_approx(xv.y));
                            const float2 dv = __fmul2_rn(
                                pv, __fadd2_rn(make_float2(__uint_as_float(draw[2 * u]), __uint_as_float(draw[2 * u + 1])),
                                               nD));
                            dk[u] = pack_bf16x2(dv.x, dv.y);
                        }
                    };
                    // one loop per (mask, bias form): the tile-uniform choices stay out of the element loop
                    auto run = [&](auto diag_c, auto sym_c) {
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            float dv[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int c = 2 * u + e;
                                const float tt = fmaf(sl2, static_cast<float>(c), nb);
                                const float b = decltype(sym_c)::value ? -fabsf(tt) : tt;
                                float x = fmaf(__uint_as_float(sraw[c]), p.c1, b + nl);
                                if (decltype(diag_c)::value && 64 * s + c > r) x = -INFINITY;  // key after the query
                                const float pv = ex2_approx(x);
                                dv[e] = pv * (__uint_as_float(draw[c]) - Di);
                            }
                            dk[u] = pack_bf16x2(dv[0], dv[1]);
                        }
                    };
                    if (!CAUSAL)
                        run(std::false_type{}, std::true_type{});
                    else if (diag)
                        run_aux(std::true_type{});
                    else
                        run_aux(std::false_type{});
                }
                tmem_st32(lane_addr + kColS + 64 * s, dk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[s]);
            }
            if (!ok) break;
            {  // the next item's row statistics load while this one's dQ goes out
                const int wn = item_index(k + 1);
                if (wn < p.num_items) load_stats(dq_item(p, wn, CAUSAL), nxt);
            }
            ok = mbar_wait(acc_full, k & 1, err, SITE_B_EW_ACC);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int row0 = t.tile * BT + quad * 32;
            if (row0 < p.N) store_acc_half<D>(lane_addr, kColAcc0, s, stg, &p.tg0, row0, t.bh, p.inv_sqrt_d);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
        }
    }

    if (warp >= 4 && lane == 0) bulk_wait_all();  // the epilogue's stores are done
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // this grid may have started while the dK/dV kernel ran; it completes only after
    // that kernel has, so stream order after the backward holds for both
    griddep_wait();
}

// ---------------------------------------------------------------- D = dO . O

// One half-warp per row (8 bf16 per lane), D / 8 lanes per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ out,
                                                       const __nv_bfloat16 *__restrict__ dout,
                                                       float *__restrict__ dsum, long long rows)
{
    constexpr int LPR = D / 8, RPW = 32 / LPR;
    griddep_launch_dependents();  // the dK/dV kernel waits for this grid before it reads D
    const int lane = threadIdx.x & 31;
    const long long row = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * RPW + lane / LPR;
    const int l = lane % LPR;
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = *reinterpret_cast<const uint4 *>(out + row * D + 8 * l);
        const uint4 b = *reinterpret_cast<const uint4 *>(dout + row * D + 8 * l);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            acc = fmaf(__uint_as_float(wa[t] << 16), __uint_as_float(wb[t] << 16), acc);
            acc = fmaf(__uint_as_float(wa[t] & 0xFFFF0000u), __uint_as_float(wb[t] & 0xFFFF0000u), acc);
        }
    }
#pragma unroll
    for (int o = LPR / 2; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (row < rows && l == 0) dsum[row] = acc;
}

// Launch with programmatic stream serialization: the grid may start on SMs the
// previous grid in the stream has left, before that grid has finished (the
// kernels order their own dependences with griddep_wait).
static cudaError_t launch_dependent(void (*kernel)(BwdParams), int grid, int smem, cudaStream_t stream,
                                    const BwdParams &p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int D, bool VAR>
cudaError_t launch_bwd_d(const void *q, const void *k, const void *v, const void *out, const float *lse,
                         const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int causal,
                         unsigned int flags, float clamp_min, float softcap_z, const Slopes &slopes, float *dsum,
                         cudaStream_t stream)
{
    using C = BwdCfg<D>;
    // The register split only balances if the kernels launch with exactly kLaunchRegs per
    // thread; prepare_kernel refuses otherwise (an unbalanced setmaxnreg.inc never returns).
    {
        const void *kerns[4] = {reinterpret_cast<const void *>(bwd_dkdv_kernel<D, VAR, true>),
                                reinterpret_cast<const void *>(bwd_dq_kernel<D, VAR, true>),
                                reinterpret_cast<const void *>(bwd_dkdv_kernel<D, VAR, false>),
                                reinterpret_cast<const void *>(bwd_dq_kernel<D, VAR, false>)};
        for (const void *kern : kerns) {
            const cudaError_t e = prepare_kernel(kern, C::kSmem, kLaunchRegs);
            if (e != cudaSuccess) return e;
        }
    }
    const long long rows = static_cast<long long>(B) * H * N;
    constexpr int kRowsPerCta = 8 * (32 / (D / 8));
    bwd_prep_kernel<D><<<static_cast<unsigned>((rows + kRowsPerCta - 1) / kRowsPerCta), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(out), static_cast<const __nv_bfloat16 *>(dout), dsum, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    BwdParams p;
    const uint64_t BH = static_cast<uint64_t>(B) * H;
    if (!encode_tmap_bf16_3d(&p.tq, q, D, N, BH, 64, BT) || !encode_tmap_bf16_3d(&p.tk, k, D, N, BH, 64, BT) ||
        !encode_tmap_bf16_3d(&p.tv, v, D, N, BH, 64, BT) || !encode_tmap_bf16_3d(&p.tdo, dout, D, N, BH, 64, BT))
        return cudaErrorInvalidValue;
    p.lse = lse;
    p.dsum = dsum;
    p.err = device_status_word();
    if (!p.err) return cudaErrorInvalidDevice;
    p.N = N;
    p.BH = static_cast<int>(BH);
    p.H = H;
    p.NT = (N + BT - 1) / BT;
    p.num_items = p.NT * p.BH;
    p.causal = causal;
    p.c1 = kLog2e / sqrtf(static_cast<float>(D));
    p.inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(D));
    p.slopes = slopes;
    p.variant = flags & (kFwdClamp | kFwdLogDist | kFwdSoftcap);
    p.clamp2 = clamp_min * kLog2e;
    p.cap_k = (flags & kFwdSoftcap) ? 2.0f * kLog2e / (sqrtf(static_cast<float>(D)) * softcap_z) : 0.f;
    p.cap_zl = softcap_z * kLog2e;
    const int grid = p.num_items < num_sms() ? p.num_items : num_sms();

    p.g0 = static_cast<__nv_bfloat16 *>(dk);
    p.g1 = static_cast<__nv_bfloat16 *>(dv);
    if (!encode_tmap_bf16_3d(&p.tg0, dk, D, N, BH, 16, 32, false) ||
        !encode_tmap_bf16_3d(&p.tg1, dv, D, N, BH, 16, 32, false))
        return cudaErrorInvalidValue;
    // large launches take the blocked work order (same items, same results)
    const bool blocked = !(flags & kFwdNominalOrder);
    p.order = blocked ? work_order(OrderKind::BwdDkDv, causal, p.BH, N, D, stream) : nullptr;
    e = launch_dependent(causal ? bwd_dkdv_kernel<D, VAR, true> : bwd_dkdv_kernel<D, VAR, false>, grid, C::kSmem,
                         stream, p);
    if (e != cudaSuccess) return e;
    p.g0 = static_cast<__nv_bfloat16 *>(dq);
    p.g1 = nullptr;
    if (!encode_tmap_bf16_3d(&p.tg0, dq, D, N, BH, 16, 32, false)) return cudaErrorInvalidValue;
    p.order = blocked ? work_order(OrderKind::BwdDq, causal, p.BH, N, D, stream) : nullptr;
    return launch_dependent(causal ? bwd_dq_kernel<D, VAR, true> : bwd_dq_kernel<D, VAR, false>, grid, C::kSmem,
                            stream, p);
}

}  // namespace

size_t bwd_workspace_bytes(int BH, int N) { return static_cast<size_t>(BH) * N * sizeof(float) + 256; }

cudaError_t launch_bwd_tc(const void *q, const void *k, const void *v, const void *out, const float *lse,
                          const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d, int causal,
                          unsigned int flags, float clamp_min, float softcap_z, const Slopes &slopes,
                          cudaStream_t stream)
{
    if (d != 128 && d != 64) return cudaErrorInvalidValue;
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, bwd_workspace_bytes(B * H, N), decode_pool(), stream);
    if (e != cudaSuccess) return e;
    float *dsum = static_cast<float *>(ws);
    const bool var = (flags & (kFwdClamp | kFwdLogDist | kFwdSoftcap)) != 0;
#define ALIBI_BWD_ARGS q, k, v, out, lse, dout, dq, dk, dv, B, H, N, causal, flags, clamp_min, softcap_z, slopes, dsum, stream
    if (d == 128)
        e = var ? launch_bwd_d<128, true>(ALIBI_BWD_ARGS) : launch_bwd_d<128, false>(ALIBI_BWD_ARGS);
    else
        e = var ? launch_bwd_d<64, true>(ALIBI_BWD_ARGS) : launch_bwd_d<64, false>(ALIBI_BWD_ARGS);
#undef ALIBI_BWD_ARGS
    const cudaError_t f = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : f;
}

}  // namespace alibi

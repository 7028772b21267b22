// Plan for skipping KV tiles whose attention weights provably underflow.
//
// "When Attention Goes Blind: Numerical Failure in ALiBi Positional Encodings"
// (arXiv 2608.03994), sec. 3.2-3.3 and sec. 5.1-5.2: once the bias -m_h (i - j)
// drives an exponent below the smallest normal number, the weight is exactly
// zero, yet a dense kernel still spends the work on those entries (the paper's
// point about steep heads acting as a sliding window). The prefill kernel
// evaluates p = 2^(x - M) with a flush-to-zero
// exponential, so an entry contributes exactly nothing when x - M < -126 (base-2
// units). This plan finds, for every work item (one (b, h) and a block of 256
// query rows), the KV tiles at the far end of the causal range where that holds
// for every row, so the kernel can leave them out with a bit-identical result.
//
// Bound, per query row i (base-2 units, c1 = log2(e)/sqrt(d), sl2 = m_h log2(e)):
//   every score satisfies  c1 q_i.k_j <= c1 |q_i| max_j |k_j|      (Cauchy-Schwarz)
//   the kernel's running max satisfies  M_i >= c1 q_i.k_i           (the diagonal
//     tile is processed first and the running max only grows)
// so a key at distance D >= (c1 (|q_i| Kmax - q_i.k_i) + 127) / sl2 has
// x - M <= -127 and its weight flushes to zero. The margin of one unit past 126
// and a relative slack on the norms cover fp32 rounding in the kernel. A KV tile
// is skipped only if this holds for every row of the item; since the bias grows
// with distance, the skipped tiles are a prefix [0, first) of the causal range.

#include "ptx.cuh"

namespace alibi {
namespace {

constexpr int kPlanRows = 256;  // query rows per work item (two 128-row tiles)

// Sum of squares / dot products of bf16 rows, LPK lanes per row (8 bf16 per lane).
template <int LPK>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = LPK / 2; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void bf16x8(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        f[2 * t] = __uint_as_float(w[t] << 16);
        f[2 * t + 1] = __uint_as_float(w[t] & 0xFFFF0000u);
    }
}

// Max squared key norm per (b, h), and per row i of the same pass |q_i|^2 and
// q_i.k_i (query and key rows share the index): a one-dimensional grid of nblk
// 256-row blocks per (b, h) (so B*H may exceed the 65535 limit of a second grid
// dimension), 256 threads, LPK lanes per row, four rows of each lane group in
// flight. rows[bh N + i] = (|q_i|^2, q_i.k_i), each sum in the same order as the
// per-row sums the plan needs, so the plan reads 8 bytes per row instead of Q and K.
template <int D>
__global__ void __launch_bounds__(256) kmax_kernel(const __nv_bfloat16 *__restrict__ q,
                                                   const __nv_bfloat16 *__restrict__ k, int N, int nblk,
                                                   unsigned int *__restrict__ kmax2_bits, float2 *__restrict__ rows)
{
    constexpr int LPK = D / 8, KPW = 32 / LPK;  // lanes per row, rows per warp pass
    constexpr int kStep = 8 * KPW;              // rows per CTA pass (8 warps)
    constexpr int kUnroll = 4;
    const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(nblk));
    const int blk = static_cast<int>(blockIdx.x - static_cast<unsigned>(bh) * nblk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LPK, l = lane % LPK;
    const size_t base = static_cast<size_t>(bh) * N * D;
    const int end = min(N, (blk + 1) * kPlanRows);
    float best = 0.f;
    // the loop index is the same for every lane of the warp (the shuffles below need
    // the whole warp); the lane's row is j0 + sub
    for (int j0 = blk * kPlanRows + warp * KPW; j0 < end; j0 += kUnroll * kStep) {
        uint4 uk[kUnroll], uq[kUnroll];
#pragma unroll
        for (int t = 0; t < kUnroll; ++t) {
            const int j = j0 + sub + t * kStep;
            if (j < end) {
                uk[t] = *reinterpret_cast<const uint4 *>(k + base + static_cast<size_t>(j) * D + 8 * l);
                uq[t] = *reinterpret_cast<const uint4 *>(q + base + static_cast<size_t>(j) * D + 8 * l);
            }
        }
#pragma unroll
        for (int t = 0; t < kUnroll; ++t) {
            const int j = j0 + sub + t * kStep;
            float kk = 0.f, qq = 0.f, qk = 0.f;
            if (j < end) {
                float fk[8], fq[8];
                bf16x8(uk[t], fk);
                bf16x8(uq[t], fq);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    kk = fmaf(fk[e], fk[e], kk);
                    qq = fmaf(fq[e], fq[e], qq);
                    qk = fmaf(fq[e], fk[e], qk);
                }
            }
            kk = group_sum<LPK>(kk);
            qq = group_sum<LPK>(qq);
            qk = group_sum<LPK>(qk);
            if (j < end) {
                best = fmaxf(best, kk);
                if (l == 0) rows[static_cast<size_t>(bh) * N + j] = make_float2(qq, qk);
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
    __shared__ float red[8];
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = red[0];
        for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
        atomicMax(kmax2_bits + bh, __float_as_uint(m));  // non-negative floats order as their bits
    }
}

// First KV tile worth computing per work item: one CTA per item, one thread per
// query row (256). info[w] = (first tile, tiles the item then spans).
__global__ void __launch_bounds__(kPlanRows) item_plan_kernel(const float2 *__restrict__ rows,
                                                              const unsigned int *__restrict__ kmax2_bits, int N,
                                                              int H, int NQB, int NQT, float c1, Slopes slopes,
                                                              int2 *__restrict__ info)
{
    const int w = blockIdx.x;
    const int bh = w / NQB, qb = w - bh * NQB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // fp32 is ample here: the bound keeps a whole unit of exponent margin, and fp32
    // rounding moves the cut by ~1e-3 tokens (~1e-3 m log2(e) exponent units).
    const float kmax = sqrtf(__uint_as_float(kmax2_bits[bh]));
    const float sl2 = slopes.log2e[bh % H];
    float cut = 3.0e38f;  // min over the item's rows of i - D_i
    const int i = qb * kPlanRows + static_cast<int>(threadIdx.x);
    if (i < N) {
        const float2 r = rows[static_cast<size_t>(bh) * N + i];
        const float qq = r.x, qk = r.y;
        // 2^-10 relative slack on the norm product and on |q.k| absorbs the rounding of
        // these sums and of the kernel's scores (both far below 2^-10 relative).
        const float slack = 1.0f + 0x1p-10f;
        const float a = c1 * (sqrtf(qq) * kmax * slack * slack - qk + fabsf(qk) * 0x1p-10f) + 127.0f;
        cut = static_cast<float>(i) - a / sl2;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) cut = fminf(cut, __shfl_xor_sync(0xffffffffu, cut, o));
    __shared__ float red[kPlanRows / 32];
    if (lane == 0) red[warp] = cut;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = red[0];
        for (int ww = 1; ww < kPlanRows / 32; ++ww) m = fminf(m, red[ww]);
        // tile jt (keys 128 jt .. 128 jt + 127) is skippable when 128 jt + 127 < m
        const int qt0 = 2 * qb, qt1 = 2 * qb + 1;
        const int n_nom = qt1 < NQT ? qt1 + 1 : qt1;
        const float y = (m - 127.0f) / 128.0f;
        int first = y > 0.0f ? static_cast<int>(ceilf(y)) : 0;
        if (first > qt0) first = qt0;  // the diagonal tiles are always computed
        info[w] = make_int2(first, n_nom - first);
    }
}

// Work order: items sorted by the tiles they span, longest first (counting sort in
// one CTA; ties in any order). plan[idx] = (item, first tile).
__global__ void __launch_bounds__(1024) plan_sort_kernel(const int2 *__restrict__ info, int items, int max_len,
                                                         int2 *__restrict__ plan)
{
    extern __shared__ int hist[];  // max_len + 1 bins
    for (int b = threadIdx.x; b <= max_len; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    for (int w = threadIdx.x; w < items; w += blockDim.x) atomicAdd(&hist[info[w].y], 1);
    __syncthreads();
    if (threadIdx.x == 0) {  // exclusive offsets, longest first (at most 12288 bins)
        int acc = 0;
        for (int b = max_len; b >= 0; --b) {
            const int c = hist[b];
            hist[b] = acc;
            acc += c;
        }
    }
    __syncthreads();
    for (int w = threadIdx.x; w < items; w += blockDim.x) {
        const int2 e = info[w];
        const int pos = atomicAdd(&hist[e.y], 1);
        plan[pos] = make_int2(w, e.x);
    }
}

// Nominal order (no sort) when the bin count does not fit: plan[idx] = (idx, first).
__global__ void plan_identity_kernel(const int2 *__restrict__ info, int items, int2 *__restrict__ plan)
{
    const int w = blockIdx.x * blockDim.x + threadIdx.x;
    if (w < items) plan[w] = make_int2(w, info[w].x);
}

}  // namespace

// Scratch of the plan: [plan | info | kmax2 | per-row sums], the last at a 256-byte
// offset.
static size_t rows_offset(int BH, int NQB)
{
    const size_t items = static_cast<size_t>(BH) * NQB;
    const size_t head = items * 2 * sizeof(int2) + static_cast<size_t>(BH) * sizeof(unsigned int);
    return (head + 255) & ~static_cast<size_t>(255);
}

size_t skip_plan_bytes(int BH, int N)
{
    const int NQB = ((N + 127) / 128 + 1) / 2;
    return 256 + rows_offset(BH, NQB) + static_cast<size_t>(BH) * N * sizeof(float2);
}

// Lays out [plan | info | kmax2 | rows] in `scratch` (skip_plan_bytes long) and fills it.
cudaError_t launch_skip_plan(const void *q, const void *k, int B, int H, int N, int d, const Slopes &slopes,
                             void *scratch, int2 **plan_out, int2 **info_out, cudaStream_t stream)
{
    const int BH = B * H, NQT = (N + 127) / 128, NQB = (NQT + 1) / 2, items = BH * NQB;
    int2 *plan = static_cast<int2 *>(scratch);
    int2 *info = plan + items;
    unsigned int *kmax2 = reinterpret_cast<unsigned int *>(info + items);
    cudaError_t e = cudaMemsetAsync(kmax2, 0, sizeof(unsigned int) * BH, stream);
    if (e != cudaSuccess) return e;
    const float c1 = 1.4426950408889634f / sqrtf(static_cast<float>(d));
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    const int nblk = (N + 255) / 256;
    const unsigned g1 = static_cast<unsigned>(nblk) * static_cast<unsigned>(BH);  // <= 2^31 - 1 (check_dims)
    float2 *rows = reinterpret_cast<float2 *>(static_cast<uint8_t *>(scratch) + rows_offset(BH, NQB));
    if (d == 128)
        kmax_kernel<128><<<g1, 256, 0, stream>>>(qb, kb, N, nblk, kmax2, rows);
    else if (d == 64)
        kmax_kernel<64><<<g1, 256, 0, stream>>>(qb, kb, N, nblk, kmax2, rows);
    else if (d == 32)
        kmax_kernel<32><<<g1, 256, 0, stream>>>(qb, kb, N, nblk, kmax2, rows);
    else if (d == 16)
        kmax_kernel<16><<<g1, 256, 0, stream>>>(qb, kb, N, nblk, kmax2, rows);
    else
        return cudaErrorInvalidValue;
    item_plan_kernel<<<items, kPlanRows, 0, stream>>>(rows, kmax2, N, H, NQB, NQT, c1, slopes, info);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int max_len = NQT;  // no item spans more tiles than there are tiles
    // one int per bin within the 48 KB of dynamic shared memory a launch gets without
    // raising the kernel's attribute; beyond that the nominal order is kept
    if ((max_len + 1) * sizeof(int) <= 48 * 1024) {
        plan_sort_kernel<<<1, 1024, (max_len + 1) * sizeof(int), stream>>>(info, items, max_len, plan);
    } else {
        plan_identity_kernel<<<(items + 255) / 256, 256, 0, stream>>>(info, items, plan);
    }
    if (plan_out) *plan_out = plan;
    if (info_out) *info_out = info;
    return cudaGetLastError();
}

}  // namespace alibi

// CUDA-core kernels of the library:
//   - fp32 prefill at reference precision (IEEE expf/logf), one warp per
//     query row, keys processed 32 at a time with an online softmax; causal,
//     or over all keys with the symmetric distance |i - j| ("ALiBi and
//     Relative Position Bias", "The mechanics");
//   - export of the fp32 attention weights from the saved LSE;
//   - the bf16 underflow counter: per head, the number of causal pairs whose
//     max-subtracted exponent is <= tau, in two passes per row (row max, then
//     count).
// Scores follow "When Attention Goes Blind: Numerical Failure in ALiBi
// Positional Encodings" (arXiv 2608.03994) sec. 3.1 eq. 1-3 with the causal
// mask of "ALiBi: Attention with Linear Biases" (abhik.ai), "From distance to
// a normalized weight"; the underflow criterion is sec. 3.2 (e^{tau} = 0,
// crossing at "<= tau") and sec. 3.3 (what the fraction counts).

#include "ptx.cuh"

namespace alibi {
namespace {

constexpr int kRowsPerBlock = 8;  // warps (query rows) per CTA in the fp32 prefill

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Scaled, biased logit of the fp32 path (shared by the prefill and the weight export so
// both see bit-identical values): dot in index order, then one FMA each.
__device__ __forceinline__ float f32_logit(const float *qs, const float *kj, int d, float scale, float slope, int dist)
{
    float dot = 0.f;
    for (int t = 0; t < d; ++t) dot = fmaf(qs[t], kj[t], dot);
    return fmaf(dot, scale, -slope * static_cast<float>(dist));
}

template <int DPL>  // d elements per lane: lane owns t = lane + 32 u
__global__ void __launch_bounds__(kRowsPerBlock * 32) fwd_f32_kernel(const float *__restrict__ q,
                                                                      const float *__restrict__ k,
                                                                      const float *__restrict__ v, float *__restrict__ out,
                                                                      float *__restrict__ lse, long long rows, int H,
                                                                      int N, int d, int causal, float scale,
                                                                      Slopes slopes)
{
    __shared__ float qsm[kRowsPerBlock][32 * DPL];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kRowsPerBlock + warp;
    if (row >= rows) return;
    const long long bh = row / N;
    const int i = static_cast<int>(row - bh * N);
    const float slope = slopes.nat[bh % H];
    const float *kb = k + bh * N * d;
    const float *vb = v + bh * N * d;
    for (int t = lane; t < d; t += 32) qsm[warp][t] = q[row * d + t];
    __syncwarp();

    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int u = 0; u < DPL; ++u) o[u] = 0.f;
    const int jlast = causal ? i : N - 1;  // last key the row attends to
    for (int j0 = 0; j0 <= jlast; j0 += 32) {
        const int j = j0 + lane;
        const float x = (j <= jlast) ? f32_logit(qsm[warp], kb + static_cast<long long>(j) * d, d, scale, slope,
                                                 abs(i - j))
                                     : -INFINITY;
        const float mn = fmaxf(m, warp_max(x));  // finite: key j0 <= jlast is always allowed
        const float alpha = expf(m - mn);        // 0 on the first block (m = -inf)
        const float pj = (j <= jlast) ? expf(x - mn) : 0.f;
        l = l * alpha + warp_sum(pj);
#pragma unroll
        for (int u = 0; u < DPL; ++u) o[u] *= alpha;
        const int jn = min(32, jlast - j0 + 1);
        for (int jj = 0; jj < jn; ++jj) {
            const float pb = __shfl_sync(0xffffffffu, pj, jj);
            const float *vr = vb + static_cast<long long>(j0 + jj) * d;
#pragma unroll
            for (int u = 0; u < DPL; ++u) {
                const int t = lane + 32 * u;
                if (t < d) o[u] = fmaf(pb, vr[t], o[u]);
            }
        }
        m = mn;
    }
#pragma unroll
    for (int u = 0; u < DPL; ++u) {
        const int t = lane + 32 * u;
        if (t < d) out[row * d + t] = o[u] / l;
    }
    if (lse && lane == 0) lse[row] = m + logf(l);
}

// P[b,h,i,j] = exp(x_ij - lse_i) for every allowed key (j <= i when causal), else 0.
// One thread per (row, j).
__global__ void probs_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                                 const float *__restrict__ lse, float *__restrict__ P, long long total, int H, int N,
                                 int d, int causal, float scale, Slopes slopes)
{
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const long long row = idx / N;
    const int j = static_cast<int>(idx - row * N);
    const long long bh = row / N;
    const int i = static_cast<int>(row - bh * N);
    float pij = 0.f;
    if (!causal || j <= i) {
        const float x = f32_logit(q + row * d, k + (bh * N + j) * d, d, scale, slopes.nat[bh % H], abs(i - j));
        pij = expf(x - lse[row]);
    }
    P[idx] = pij;
}

// ------------------------------------------------------------------ underflow

constexpr int kUfRows = 128;  // query rows per CTA (one per thread)
constexpr int kUfKeys = 32;   // keys per shared-memory tile

template <int D>
__global__ void __launch_bounds__(kUfRows) underflow_kernel(const __nv_bfloat16 *__restrict__ q,
                                                            const __nv_bfloat16 *__restrict__ k,
                                                            unsigned long long *__restrict__ counts, int H, int N,
                                                            float tau, float scale, Slopes slopes)
{
    __shared__ __align__(16) float ks[kUfKeys][D];
    __shared__ unsigned long long red[kUfRows / 32];
    // one-dimensional grid (B*H may exceed the 65535 limit of the y dimension)
    const int nrb = (N + kUfRows - 1) / kUfRows;
    const int bh = static_cast<int>(blockIdx.x / nrb);
    const int r0 = static_cast<int>(blockIdx.x - bh * nrb) * kUfRows;
    const int i = r0 + threadIdx.x;
    const bool valid = i < N;
    const float slope = slopes.nat[bh % H];
    const __nv_bfloat16 *kb = k + static_cast<size_t>(bh) * N * D;

    float qr[D];
    {
        const __nv_bfloat16 *qi = q + (static_cast<size_t>(bh) * N + (valid ? i : 0)) * D;
#pragma unroll
        for (int t = 0; t < D; ++t) qr[t] = __bfloat162float(qi[t]);
    }
    const int jmax = min(N - 1, r0 + kUfRows - 1);  // last key any row of this CTA needs

    float M = -INFINITY;
    unsigned long long cnt = 0;
    for (int pass = 0; pass < 2; ++pass) {
        for (int j0 = 0; j0 <= jmax; j0 += kUfKeys) {
            __syncthreads();
            for (int e = threadIdx.x; e < kUfKeys * D; e += kUfRows) {
                const int jj = e / D, t = e - jj * D;
                const int j = j0 + jj;
                ks[jj][t] = (j <= jmax) ? __bfloat162float(kb[static_cast<size_t>(j) * D + t]) : 0.f;
            }
            __syncthreads();
            if (!valid) continue;
            const int jn = min(kUfKeys, i - j0 + 1);
            for (int jj = 0; jj < jn; ++jj) {
                float dot = 0.f;
#pragma unroll
                for (int t = 0; t < D; t += 4) {
                    const float4 kv = *reinterpret_cast<const float4 *>(&ks[jj][t]);
                    dot = fmaf(qr[t], kv.x, dot);
                    dot = fmaf(qr[t + 1], kv.y, dot);
                    dot = fmaf(qr[t + 2], kv.z, dot);
                    dot = fmaf(qr[t + 3], kv.w, dot);
                }
                const float x = fmaf(dot, scale, -slope * static_cast<float>(i - (j0 + jj)));
                if (pass == 0)
                    M = fmaxf(M, x);
                else
                    cnt += (x - M <= tau) ? 1ull : 0ull;
            }
        }
    }
    // block reduction, one atomic per CTA
#pragma unroll
    for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0;
        for (int w = 0; w < kUfRows / 32; ++w) s += red[w];
        atomicAdd(&counts[bh % H], s);
    }
}

// Decode row (query at position L-1 against keys 0..L-1): one CTA per (b, h), 256
// threads, LPK = D/8 lanes per key row (16-byte loads). Pass 1 takes the row max of
// x_j = q.k_j / sqrt(d) - m_h (L-1-j), pass 2 counts the keys with x_j - M <= tau.
template <int D>
__global__ void __launch_bounds__(256) decode_underflow_kernel(const __nv_bfloat16 *__restrict__ q,
                                                               const __nv_bfloat16 *__restrict__ k,
                                                               unsigned long long *__restrict__ counts, int H, int L,
                                                               float tau, float scale, Slopes slopes)
{
    constexpr int LPK = D / 8, KPW = 32 / LPK;  // lanes per key, keys per warp pass
    __shared__ float redf[8];
    __shared__ unsigned long long redc[8];
    const int bh = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LPK, l = lane % LPK;
    const float slope = slopes.nat[bh % H];
    const __nv_bfloat16 *kb = k + static_cast<size_t>(bh) * L * D;
    float qf[8];
    {
        const uint4 u = *reinterpret_cast<const uint4 *>(q + static_cast<size_t>(bh) * D + 8 * l);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            qf[2 * t] = __uint_as_float(w[t] << 16);
            qf[2 * t + 1] = __uint_as_float(w[t] & 0xFFFF0000u);
        }
    }
    float M = -INFINITY;
    unsigned long long cnt = 0;
    for (int pass = 0; pass < 2; ++pass) {
        for (int j0 = warp * KPW; j0 < L; j0 += 8 * KPW) {
            const int j = j0 + sub;
            float dot = 0.f;
            if (j < L) {
                const uint4 u = *reinterpret_cast<const uint4 *>(kb + static_cast<size_t>(j) * D + 8 * l);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    dot = fmaf(qf[2 * t], __uint_as_float(w[t] << 16), dot);
                    dot = fmaf(qf[2 * t + 1], __uint_as_float(w[t] & 0xFFFF0000u), dot);
                }
            }
#pragma unroll
            for (int o = LPK / 2; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            if (j < L && l == 0) {
                const float x = fmaf(dot, scale, -slope * static_cast<float>(L - 1 - j));
                if (pass == 0)
                    M = fmaxf(M, x);
                else
                    cnt += (x - M <= tau) ? 1ull : 0ull;
            }
        }
        if (pass == 0) {  // CTA-wide row max
#pragma unroll
            for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            if (lane == 0) redf[warp] = M;
            __syncthreads();
            M = redf[0];
            for (int w = 1; w < 8; ++w) M = fmaxf(M, redf[w]);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) redc[warp] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0;
        for (int w = 0; w < 8; ++w) s += redc[w];
        atomicAdd(&counts[bh % H], s);
    }
}

// Waits on a barrier nobody arrives on: the bounded wait must give up and record
// a timeout (failure-path self-test).
__global__ void selftest_timeout_kernel(uint32_t *err)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        cta_err_init(kWaitLimitNs);
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait(&bar, 0, err, 0x901);
    }
}

}  // namespace

cudaError_t launch_selftest_timeout(cudaStream_t stream)
{
    uint32_t *err = device_status_word();
    if (!err) return cudaErrorInvalidDevice;
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *out, float *lse, int B, int H,
                           int N, int d, int causal, const Slopes &slopes, cudaStream_t stream)
{
    const long long rows = static_cast<long long>(B) * H * N;
    const unsigned grid = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    const float scale = 1.0f / sqrtf(static_cast<float>(d));
    const int dpl = (d + 31) / 32;
#define ALIBI_F32_CASE(X)                                                                                        \
    case X:                                                                                                      \
        fwd_f32_kernel<X><<<grid, kRowsPerBlock * 32, 0, stream>>>(q, k, v, out, lse, rows, H, N, d, causal, scale, \
                                                                    slopes);                               \
        break;
    switch (dpl) {
        ALIBI_F32_CASE(1)
        ALIBI_F32_CASE(2)
        ALIBI_F32_CASE(3)
        ALIBI_F32_CASE(4)
        ALIBI_F32_CASE(5)
        ALIBI_F32_CASE(6)
        ALIBI_F32_CASE(7)
        ALIBI_F32_CASE(8)
        default:
            return cudaErrorInvalidValue;
    }
#undef ALIBI_F32_CASE
    return cudaGetLastError();
}

cudaError_t launch_probs_f32(const float *q, const float *k, const float *lse, float *P, int B, int H, int N, int d,
                             int causal, const Slopes &slopes, cudaStream_t stream)
{
    const long long total = static_cast<long long>(B) * H * N * N;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    probs_f32_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(q, k, lse, P, total, H, N, d, causal,
                                                                            1.0f / sqrtf(static_cast<float>(d)),
                                                                            slopes);
    return cudaGetLastError();
}

cudaError_t launch_decode_underflow(const void *q, const void *kc, int B, int H, int L, int d, float tau,
                                    unsigned long long *counts, const Slopes &slopes, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(unsigned long long) * H, stream);
    if (e != cudaSuccess) return e;
    const long long BH = static_cast<long long>(B) * H;
    if (BH > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(BH);
    const float scale = 1.0f / sqrtf(static_cast<float>(d));
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(kc);
    if (d == 128)
        decode_underflow_kernel<128><<<grid, 256, 0, stream>>>(qb, kb, counts, H, L, tau, scale, slopes);
    else if (d == 64)
        decode_underflow_kernel<64><<<grid, 256, 0, stream>>>(qb, kb, counts, H, L, tau, scale, slopes);
    else if (d == 32)
        decode_underflow_kernel<32><<<grid, 256, 0, stream>>>(qb, kb, counts, H, L, tau, scale, slopes);
    else if (d == 16)
        decode_underflow_kernel<16><<<grid, 256, 0, stream>>>(qb, kb, counts, H, L, tau, scale, slopes);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_underflow(const void *q, const void *k, int B, int H, int N, int d, float tau,
                             unsigned long long *counts, const Slopes &slopes, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(unsigned long long) * H, stream);
    if (e != cudaSuccess) return e;
    const long long nblocks = static_cast<long long>((N + kUfRows - 1) / kUfRows) * B * H;
    if (nblocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(nblocks);
    const float scale = 1.0f / sqrtf(static_cast<float>(d));
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    if (d == 128)
        underflow_kernel<128><<<grid, kUfRows, 0, stream>>>(qb, kb, counts, H, N, tau, scale, slopes);
    else if (d == 64)
        underflow_kernel<64><<<grid, kUfRows, 0, stream>>>(qb, kb, counts, H, N, tau, scale, slopes);
    else if (d == 32)
        underflow_kernel<32><<<grid, kUfRows, 0, stream>>>(qb, kb, counts, H, N, tau, scale, slopes);
    else if (d == 16)
        underflow_kernel<16><<<grid, kUfRows, 0, stream>>>(qb, kb, counts, H, N, tau, scale, slopes);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace alibi

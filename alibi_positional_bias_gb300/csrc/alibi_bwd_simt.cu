// fp32 backward at reference precision (CUDA cores, IEEE expf): the same
// gradients as the tensor-core backward (dQ, dK, dV of sum(dO * O) for the
// ALiBi attention of "When Attention Goes Blind" sec. 3.1 eq. 1-4, causal or
// with the symmetric |i - j| bias), every product and sum in fp32.
//   bwd_f32_dq_kernel   one warp per query row i: D_i = dO_i . O_i (stored for
//                       the second kernel), then dQ_i = sum_j dS_ij k_j / sqrt(d)
//   bwd_f32_dkv_kernel  one warp per key j: dK_j = sum_i dS_ij q_i / sqrt(d),
//                       dV_j = sum_i P_ij dO_i
// with P_ij = exp(x_ij - LSE_i) from the forward's LSE and
// dS_ij = P_ij (dO_i . v_j - D_i).

#include "ptx.cuh"

namespace alibi {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_sum_b(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float dot_f32(const float *a, const float *b, int d)
{
    float s = 0.f;
    for (int t = 0; t < d; ++t) s = fmaf(a[t], b[t], s);
    return s;
}

// Logit of the fp32 forward path: dot in index order, then one FMA with the bias.
__device__ __forceinline__ float bwd_logit(const float *qi, const float *kj, int d, float scale, float slope, int i,
                                           int j)
{
    return fmaf(dot_f32(qi, kj, d), scale, -slope * static_cast<float>(abs(i - j)));
}

template <int DPL>
__global__ void __launch_bounds__(kWarps * 32) bwd_f32_dq_kernel(const float *__restrict__ q, const float *__restrict__ k,
                                                                 const float *__restrict__ v, const float *__restrict__ o,
                                                                 const float *__restrict__ lse,
                                                                 const float *__restrict__ dout, float *__restrict__ dq,
                                                                 float *__restrict__ dsum, long long rows, int H, int N,
                                                                 int d, int causal, float scale, Slopes slopes)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kWarps + warp;
    if (row >= rows) return;
    const long long bh = row / N;
    const int i = static_cast<int>(row - bh * N);
    const float slope = slopes.nat[bh % H];
    const float *kb = k + bh * N * d, *vb = v + bh * N * d;
    const float *qi = q + row * d, *doi = dout + row * d;
    float part = 0.f;
    for (int t = lane; t < d; t += 32) part = fmaf(doi[t], o[row * d + t], part);
    const float Di = warp_sum_b(part);
    if (lane == 0) dsum[row] = Di;
    const float li = lse[row];
    float acc[DPL];
#pragma unroll
    for (int u = 0; u < DPL; ++u) acc[u] = 0.f;
    const int jlast = causal ? i : N - 1;
    for (int j0 = 0; j0 <= jlast; j0 += 32) {
        const int j = j0 + lane;
        float ds = 0.f;
        if (j <= jlast) {
            const float pij = expf(bwd_logit(qi, kb + static_cast<long long>(j) * d, d, scale, slope, i, j) - li);
            ds = pij * (dot_f32(doi, vb + static_cast<long long>(j) * d, d) - Di);
        }
        const int jn = min(32, jlast - j0 + 1);
        for (int jj = 0; jj < jn; ++jj) {
            const float b = __shfl_sync(0xffffffffu, ds, jj);
            const float *kr = kb + static_cast<long long>(j0 + jj) * d;
#pragma unroll
            for (int u = 0; u < DPL; ++u) {
                const int t = lane + 32 * u;
                if (t < d) acc[u] = fmaf(b, kr[t], acc[u]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < DPL; ++u) {
        const int t = lane + 32 * u;
        if (t < d) dq[row * d + t] = acc[u] * scale;
    }
}

template <int DPL>
__global__ void __launch_bounds__(kWarps * 32) bwd_f32_dkv_kernel(const float *__restrict__ q, const float *__restrict__ k,
                                                                  const float *__restrict__ v,
                                                                  const float *__restrict__ lse,
                                                                  const float *__restrict__ dout,
                                                                  const float *__restrict__ dsum, float *__restrict__ dk,
                                                                  float *__restrict__ dv, long long rows, int H, int N,
                                                                  int d, int causal, float scale, Slopes slopes)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long col = static_cast<long long>(blockIdx.x) * kWarps + warp;  // flat key index
    if (col >= rows) return;
    const long long bh = col / N;
    const int j = static_cast<int>(col - bh * N);
    const float slope = slopes.nat[bh % H];
    const float *qb = q + bh * N * d, *ob = dout + bh * N * d;
    const float *kj = k + col * d, *vj = v + col * d;
    const float *lb = lse + bh * N, *db = dsum + bh * N;
    float ak[DPL], av[DPL];
#pragma unroll
    for (int u = 0; u < DPL; ++u) ak[u] = av[u] = 0.f;
    const int ifirst = causal ? j : 0;
    for (int i0 = ifirst; i0 < N; i0 += 32) {
        const int i = i0 + lane;
        float pij = 0.f, ds = 0.f;
        if (i < N) {
            const float *qi = qb + static_cast<long long>(i) * d;
            pij = expf(bwd_logit(qi, kj, d, scale, slope, i, j) - lb[i]);
            ds = pij * (dot_f32(ob + static_cast<long long>(i) * d, vj, d) - db[i]);
        }
        const int in = min(32, N - i0);
        for (int ii = 0; ii < in; ++ii) {
            const float bp = __shfl_sync(0xffffffffu, pij, ii), bs = __shfl_sync(0xffffffffu, ds, ii);
            const float *qr = qb + static_cast<long long>(i0 + ii) * d, *orow = ob + static_cast<long long>(i0 + ii) * d;
#pragma unroll
            for (int u = 0; u < DPL; ++u) {
                const int t = lane + 32 * u;
                if (t < d) {
                    ak[u] = fmaf(bs, qr[t], ak[u]);
                    av[u] = fmaf(bp, orow[t], av[u]);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < DPL; ++u) {
        const int t = lane + 32 * u;
        if (t < d) {
            dk[col * d + t] = ak[u] * scale;
            dv[col * d + t] = av[u];
        }
    }
}

}  // namespace

cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *out, const float *lse,
                           const float *dout, float *dq, float *dk, float *dv, int B, int H, int N, int d, int causal,
                           const Slopes &slopes, cudaStream_t stream)
{
    const long long rows = static_cast<long long>(B) * H * N;
    const unsigned grid = static_cast<unsigned>((rows + kWarps - 1) / kWarps);
    const float scale = 1.0f / sqrtf(static_cast<float>(d));
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, static_cast<size_t>(rows) * sizeof(float) + 256, decode_pool(), stream);
    if (e != cudaSuccess) return e;
    float *dsum = static_cast<float *>(ws);
    const int dpl = (d + 31) / 32;
#define ALIBI_BWD_F32_CASE(X)                                                                                    \
    case X:                                                                                                      \
        bwd_f32_dq_kernel<X><<<grid, kWarps * 32, 0, stream>>>(q, k, v, out, lse, dout, dq, dsum, rows, H, N, d, \
                                                               causal, scale, slopes);                           \
        bwd_f32_dkv_kernel<X><<<grid, kWarps * 32, 0, stream>>>(q, k, v, lse, dout, dsum, dk, dv, rows, H, N, d, \
                                                                causal, scale, slopes);                          \
        break;
    switch (dpl) {
        ALIBI_BWD_F32_CASE(1)
        ALIBI_BWD_F32_CASE(2)
        ALIBI_BWD_F32_CASE(3)
        ALIBI_BWD_F32_CASE(4)
        ALIBI_BWD_F32_CASE(5)
        ALIBI_BWD_F32_CASE(6)
        ALIBI_BWD_F32_CASE(7)
        ALIBI_BWD_F32_CASE(8)
        default:
            e = cudaErrorInvalidValue;
    }
#undef ALIBI_BWD_F32_CASE
    if (e == cudaSuccess) e = cudaGetLastError();
    const cudaError_t f = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : f;
}

}  // namespace alibi

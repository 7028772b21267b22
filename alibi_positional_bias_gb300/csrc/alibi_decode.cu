// ALiBi decode: one new query per (b, h) against a bf16 KV cache of L positions.
//
// The query sits at its true sequence position L - 1 ("ALiBi: Attention with
// Linear Biases" (abhik.ai), the KV-cache paragraph after the full-sequence
// example), so key j has bias -m_h (L - 1 - j):
//   s_j = q.k_j / sqrt(d) - m_h (L - 1 - j),  out = sum_j softmax_j(s) v_j
// with the max-shifted softmax of "When Attention Goes Blind" (arXiv
// 2608.03994), App. B.1, evaluated online and merged across splits.
//
// Memory-bound design: the cache is streamed once with 16-byte non-caching
// loads. A group of d/8 lanes owns one key row (8 bf16 per lane: 16 lanes for
// d = 128, 8 for 64, 4 for 32, 2 for 16), so a warp-wide load covers 32/(d/8)
// adjacent rows (512 contiguous bytes). Each lane issues 8 K and 8 V loads
// before using them, keeping ~8 KB per warp in flight at every d. One CTA per
// (b, h) and split (one-dimensional grid, splits of a head adjacent); each CTA (8 warps) streams a contiguous slice of the cache,
// merges its warps' partial softmaxes in shared memory, and either writes the
// output (one split) or an fp32 partial (m, l, o[d]). With several splits, the
// CTA that finishes a (b, h) last (a per-(b, h) counter it increments after a
// device-wide fence) merges that head's partials and writes its output, so no
// CTA ever waits for another and no second kernel is launched.
//
// Skipping ("When Attention Goes Blind" sec. 3.2-3.3 and 5.2: past its blindness
// distance a head's weights are exactly zero): with per-64-key-block maximum key
// norms (kv_block_norms_kernel, kept by the caller alongside the cache), a warp
// step is left out when every key j in it satisfies, in base-2 units,
//   c1 |q| max|k| - m log2(e) (L - 1 - j) <= x_last - 127
// where x_last is the last key's logit, a lower bound of the final row max:
// each such weight is below 2^-127 of the largest one, i.e. below the fp32
// resolution of the sum, and its K and V rows are never read.

#include "ptx.cuh"

namespace alibi {
namespace {

constexpr int kWarps = 8;
constexpr int kKeysPerGroup = 8;  // keys per lane group per step

template <int D>
struct DecCfg {
    static constexpr int kLanesPerRow = D / 8;              // 8 bf16 per lane
    static constexpr int kGroups = 32 / kLanesPerRow;       // key rows per warp-wide load
    static constexpr int kKeysPerWarp = kGroups * kKeysPerGroup;
    static constexpr int kPartStride = D + 4;               // floats per partial: m, l, pad, pad, o[d]
};

struct DecodeParams {
    const __nv_bfloat16 *q, *k, *v;
    __nv_bfloat16 *out;
    float *part;  // [BH][splits][kPartStride], used when splits > 1
    unsigned *count;  // [BH] splits finished per (b, h), zero between calls; used when splits > 1
    const float *knorm;  // optional [BH][nblk] max key norm per 64-key block: enables skipping
    int H, L, splits, chunk, nblk;
    float c1;  // log2(e) / sqrt(d)
    Slopes slopes;
};

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        f[2 * t] = __uint_as_float(w[t] << 16);
        f[2 * t + 1] = __uint_as_float(w[t] & 0xFFFF0000u);
    }
}

// One warp merges the splits' partial softmaxes of one (b, h) (lane t covers
// o[4t .. 4t + 3]); the partials are read through L2 (written by other CTAs).
template <int D>
__device__ __forceinline__ void merge_partials(const float *base, int splits, __nv_bfloat16 *out_row, int lane)
{
    constexpr int kStride = DecCfg<D>::kPartStride;
    float M = -INFINITY;
    for (int s = lane; s < splits; s += 32) M = fmaxf(M, __ldcg(base + s * kStride));
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    // lanes own 4 output columns each; the partials of 8 splits are loaded together
    const bool mine = 4 * lane < D;
    float Lsum = 0.f, O[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < splits; s0 += 8) {
        float ms[8], ls[8];
        float4 ov[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool in = s0 + j < splits;
            const float *ps = base + (in ? s0 + j : 0) * kStride;
            ms[j] = in ? __ldcg(ps) : -INFINITY;
            ls[j] = in ? __ldcg(ps + 1) : 0.f;
            ov[j] = (in && mine) ? __ldcg(reinterpret_cast<const float4 *>(ps + 4 + 4 * lane))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float a = (ms[j] == -INFINITY) ? 0.f : ex2_approx(ms[j] - M);
            Lsum = fmaf(ls[j], a, Lsum);
            O[0] = fmaf(ov[j].x, a, O[0]);
            O[1] = fmaf(ov[j].y, a, O[1]);
            O[2] = fmaf(ov[j].z, a, O[2]);
            O[3] = fmaf(ov[j].w, a, O[3]);
        }
    }
    if (!mine) return;
    const float inv = 1.0f / Lsum;
    __nv_bfloat162 r0 = __floats2bfloat162_rn(O[0] * inv, O[1] * inv);
    __nv_bfloat162 r1 = __floats2bfloat162_rn(O[2] * inv, O[3] * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&r0);
    pk.y = *reinterpret_cast<uint32_t *>(&r1);
    *reinterpret_cast<uint2 *>(out_row + 4 * lane) = pk;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32, 2) decode_kernel(const __grid_constant__ DecodeParams p)
{
    using C = DecCfg<D>;
    constexpr int LPR = C::kLanesPerRow;
    __shared__ float sm_m[kWarps], sm_l[kWarps];
    __shared__ float sm_o[kWarps][D];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane / LPR, l16 = lane % LPR;  // lane group (key row) and slice within the row
    // one-dimensional grid (B*H may exceed the 65535 limit of the y dimension): the
    // splits of one (b, h) are adjacent
    const int bh = static_cast<int>(blockIdx.x / p.splits), split = static_cast<int>(blockIdx.x - bh * p.splits);
    const int h = bh % p.H;
    const float sl2 = p.slopes.log2e[h];
    const int pos = p.L - 1;
    const int kbeg = split * p.chunk;
    const int kend = min(p.L, kbeg + p.chunk);

    // this lane's 8 query elements (d slice [8 l16, 8 l16 + 8)), pre-scaled to log2 units
    float qf[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(p.q + static_cast<size_t>(bh) * D + 8 * l16), qf);
#pragma unroll
    for (int t = 0; t < 8; ++t) qf[t] *= p.c1;

    const __nv_bfloat16 *kbase = p.k + static_cast<size_t>(bh) * p.L * D + 8 * l16;
    const __nv_bfloat16 *vbase = p.v + static_cast<size_t>(bh) * p.L * D + 8 * l16;

    float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) o[t] = 0.f;

    // Skip set-up: |q| c1 and the last key's logit (both the same in every lane group).
    const bool skip = p.knorm != nullptr;
    float skip_a = 0.f;  // c1 |q| (1 + 2^-10)^2: multiplies a block's max key norm
    float skip_b = 0.f;  // -x_last + |x_last| 2^-10 + 127: with the above, the bias a step must exceed
    const float *kn = skip ? p.knorm + static_cast<size_t>(bh) * p.nblk : nullptr;
    if (skip) {
        float ss = 0.f, dl = 0.f;
        float kf[8];
        bf16x8_to_f32(ld_stream(kbase + static_cast<size_t>(pos) * D), kf);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            ss = fmaf(qf[t], qf[t], ss);
            dl = fmaf(qf[t], kf[t], dl);
        }
#pragma unroll
        for (int off = LPR / 2; off; off >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
            dl += __shfl_xor_sync(0xffffffffu, dl, off);
        }
        const float slack = 1.0f + 0x1p-10f;
        skip_a = sqrtf(ss) * slack * slack;
        skip_b = -dl + fabsf(dl) * 0x1p-10f + 127.0f;
    }
    // max key norm over the norm blocks a warp step [b, b + KPW) touches
    auto step_norm = [&](int b) -> float {
        const int b0 = b >> 6, b1 = min((b + C::kKeysPerWarp - 1) >> 6, p.nblk - 1);
        return fmaxf(__ldg(kn + b0), __ldg(kn + b1));
    };
    const int first = kbeg + warp * C::kKeysPerWarp, stride = kWarps * C::kKeysPerWarp;
    float kn_cur = (skip && first < kend) ? step_norm(first) : 0.f;

    for (int blk = first; blk < kend; blk += stride) {
        // next step's norm fetched one step ahead, off the load path
        const float kn_nxt = (skip && blk + stride < kend) ? step_norm(blk + stride) : 0.f;
        const bool drop = skip && sl2 * static_cast<float>(pos - min(blk + C::kKeysPerWarp - 1, kend - 1)) >=
                                      fmaf(skip_a, kn_cur, skip_b);
        kn_cur = kn_nxt;
        if (drop) continue;  // every weight of this step is below 2^-127 of the row's largest
        uint4 kr[kKeysPerGroup], vr[kKeysPerGroup];
#pragma unroll
        for (int u = 0; u < kKeysPerGroup; ++u) {
            const int key = blk + C::kGroups * u + half;
            if (key < kend) {
                kr[u] = ld_stream(kbase + static_cast<size_t>(key) * D);
                vr[u] = ld_stream(vbase + static_cast<size_t>(key) * D);
            } else {
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
            }
        }
        float x[kKeysPerGroup];
        float mt = -INFINITY;
#pragma unroll
        for (int u = 0; u < kKeysPerGroup; ++u) {
            float kf[8];
            bf16x8_to_f32(kr[u], kf);
            float dot = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) dot = fmaf(qf[t], kf[t], dot);
#pragma unroll
            for (int off = LPR / 2; off; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const int key = blk + C::kGroups * u + half;
            x[u] = (key < kend) ? fmaf(-sl2, static_cast<float>(pos - key), dot) : -INFINITY;
            mt = fmaxf(mt, x[u]);
        }
        if (mt > -INFINITY) {  // this lane group saw at least one key in range
            const float mn = fmaxf(m, mt);
            const float alpha = ex2_approx(m - mn);  // 0 while m is still -inf
            m = mn;
            l *= alpha;
#pragma unroll
            for (int t = 0; t < 8; ++t) o[t] *= alpha;
#pragma unroll
            for (int u = 0; u < kKeysPerGroup; ++u) {
                const float pu = ex2_approx(x[u] - m);
                l += pu;
                float vf[8];
                bf16x8_to_f32(vr[u], vf);
#pragma unroll
                for (int t = 0; t < 8; ++t) o[t] = fmaf(pu, vf[t], o[t]);
            }
        }
    }

    // merge the lane groups (lanes l16 + LPR g own the same d slice for every g)
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off);
        const float lo = __shfl_xor_sync(0xffffffffu, l, off);
        const float mn = fmaxf(m, mo);
        const float a = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
        const float b = (mo == -INFINITY) ? 0.f : ex2_approx(mo - mn);
        l = l * a + lo * b;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float oo = __shfl_xor_sync(0xffffffffu, o[t], off);
            o[t] = o[t] * a + oo * b;
        }
        m = mn;
    }
    if (lane < LPR) {
#pragma unroll
        for (int t = 0; t < 8; ++t) sm_o[warp][8 * l16 + t] = o[t];
        if (lane == 0) {
            sm_m[warp] = m;
            sm_l[warp] = l;
        }
    }
    __syncthreads();
    if (threadIdx.x < D) {
        const int t = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w]);
        float Lsum = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float a = (sm_m[w] == -INFINITY) ? 0.f : ex2_approx(sm_m[w] - M);
            Lsum = fmaf(sm_l[w], a, Lsum);
            O = fmaf(sm_o[w][t], a, O);
        }
        if (p.splits == 1) {
            p.out[static_cast<size_t>(bh) * D + t] = __float2bfloat16_rn(O / Lsum);
        } else {
            float *dst = p.part + (static_cast<size_t>(bh) * p.splits + split) * C::kPartStride;
            if (t == 0) {
                dst[0] = M;
                dst[1] = Lsum;
            }
            dst[4 + t] = O;
        }
    }
    if (p.splits == 1) return;
    // Count this split as done once its partial is visible device-wide; the CTA that
    // counts a (b, h) last merges it (no CTA waits for another) and re-arms the counter.
    __shared__ bool last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(p.count + bh, 1u) == static_cast<unsigned>(p.splits - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();  // the other splits' partials, counted before this CTA, are read after it
    if (warp == 0)
        merge_partials<D>(p.part + static_cast<size_t>(bh) * p.splits * C::kPartStride, p.splits,
                          p.out + static_cast<size_t>(bh) * D, lane);
    if (threadIdx.x == 0) p.count[bh] = 0u;  // zero again for the next call that uses this buffer
}

// Maximum key norm of each 64-key block of the cache: one CTA per (b, h) and block
// (one-dimensional grid), 256 threads, d/8 lanes per key. Blocks [blk_begin, nblk) of every (b, h).
template <int D>
__global__ void __launch_bounds__(256) kv_block_norms_kernel(const __nv_bfloat16 *__restrict__ k, float *__restrict__ knorm,
                                                             int L, int nblk, int blk_begin)
{
    constexpr int LPR = D / 8, RPW = 32 / LPR;
    __shared__ float red[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = nblk - blk_begin;  // one-dimensional grid: the blocks of one (b, h) are adjacent
    const int bh = static_cast<int>(blockIdx.x / nb), b = blk_begin + static_cast<int>(blockIdx.x - bh * nb);
    const int g = lane / LPR, l = lane % LPR;
    const __nv_bfloat16 *kb = k + static_cast<size_t>(bh) * L * D + 8 * l;
    float best = 0.f;
    // uniform trip count: every lane takes part in the shuffles
    for (int j0 = b * 64 + warp * RPW; j0 < b * 64 + 64; j0 += 8 * RPW) {
        const int j = j0 + g;
        float ss = 0.f;
        if (j < L) {
            float kf[8];
            bf16x8_to_f32(ld_stream(kb + static_cast<size_t>(j) * D), kf);
#pragma unroll
            for (int t = 0; t < 8; ++t) ss = fmaf(kf[t], kf[t], ss);
        }
        // the row's sum of squares over its d/8 lanes
#pragma unroll
        for (int off = LPR / 2; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        best = fmaxf(best, ss);
    }
    // max over the rows this warp saw
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, off));
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mx = red[0];
        for (int w = 1; w < 8; ++w) mx = fmaxf(mx, red[w]);
        knorm[static_cast<size_t>(bh) * nblk + b] = sqrtf(mx);
    }
}

}  // namespace

cudaError_t launch_kv_block_norms(const void *kc, float *knorm, int B, int H, int L, int d, int blk_begin,
                                  cudaStream_t stream)
{
    const int nblk = (L + 63) / 64;
    if (blk_begin >= nblk) return cudaSuccess;
    const long long nblocks = static_cast<long long>(nblk - blk_begin) * B * H;
    if (nblocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(nblocks);
    const auto *k = static_cast<const __nv_bfloat16 *>(kc);
    switch (d) {
        case 128: kv_block_norms_kernel<128><<<grid, 256, 0, stream>>>(k, knorm, L, nblk, blk_begin); break;
        case 64: kv_block_norms_kernel<64><<<grid, 256, 0, stream>>>(k, knorm, L, nblk, blk_begin); break;
        case 32: kv_block_norms_kernel<32><<<grid, 256, 0, stream>>>(k, knorm, L, nblk, blk_begin); break;
        case 16: kv_block_norms_kernel<16><<<grid, 256, 0, stream>>>(k, knorm, L, nblk, blk_begin); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// Split count: with eight or more waves of whole heads (two resident CTAs per SM)
// every SM streams whole heads and there is nothing to merge; with fewer, each
// head's cache is cut into the number of slices that minimises (waves of CTAs) x
// (keys per CTA + a fixed per-CTA cost of 256 keys) plus the merge, slices of at
// least 256 keys.
int decode_splits(int BH, int L)
{
    const long long R = 2LL * num_sms();
    if (BH >= 8 * R) return 1;
    const int max_s = (L + 255) / 256;
    int best = 1;
    long long best_cost = -1;
    for (int s = 1; s <= max_s && s <= 4096; ++s) {
        const long long waves = (static_cast<long long>(BH) * s + R - 1) / R;
        // a split also costs its merge: the partials and the merging CTA's pass (~512 keys)
        const long long cost = waves * ((L + s - 1) / s + 256) + (s > 1 ? 512 : 0);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

size_t decode_partials_bytes(int BH, int splits, int d)
{
    return splits > 1 ? static_cast<size_t>(BH) * splits * (d + 4) * sizeof(float) : 0;
}

size_t decode_counters_bytes(int BH, int splits) { return splits > 1 ? static_cast<size_t>(BH) * sizeof(unsigned) : 0; }

bool decode_supports(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

template <int D>
static cudaError_t launch_decode_d(const void *q, const void *kc, const void *vc, const float *knorm, void *out, int B,
                                   int H, int L, const Slopes &slopes, int splits, float *partials, unsigned *counters,
                                   cudaStream_t stream)
{
    using C = DecCfg<D>;
    DecodeParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(kc);
    p.v = static_cast<const __nv_bfloat16 *>(vc);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.part = partials;
    p.count = counters;
    p.H = H;
    p.L = L;
    p.splits = splits;
    p.chunk = (L + splits - 1) / splits;
    p.chunk = (p.chunk + C::kKeysPerWarp - 1) / C::kKeysPerWarp * C::kKeysPerWarp;
    p.c1 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    p.slopes = slopes;
    const int BH = B * H;
    p.knorm = knorm;
    p.nblk = (L + 63) / 64;
    // recompute splits so that no split is empty after rounding the chunk
    p.splits = (L + p.chunk - 1) / p.chunk;
    if (p.splits > splits) return cudaErrorInvalidValue;
    const long long nblocks = static_cast<long long>(p.splits) * BH;
    if (nblocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(nblocks);
    if (p.splits > 1 && (!partials || !counters)) return cudaErrorInvalidValue;
    decode_kernel<D><<<grid, kWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode_with(const void *q, const void *kc, const void *vc, const float *knorm, void *out, int B,
                               int H, int L, int d, const Slopes &slopes, int splits, float *partials,
                               unsigned *counters, cudaStream_t stream)
{
    switch (d) {
        case 128:
            return launch_decode_d<128>(q, kc, vc, knorm, out, B, H, L, slopes, splits, partials, counters, stream);
        case 64:
            return launch_decode_d<64>(q, kc, vc, knorm, out, B, H, L, slopes, splits, partials, counters, stream);
        case 32:
            return launch_decode_d<32>(q, kc, vc, knorm, out, B, H, L, slopes, splits, partials, counters, stream);
        case 16:
            return launch_decode_d<16>(q, kc, vc, knorm, out, B, H, L, slopes, splits, partials, counters, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode(const void *q, const void *kc, const void *vc, const float *knorm, void *out, int B, int H,
                          int L, int d, const Slopes &slopes, cudaStream_t stream)
{
    if (!decode_supports(d)) return cudaErrorInvalidValue;
    const int BH = B * H;
    const int splits = decode_splits(BH, L);
    if (splits == 1)
        return launch_decode_with(q, kc, vc, knorm, out, B, H, L, d, slopes, 1, nullptr, nullptr, stream);
    // partials, then the per-(b, h) counters (zeroed here: pool memory holds whatever its last user left)
    const size_t pb = (decode_partials_bytes(BH, splits, d) + 255) & ~size_t(255);
    const size_t cb = decode_counters_bytes(BH, splits);
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, pb + cb, decode_pool(), stream);
    if (e != cudaSuccess) return e;
    unsigned *counters = reinterpret_cast<unsigned *>(static_cast<char *>(ws) + pb);
    e = cudaMemsetAsync(counters, 0, cb, stream);
    if (e == cudaSuccess)
        e = launch_decode_with(q, kc, vc, knorm, out, B, H, L, d, slopes, splits, static_cast<float *>(ws), counters,
                               stream);
    cudaError_t f = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : f;
}

}  // namespace alibi

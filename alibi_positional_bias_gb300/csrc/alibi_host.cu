// Host side of the C ABI declared in include/alibi.h: argument validation,
// the ALiBi slope schedule, TMA tensor-map encoding, per-device state (status
// word, SM count, decode memory pool) and the extern "C" entry points.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "alibi.h"
#include "internal.h"
#include "work_order.h"

namespace alibi {

// Device status word: [0] = ALIBI_DEV_* bits, [1] = first failing site.
__device__ uint32_t g_status[2];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
int g_l2[kMaxDevices] = {};
cudaMemPool_t g_pool[kMaxDevices] = {};

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Slope exponent of head h as 2^(-num/den): "ALiBi: Attention with Linear
// Biases" (abhik.ai), "Different heads, different distance penalties".
void slope_exponent(int H, int h, int *num, int *den)
{
    int c = 1;
    while (c * 2 <= H) c *= 2;  // largest power of two <= H
    if (h < c) {
        *num = 8 * (h + 1);
        *den = c;
    } else {
        *num = 8 * (2 * (h - c) + 1);  // every other entry of the 2c schedule
        *den = 2 * c;
    }
}

// 2^(-num/den) rounded once to fp32: the integer part of the exponent is
// applied exactly with ldexp, the fractional part in long double.
float slope_value(int num, int den)
{
    const int whole = num / den, frac = num % den;
    const long double f = exp2l(-static_cast<long double>(frac) / static_cast<long double>(den));
    return static_cast<float>(ldexpl(f, -whole));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int to_status(cudaError_t e)
{
    return e == cudaSuccess ? ALIBI_OK : ALIBI_ERR_CUDA;
}

}  // namespace

uint32_t *device_status_word()
{
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<uint32_t *>(p);
    }
    return g_status_ptr[dev];
}

int num_sms()
{
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

int l2_bytes()
{
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_l2[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n < 1) n = -1;
        g_l2[dev] = n;
    }
    return g_l2[dev];
}

// Blocked work-order tables (work_order.h), one per (device, kind, mask, B*H, N,
// grid), built on the first launch of that shape and kept for the life of the
// process. Shapes for which the nominal order is kept are remembered too (null
// entries).
const int2 *work_order(OrderKind kind, int causal, int BH, int N, int dr, cudaStream_t stream)
{
    constexpr size_t kMaxTables = 256;               // cached shapes, null entries included
    constexpr size_t kMaxBytes = size_t(256) << 20;  // device memory held by the tables
    constexpr int64_t kMaxItems = int64_t(1) << 24;
    const int NQT = (N + 127) / 128;
    // items per head: prefill blocks of two Q tiles, or the backward's single tiles
    const int per_head = kind == OrderKind::Prefill ? (NQT + 1) / 2 : NQT;
    const int64_t n = static_cast<int64_t>(BH) * per_head;
    // only where the nominal order re-reads a head's streamed tiles (K and V, or Q
    // and dO) from DRAM: B*H heads of them above half the L2 (the resident tiles,
    // the outputs and the far half of the cache take the rest); for the prefill at
    // most 16 blocks of 256 rows per head (with 32 or more its blocked order measured
    // up to 3% slower: a head's items are long enough that the nominal order reuses
    // its tiles), while the backward's kernels gained at every length measured (3-12%
    // from 8K to 64K rows)
    const int l2 = l2_bytes();
    if (NQT < 2 || (kind == OrderKind::Prefill && NQT > 32) || n > kMaxItems || l2 <= 0) return nullptr;
    if (4.0 * BH * static_cast<double>(N) * dr <= 0.5 * static_cast<double>(l2)) return nullptr;
    const int dev = current_device();
    if (dev < 0) return nullptr;
    const int G = static_cast<int>(std::min<int64_t>(n, num_sms()));
    using Key = std::tuple<int, int, int, int, int, int>;
    static std::map<Key, int2 *> tables;
    static size_t held_bytes = 0;
    static std::mutex mu;
    const Key key(dev, static_cast<int>(kind), causal, BH, N, G);
    std::lock_guard<std::mutex> g(mu);
    const auto it = tables.find(key);
    if (it != tables.end()) return it->second;
    if (tables.size() >= kMaxTables) return nullptr;
    // the table is built outside any stream capture (a captured launch of a new
    // shape keeps the nominal order, with identical results)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return nullptr;
    }
    const std::vector<int64_t> sched = !causal                      ? order::choose_uniform(BH, per_head, G)
                                       : kind == OrderKind::Prefill ? order::choose(BH, per_head, NQT, G)
                                                                    : order::choose_single(BH, per_head, G);
    const size_t bytes = sched.size() * sizeof(int2);
    if (sched.empty() || held_bytes + bytes > kMaxBytes) {
        tables[key] = nullptr;
        return nullptr;
    }
    // entries (b h * per_head + index, 0): the prefill's block index is the rank;
    // the backward's rank r is query tile r (dQ) or KV tile NT-1-r (dK/dV)
    std::vector<int2> h(sched.size());
    for (size_t i = 0; i < sched.size(); ++i) {
        const int64_t bh = sched[i] / per_head, r = sched[i] - bh * per_head;
        const int64_t idx = kind == OrderKind::BwdDkDv ? per_head - 1 - r : r;
        h[i] = make_int2(static_cast<int>(bh * per_head + idx), 0);
    }
    // upload on a private stream and wait for it, so the table is complete before
    // any stream can launch with it; relaxed capture mode keeps another thread's
    // capture from refusing these calls
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    int2 *d = nullptr;
    cudaStream_t up = nullptr;
    bool ok = cudaMalloc(&d, bytes) == cudaSuccess &&
              cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking) == cudaSuccess &&
              cudaMemcpyAsync(d, h.data(), bytes, cudaMemcpyHostToDevice, up) == cudaSuccess &&
              cudaStreamSynchronize(up) == cudaSuccess;
    if (up) cudaStreamDestroy(up);
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (!ok) {
        if (d) cudaFree(d);
        cudaGetLastError();  // a failed table only means the nominal order
        return nullptr;
    }
    tables[key] = d;
    held_bytes += bytes;
    return d;
}

cudaError_t prepare_kernel(const void *func, int smem, uint32_t regs)
{
    struct Prepared {
        int dev;
        const void *func;
    };
    static Prepared done[256];
    static int ndone = 0;
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_mu);
    for (int i = 0; i < ndone; ++i)
        if (done[i].dev == dev && done[i].func == func) return cudaSuccess;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, func);
    if (e != cudaSuccess) return e;
    if (regs != 0 && fa.numRegs != static_cast<int>(regs)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (ndone < 256) done[ndone++] = {dev, func};  // a full table only repeats the (idempotent) set-up
    return cudaSuccess;
}

cudaMemPool_t decode_pool()
{
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_pool[dev]) {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
        // keep freed blocks in this pool: the partials buffer is reused call after call
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pool[dev] = pool;
    }
    return g_pool[dev];
}

// The schedule is evaluated in long double, which some hosts (Arm) emulate in
// software at about half a microsecond per value, so each head count's table is
// computed once per process and copied on later calls (the same values).
namespace {
std::atomic<const Slopes *> g_slope_cache[kMaxHeads + 1];

void compute_slopes(int H, Slopes *s)
{
    for (int h = 0; h < H && h < kMaxHeads; ++h) {
        int num, den;
        slope_exponent(H, h, &num, &den);
        s->nat[h] = slope_value(num, den);
        s->log2e[h] = static_cast<float>(static_cast<double>(s->nat[h]) * 1.4426950408889634);
    }
}
}  // namespace

void fill_slopes(int H, Slopes *s)
{
    if (H < 1 || H > kMaxHeads) return compute_slopes(H, s);
    const Slopes *c = g_slope_cache[H].load(std::memory_order_acquire);
    if (!c) {
        Slopes *fresh = new Slopes;
        compute_slopes(H, fresh);
        const Slopes *expected = nullptr;
        if (g_slope_cache[H].compare_exchange_strong(expected, fresh, std::memory_order_acq_rel)) {
            c = fresh;
        } else {  // another thread published the same table first
            delete fresh;
            c = expected;
        }
    }
    std::memcpy(s->nat, c->nat, sizeof(float) * static_cast<size_t>(H));
    std::memcpy(s->log2e, c->log2e, sizeof(float) * static_cast<size_t>(H));
}

void fill_slopes_from(int H, const float *nat, Slopes *s)
{
    for (int h = 0; h < H && h < kMaxHeads; ++h) {
        s->nat[h] = nat[h];
        s->log2e[h] = static_cast<float>(static_cast<double>(nat[h]) * 1.4426950408889634);
    }
}

bool encode_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                         uint32_t box0, uint32_t box1, bool swizzle128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {dim0, dim1, dim2};
    const cuuint64_t strides[2] = {dim0 * 2, dim0 * dim1 * 2};  // bytes, dims 1 and 2
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace alibi

using namespace alibi;

static_assert(kFwdSkipUnderflow == ALIBI_FWD_SKIP_UNDERFLOW && kFwdClamp == ALIBI_FWD_CLAMP &&
                  kFwdLogDist == ALIBI_FWD_LOGDIST && kFwdSoftcap == ALIBI_FWD_SOFTCAP &&
                  kFwdNominalOrder == ALIBI_FWD_NOMINAL_ORDER,
              "flag values of the C ABI");

extern "C" {

int alibi_version(void) { return 100; }

const char *alibi_status_str(int status)
{
    switch (status) {
        case ALIBI_OK: return "ALIBI_OK";
        case ALIBI_ERR_INVALID: return "ALIBI_ERR_INVALID: invalid argument";
        case ALIBI_ERR_UNSUPPORTED: return "ALIBI_ERR_UNSUPPORTED: unsupported shape or option";
        case ALIBI_ERR_CUDA: return "ALIBI_ERR_CUDA: CUDA call or kernel launch failed";
        case ALIBI_ERR_TIMEOUT: return "ALIBI_ERR_TIMEOUT: a bounded device-side wait expired";
        case ALIBI_ERR_CHECK: return "ALIBI_ERR_CHECK: a debug-build address check failed";
        default: return "unknown alibi status";
    }
}

int alibi_slopes(int H, float *out_host)
{
    if (!out_host || H < 1 || H > 4096) return ALIBI_ERR_INVALID;
    for (int h = 0; h < H; ++h) {
        int num, den;
        slope_exponent(H, h, &num, &den);
        out_host[h] = slope_value(num, den);
    }
    return ALIBI_OK;
}

int alibi_slopes_explicit(int H, double delta_first, double delta_last, double tau, int log_distance,
                          float *out_host)
{
    if (!out_host || H < 1 || H > 4096 || (log_distance != 0 && log_distance != 1)) return ALIBI_ERR_INVALID;
    if (!(delta_first > 0.0) || !(delta_last > 0.0) || !(tau < 0.0)) return ALIBI_ERR_INVALID;
    if (!std::isfinite(delta_first) || !std::isfinite(delta_last) || !std::isfinite(tau)) return ALIBI_ERR_INVALID;
    // geometric targets in log space: ln delta_h = ln delta_first + (h / (H - 1)) ln(delta_last / delta_first)
    const double l0 = std::log(delta_first), span = std::log(delta_last) - l0;
    for (int h = 0; h < H; ++h) {
        const double delta = H > 1 ? std::exp(l0 + span * h / (H - 1)) : delta_first;
        // slope whose zero-logit bias reaches tau exactly at the target distance
        const double dist = log_distance ? std::log1p(delta) : delta;
        out_host[h] = static_cast<float>(-tau / dist);
    }
    return ALIBI_OK;
}

static int check_dims(int B, int H, int N, int d)
{
    if (B < 1 || H < 1 || N < 1 || d < 1) return ALIBI_ERR_INVALID;
    if (H > kMaxHeads) return ALIBI_ERR_UNSUPPORTED;
    // flat indices stay below 2^31 rows per (b, h) and 2^24 positions (exact in fp32)
    if (N > (1 << 24) || static_cast<long long>(B) * H > (1LL << 31) - 1) return ALIBI_ERR_UNSUPPORTED;
    // prefill work items and 256-key blocks of every (b, h) are counted in int
    if (static_cast<long long>(B) * H * ((N + 255) / 256) > (1LL << 31) - 1) return ALIBI_ERR_UNSUPPORTED;
    return ALIBI_OK;
}

int alibi_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int N, int d,
                   int causal, void *stream)
{
    return alibi_attn_fwd_ex(q, k, v, out, lse, B, H, N, d, causal, nullptr, stream);
}

// Caller-chosen slopes must be finite and non-negative (a zero slope is plain
// attention; a negative one would reward distance).
static bool slopes_ok(int H, const float *m)
{
    for (int h = 0; h < H; ++h)
        if (!std::isfinite(m[h]) || m[h] < 0.0f) return false;
    return true;
}

int alibi_attn_fwd_ex(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int N,
                      int d, int causal, const alibi_fwd_options *opt, void *stream)
{
    const alibi_fwd_options none = {0u, 0.0f, 0.0f, nullptr};
    if (!opt) opt = &none;
    const unsigned int flags = opt->flags;
    const float clamp_min = opt->clamp_min, softcap_z = opt->softcap_z;
    if (!q || !k || !v || !out) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (lse && !aligned16(lse)))
        return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, N, d);
    if (st != ALIBI_OK) return st;
    if (causal != 0 && causal != 1) return ALIBI_ERR_INVALID;
    if (d != 16 && d != 32 && d != 64 && d != 128) return ALIBI_ERR_UNSUPPORTED;
    const unsigned int known =
        ALIBI_FWD_SKIP_UNDERFLOW | ALIBI_FWD_CLAMP | ALIBI_FWD_LOGDIST | ALIBI_FWD_SOFTCAP | ALIBI_FWD_NOMINAL_ORDER;
    if (flags & ~known) return ALIBI_ERR_INVALID;
    if ((flags & ALIBI_FWD_CLAMP) && !(clamp_min < 0.0f)) return ALIBI_ERR_INVALID;
    if ((flags & ALIBI_FWD_SOFTCAP) && !(softcap_z > 0.0f && std::isfinite(softcap_z))) return ALIBI_ERR_INVALID;
    if ((flags & ALIBI_FWD_SKIP_UNDERFLOW) && (flags & (ALIBI_FWD_CLAMP | ALIBI_FWD_LOGDIST | ALIBI_FWD_SOFTCAP)))
        return ALIBI_ERR_INVALID;
    // the skip bound follows the causal range (tiles left of the diagonal)
    if ((flags & ALIBI_FWD_SKIP_UNDERFLOW) && !causal) return ALIBI_ERR_UNSUPPORTED;
    if (opt->slopes && !slopes_ok(H, opt->slopes)) return ALIBI_ERR_INVALID;
    Slopes s;
    if (opt->slopes)
        fill_slopes_from(H, opt->slopes, &s);
    else
        fill_slopes(H, &s);
    return to_status(launch_fwd_tc(q, k, v, out, lse, B, H, N, d, causal, flags, clamp_min, softcap_z, s,
                                   static_cast<cudaStream_t>(stream)));
}

int alibi_attn_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse, const void *dout,
                   void *dq, void *dk, void *dv, int B, int H, int N, int d, int causal, const alibi_fwd_options *opt,
                   void *stream)
{
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, N, d);
    if (st != ALIBI_OK) return st;
    if (causal != 0 && causal != 1) return ALIBI_ERR_INVALID;
    if (d != 64 && d != 128) return ALIBI_ERR_UNSUPPORTED;
    const alibi_fwd_options none = {0u, 0.0f, 0.0f, nullptr};
    if (!opt) opt = &none;
    const unsigned int mit = ALIBI_FWD_CLAMP | ALIBI_FWD_LOGDIST | ALIBI_FWD_SOFTCAP;
    // ALIBI_FWD_NOMINAL_ORDER keeps the nominal work order of the backward's kernels too
    if (opt->flags & ~(mit | ALIBI_FWD_SKIP_UNDERFLOW | ALIBI_FWD_NOMINAL_ORDER)) return ALIBI_ERR_INVALID;
    if (opt->flags & ALIBI_FWD_SKIP_UNDERFLOW) return ALIBI_ERR_UNSUPPORTED;
    if ((opt->flags & ALIBI_FWD_CLAMP) && !(opt->clamp_min < 0.0f)) return ALIBI_ERR_INVALID;
    if ((opt->flags & ALIBI_FWD_SOFTCAP) && !(opt->softcap_z > 0.0f && std::isfinite(opt->softcap_z)))
        return ALIBI_ERR_INVALID;
    if (opt->slopes && !slopes_ok(H, opt->slopes)) return ALIBI_ERR_INVALID;
    Slopes s;
    if (opt->slopes)
        fill_slopes_from(H, opt->slopes, &s);
    else
        fill_slopes(H, &s);
    return to_status(launch_bwd_tc(q, k, v, out, lse, dout, dq, dk, dv, B, H, N, d, causal, opt->flags,
                                   opt->clamp_min, opt->softcap_z, s, static_cast<cudaStream_t>(stream)));
}

int alibi_attn_bwd_f32(const float *q, const float *k, const float *v, const float *out, const float *lse,
                       const float *dout, float *dq, float *dk, float *dv, int B, int H, int N, int d, int causal,
                       void *stream)
{
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, N, d);
    if (st != ALIBI_OK) return st;
    if (causal != 0 && causal != 1) return ALIBI_ERR_INVALID;
    if (d > 256) return ALIBI_ERR_UNSUPPORTED;
    Slopes s;
    fill_slopes(H, &s);
    return to_status(launch_bwd_f32(q, k, v, out, lse, dout, dq, dk, dv, B, H, N, d, causal, s,
                                    static_cast<cudaStream_t>(stream)));
}

int alibi_attn_skip_plan(const void *q, const void *k, int B, int H, int N, int d, const float *slopes,
                         int *first_tile, void *stream)
{
    if (!q || !k || !first_tile) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(first_tile) & 3u)) return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, N, d);
    if (st != ALIBI_OK) return st;
    if (d != 16 && d != 32 && d != 64 && d != 128) return ALIBI_ERR_UNSUPPORTED;
    if (slopes && !slopes_ok(H, slopes)) return ALIBI_ERR_INVALID;
    Slopes s;
    if (slopes)
        fill_slopes_from(H, slopes, &s);
    else
        fill_slopes(H, &s);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int NQB = ((N + 127) / 128 + 1) / 2, items = B * H * NQB;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, skip_plan_bytes(B * H, N), decode_pool(), cs) != cudaSuccess)
        return ALIBI_ERR_CUDA;
    int2 *info = nullptr;
    cudaError_t e = launch_skip_plan(q, k, B, H, N, d, s, ws, nullptr, &info, cs);
    // first tiles are the .x fields of the int2 info records
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(first_tile, sizeof(int), info, sizeof(int2), sizeof(int), items,
                              cudaMemcpyDeviceToDevice, cs);
    const cudaError_t f = cudaFreeAsync(ws, cs);
    return to_status(e != cudaSuccess ? e : f);
}

int alibi_attn_fwd_f32(const float *q, const float *k, const float *v, float *out, float *lse, int B, int H, int N,
                       int d, int causal, void *stream)
{
    if (!q || !k || !v || !out) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (lse && !aligned16(lse)))
        return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, N, d);
    if (st != ALIBI_OK) return st;
    if (causal != 0 && causal != 1) return ALIBI_ERR_INVALID;
    if (d > 256) return ALIBI_ERR_UNSUPPORTED;
    Slopes s;
    fill_slopes(H, &s);
    return to_status(launch_fwd_f32(q, k, v, out, lse, B, H, N, d, causal, s, static_cast<cudaStream_t>(stream)));
}

int alibi_attn_decode(const void *q, const void *kcache, const void *vcache, void *out, int B, int H, int L, int d,
                      void *stream)
{
    if (!q || !kcache || !vcache || !out) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out)) return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, L, d);
    if (st != ALIBI_OK) return st;
    if (!decode_supports(d)) return ALIBI_ERR_UNSUPPORTED;
    Slopes s;
    fill_slopes(H, &s);
    return to_status(launch_decode(q, kcache, vcache, nullptr, out, B, H, L, d, s, static_cast<cudaStream_t>(stream)));
}

int alibi_kv_block_norms(const void *kcache, float *knorm, int B, int H, int L, int d, int blk_begin, void *stream)
{
    if (!kcache || !knorm) return ALIBI_ERR_INVALID;
    if (!aligned16(kcache) || (reinterpret_cast<uintptr_t>(knorm) & 3u)) return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, L, d);
    if (st != ALIBI_OK) return st;
    if (!decode_supports(d)) return ALIBI_ERR_UNSUPPORTED;
    if (blk_begin < 0 || blk_begin > (L + 63) / 64) return ALIBI_ERR_INVALID;
    return to_status(launch_kv_block_norms(kcache, knorm, B, H, L, d, blk_begin, static_cast<cudaStream_t>(stream)));
}

int alibi_attn_decode_skip(const void *q, const void *kcache, const void *vcache, const float *knorm, void *out, int B,
                           int H, int L, int d, void *stream)
{
    if (!q || !kcache || !vcache || !knorm || !out) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(knorm) & 3u))
        return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, L, d);
    if (st != ALIBI_OK) return st;
    if (!decode_supports(d)) return ALIBI_ERR_UNSUPPORTED;
    Slopes s;
    fill_slopes(H, &s);
    return to_status(launch_decode(q, kcache, vcache, knorm, out, B, H, L, d, s, static_cast<cudaStream_t>(stream)));
}

int alibi_attn_decode_splits(int B, int H, int L, int d)
{
    int st = check_dims(B, H, L, d);
    if (st != ALIBI_OK) return st;
    if (!decode_supports(d)) return ALIBI_ERR_UNSUPPORTED;
    return decode_splits(B * H, L);
}

int alibi_attn_probs_f32(const float *q, const float *k, const float *lse, float *P, int B, int H, int N, int d,
                         void *stream)
{
    return alibi_attn_probs_f32_ex(q, k, lse, P, B, H, N, d, 1, stream);
}

int alibi_attn_probs_f32_ex(const float *q, const float *k, const float *lse, float *P, int B, int H, int N, int d,
                            int causal, void *stream)
{
    if (!q || !k || !lse || !P) return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, N, d);
    if (st != ALIBI_OK) return st;
    if (causal != 0 && causal != 1) return ALIBI_ERR_INVALID;
    if (d > 256) return ALIBI_ERR_UNSUPPORTED;
    Slopes s;
    fill_slopes(H, &s);
    return to_status(launch_probs_f32(q, k, lse, P, B, H, N, d, causal, s, static_cast<cudaStream_t>(stream)));
}

int alibi_attn_underflow_bf16(const void *q, const void *k, int B, int H, int N, int d, float tau,
                              unsigned long long *counts, void *stream)
{
    if (!q || !k || !counts) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(counts) & 7u)) return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, N, d);
    if (st != ALIBI_OK) return st;
    if (d != 16 && d != 32 && d != 64 && d != 128) return ALIBI_ERR_UNSUPPORTED;
    if (!std::isfinite(tau)) return ALIBI_ERR_INVALID;
    Slopes s;
    fill_slopes(H, &s);
    return to_status(launch_underflow(q, k, B, H, N, d, tau, counts, s, static_cast<cudaStream_t>(stream)));
}

int alibi_decode_underflow_bf16(const void *q, const void *kcache, int B, int H, int L, int d, float tau,
                                unsigned long long *counts, void *stream)
{
    if (!q || !kcache || !counts) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(kcache) || (reinterpret_cast<uintptr_t>(counts) & 7u)) return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, L, d);
    if (st != ALIBI_OK) return st;
    if (d != 16 && d != 32 && d != 64 && d != 128) return ALIBI_ERR_UNSUPPORTED;
    if (!std::isfinite(tau)) return ALIBI_ERR_INVALID;
    Slopes s;
    fill_slopes(H, &s);
    return to_status(launch_decode_underflow(q, kcache, B, H, L, d, tau, counts, s, static_cast<cudaStream_t>(stream)));
}

int alibi_selftest_fwd_timeout(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                               int N, int d, int wait_us, void *stream)
{
    if (!q || !k || !v || !out) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (lse && !aligned16(lse)))
        return ALIBI_ERR_INVALID;
    int st = check_dims(B, H, N, d);
    if (st != ALIBI_OK) return st;
    if (d != 16 && d != 32 && d != 64 && d != 128) return ALIBI_ERR_UNSUPPORTED;
    if (wait_us < 1 || wait_us > 1000000) return ALIBI_ERR_INVALID;
    Slopes s;
    fill_slopes(H, &s);
    return to_status(launch_fwd_tc(q, k, v, out, lse, B, H, N, d, 1, 0u, 0.0f, 0.0f, s,
                                   static_cast<cudaStream_t>(stream), static_cast<uint64_t>(wait_us) * 1000u));
}

int alibi_selftest_timeout(void *stream)
{
    return to_status(launch_selftest_timeout(static_cast<cudaStream_t>(stream)));
}

int alibi_check_error(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ALIBI_ERR_CUDA;
    uint32_t *w = device_status_word();
    if (!w) return ALIBI_ERR_CUDA;
    uint32_t h[2] = {0, 0};
    if (cudaMemcpy(h, w, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ALIBI_ERR_CUDA;
    if (h[0] != 0u && cudaMemset(w, 0, sizeof(h)) != cudaSuccess) return ALIBI_ERR_CUDA;
    if (h[0] & ALIBI_DEV_CHECK) return ALIBI_ERR_CHECK;
    if (h[0] & ALIBI_DEV_TIMEOUT) return ALIBI_ERR_TIMEOUT;
    if (h[0] != 0u) return ALIBI_ERR_CUDA;
    return ALIBI_OK;
}

}  // extern "C"

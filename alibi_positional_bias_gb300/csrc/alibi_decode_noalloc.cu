// Decode for callers that cannot allocate device memory.
//
// alibi_attn_decode takes its split-K partials buffer from a stream-ordered
// memory pool when it splits the KV cache. Some callers cannot let a library
// allocate: a serving process whose own allocator has reserved the whole GPU
// up front (an extra driver allocation fails or fragments it), a real-time
// decode loop where the latency and possible synchronisation of an allocation
// are not allowed, or an embedding runtime that forbids device allocations
// outside its own arena. This entry point runs the same decode kernels with
// the partials in a fixed buffer compiled into the library, and allocates
// nothing itself.

#include <mutex>

#include "alibi.h"
#include "internal.h"

namespace alibi {
namespace {

// Fixed scratch for the split-K partials (4 MiB). Every GPU that loads the
// library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];
// Per-(b, h) split counters: zero when the library loads, and every call leaves
// them zero again (the CTA that merges a (b, h) resets its counter). 4 MiB of
// partials hold at most 26214 (b, h) pairs with two or more splits.
constexpr int kNoAllocCounters = 32768;
static __device__ unsigned g_noalloc_counters[kNoAllocCounters];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_scratch_addr[kMaxDevices] = {};
unsigned *g_counters_addr[kMaxDevices] = {};

// One-time set-up per device, with that device current: in host code the
// array's name is only a host-side stand-in, so the kernel must be given the
// device address the runtime reports for it.
cudaError_t scratch_address(float **addr, unsigned **counters)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr, *c = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        e = cudaGetSymbolAddress(&c, g_noalloc_counters);
        if (e != cudaSuccess) return e;
        g_counters_addr[dev] = static_cast<unsigned *>(c);
        g_scratch_addr[dev] = static_cast<float *>(p);
    }
    *addr = g_scratch_addr[dev];
    *counters = g_counters_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace alibi

using namespace alibi;

extern "C" int alibi_attn_decode_noalloc(const void *q, const void *kcache, const void *vcache, void *out, int B,
                                         int H, int L, int d, void *stream)
{
    if (!q || !kcache || !vcache || !out) return ALIBI_ERR_INVALID;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out)) return ALIBI_ERR_INVALID;
    if (B < 1 || H < 1 || L < 1 || d < 1) return ALIBI_ERR_INVALID;
    if (H > kMaxHeads || L > (1 << 24) || static_cast<long long>(B) * H > (1LL << 31) - 1)
        return ALIBI_ERR_UNSUPPORTED;
    if (!decode_supports(d)) return ALIBI_ERR_UNSUPPORTED;
    // same split plan as alibi_attn_decode, so both give the same result
    const int splits = decode_splits(B * H, L);
    if (decode_partials_bytes(B * H, splits, d) > kNoAllocScratchBytes) return ALIBI_ERR_UNSUPPORTED;
    if (splits > 1 && B * H > kNoAllocCounters) return ALIBI_ERR_UNSUPPORTED;
    float *scratch = nullptr;
    unsigned *counters = nullptr;
    if (scratch_address(&scratch, &counters) != cudaSuccess) return ALIBI_ERR_CUDA;
    Slopes s;
    fill_slopes(H, &s);
    // Every partial the merge reads is written earlier in the same call, so the
    // buffer needs no clearing; what the previous call left there is overwritten.
    // The counters are zero between calls (each call's merging CTAs reset theirs).
    const cudaError_t e = launch_decode_with(q, kcache, vcache, nullptr, out, B, H, L, d, s, splits,
                                             splits > 1 ? scratch : nullptr, splits > 1 ? counters : nullptr,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ALIBI_OK : ALIBI_ERR_CUDA;
}

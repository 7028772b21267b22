// Internal declarations shared by the host entry points and the kernel units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace alibi {

// Device status word bits (word 0) and the first failing site (word 1).
constexpr uint32_t ALIBI_DEV_TIMEOUT = 1u;
constexpr uint32_t ALIBI_DEV_BADSTATE = 2u;
constexpr uint32_t ALIBI_DEV_CHECK = 4u;  // a debug-checks build found a bad address (checks.h)

// Every device-side wait gives up after this long (ns).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Largest head count the kernels accept (slopes travel as kernel parameters).
constexpr int kMaxHeads = 256;

struct Slopes {
    float log2e[kMaxHeads];  // m_h * log2(e): the bias in base-2 exponent units
    float nat[kMaxHeads];    // m_h in natural-log units
};

// Host helpers (alibi_host.cu).
uint32_t *device_status_word();  // per current device, 2 words
void fill_slopes(int H, Slopes *s);
void fill_slopes_from(int H, const float *nat, Slopes *s);  // caller-chosen slopes (natural-log units)
int num_sms();                   // of the current device
int l2_bytes();                  // L2 size of the current device
// Blocked work order (work_order.h) of a dense launch over B*H heads of N rows,
// head size dr, causal or not: the prefill, or one of the backward's two kernels.
// A device table of (item, 0) entries cached per device and shape, or null for
// the nominal order (the streamed tiles fit in L2, the model prefers it, or the
// stream is being captured before the shape's table exists).
enum class OrderKind { Prefill = 0, BwdDkDv = 1, BwdDq = 2 };
const int2 *work_order(OrderKind kind, int causal, int BH, int N, int dr, cudaStream_t stream);
// Once per (current device, kernel): check that `func` compiled to `regs` registers
// per thread (0: any count) and raise its dynamic shared-memory limit to `smem`
// bytes. Function attributes belong to each device's context, so a process that
// runs on several devices prepares each one.
cudaError_t prepare_kernel(const void *func, int smem, uint32_t regs);
cudaMemPool_t decode_pool();     // library-owned stream-ordered pool of the current device
// 3-D TMA map over a [dim2, dim1, dim0] bf16 tensor (dim0 fastest), box {box0, box1, 1},
// zero fill out of bounds; 128-byte swizzle, or none (plain row-major boxes, as the
// epilogue's bulk stores use).
bool encode_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                         uint32_t box0, uint32_t box1, bool swizzle128 = true);

// Decode split plan (alibi_decode.cu): number of KV splits for B*H heads of length L.
int decode_splits(int BH, int L);
// Bytes of split-K partials the decode needs for that plan (0 when it does not split).
size_t decode_partials_bytes(int BH, int splits, int d);
// Bytes of per-(b, h) split counters for that plan (0 when it does not split).
size_t decode_counters_bytes(int BH, int splits);
// Head sizes the decode kernels are built for (16, 32, 64, 128).
bool decode_supports(int d);
// Launch the decode kernel with caller-provided partials and counters (used when
// splits > 1). The counters must be zero at launch; the kernel leaves them zero.
cudaError_t launch_decode_with(const void *q, const void *kc, const void *vc, const float *knorm, void *out, int B,
                               int H, int L, int d, const Slopes &slopes, int splits, float *partials,
                               unsigned *counters, cudaStream_t stream);
// Maximum key norm per 64-key block, blocks [blk_begin, ceil(L/64)) of every (b, h).
cudaError_t launch_kv_block_norms(const void *kc, float *knorm, int B, int H, int L, int d, int blk_begin,
                                  cudaStream_t stream);

// Prefill flags (the values of ALIBI_FWD_* in alibi.h).
constexpr unsigned int kFwdSkipUnderflow = 1u;
constexpr unsigned int kFwdClamp = 2u;
constexpr unsigned int kFwdLogDist = 4u;
constexpr unsigned int kFwdSoftcap = 8u;
constexpr unsigned int kFwdNominalOrder = 16u;

// Underflow-skip plan (alibi_skip.cu): scratch size for B*H heads of N rows, and the
// launch that fills it ([plan | info | key norms | per-row |q|^2 and q.k]).
size_t skip_plan_bytes(int BH, int N);
cudaError_t launch_skip_plan(const void *q, const void *k, int B, int H, int N, int d, const Slopes &slopes,
                             void *scratch, int2 **plan_out, int2 **info_out, cudaStream_t stream);

// Kernel launchers; each returns a cudaError_t from the launch.
cudaError_t launch_fwd_tc(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                          int N, int d, int causal, unsigned int flags, float clamp_min, float softcap_z, const Slopes &slopes,
                          cudaStream_t stream, uint64_t test_wait_ns = 0);
cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *out, float *lse, int B,
                           int H, int N, int d, int causal, const Slopes &slopes, cudaStream_t stream);
cudaError_t launch_probs_f32(const float *q, const float *k, const float *lse, float *P, int B, int H, int N,
                             int d, int causal, const Slopes &slopes, cudaStream_t stream);
cudaError_t launch_decode(const void *q, const void *kc, const void *vc, const float *knorm, void *out, int B, int H,
                          int L, int d, const Slopes &slopes, cudaStream_t stream);
cudaError_t launch_bwd_tc(const void *q, const void *k, const void *v, const void *out, const float *lse,
                          const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d, int causal,
                          unsigned int flags, float clamp_min, float softcap_z, const Slopes &slopes,
                          cudaStream_t stream);
cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *out, const float *lse,
                           const float *dout, float *dq, float *dk, float *dv, int B, int H, int N, int d, int causal,
                           const Slopes &slopes, cudaStream_t stream);
cudaError_t launch_selftest_timeout(cudaStream_t stream);
cudaError_t launch_underflow(const void *q, const void *k, int B, int H, int N, int d, float tau,
                             unsigned long long *counts, const Slopes &slopes, cudaStream_t stream);
cudaError_t launch_decode_underflow(const void *q, const void *kc, int B, int H, int L, int d, float tau,
                                    unsigned long long *counts, const Slopes &slopes, cudaStream_t stream);

}  // namespace alibi

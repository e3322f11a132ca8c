// common.cuh -- shared device helpers and the internal launcher interface of
// the ZETA library.  Nothing here is exported; the C ABI is include/zeta.h.
#pragma once

#include <atomic>
#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/zeta.h"

#define ZETA_API extern "C" __attribute__((visibility("default")))

namespace zeta {

constexpr int kMaxDK = 8;
constexpr int kMaxDV = 256;
constexpr int kMaxChunks = 1024;
constexpr unsigned kFull = 0xffffffffu;

// Validated view of a problem, with derived sizes in 64-bit.
struct Prob {
    int B, H, N, dK, dV, k, C, bits;
    int vdt;
    int64_t S;        // slices B*H
    int64_t n;        // chunks N / C
    int64_t T;        // prefix entries per slice
    int code64;       // 1 when d_K*bits > 32
    int wk;           // weight kernel (kWCauchy, kWSoftmax, kWInvEuclid)
};

// Launch set-up done once per device (for example cudaFuncSetAttribute, which
// applies to a function on the current device only): one bit per device id
// below 64 records that it ran; threads that race may both run it (the set-up
// calls used with it are idempotent).
struct PerDeviceOnce {
    std::atomic<uint64_t> done{0};
    template <typename Fn>
    cudaError_t run(Fn &&fn) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
        if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
        e = fn();
        if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
        return e;
    }
};

// A named NVTX range for the duration of one C-ABI call (host side: the
// checks and the launches it enqueues); a no-op when no tool is attached.
struct CallRange {
    explicit CallRange(const char *name);
    ~CallRange();
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

// Record the first device-side error in an optional status word.
__device__ __forceinline__ void set_status(int32_t *st, int code) {
    if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <typename T> struct VT;
template <> struct VT<float> {
    static __device__ __forceinline__ float ld(const float *p) { return *p; }
    static __device__ __forceinline__ void st(float *p, float x) { *p = x; }
};
template <> struct VT<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

// Cauchy weight 1 / (1 + d2 * inv_g2) in float32 with a correctly rounded
// reciprocal.
__device__ __forceinline__ float cauchy_w(float d2, float inv_g2) {
    return __frcp_rn(__fmaf_rn(d2, inv_g2, 1.0f));
}

// Weight kernels of the attended set (the low bits of zeta_problem_t.flags):
// the Cauchy softmax of the method, and the two kernels it is compared with in
// the OpenReview discussion, reply A3 "Justification for Euclidean Distance
// Claim": softmax of -d2 / gamma^2 (weights exp((m - d2) / gamma^2) with a
// per-query shift m = the smallest d2 of the attended set, which leaves the
// normalised weights unchanged) and inverse Euclidean 1 / sqrt(d2 + 1e-12).
constexpr int kWCauchy = 0, kWSoftmax = 1, kWInvEuclid = 2;
constexpr float kInvEps2 = 1e-12f;

template <int WK>
__device__ __forceinline__ float weight_of(float d2, float m, float inv_g2) {
    if constexpr (WK == kWSoftmax) return expf((m - d2) * inv_g2);
    else if constexpr (WK == kWInvEuclid) return __frsqrt_rn(d2 + kInvEps2);
    else return cauchy_w(d2, inv_g2);
}

// -dw/d(d2) as a function of the weight.
template <int WK>
__device__ __forceinline__ float neg_dw_dd2(float w, float inv_g2) {
    if constexpr (WK == kWSoftmax) return w * inv_g2;
    else if constexpr (WK == kWInvEuclid) return 0.5f * w * w * w;
    else return w * w * inv_g2;
}

// dw/dgamma (for the softmax with the shift held fixed; the shift's own
// derivative cancels in the normalised weights).
template <int WK>
__device__ __forceinline__ float dw_dgamma(float w, float d2, float m, float inv_g2, float inv_g) {
    if constexpr (WK == kWSoftmax) return 2.f * w * (d2 - m) * inv_g2 * inv_g;
    else if constexpr (WK == kWInvEuclid) return 0.f;
    else return 2.f * w * (1.f - w) * inv_g;
}

// ----------------------------------------------------------- launchers ---
// Each returns cudaGetLastError() after enqueueing on `st`.

cudaError_t launch_encode(const Prob &p, const float *x, void *codes, cudaStream_t st);

size_t sort_ws_bytes(const Prob &p);
cudaError_t launch_sort_chunks(const Prob &p, const void *key_codes, void *prefix_codes,
                               int32_t *prefix_idx, void *ws, cudaStream_t st);

cudaError_t launch_select(const Prob &p, const void *q_codes, const void *prefix_codes,
                          const int32_t *prefix_idx, int32_t *idx, cudaStream_t st);
cudaError_t launch_encode_curves(const Prob &p, const float *x, int curves, const int32_t *axes,
                                 void *codes, cudaStream_t st);
cudaError_t launch_select_curves(const Prob &p, int curves, const void *q_codes,
                                 const void *prefix_codes, const int32_t *prefix_idx,
                                 int32_t *idx, cudaStream_t st);

// Two-layer projection + encode on tcgen05 (F = 64, D % 64 == 0, H % 4 == 0).
bool project_tc_supported(const Prob &p, int D, int F);
cudaError_t launch_project_tc(const Prob &p, int D, const void *x, const void *w1,
                              const float *b1, const float *w2, const float *b2, float *q,
                              float *k, void *q_codes, void *k_codes, int32_t *status,
                              cudaStream_t st);

cudaError_t launch_attend_fwd(const Prob &p, const float *q, const float *k, const void *v,
                              const float *gamma, const int32_t *idx, void *out, float *rowsum,
                              int32_t *status, cudaStream_t st);

// The bounded mbarrier wait on a barrier that is (arrive != 0) or is not
// completed; a wait that gives up records ZETA_ERR_DEVICE_TIMEOUT.
cudaError_t launch_bounded_wait_check(uint32_t limit, int arrive, int32_t *status,
                                      cudaStream_t st);

// Select + attend in one call (fused kernel on the tensor-core shapes).
cudaError_t launch_select_attend_fwd(const Prob &p, const float *q, const float *k,
                                     const void *v, const float *gamma, const void *q_codes,
                                     const void *prefix_codes, const int32_t *prefix_idx,
                                     int32_t *idx, void *out, float *rowsum, int32_t *status,
                                     cudaStream_t st);

// Tensor-core forward for bf16 values, d_V = 64, d_K <= 4.
bool attend_fwd_tc_supported(const Prob &p);
cudaError_t launch_attend_fwd_tc(const Prob &p, const float *q, const float *k, const void *v,
                                 const float *gamma, const int32_t *idx, void *out,
                                 float *rowsum, int32_t *status, cudaStream_t st);

// Tensor-core backward kernels for bf16 values, d_V = 64, d_K <= 4.
bool attend_bwd_tc_supported(const Prob &p);
size_t bwd_tc_rec_bytes(const Prob &p);
cudaError_t launch_bwd_query_tc(const Prob &p, const float *q, const float *k, const void *v,
                                const float *gamma, const int32_t *idx, const void *dout,
                                float *dq, void *rec, float *dg_part, int32_t *status,
                                cudaStream_t st);
// csr_q holds the queries of every key's list (masked with csr_mask).
// csr_q: the sorted list words (packed (key << 16) | query, csr_k null) or the
// queries of the sorted (key, query) pairs with csr_k their keys; csr_mask
// takes the query out of a word.  off: per segment, the first list position of
// each key (kgs = 0, N + 1 entries) or of each 8-key group (kgs = 3, N / 8 + 1
// entries; C a multiple of 8).
// own_dv / own_dk: the own-chunk partial sums from launch_bwd_key_own_tc05, or
// null for the key kernel to compute its own-chunk block itself.
cudaError_t launch_bwd_key_tc(const Prob &p, const float *k, const void *v, const float *gamma,
                              const void *dout, const void *rec, const uint32_t *csr_q,
                              const uint32_t *csr_k, uint32_t csr_mask, int kgs,
                              const uint32_t *off, int64_t csr_stride,
                              float *dk, void *dv, const float *own_dv, const float *own_dk,
                              cudaStream_t st);
// The key side's own-chunk block on tcgen05 (C a multiple of 128, N of C;
// cudaErrorNotSupported when the driver offers no tensor-map encoder or k, v
// or dout is not 16-byte aligned):
// per key, dv (64 floats) and dk (4 floats) into own_dv / own_dk, without the
// Cauchy constant.
bool bwd_own_tc05_supported(const Prob &p);
cudaError_t launch_bwd_key_own_tc05(const Prob &p, const float *k, const void *v,
                                    const float *gamma, const void *dout, const void *rec,
                                    float *own_dv, float *own_dk, int32_t *status,
                                    cudaStream_t st);

size_t bwd_ws_bytes(const Prob &p);
cudaError_t launch_attend_bwd(const Prob &p, const float *q, const float *k, const void *v,
                              const float *gamma, const int32_t *idx, const void *dout, float *dq,
                              float *dk, void *dv, float *dgamma, void *ws, int32_t *status,
                              cudaStream_t st);

// Segmented stable LSD radix sort of (key, value) pairs, 8-bit digits.
// Slices of `len` items each, laid out `stride` apart.
struct RadixWs {
    void *keys[2];          // ping-pong key buffers, S * stride keys each
    uint32_t *vals[2];      // ping-pong value buffers
    uint32_t *hist;         // S * tiles * 256
    uint32_t *seglen;       // S, valid items per slice (filtered sources)
};

constexpr int kRadixThreads = 512;
constexpr int kRadixItems = 8;
constexpr int kRadixTile = kRadixThreads * kRadixItems;

inline int64_t radix_tiles(int64_t len) { return (len + kRadixTile - 1) / kRadixTile; }

// Sort codes (values = position in slice).  Result lands in keys[out_buf].
template <typename K>
cudaError_t radix_sort_codes(const K *codes, int64_t S, int64_t N, int key_bits, RadixWs &ws,
                             int *out_buf, cudaStream_t st);

// Sort the valid entries of an int32 index array [S][N*k] by index value,
// values = entry / k (the query i).  Entries equal to -1 are dropped; other
// entries outside [0, chunk start of i) are dropped and flagged in `status`.
// Per-slice counts land in ws.seglen.
cudaError_t radix_sort_idx(const int32_t *idx, int64_t S, int64_t N, int k, int C, RadixWs &ws,
                           int *out_buf, int32_t *status, cudaStream_t st);

// The same transpose for N <= 65536 with each entry packed as (key << 16) |
// query in one 32-bit word (keys only, no value array); sorted words land in
// ws.keys[*out_buf].  groups: ordered by key / 8 only (the entries of an
// 8-key group contiguous, in query order, their keys mixed).
cudaError_t radix_sort_idx_packed(const int32_t *idx, int64_t S, int64_t N, int k, int C,
                                  bool groups, RadixWs &ws, int *out_buf, int32_t *status,
                                  cudaStream_t st);

// Carve aligned sub-buffers out of a workspace.
struct Carver {
    char *base;
    size_t off = 0;
    explicit Carver(void *b) : base(static_cast<char *>(b)) {}
    template <typename T> T *take(size_t count) {
        off = (off + 255) & ~size_t(255);
        T *r = reinterpret_cast<T *>(base ? base + off : nullptr);
        off += count * sizeof(T);
        return r;
    }
    size_t bytes() const { return (off + 255) & ~size_t(255); }
};

}  // namespace zeta

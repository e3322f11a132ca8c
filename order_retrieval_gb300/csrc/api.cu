// api.cu -- the exported C ABI (include/zeta.h): argument checks and dispatch.
//
// Every check runs on the host before any CUDA call, so an invalid request
// returns a status without touching the device (and works without a GPU).
#include <climits>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"

zeta::CallRange::CallRange(const char *name) { nvtxRangePushA(name); }
zeta::CallRange::~CallRange() { nvtxRangePop(); }

using zeta::Prob;

namespace {

// Structural checks shared by every call; fills the derived sizes.
zeta_status_t check_problem(const zeta_problem_t *pp, Prob *out) {
    if (!pp) return ZETA_ERR_INVALID_ARG;
    const zeta_problem_t &p = *pp;
    if (p.B < 0 || p.H < 0 || p.N < 0) return ZETA_ERR_INVALID_ARG;
    if (p.d_K < 1 || p.bits < 1 || p.C < 1 || p.k < 1 || p.d_V < 1) return ZETA_ERR_INVALID_ARG;
    if ((int64_t)p.d_K * p.bits > 64) return ZETA_ERR_INVALID_ARG;
    if (p.d_K > zeta::kMaxDK || p.bits > 24) return ZETA_ERR_UNSUPPORTED;
    if (p.d_V > zeta::kMaxDV) return ZETA_ERR_UNSUPPORTED;
    if (p.N % p.C != 0) return ZETA_ERR_INVALID_ARG;
    if (p.k > p.C) return ZETA_ERR_INVALID_ARG;
    if (p.v_dtype != ZETA_F32 && p.v_dtype != ZETA_BF16) return ZETA_ERR_INVALID_ARG;
    if ((p.flags & ~3u) != 0 || (p.flags & 3u) == 3u) return ZETA_ERR_UNSUPPORTED;
    const int64_t S = (int64_t)p.B * p.H;
    if (S > 65535) return ZETA_ERR_UNSUPPORTED;            // slices ride on gridDim.y
    if ((int64_t)p.N * p.k > INT32_MAX) return ZETA_ERR_UNSUPPORTED;
    Prob r;
    r.B = p.B; r.H = p.H; r.N = p.N; r.dK = p.d_K; r.dV = p.d_V; r.k = p.k; r.C = p.C;
    r.bits = p.bits; r.vdt = p.v_dtype;
    r.S = S;
    r.n = p.N / p.C;
    r.T = (int64_t)p.C * r.n * (r.n - 1) / 2;
    r.code64 = p.d_K * p.bits > 32;
    r.wk = (int)(p.flags & 3u);
    *out = r;
    return ZETA_OK;
}

bool empty(const Prob &p) { return p.S == 0 || p.N == 0; }

zeta_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? ZETA_OK : ZETA_ERR_CUDA; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

ZETA_API size_t zeta_code_bytes(const zeta_problem_t *p) {
    Prob pr;
    if (check_problem(p, &pr) != ZETA_OK) return 0;
    return pr.code64 ? 8 : 4;
}

ZETA_API int64_t zeta_prefix_entries(const zeta_problem_t *p) {
    Prob pr;
    if (check_problem(p, &pr) != ZETA_OK) return -1;
    return pr.T;
}

ZETA_API size_t zeta_sort_workspace_bytes(const zeta_problem_t *p) {
    Prob pr;
    if (check_problem(p, &pr) != ZETA_OK) return 0;
    return zeta::sort_ws_bytes(pr);
}

ZETA_API size_t zeta_bwd_workspace_bytes(const zeta_problem_t *p) {
    Prob pr;
    if (check_problem(p, &pr) != ZETA_OK) return 0;
    return zeta::bwd_ws_bytes(pr);
}

ZETA_API const char *zeta_status_string(zeta_status_t s) {
    switch (s) {
        case ZETA_OK: return "ZETA_OK";
        case ZETA_ERR_INVALID_ARG: return "ZETA_ERR_INVALID_ARG";
        case ZETA_ERR_UNSUPPORTED: return "ZETA_ERR_UNSUPPORTED";
        case ZETA_ERR_WORKSPACE: return "ZETA_ERR_WORKSPACE";
        case ZETA_ERR_CUDA: return "ZETA_ERR_CUDA";
        case ZETA_ERR_DEVICE_TIMEOUT: return "ZETA_ERR_DEVICE_TIMEOUT";
        case ZETA_ERR_BOUNDS: return "ZETA_ERR_BOUNDS";
    }
    return "ZETA_ERR_UNKNOWN";
}

ZETA_API zeta_status_t zeta_encode(const zeta_problem_t *p, const float *x, void *codes,
                                   cudaStream_t stream) {
    zeta::CallRange range_("zeta_encode");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (empty(pr)) return ZETA_OK;
    if (!x || !codes) return ZETA_ERR_INVALID_ARG;
    return from_cuda(zeta::launch_encode(pr, x, codes, stream));
}

ZETA_API zeta_status_t zeta_sort_chunks(const zeta_problem_t *p, const void *key_codes,
                                        void *prefix_codes, int32_t *prefix_idx, void *workspace,
                                        size_t ws_bytes, cudaStream_t stream) {
    zeta::CallRange range_("zeta_sort_chunks");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (pr.n > zeta::kMaxChunks) return ZETA_ERR_UNSUPPORTED;
    if (empty(pr) || pr.T == 0) return ZETA_OK;
    if (!key_codes || !prefix_codes || !prefix_idx) return ZETA_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < zeta::sort_ws_bytes(pr)) return ZETA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ZETA_ERR_WORKSPACE;
    return from_cuda(zeta::launch_sort_chunks(pr, key_codes, prefix_codes, prefix_idx, workspace,
                                              stream));
}

ZETA_API zeta_status_t zeta_select_topk(const zeta_problem_t *p, const void *q_codes,
                                        const void *prefix_codes, const int32_t *prefix_idx,
                                        int32_t *idx, cudaStream_t stream) {
    zeta::CallRange range_("zeta_select_topk");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (empty(pr)) return ZETA_OK;
    if (!q_codes || !idx) return ZETA_ERR_INVALID_ARG;
    if (pr.T > 0 && (!prefix_codes || !prefix_idx)) return ZETA_ERR_INVALID_ARG;
    return from_cuda(zeta::launch_select(pr, q_codes, prefix_codes, prefix_idx, idx, stream));
}

ZETA_API zeta_status_t zeta_encode_curves(const zeta_problem_t *p, const float *x,
                                          int32_t curves, const int32_t *axes, void *codes,
                                          cudaStream_t stream) {
    zeta::CallRange range_("zeta_encode_curves");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (curves < 1 || curves > 8 || !axes) return ZETA_ERR_INVALID_ARG;
    for (int m = 0; m < curves; ++m) {
        unsigned seen = 0;
        for (int d = 0; d < pr.dK; ++d) {
            const int32_t a = axes[m * pr.dK + d];
            if (a < 0 || a >= pr.dK || (seen >> a) & 1u) return ZETA_ERR_INVALID_ARG;
            seen |= 1u << a;
        }
    }
    if (empty(pr)) return ZETA_OK;
    if (!x || !codes) return ZETA_ERR_INVALID_ARG;
    return from_cuda(zeta::launch_encode_curves(pr, x, curves, axes, codes, stream));
}

ZETA_API zeta_status_t zeta_select_topk_curves(const zeta_problem_t *p, int32_t curves,
                                               const void *q_codes, const void *prefix_codes,
                                               const int32_t *prefix_idx, int32_t *idx,
                                               cudaStream_t stream) {
    zeta::CallRange range_("zeta_select_topk_curves");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (curves < 1 || curves > 8 || pr.k / curves < 1) return ZETA_ERR_INVALID_ARG;
    if (pr.k > 256) return ZETA_ERR_UNSUPPORTED;
    if (pr.S * curves > 65535) return ZETA_ERR_UNSUPPORTED;
    if (empty(pr)) return ZETA_OK;
    if (!q_codes || !idx) return ZETA_ERR_INVALID_ARG;
    if (pr.T > 0 && (!prefix_codes || !prefix_idx)) return ZETA_ERR_INVALID_ARG;
    return from_cuda(
        zeta::launch_select_curves(pr, curves, q_codes, prefix_codes, prefix_idx, idx, stream));
}

ZETA_API zeta_status_t zeta_project_encode(const zeta_problem_t *p, const zeta_proj_t *pj,
                                           const void *x, const void *w1, const float *b1,
                                           const float *w2, const float *b2, float *q, float *k,
                                           void *q_codes, void *k_codes, int32_t *dev_status,
                                           cudaStream_t stream) {
    zeta::CallRange range_("zeta_project_encode");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (!pj || pj->D < 1 || pj->F < 1) return ZETA_ERR_INVALID_ARG;
    if (empty(pr)) return ZETA_OK;
    if (!x || !w1 || !b1 || !w2 || !b2 || !q || !k || !q_codes || !k_codes)
        return ZETA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w1)) return ZETA_ERR_INVALID_ARG;
    if (!zeta::project_tc_supported(pr, pj->D, pj->F)) return ZETA_ERR_UNSUPPORTED;
    return from_cuda(zeta::launch_project_tc(pr, pj->D, x, w1, b1, w2, b2, q, k, q_codes,
                                             k_codes, dev_status, stream));
}

ZETA_API zeta_status_t zeta_attend_fwd(const zeta_problem_t *p, const float *q, const float *k,
                                       const void *v, const float *gamma, const int32_t *idx,
                                       void *out, float *rowsum, int32_t *dev_status,
                                       cudaStream_t stream) {
    zeta::CallRange range_("zeta_attend_fwd");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (empty(pr)) return ZETA_OK;
    if (!q || !k || !v || !gamma || !idx || !out || !rowsum) return ZETA_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(out)) return ZETA_ERR_INVALID_ARG;
    return from_cuda(
        zeta::launch_attend_fwd(pr, q, k, v, gamma, idx, out, rowsum, dev_status, stream));
}

ZETA_API zeta_status_t zeta_select_attend_fwd(const zeta_problem_t *p, const float *q,
                                              const float *k, const void *v, const float *gamma,
                                              const void *q_codes, const void *prefix_codes,
                                              const int32_t *prefix_idx, int32_t *idx, void *out,
                                              float *rowsum, int32_t *dev_status,
                                              cudaStream_t stream) {
    zeta::CallRange range_("zeta_select_attend_fwd");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (empty(pr)) return ZETA_OK;
    if (!q || !k || !v || !gamma || !q_codes || !idx || !out || !rowsum)
        return ZETA_ERR_INVALID_ARG;
    if (pr.T > 0 && (!prefix_codes || !prefix_idx)) return ZETA_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(out)) return ZETA_ERR_INVALID_ARG;
    return from_cuda(zeta::launch_select_attend_fwd(pr, q, k, v, gamma, q_codes, prefix_codes,
                                                    prefix_idx, idx, out, rowsum, dev_status,
                                                    stream));
}

ZETA_API zeta_status_t zeta_attend_bwd(const zeta_problem_t *p, const float *q, const float *k,
                                       const void *v, const float *gamma, const int32_t *idx,
                                       const void *dout, float *dq, float *dk, void *dv,
                                       float *dgamma, void *workspace, size_t ws_bytes,
                                       int32_t *dev_status, cudaStream_t stream) {
    zeta::CallRange range_("zeta_attend_bwd");
    Prob pr;
    zeta_status_t s = check_problem(p, &pr);
    if (s != ZETA_OK) return s;
    if (empty(pr)) {
        if (pr.H > 0 && !dgamma) return ZETA_ERR_INVALID_ARG;
        if (pr.H > 0) return from_cuda(cudaMemsetAsync(dgamma, 0, sizeof(float) * pr.H, stream));
        return ZETA_OK;
    }
    if (!q || !k || !v || !gamma || !idx || !dout || !dq || !dk || !dv || !dgamma)
        return ZETA_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(dout) || !aligned16(dv)) return ZETA_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < zeta::bwd_ws_bytes(pr)) return ZETA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ZETA_ERR_WORKSPACE;
    return from_cuda(zeta::launch_attend_bwd(pr, q, k, v, gamma, idx, dout, dq, dk, dv, dgamma,
                                             workspace, dev_status, stream));
}

ZETA_API zeta_status_t zeta_check_bounded_wait(uint32_t iterations, int32_t arrive,
                                               int32_t *dev_status, cudaStream_t stream) {
    zeta::CallRange range_("zeta_check_bounded_wait");
    if (!dev_status || iterations == 0) return ZETA_ERR_INVALID_ARG;
    return from_cuda(zeta::launch_bounded_wait_check(iterations, arrive, dev_status, stream));
}

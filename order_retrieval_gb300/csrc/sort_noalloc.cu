// sort_noalloc.cu -- zeta_sort_chunks for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc at the point where they need the sorted
// prefixes: code running inside a custom allocator or a memory-pool callback,
// plug-ins whose host framework owns every device allocation, or processes
// that must keep their device footprint fixed after start-up.  For them this
// entry point takes no workspace argument and allocates nothing: its scratch
// is one file-scope __device__ array of fixed size, which every GPU that loads
// this code holds until the process exits.
//
// Host code cannot use the array's name as a device address, so the address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) and cached.  The actual work is the ordinary zeta_sort_chunks call
// given that scratch.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;     // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_sort_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_sort_scratch on the current device (looked up once).
zeta_status_t scratch_on_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZETA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ZETA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_sort_scratch) != cudaSuccess || !p) return ZETA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return ZETA_OK;
}

}  // namespace

ZETA_API zeta_status_t zeta_sort_chunks_noalloc(const zeta_problem_t *p, const void *key_codes,
                                                void *prefix_codes, int32_t *prefix_idx,
                                                cudaStream_t stream) {
    zeta::CallRange range_("zeta_sort_chunks_noalloc");
    // Every check of zeta_sort_chunks first, with no workspace: that call
    // returns before launching anything, with ZETA_OK when there is nothing to
    // sort (an empty problem, or fewer than two chunks), its own error for an
    // invalid or unsupported problem, and ZETA_ERR_WORKSPACE when the problem
    // is valid and needs scratch.  Only then is the scratch size compared.
    const zeta_status_t pre =
        zeta_sort_chunks(p, key_codes, prefix_codes, prefix_idx, nullptr, 0, stream);
    if (pre != ZETA_ERR_WORKSPACE) return pre;
    if (zeta_sort_workspace_bytes(p) > kNoallocScratchBytes) return ZETA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const zeta_status_t s = scratch_on_current_device(&scratch);
    if (s != ZETA_OK) return s;
    return zeta_sort_chunks(p, key_codes, prefix_codes, prefix_idx, scratch,
                            kNoallocScratchBytes, stream);
}

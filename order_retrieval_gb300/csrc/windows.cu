// windows.cu -- the key side's lists of the backward, read off the windows
// themselves instead of sorting idx.
//
// Under the selection rule of "ZETA: Leveraging Z-order Curves for Efficient
// Top-k Attention" (OpenReview reply A3: binary search of the insertion
// position in the sorted prefix; reply A2 "Clarification": the window centred
// at that position), the window of query i in chunk c is one contiguous run of
// its prefix: positions [start_i, start_i + k) of prefix c.  The queries of
// chunk c that selected the key at position p are therefore those with
// start_i in (p - k, p], and once the chunk's queries are ordered by
// (start, index) they form one contiguous range of that order.
//
// win_build, one CTA per (chunk c >= 1, slice):
//   1. inv[c][j] = position of key j in prefix c, for every j < cC (a scatter
//      of the prefix's own permutation; the CTA reads back only its region);
//   2. start_i = inv[c][idx_i[0]] for the chunk's queries; the row's last entry
//      must be the prefix entry at start_i + k - 1 (else ZETA_ERR_INVALID_ARG
//      goes to the status word: the rows are not windows of this prefix);
//   3. the chunk's queries sorted by (start_i, i) in shared memory (bitonic),
//      written to ord[cC .. cC + C);
//   4. for every position p of prefix c, with cnt(x) = #{i : start_i <= x}:
//      lo = cnt(p - k), len = cnt(p) - lo, and the word (lo << 16) | len stored
//      for the key j at p in key-major order: word kmaj(j) + (c - chunk(j) - 1),
//      so a key's ranges over the later chunks are adjacent and the ranges of
//      adjacent keys follow each other (the table has T words, like a prefix
//      table).
// The backward's key kernel walks these ranges (chunk by chunk, each range in
// ord order), so every key's sums run in a fixed order.
#include "common.cuh"

namespace zeta {
namespace {

constexpr int kWinThreads = 512;

__device__ __forceinline__ int64_t prefix_off(int64_t C, int64_t c) { return C * c * (c - 1) / 2; }

// Number of sorted starts <= x (x may be negative).
__device__ __forceinline__ int count_le(const uint32_t *sst, int C, int64_t x) {
    if (x < 0) return 0;
    int lo = 0, hi = C;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)sst[mid] <= x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kWinThreads)
win_build(const int32_t *__restrict__ pidx, const int32_t *__restrict__ idx,
          int32_t *__restrict__ inv, int32_t *__restrict__ ord, uint32_t *__restrict__ rw,
          int32_t *status, int N, int C, int k, int n, int64_t T, int P) {
    extern __shared__ __align__(16) unsigned char win_smem[];
    uint64_t *key = reinterpret_cast<uint64_t *>(win_smem);          // P sort keys
    uint32_t *sst = reinterpret_cast<uint32_t *>(key + P);           // C sorted starts
    const int c = blockIdx.x + 1;
    const int64_t seg = blockIdx.y;
    const int64_t cC = (int64_t)c * C;
    const int32_t *pc = pidx + seg * T + prefix_off(C, c);
    int32_t *ic = inv + seg * T + prefix_off(C, c);
    // 1. inverse of prefix c's permutation
    for (int64_t p = threadIdx.x; p < cC; p += blockDim.x) {
        const int32_t j = pc[p];
        if (j >= 0 && j < cC) ic[j] = (int32_t)p;
    }
    __syncthreads();
    // 2. window starts of the chunk's queries, checked against the prefix
    for (int t = threadIdx.x; t < P; t += blockDim.x) {
        uint64_t kv = ~uint64_t(0);
        if (t < C) {
            const int64_t i = cC + t;
            const int32_t *row = idx + (seg * N + i) * (int64_t)k;
            const int32_t j0 = row[0];
            int64_t start = 0;
            bool ok = j0 >= 0 && j0 < cC;
            if (ok) {
                start = ic[j0];
                ok = start >= 0 && start + k <= cC && row[k - 1] == pc[start + k - 1];
            }
            if (!ok) {
                set_status(status, ZETA_ERR_INVALID_ARG);
                start = 0;
            }
            kv = ((uint64_t)start << 32) | (uint32_t)t;
        }
        key[t] = kv;
    }
    __syncthreads();
    // 3. bitonic sort of the P keys (padding sorts last)
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = threadIdx.x; t < P / 2; t += blockDim.x) {
                const int lo = 2 * stride * (t / stride) + (t % stride);
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const uint64_t a = key[lo], b = key[hi];
                if ((a > b) == up) {
                    key[lo] = b;
                    key[hi] = a;
                }
            }
            __syncthreads();
        }
    }
    int32_t *oc = ord + seg * N + cC;
    for (int r = threadIdx.x; r < C; r += blockDim.x) {
        const uint64_t kv = key[r];
        sst[r] = (uint32_t)(kv >> 32);
        oc[r] = (int32_t)(cC + (uint32_t)kv);
    }
    __syncthreads();
    // 4. the range of every position's key, four consecutive positions a thread
    uint32_t *rs = rw + seg * T;
    const int64_t nm1 = n - 1;
    for (int64_t p0 = 4 * (int64_t)threadIdx.x; p0 < cC; p0 += 4 * (int64_t)blockDim.x) {
        int hi = count_le(sst, C, p0);
        int lo = count_le(sst, C, p0 - k);
        for (int e = 0; e < 4 && p0 + e < cC; ++e) {
            const int64_t p = p0 + e;
            if (e > 0) {
                while (hi < C && (int64_t)sst[hi] <= p) ++hi;
                while (lo < C && (int64_t)sst[lo] <= p - k) ++lo;
            }
            const int32_t j = pc[p];
            if (j < 0 || j >= cC) continue;
            const int64_t cj = j / C;
            const int64_t kmaj = (int64_t)C * (cj * nm1 - cj * (cj - 1) / 2) +
                                 (j - cj * C) * (nm1 - cj);
            rs[kmaj + (c - cj - 1)] = ((uint32_t)lo << 16) | (uint32_t)(hi - lo);
        }
    }
}

}  // namespace

bool win_lists_supported(const Prob &p) { return p.C <= kWinMaxC && p.n >= 2; }

size_t win_ws_bytes(const Prob &p) {
    Carver cv(nullptr);
    cv.take<int32_t>(p.S * p.T);         // inv
    cv.take<int32_t>(p.S * p.N);         // ord
    cv.take<uint32_t>(p.S * p.T);        // range words
    return cv.bytes();
}

WinLists carve_win(const Prob &p, void *base) {
    Carver cv(base);
    WinLists w;
    w.inv = cv.take<int32_t>(p.S * p.T);
    w.ord = cv.take<int32_t>(p.S * p.N);
    w.rw = cv.take<uint32_t>(p.S * p.T);
    return w;
}

cudaError_t launch_win_build(const Prob &p, const int32_t *prefix_idx, const int32_t *idx,
                             const WinLists &w, int32_t *status, cudaStream_t st) {
    int P = 1;
    while (P < p.C) P <<= 1;
    const size_t smem = sizeof(uint64_t) * P + sizeof(uint32_t) * p.C;
    win_build<<<dim3((unsigned)(p.n - 1), (unsigned)p.S), kWinThreads, smem, st>>>(
        prefix_idx, idx, w.inv, w.ord, w.rw, status, p.N, p.C, p.k, (int)p.n, p.T, P);
    return cudaGetLastError();
}

}  // namespace zeta

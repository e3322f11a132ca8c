// radix.cu -- segmented, stable LSD radix sort of (key, value) pairs.
//
// The pages sort Z-order codes with "an efficiently implemented radix sorting
// operation" (OpenReview discussion of "ZETA: Leveraging Z-order Curves for
// Efficient Top-k Attention", reply A3 "Chunking ... & Where efficiency is
// coming from").  Here each (b, h) slice is one segment.  Every 8-bit digit pass
// is three launches with no inter-block waiting (reduce, then scan, then
// scatter), so nothing spins and the order is deterministic:
//   upsweep   per tile of 2048 items: digit histogram -> hist[seg][digit][tile]
//   scan      per segment: exclusive scan of hist in (digit, tile) order
//   downsweep per tile: stable rank of every item among equal digits (warp
//             match + per-warp counters), scatter to hist offset + rank.
#include "common.cuh"

namespace zeta {
namespace {

template <typename K>
struct CodesSrc {          // first pass over Z codes: value = position
    const K *codes;
    int64_t N;
    __device__ int64_t len(int64_t) const { return N; }
    __device__ bool load(int64_t seg, int64_t p, K &key, uint32_t &val, int32_t *) const {
        key = codes[seg * N + p];
        val = static_cast<uint32_t>(p);
        return true;
    }
};

template <typename K>
struct PairsSrc {          // later passes: ping-pong buffers
    const K *keys;
    const uint32_t *vals;
    int64_t stride;
    const uint32_t *seglen;
    __device__ int64_t len(int64_t seg) const { return seglen ? (int64_t)seglen[seg] : stride; }
    __device__ bool load(int64_t seg, int64_t p, K &key, uint32_t &val, int32_t *) const {
        key = keys[seg * stride + p];
        val = vals[seg * stride + p];
        return true;
    }
};

struct IdxSrc {            // window indices: key = selected key, value = query
    const int32_t *idx;
    int64_t N;
    int k;
    int C;
    __device__ int64_t len(int64_t) const { return N * k; }
    __device__ bool load(int64_t seg, int64_t p, uint32_t &key, uint32_t &val, int32_t *st) const {
        const int32_t j = idx[seg * N * k + p];
        if (j == -1) return false;
        const int32_t i = static_cast<int32_t>(p / k);
        if (j < 0 || j >= (i / C) * C) { set_status(st, ZETA_ERR_BOUNDS); return false; }
        key = static_cast<uint32_t>(j);
        val = static_cast<uint32_t>(i);
        return true;
    }
};

template <typename K, typename Src>
__global__ void __launch_bounds__(kRadixThreads)
radix_upsweep(Src src, int shift, uint32_t *__restrict__ hist, int64_t tiles, int32_t *status) {
    __shared__ uint32_t sh[256];
    const int64_t seg = blockIdx.y, tile = blockIdx.x;
    sh[threadIdx.x] = 0;
    __syncthreads();
    const int64_t len = src.len(seg);
    const int64_t base = tile * kRadixTile;
    for (int r = 0; r < kRadixItems; ++r) {
        int64_t p = base + r * kRadixThreads + threadIdx.x;
        if (p < len) {
            K key;
            uint32_t val;
            if (src.load(seg, p, key, val, status))
                atomicAdd(&sh[(unsigned)(key >> shift) & 255u], 1u);
        }
    }
    __syncthreads();
    hist[(seg * 256 + threadIdx.x) * tiles + tile] = sh[threadIdx.x];
}

// Exclusive scan of one segment's 256*tiles counters; total -> seglen[seg].
__global__ void __launch_bounds__(1024)
radix_scan(uint32_t *__restrict__ hist, int64_t tiles, uint32_t *seglen) {
    __shared__ uint32_t warp_sum[32];
    const int64_t L = 256 * tiles;
    uint32_t *h = hist + blockIdx.x * L;
    const int64_t per = (L + 1023) / 1024;
    const int64_t beg = threadIdx.x * per;
    const int64_t end = beg + per < L ? beg + per : L;
    uint32_t sum = 0;
    for (int64_t i = beg; i < end; ++i) sum += h[i];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t inc = sum;
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_sum[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        uint32_t x = warp_sum[lane], s = x;
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(kFull, s, o);
            if (lane >= o) s += y;
        }
        warp_sum[lane] = s - x;    // exclusive warp offsets
    }
    __syncthreads();
    uint32_t run = warp_sum[wid] + inc - sum;
    for (int64_t i = beg; i < end; ++i) {
        uint32_t t = h[i];
        h[i] = run;
        run += t;
    }
    if (threadIdx.x == 1023 && seglen) seglen[blockIdx.x] = run;
}

template <typename K, typename Src>
__global__ void __launch_bounds__(kRadixThreads)
radix_downsweep(Src src, int shift, const uint32_t *__restrict__ hist, int64_t tiles,
                K *__restrict__ keys_out, uint32_t *__restrict__ vals_out, int64_t out_stride) {
    constexpr int W = kRadixThreads / 32;
    __shared__ uint32_t soff[256];
    __shared__ uint16_t wcnt[W][256];
    const int64_t seg = blockIdx.y, tile = blockIdx.x;
    const int64_t len = src.len(seg);
    const int64_t base = tile * kRadixTile;
    if (base >= len) return;
    soff[threadIdx.x] = hist[(seg * 256 + threadIdx.x) * tiles + tile];
    for (int w = 0; w < W; ++w) wcnt[w][threadIdx.x] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned lt = lanemask_lt();
    K key[kRadixItems];
    uint32_t val[kRadixItems];
    int dig[kRadixItems];
    uint32_t rank[kRadixItems];
#pragma unroll
    for (int r = 0; r < kRadixItems; ++r) {
        const int64_t p = base + w * (32 * kRadixItems) + r * 32 + lane;
        bool ok = false;
        if (p < len) ok = src.load(seg, p, key[r], val[r], nullptr);
        dig[r] = ok ? (int)((unsigned)(key[r] >> shift) & 255u) : 256;
        const unsigned peers = __match_any_sync(kFull, dig[r]);
        uint32_t cur = 0;
        if (ok) cur = wcnt[w][dig[r]];
        __syncwarp();
        if (ok) {
            rank[r] = cur + __popc(peers & lt);
            if ((peers & lt) == 0) wcnt[w][dig[r]] = (uint16_t)(cur + __popc(peers));
        }
        __syncwarp();
    }
    __syncthreads();
    {
        uint32_t run = 0;
        for (int ww = 0; ww < W; ++ww) {
            uint32_t c = wcnt[ww][threadIdx.x];
            wcnt[ww][threadIdx.x] = (uint16_t)run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRadixItems; ++r) {
        if (dig[r] < 256) {
            const int64_t dst = (int64_t)soff[dig[r]] + wcnt[w][dig[r]] + rank[r];
            keys_out[seg * out_stride + dst] = key[r];
            vals_out[seg * out_stride + dst] = val[r];
        }
    }
}

template <typename K, typename Src>
cudaError_t run_pass(const Src &src, int shift, int64_t S, int64_t maxlen, RadixWs &ws, int nxt,
                     int64_t out_stride, uint32_t *seglen_out, int32_t *status, cudaStream_t st) {
    const int64_t tiles = radix_tiles(maxlen);
    dim3 grid((unsigned)tiles, (unsigned)S);
    radix_upsweep<K, Src><<<grid, kRadixThreads, 0, st>>>(src, shift, ws.hist, tiles, status);
    radix_scan<<<(unsigned)S, 1024, 0, st>>>(ws.hist, tiles, seglen_out);
    radix_downsweep<K, Src><<<grid, kRadixThreads, 0, st>>>(
        src, shift, ws.hist, tiles, static_cast<K *>(ws.keys[nxt]), ws.vals[nxt], out_stride);
    return cudaGetLastError();
}

}  // namespace

template <typename K>
cudaError_t radix_sort_codes(const K *codes, int64_t S, int64_t N, int key_bits, RadixWs &ws,
                             int *out_buf, cudaStream_t st) {
    int passes = (key_bits + 7) / 8;
    if (passes < 1) passes = 1;
    int cur = -1;
    for (int ps = 0; ps < passes; ++ps) {
        const int nxt = cur == 0 ? 1 : 0;
        cudaError_t e;
        if (ps == 0)
            e = run_pass<K>(CodesSrc<K>{codes, N}, 0, S, N, ws, nxt, N, nullptr, nullptr, st);
        else
            e = run_pass<K>(PairsSrc<K>{static_cast<const K *>(ws.keys[cur]), ws.vals[cur], N, nullptr},
                            8 * ps, S, N, ws, nxt, N, nullptr, nullptr, st);
        if (e != cudaSuccess) return e;
        cur = nxt;
    }
    *out_buf = cur;
    return cudaSuccess;
}

template cudaError_t radix_sort_codes<uint32_t>(const uint32_t *, int64_t, int64_t, int, RadixWs &,
                                                int *, cudaStream_t);
template cudaError_t radix_sort_codes<uint64_t>(const uint64_t *, int64_t, int64_t, int, RadixWs &,
                                                int *, cudaStream_t);

cudaError_t radix_sort_idx(const int32_t *idx, int64_t S, int64_t N, int k, int C, RadixWs &ws,
                           int *out_buf, int32_t *status, cudaStream_t st) {
    int key_bits = 0;
    while (key_bits < 32 && (int64_t(1) << key_bits) < N) ++key_bits;
    int passes = (key_bits + 7) / 8;
    if (passes < 1) passes = 1;
    const int64_t L = N * (int64_t)k;
    int cur = -1;
    for (int ps = 0; ps < passes; ++ps) {
        const int nxt = cur == 0 ? 1 : 0;
        cudaError_t e;
        if (ps == 0)
            e = run_pass<uint32_t>(IdxSrc{idx, N, k, C}, 0, S, L, ws, nxt, L, ws.seglen, status, st);
        else
            e = run_pass<uint32_t>(
                PairsSrc<uint32_t>{static_cast<const uint32_t *>(ws.keys[cur]), ws.vals[cur], L,
                                   ws.seglen},
                8 * ps, S, L, ws, nxt, L, nullptr, nullptr, st);
        if (e != cudaSuccess) return e;
        cur = nxt;
    }
    *out_buf = cur;
    return cudaSuccess;
}

}  // namespace zeta

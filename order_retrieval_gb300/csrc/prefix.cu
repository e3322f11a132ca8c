// prefix.cu -- sorted causal prefixes and the top-k window select.
//
// Passages (OpenReview discussion of "ZETA: Leveraging Z-order Curves for
// Efficient Top-k Attention"): reply A3 "Chunking ... & Where efficiency is
// coming from" (radix sort of the Z codes, binary search of the query's
// insertion position) and reply A2 "Clarification" (the window centred at the
// insertion position holds the nearest neighbours); atlas.scime.ai summary,
// "Approach" (keys are sorted and chunked so that every query searches its
// causal past in parallel).
//
// Prefix build.  Prefix c is the keys of chunks 0..c-1 in (code, index) order.
// All of them are produced at once from ONE sorted order of the whole slice:
// sort the slice by (code, index) (radix sort, values = token index), then
// prefix c is the stable filter "chunk(index) < c" of that order.  A tile of the
// sorted slice is read once and written into every prefix that contains it:
//   count   per tile: how many items of each chunk it holds -> cum[c] = #(< c)
//   base    per (slice, c): exclusive scan of cum over tiles
//   scatter per tile: for every c, warp ballots rank the qualifying items;
//           each warp store writes a contiguous run of prefix c.
// Reads are one pass over the sorted slice; writes are the table itself.
//
// Select.  One lane finds one query's upper bound (of its code in its chunk's
// prefix), then the warp copies the 32 windows with coalesced loads.  When a
// block's 256 queries lie in one chunk (C a multiple of 256), the search runs
// in two levels: the first code of every block of 2^fsh prefix entries is
// staged in shared memory and searched there, then the query's block in global
// memory (its probes after the first hit L1); otherwise one binary search over
// the prefix.  Both give the same upper bound.
#include "common.cuh"

namespace zeta {
namespace {

constexpr int kPT = 1024;           // items per prefix tile
constexpr int kPThreads = 256;
constexpr int kPItems = kPT / kPThreads;
constexpr int kPWarps = kPThreads / 32;

__global__ void __launch_bounds__(kPThreads)
prefix_count(const uint32_t *__restrict__ sidx, int64_t N, int C, int n, int64_t tiles,
             uint32_t *__restrict__ cnt) {
    __shared__ uint32_t h[kMaxChunks + 1];
    const int64_t seg = blockIdx.y, tile = blockIdx.x;
    for (int c = threadIdx.x; c <= n; c += kPThreads) h[c] = 0;
    __syncthreads();
    for (int r = 0; r < kPItems; ++r) {
        const int64_t p = tile * kPT + r * kPThreads + threadIdx.x;
        if (p < N) atomicAdd(&h[sidx[seg * N + p] / (uint32_t)C], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {           // exclusive scan over c = 0..n by one warp
        const int lane = threadIdx.x;
        const int per = (n + 1 + 31) / 32;
        const int beg = lane * per;
        uint32_t s = 0;
        for (int c = beg; c < beg + per && c <= n; ++c) s += h[c];
        uint32_t inc = s;
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += y;
        }
        uint32_t run = inc - s;
        for (int c = beg; c < beg + per && c <= n; ++c) {
            uint32_t t = h[c];
            h[c] = run;
            run += t;
        }
    }
    __syncthreads();
    uint32_t *out = cnt + (seg * tiles + tile) * (int64_t)(n + 1);
    for (int c = threadIdx.x; c <= n; c += kPThreads) out[c] = h[c];
}

// Exclusive scan over tiles for every c.  Block (32, 32): x = c, y = tile range.
__global__ void prefix_base(uint32_t *__restrict__ cnt, int n, int64_t tiles) {
    __shared__ uint32_t part[32][33];
    const int64_t seg = blockIdx.y;
    const int c = blockIdx.x * 32 + threadIdx.x;
    const int64_t per = (tiles + 31) / 32;
    const int64_t t0 = threadIdx.y * per;
    const int64_t t1 = t0 + per < tiles ? t0 + per : tiles;
    uint32_t *base = cnt + seg * tiles * (int64_t)(n + 1);
    uint32_t s = 0;
    if (c <= n)
        for (int64_t t = t0; t < t1; ++t) s += base[t * (n + 1) + c];
    part[threadIdx.y][threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.y == 0) {
        uint32_t run = 0;
        for (int y = 0; y < 32; ++y) {
            uint32_t x = part[y][threadIdx.x];
            part[y][threadIdx.x] = run;
            run += x;
        }
    }
    __syncthreads();
    uint32_t run = part[threadIdx.y][threadIdx.x];
    if (c <= n)
        for (int64_t t = t0; t < t1; ++t) {
            uint32_t x = base[t * (n + 1) + c];
            base[t * (n + 1) + c] = run;
            run += x;
        }
}

template <typename K>
__global__ void __launch_bounds__(kPThreads)
prefix_scatter(const K *__restrict__ skey, const uint32_t *__restrict__ sidx, int64_t N, int C,
               int n, int64_t tiles, int64_t T, const uint32_t *__restrict__ cnt,
               K *__restrict__ pcodes, int32_t *__restrict__ pidx) {
    __shared__ uint32_t tbase[kMaxChunks + 1];
    __shared__ uint32_t wh[kPWarps][kMaxChunks + 1];
    const int64_t seg = blockIdx.y, tile = blockIdx.x;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t *cb = cnt + (seg * tiles + tile) * (int64_t)(n + 1);
    for (int c = threadIdx.x; c <= n; c += kPThreads) {
        tbase[c] = cb[c];
        for (int ww = 0; ww < kPWarps; ++ww) wh[ww][c] = 0;
    }
    __syncthreads();
    K key[kPItems];
    int32_t idx[kPItems];
    int ch[kPItems];
    int minch = n;
#pragma unroll
    for (int r = 0; r < kPItems; ++r) {
        const int64_t p = tile * kPT + w * (32 * kPItems) + r * 32 + lane;
        if (p < N) {
            key[r] = skey[seg * N + p];
            idx[r] = (int32_t)sidx[seg * N + p];
            ch[r] = idx[r] / C;
            atomicAdd(&wh[w][ch[r]], 1u);
        } else {
            ch[r] = n;            // never qualifies
        }
        minch = min(minch, ch[r]);
    }
    __syncwarp();
    {   // per-warp exclusive scan over c: wh[w][c] = #items of this warp with chunk < c
        const int per = (n + 1 + 31) / 32;
        const int beg = lane * per;
        uint32_t s = 0;
        for (int c = beg; c < beg + per && c <= n; ++c) s += wh[w][c];
        uint32_t inc = s;
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += y;
        }
        uint32_t run = inc - s;
        for (int c = beg; c < beg + per && c <= n; ++c) {
            uint32_t t = wh[w][c];
            wh[w][c] = run;
            run += t;
        }
    }
    __syncthreads();
    for (int c = threadIdx.x; c <= n; c += kPThreads) {   // exclusive over warps
        uint32_t run = 0;
        for (int ww = 0; ww < kPWarps; ++ww) {
            uint32_t x = wh[ww][c];
            wh[ww][c] = run;
            run += x;
        }
    }
    __syncthreads();
    for (int o = 16; o > 0; o >>= 1) minch = min(minch, __shfl_xor_sync(kFull, minch, o));
    const unsigned lt = lanemask_lt();
    K *pc = pcodes + seg * T;
    int32_t *pi = pidx + seg * T;
    for (int c = minch + 1; c < n; ++c) {
        const int64_t off = (int64_t)C * c * (c - 1) / 2;
        uint32_t run = tbase[c] + wh[w][c];
#pragma unroll
        for (int r = 0; r < kPItems; ++r) {
            const bool q = ch[r] < c;
            const unsigned m = __ballot_sync(kFull, q);
            if (q) {
                const int64_t pos = off + run + __popc(m & lt);
                pc[pos] = key[r];
                pi[pos] = idx[r];
            }
            run += __popc(m);
        }
    }
}

constexpr int kSelThreads = 256;
constexpr int kSelFence = 2048;                            // fences per block, at most

template <typename K>
__global__ void __launch_bounds__(kSelThreads)
select_kernel(const K *__restrict__ qc, const K *__restrict__ pc,
              const int32_t *__restrict__ pidx, int32_t *__restrict__ out, int64_t S, int N,
              int C, int k, int64_t T, int fenced) {
    __shared__ K fence[kSelFence];
    const int64_t wpr = (N + 31) / 32;                    // warps per slice
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (fenced) {
        // all 256 queries of this block are in one chunk c (C % 256 == 0, N % 256 == 0)
        const int64_t gb = blockIdx.x * (int64_t)(kSelThreads / 32);
        const int64_t seg = gb / wpr;
        const int c = (int)((gb % wpr) * 32 / C);
        if (c >= 1) {
            const int M = c * C;
            const K *p = pc + seg * T + (int64_t)C * c * (c - 1) / 2;
            int fsh = 6;
            while ((M >> fsh) >= kSelFence) ++fsh;
            const int nf = (M + (1 << fsh) - 1) >> fsh;
            for (int f = threadIdx.x; f < nf; f += kSelThreads) fence[f] = p[(int64_t)f << fsh];
            __syncthreads();
            const int qb = (int)(gw % wpr) * 32;
            const K x = qc[seg * N + qb + lane];
            int lo = 0, hi = nf;                           // fences with code <= x
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (fence[mid] <= x) lo = mid + 1; else hi = mid;
            }
            int r = 0;
            if (lo > 0) {                                  // entry b0 <= x; later blocks > x
                const int b0 = (lo - 1) << fsh;
                int a = b0 + 1, b = min(M, b0 + (1 << fsh));
                while (a < b) {
                    const int mid = (a + b) >> 1;
                    if (p[mid] <= x) a = mid + 1; else b = mid;
                }
                r = a;
            }
            int start = r - (k + 1) / 2;
            start = start < 0 ? 0 : start;
            start = start > M - k ? M - k : start;
            // the warp copies its 32 windows: their rows are 32 k consecutive
            // words of idx, written in order; word f is entry f % k of query
            // f / k, whose window start comes from that query's lane
            const int32_t *pi = pidx + seg * T + (int64_t)C * c * (c - 1) / 2;
            int32_t *o = out + (seg * N + qb) * (int64_t)k;
            int qq = 0, t = lane;
            while (t >= k) { t -= k; ++qq; }
#pragma unroll 4
            for (int f = lane; f < 32 * k; f += 32) {
                const int s = __shfl_sync(kFull, start, qq);
                o[f] = pi[s + t];
                t += 32;
                while (t >= k) { t -= k; ++qq; }
            }
            return;
        }
        // chunk 0: falls through to the plain path (every row is -1)
    }
    if (gw >= S * wpr) return;                            // whole warp exits together
    const int64_t seg = gw / wpr;
    const int qb = (int)(gw % wpr) * 32;
    const int i = qb + lane;
    int start = -1;
    if (i < N) {
        const int c = i / C;
        if (c >= 1) {
            const int M = c * C;
            const K *p = pc + seg * T + (int64_t)C * c * (c - 1) / 2;
            const K x = qc[seg * N + i];
            int lo = 0, hi = M;                            // upper bound
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (p[mid] <= x) lo = mid + 1; else hi = mid;
            }
            start = lo - (k + 1) / 2;
            start = start < 0 ? 0 : start;
            start = start > M - k ? M - k : start;
        }
    }
    // the warp's windows as one run of last * k words (as in the fenced path;
    // here the queries may lie in different chunks, and chunk 0's rows are -1)
    const int last = min(32, N - qb);
    const int total = last * k;
    int32_t *o = out + (seg * N + qb) * (int64_t)k;
    int qq = 0, t = lane;
    while (t >= k) { t -= k; ++qq; }
    for (int f0 = 0; f0 < total; f0 += 32) {
        const int s = __shfl_sync(kFull, start, qq & 31);
        const int f = f0 + lane;
        if (f < total) {
            const int c2 = (qb + qq) / C;
            o[f] = s < 0 ? -1 : pidx[seg * T + (int64_t)C * c2 * (c2 - 1) / 2 + s + t];
        }
        t += 32;
        while (t >= k) { t -= k; ++qq; }
    }
}

}  // namespace

size_t sort_ws_bytes(const Prob &p) {
    Carver cv(nullptr);
    const size_t cb = p.code64 ? 8 : 4;
    const int64_t items = p.S * p.N;
    cv.take<char>(items * cb);
    cv.take<char>(items * cb);
    cv.take<uint32_t>(items);
    cv.take<uint32_t>(items);
    cv.take<uint32_t>(p.S * radix_tiles(p.N) * 256);
    cv.take<uint32_t>(p.S);
    const int64_t tiles2 = (p.N + kPT - 1) / kPT;
    cv.take<uint32_t>(p.S * tiles2 * (p.n + 1));
    return cv.bytes();
}

template <typename K>
static cudaError_t sort_impl(const Prob &p, const K *kc, K *pcodes, int32_t *pidx, void *ws,
                             cudaStream_t st) {
    Carver cv(ws);
    RadixWs rw;
    const int64_t items = p.S * p.N;
    rw.keys[0] = cv.take<K>(items);
    rw.keys[1] = cv.take<K>(items);
    rw.vals[0] = cv.take<uint32_t>(items);
    rw.vals[1] = cv.take<uint32_t>(items);
    rw.hist = cv.take<uint32_t>(p.S * radix_tiles(p.N) * 256);
    rw.seglen = cv.take<uint32_t>(p.S);
    const int64_t tiles2 = (p.N + kPT - 1) / kPT;
    uint32_t *cnt = cv.take<uint32_t>(p.S * tiles2 * (p.n + 1));
    if (p.n < 2) return cudaGetLastError();              // no prefix to build
    int ob = 0;
    cudaError_t e = radix_sort_codes<K>(kc, p.S, p.N, p.dK * p.bits, rw, &ob, st);
    if (e != cudaSuccess) return e;
    const K *skey = static_cast<const K *>(rw.keys[ob]);
    const uint32_t *sidx = rw.vals[ob];
    const int n = (int)p.n;
    prefix_count<<<dim3((unsigned)tiles2, (unsigned)p.S), kPThreads, 0, st>>>(sidx, p.N, p.C, n,
                                                                           tiles2, cnt);
    prefix_base<<<dim3((unsigned)((n + 1 + 31) / 32), (unsigned)p.S), dim3(32, 32), 0, st>>>(
        cnt, n, tiles2);
    prefix_scatter<K><<<dim3((unsigned)tiles2, (unsigned)p.S), kPThreads, 0, st>>>(
        skey, sidx, p.N, p.C, n, tiles2, p.T, cnt, pcodes, pidx);
    return cudaGetLastError();
}

cudaError_t launch_sort_chunks(const Prob &p, const void *key_codes, void *prefix_codes,
                               int32_t *prefix_idx, void *ws, cudaStream_t st) {
    if (p.code64)
        return sort_impl<uint64_t>(p, static_cast<const uint64_t *>(key_codes),
                                   static_cast<uint64_t *>(prefix_codes), prefix_idx, ws, st);
    return sort_impl<uint32_t>(p, static_cast<const uint32_t *>(key_codes),
                               static_cast<uint32_t *>(prefix_codes), prefix_idx, ws, st);
}

cudaError_t launch_select(const Prob &p, const void *q_codes, const void *prefix_codes,
                          const int32_t *prefix_idx, int32_t *idx, cudaStream_t st) {
    const int64_t warps = p.S * ((p.N + 31) / 32);
    const int threads = kSelThreads;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    // every block's 256 queries in one chunk of one slice: the two-level search
    const int fenced = (p.C % kSelThreads == 0 && p.N % kSelThreads == 0) ? 1 : 0;
    if (p.code64)
        select_kernel<uint64_t><<<(unsigned)blocks, threads, 0, st>>>(
            static_cast<const uint64_t *>(q_codes), static_cast<const uint64_t *>(prefix_codes),
            prefix_idx, idx, p.S, p.N, p.C, p.k, p.T, fenced);
    else
        select_kernel<uint32_t><<<(unsigned)blocks, threads, 0, st>>>(
            static_cast<const uint32_t *>(q_codes), static_cast<const uint32_t *>(prefix_codes),
            prefix_idx, idx, p.S, p.N, p.C, p.k, p.T, fenced);
    return cudaGetLastError();
}

}  // namespace zeta

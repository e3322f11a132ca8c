// radix.cu -- segmented, stable LSD radix sort of (key, value) pairs (8-bit
// digits; the transpose of idx can take a 5-bit digit for its first pass).
//
// The pages sort the Z-order codes with a radix sort (OpenReview discussion of
// "ZETA: Leveraging Z-order Curves for Efficient Top-k Attention", reply A3
// "Chunking ... & Where efficiency is coming from").  Here each (b, h) slice is
// one segment.  Every 8-bit digit pass
// is three launches with no inter-block waiting (reduce, then scan, then
// scatter), so nothing spins and the order is deterministic:
//   upsweep   per tile of 4096 items: digit histogram -> hist[seg][tile][digit]
//   scan      per segment: exclusive scan of hist in (digit, tile) order
//   downsweep per tile: stable rank of every item among equal digits (digit
//             groups from ballots + per-warp counters bumped by one lane per
//             group),
//             scatter to hist offset + rank.
#include "common.cuh"

namespace zeta {
namespace {

// Every source hands a thread the items p0, p0 + 32, ..., p0 + 32 (R - 1) of a
// segment (a warp reads 32 consecutive items per load), all loads issued before
// any is used; ok[r] is false past the segment's end and for skipped items.
template <int R, typename Src, typename K>
__device__ __forceinline__ void load_plain(const Src &s, int64_t seg, int64_t p0, int64_t len,
                                           K (&key)[R], uint32_t (&val)[R], bool (&ok)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t p = p0 + 32 * r;
        ok[r] = p < len;
        if (ok[r]) s.load1(seg, p, key[r], val[r]);
    }
}

template <typename K>
struct CodesSrc {          // first pass over Z codes: value = position
    static constexpr bool kHasVal = true;
    static constexpr int kDownBlocks = 2;   // CTAs per SM the downsweep is built for
    const K *codes;
    int64_t N;
    __device__ int64_t len(int64_t) const { return N; }
    __device__ void load1(int64_t seg, int64_t p, K &key, uint32_t &val) const {
        key = codes[seg * N + p];
        val = static_cast<uint32_t>(p);
    }
    template <int R>
    __device__ void load_run(int64_t seg, int64_t p0, int64_t len, K (&key)[R], uint32_t (&val)[R],
                             bool (&ok)[R], int32_t *) const {
        load_plain(*this, seg, p0, len, key, val, ok);
    }
};

template <typename K>
struct PairsSrc {          // later passes: ping-pong buffers
    static constexpr bool kHasVal = true;
    static constexpr int kDownBlocks = 2;   // CTAs per SM the downsweep is built for
    const K *keys;
    const uint32_t *vals;
    int64_t stride;
    const uint32_t *seglen;
    __device__ int64_t len(int64_t seg) const { return seglen ? (int64_t)seglen[seg] : stride; }
    __device__ void load1(int64_t seg, int64_t p, K &key, uint32_t &val) const {
        key = keys[seg * stride + p];
        val = vals[seg * stride + p];
    }
    template <int R>
    __device__ void load_run(int64_t seg, int64_t p0, int64_t len, K (&key)[R], uint32_t (&val)[R],
                             bool (&ok)[R], int32_t *) const {
        load_plain(*this, seg, p0, len, key, val, ok);
    }
};

// Query and chunk start of window slot p (p = i k + t): i = p / k and
// cC = C floor(i / C).  Below 2^24 the quotients come from a float reciprocal and
// one integer correction: p and i are exact in float, the product carries a
// relative error under 2^-23, so for d >= 2 the truncated estimate is within one
// of the quotient (for d = 1 the reciprocal and the product are exact); the
// remainder's sign and size then fix it.  Larger slots fall back to integer
// division.
struct SlotDiv {
    uint32_t k, C;
    float inv_k, inv_C;
    bool fast;                // N k <= 2^24
    uint32_t a32, b32;        // 32 = a32 k + b32
    static __device__ __forceinline__ uint32_t quot(uint32_t n, uint32_t d, float inv_d) {
        uint32_t q = __float2uint_rz(__uint2float_rn(n) * inv_d);
        const int64_t r = (int64_t)n - (int64_t)q * d;
        if (r < 0) --q;
        else if (r >= (int64_t)d) ++q;
        return q;
    }
    __device__ __forceinline__ void split(uint32_t p, uint32_t &i, uint32_t &cC) const {
        if (fast) {
            i = quot(p, k, inv_k);
            cC = quot(i, C, inv_C) * C;
        } else {
            i = p / k;
            cC = i - i % C;
        }
    }
};
inline SlotDiv slot_div(int64_t N, int k, int C) {
    return SlotDiv{(uint32_t)k, (uint32_t)C, 1.0f / (float)k, 1.0f / (float)C,
                   N * (int64_t)k <= (int64_t(1) << 24), 32u / (uint32_t)k, 32u % (uint32_t)k};
}

// Query and chunk start of the slots p0, p0 + 32, p0 + 64, ... of one thread:
// one division for the first, then each step adds 32 = a32 k + b32 to the
// remainder (one carry at most, as b32 < k) and moves the chunk start on by C
// while the query has passed the chunk's end (at most 33 queries per step).
struct SlotRun {
    uint32_t i, rem, cC;
    __device__ __forceinline__ SlotRun(const SlotDiv &dv, uint32_t p0) {
        dv.split(p0, i, cC);
        rem = p0 - i * dv.k;
    }
    __device__ __forceinline__ void next(const SlotDiv &dv) {
        i += dv.a32;
        rem += dv.b32;
        if (rem >= dv.k) {
            rem -= dv.k;
            ++i;
        }
        while (i >= cC + dv.C) cC += dv.C;
    }
};

struct IdxSrc {            // window indices: key = selected key, value = query
    static constexpr bool kHasVal = true;
    static constexpr int kDownBlocks = 2;   // CTAs per SM the downsweep is built for
    const int32_t *idx;
    int64_t N;
    int k;
    SlotDiv dv;
    __device__ int64_t len(int64_t) const { return N * k; }
    template <int R>
    __device__ void load_run(int64_t seg, int64_t p0, int64_t len, uint32_t (&key)[R],
                             uint32_t (&val)[R], bool (&ok)[R], int32_t *st) const {
        int32_t j[R];
#pragma unroll
        for (int r = 0; r < R; ++r) j[r] = p0 + 32 * r < len ? idx[seg * N * k + p0 + 32 * r] : -1;
        SlotRun sr(dv, static_cast<uint32_t>(p0));                                 // N*k < 2^31
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r > 0) sr.next(dv);
            ok[r] = j[r] != -1;
            if (ok[r] && static_cast<uint32_t>(j[r]) >= sr.cC) {
                set_status(st, ZETA_ERR_BOUNDS);
                ok[r] = false;
            }
            key[r] = static_cast<uint32_t>(j[r]);
            val[r] = sr.i;
        }
    }
};

// Window indices packed into one word, (key << 16) | query, when N <= 2^16:
// sorting the words on their top 16 bits is the stable transpose by key, and
// no separate value array moves.
struct PackedIdxSrc {
    static constexpr bool kHasVal = false;
    static constexpr int kDownBlocks = 3;   // CTAs per SM the downsweep is built for
    const int32_t *idx;
    int64_t N;
    int k;
    SlotDiv dv;
    __device__ int64_t len(int64_t) const { return N * k; }
    template <int R>
    __device__ void load_run(int64_t seg, int64_t p0, int64_t len, uint32_t (&key)[R],
                             uint32_t (&)[R], bool (&ok)[R], int32_t *st) const {
        int32_t j[R];
#pragma unroll
        for (int r = 0; r < R; ++r) j[r] = p0 + 32 * r < len ? idx[seg * N * k + p0 + 32 * r] : -1;
        SlotRun sr(dv, static_cast<uint32_t>(p0));
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r > 0) sr.next(dv);
            ok[r] = j[r] != -1;
            if (ok[r] && static_cast<uint32_t>(j[r]) >= sr.cC) {
                set_status(st, ZETA_ERR_BOUNDS);
                ok[r] = false;
            }
            key[r] = (static_cast<uint32_t>(j[r]) << 16) | sr.i;
        }
    }
};

struct PackedSrc {         // later passes over packed words
    static constexpr bool kHasVal = false;
    static constexpr int kDownBlocks = 3;   // CTAs per SM the downsweep is built for
    const uint32_t *keys;
    int64_t stride;
    const uint32_t *seglen;
    __device__ int64_t len(int64_t seg) const { return (int64_t)seglen[seg]; }
    __device__ void load1(int64_t seg, int64_t p, uint32_t &key, uint32_t &) const {
        key = keys[seg * stride + p];
    }
    template <int R>
    __device__ void load_run(int64_t seg, int64_t p0, int64_t len, uint32_t (&key)[R],
                             uint32_t (&val)[R], bool (&ok)[R], int32_t *) const {
        load_plain(*this, seg, p0, len, key, val, ok);
    }
};

template <typename K, typename Src, int DB>
__global__ void __launch_bounds__(kRadixThreads)
radix_upsweep(Src src, int shift, uint32_t *__restrict__ hist, int64_t tiles, int32_t *status) {
    constexpr unsigned kMask = (1u << DB) - 1u;
    __shared__ uint32_t sh[256];
    const int64_t seg = blockIdx.y, tile = blockIdx.x;
    if (threadIdx.x < 256) sh[threadIdx.x] = 0;
    __syncthreads();
    const int64_t len = src.len(seg);
    const int64_t base = tile * kRadixTile;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    K key[kRadixItems];
    uint32_t val[kRadixItems];
    bool ok[kRadixItems];
    src.load_run(seg, base + w * (32 * kRadixItems) + lane, len, key, val, ok, status);
#pragma unroll
    for (int r = 0; r < kRadixItems; ++r)
        if (ok[r]) atomicAdd(&sh[(unsigned)(key[r] >> shift) & kMask], 1u);
    __syncthreads();
    if (threadIdx.x < 256) hist[(seg * tiles + tile) * 256 + threadIdx.x] = sh[threadIdx.x];
}

// Exclusive scan of one segment's counters in (digit, tile) order, stored as
// hist[seg][tile][digit]; total -> seglen[seg].  1024 threads = 256 digits x 4
// tile ranges; every load row is one coalesced 1 KB line.
__global__ void __launch_bounds__(1024)
radix_scan(uint32_t *__restrict__ hist, int64_t tiles, uint32_t *seglen) {
    __shared__ uint32_t part[4][256];
    __shared__ uint32_t dsum[256];
    const int d = threadIdx.x & 255, qtr = threadIdx.x >> 8;
    uint32_t *h = hist + blockIdx.x * tiles * 256;
    const int64_t per = (tiles + 3) / 4;
    const int64_t t0 = qtr * per;
    const int64_t t1 = t0 + per < tiles ? t0 + per : tiles;
    uint32_t s = 0;
#pragma unroll 8
    for (int64_t t = t0; t < t1; ++t) s += h[t * 256 + d];
    part[qtr][d] = s;
    __syncthreads();
    if (threadIdx.x < 256) {
        const uint32_t tot = part[0][d] + part[1][d] + part[2][d] + part[3][d];
        // exclusive scan of the 256 digit totals by warps of 32 + a second level
        const int lane = d & 31, w = d >> 5;
        uint32_t inc = tot;
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += y;
        }
        dsum[d] = inc;                        // inclusive within the warp
        __syncwarp();
        (void)w;
    }
    __syncthreads();
    if (threadIdx.x == 0) {                   // carry across the 8 warps
        uint32_t carry = 0;
        for (int w = 0; w < 8; ++w) {
            const uint32_t last = dsum[w * 32 + 31];
            for (int l = 0; l < 32; ++l) dsum[w * 32 + l] += carry;
            carry += last;
        }
        if (seglen) seglen[blockIdx.x] = carry;
    }
    __syncthreads();
    const uint32_t tot_d = part[0][d] + part[1][d] + part[2][d] + part[3][d];
    uint32_t run = dsum[d] - tot_d;           // exclusive digit base
    for (int q = 0; q < qtr; ++q) run += part[q][d];
#pragma unroll 8
    for (int64_t t = t0; t < t1; ++t) {
        const uint32_t x = h[t * 256 + d];
        h[t * 256 + d] = run;
        run += x;
    }
}

// Shared memory of one downsweep tile: the tile's items staged in digit order.
template <typename K>
constexpr size_t downsweep_smem() {
    return sizeof(K) * kRadixTile + sizeof(uint32_t) * kRadixTile;
}

template <typename K, typename Src, int DB>
__global__ void __launch_bounds__(kRadixThreads, Src::kDownBlocks)
radix_downsweep(Src src, int shift, const uint32_t *__restrict__ hist, int64_t tiles,
                K *__restrict__ keys_out, uint32_t *__restrict__ vals_out, int64_t out_stride) {
    constexpr unsigned kMask = (1u << DB) - 1u;
    constexpr int W = kRadixThreads / 32;
    __shared__ uint32_t soff[256];          // global start of each digit's run of this tile
    __shared__ uint32_t tds[256];           // tile-local start of each digit
    __shared__ uint32_t wsum[8];
    __shared__ uint32_t s_total;            // items of this tile that are sorted
    __shared__ uint32_t wcnt[W][256];
    extern __shared__ __align__(16) unsigned char stage_raw[];
    K *skey = reinterpret_cast<K *>(stage_raw);
    uint32_t *sval = reinterpret_cast<uint32_t *>(stage_raw + sizeof(K) * kRadixTile);
    const int64_t seg = blockIdx.y, tile = blockIdx.x;
    const int64_t len = src.len(seg);
    const int64_t base = tile * kRadixTile;
    if (base >= len) return;
    if (threadIdx.x < 256) soff[threadIdx.x] = hist[(seg * tiles + tile) * 256 + threadIdx.x];
    for (int x = threadIdx.x; x < W * 256; x += kRadixThreads) (&wcnt[0][0])[x] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned lt = lanemask_lt();
    K key[kRadixItems];
    uint32_t val[kRadixItems];
    bool ok[kRadixItems];
    int dig[kRadixItems];
    uint32_t rank[kRadixItems];
    src.load_run(seg, base + w * (32 * kRadixItems) + lane, len, key, val, ok, nullptr);
#pragma unroll
    for (int r = 0; r < kRadixItems; ++r)
        dig[r] = ok[r] ? (int)((unsigned)(key[r] >> shift) & kMask) : 256;
#pragma unroll
    for (int r = 0; r < kRadixItems; ++r) {
        // lanes with this lane's digit: one ballot per digit bit (far
        // cheaper here than a warp match); the lowest lane of each group bumps
        // the warp's counter for that digit and hands the old count to its group
        // (a warp's atomics on one counter take effect in program order, so
        // items keep their order)
        unsigned peers = __ballot_sync(kFull, dig[r] < 256);
#pragma unroll
        for (int b = 0; b < DB; ++b) {
            const unsigned bal = __ballot_sync(kFull, (dig[r] >> b) & 1);
            peers &= ((dig[r] >> b) & 1) ? bal : ~bal;
        }
        const int leader = __ffs(peers) - 1;
        uint32_t old = 0;
        if (dig[r] < 256 && lane == leader) old = atomicAdd(&wcnt[w][dig[r]], __popc(peers));
        old = __shfl_sync(kFull, old, leader);
        rank[r] = old + __popc(peers & lt);
    }
    __syncthreads();
    if (threadIdx.x < 256) {                // per digit: warp offsets, then the tile total
        const int d = threadIdx.x;
        uint32_t run = 0;
        for (int ww = 0; ww < W; ++ww) {
            const uint32_t c = wcnt[ww][d];
            wcnt[ww][d] = run;
            run += c;
        }
        uint32_t inc = run;                 // exclusive scan of tile totals over digits
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) wsum[w] = inc;
        tds[d] = inc - run;
        if (d == 255) s_total = inc;        // inclusive within the last warp
    }
    __syncthreads();
    if (threadIdx.x < 256) {
        uint32_t carry = 0;
        for (int ww = 0; ww < (threadIdx.x >> 5); ++ww) carry += wsum[ww];
        tds[threadIdx.x] += carry;
        if (threadIdx.x == 255) s_total += carry;
    }
    __syncthreads();
    const uint32_t nvalid = s_total;
    // stage the items in digit order
#pragma unroll
    for (int r = 0; r < kRadixItems; ++r) {
        if (dig[r] < 256) {
            const uint32_t tp = tds[dig[r]] + wcnt[w][dig[r]] + rank[r];
            skey[tp] = key[r];
            if constexpr (Src::kHasVal) sval[tp] = val[r];
        }
    }
    __syncthreads();
    // write each digit's run of the tile contiguously
    for (uint32_t t = threadIdx.x; t < nvalid; t += kRadixThreads) {
        const K kk = skey[t];
        const int d = (int)((unsigned)(kk >> shift) & kMask);
        const int64_t dst = (int64_t)soff[d] + (t - tds[d]);
        keys_out[seg * out_stride + dst] = kk;
        if constexpr (Src::kHasVal) vals_out[seg * out_stride + dst] = sval[t];
    }
}

template <typename K, typename Src, int DB = 8>
cudaError_t run_pass(const Src &src, int shift, int64_t S, int64_t maxlen, RadixWs &ws, int nxt,
                     int64_t out_stride, uint32_t *seglen_out, int32_t *status, cudaStream_t st) {
    const int64_t tiles = radix_tiles(maxlen);
    dim3 grid((unsigned)tiles, (unsigned)S);
    radix_upsweep<K, Src, DB><<<grid, kRadixThreads, 0, st>>>(src, shift, ws.hist, tiles, status);
    radix_scan<<<(unsigned)S, 1024, 0, st>>>(ws.hist, tiles, seglen_out);
    static PerDeviceOnce smem_once;          // run once per device, outside any capture
    cudaError_t e = smem_once.run([] {
        return cudaFuncSetAttribute(radix_downsweep<K, Src, DB>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)downsweep_smem<K>());
    });
    if (e != cudaSuccess) return e;
    radix_downsweep<K, Src, DB><<<grid, kRadixThreads, downsweep_smem<K>(), st>>>(
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
            e = run_pass<uint32_t>(IdxSrc{idx, N, k, slot_div(N, k, C)}, 0, S, L, ws, nxt, L, ws.seglen, status, st);
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

cudaError_t radix_sort_idx_packed(const int32_t *idx, int64_t S, int64_t N, int k, int C,
                                  bool groups, RadixWs &ws, int *out_buf, int32_t *status,
                                  cudaStream_t st) {
    const int64_t L = N * (int64_t)k;
    // by key: bits 16-23 then 24-31 of the words; by 8-key group: bits 19-23
    // (a 5-bit digit) then 24-31
    cudaError_t e = groups
        ? run_pass<uint32_t, PackedIdxSrc, 5>(PackedIdxSrc{idx, N, k, slot_div(N, k, C)}, 19, S, L,
                                               ws, 0, L, ws.seglen, status, st)
        : run_pass<uint32_t>(PackedIdxSrc{idx, N, k, slot_div(N, k, C)}, 16, S, L, ws, 0, L,
                             ws.seglen, status, st);
    if (e != cudaSuccess) return e;
    e = run_pass<uint32_t>(PackedSrc{static_cast<const uint32_t *>(ws.keys[0]), L, ws.seglen}, 24,
                           S, L, ws, 1, L, nullptr, nullptr, st);
    if (e != cudaSuccess) return e;
    *out_buf = 1;
    return cudaSuccess;
}

}  // namespace zeta

// common.cuh -- device helpers shared by the compression kernels, and the
// host-side launch bookkeeping (error text, launch counting, event tracing).
//
// Floating point: every element-wise operation uses an explicit
// round-to-nearest intrinsic (__fadd_rn, __fmul_rn, ...), which the compiler
// never contracts into an FMA, and the library is also built with
// -fmad=false.  Results are therefore bit-reproducible and independent of
// launch shape.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gcsgd.h"

namespace gcsgd {

constexpr unsigned kFull = 0xffffffffu;

// |x| as an order-preserving key: for finite floats the unsigned order of
// these bit patterns is the order of |x|; +0 and -0 share key 0.
__device__ __forceinline__ uint32_t mag_key(float x) { return __float_as_uint(x) & 0x7fffffffu; }

// Entries DGC sends from a segment of n values: max(1, ceil(density*n)) in
// fp64, capped at n.  Host and device evaluate the same IEEE expression.
__host__ __device__ inline uint32_t dgc_k_of(double density, uint64_t n) {
    if (n == 0) return 0;
    double kd = ceil(density * (double)n);
    uint64_t k = kd < 1.0 ? 1 : (uint64_t)kd;
    if (k > n) k = n;
    return (uint32_t)k;
}

// Exclusive block-wide prefix sum of a 64-bit value (NT threads, NT a
// multiple of 32, at most 1024).  `scratch` holds NT/32 + 1 words of shared
// memory.  Returns the exclusive prefix; *total receives the block sum.
// Contains __syncthreads(): every thread of the block must call it.
template <int NT>
__device__ __forceinline__ uint64_t block_exclusive_scan(uint64_t x, uint64_t* scratch, uint64_t* total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t inc = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint64_t y = __shfl_up_sync(kFull, inc, d);
        if (lane >= d) inc += y;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        uint64_t w = lane < NW ? scratch[lane] : 0;
        uint64_t winc = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            uint64_t y = __shfl_up_sync(kFull, winc, d);
            if (lane >= d) winc += y;
        }
        if (lane < NW) scratch[lane] = winc - w;
        if (lane == NW - 1) scratch[NW] = winc;
    }
    __syncthreads();
    uint64_t res = scratch[warp] + inc - x;
    *total = scratch[NW];
    __syncthreads();
    return res;
}

// Result of a descending selection on 31-bit magnitude keys.
struct SelectResult {
    uint32_t thresh;   // key of the rank-th largest item
    uint32_t greater;  // items with key > thresh
    uint32_t ties;     // items with key == thresh to take (1 .. count(== thresh))
};

// Keys the selection keeps after its first digit (the first digit's bucket
// usually holds a small fraction of the items).
constexpr int kCandMax = 2048;

// Shared-memory scratch of radix_select_desc.
struct RadixSmem {
    uint32_t hist[2048];
    uint32_t cand[kCandMax];
    uint64_t scan[33];
    uint32_t sel[4];
};

// First digit of a key: bits [30:20] (exponent and three mantissa bits).
__device__ __forceinline__ void radix_hist_add(RadixSmem& rs, uint32_t key) { atomicAdd(&rs.hist[key >> 20], 1u); }

// hist[bin] += 1 for every lane with `hit`, lanes with the same bin summed
// first, so a warp issues one shared atomic per distinct bin (keys near a
// selection threshold crowd into a few bins).  Called by the whole warp.
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t bin, bool hit) {
    const unsigned m = __match_any_sync(0xffffffffu, hit ? bin : 0xffffffffu);
    if (hit && (threadIdx.x & 31) == (unsigned)__ffs(m) - 1u) atomicAdd(&hist[bin], (uint32_t)__popc(m));
}

template <int NT>
__device__ __forceinline__ void radix_hist_clear(RadixSmem& rs) {
    for (int b = threadIdx.x; b < 2048; b += NT) rs.hist[b] = 0;
}

// Histogram of digit (key >> shift) & (nb - 1) over the keys whose bits under
// pmask equal prefix.  GLOBAL (keys loaded from global memory, many of them
// near the threshold): eight loads in flight per thread and warp-aggregated
// adds; else four and plain shared atomics.  Ends synchronised.
template <int NT, bool GLOBAL, class Load>
__device__ void radix_count(RadixSmem& rs, Load load, uint64_t count, uint32_t pmask, uint32_t prefix, int shift,
                            int nb) {
    constexpr int LPT = GLOBAL ? 8 : 4;
    for (int b = threadIdx.x; b < nb; b += NT) rs.hist[b] = 0;
    __syncthreads();
    for (uint64_t base = 0; base < count; base += LPT * (uint64_t)NT) {
        uint32_t key[LPT];
        bool ok[LPT];
#pragma unroll
        for (int j = 0; j < LPT; ++j) {  // independent loads in flight
            const uint64_t i = base + (uint64_t)j * NT + threadIdx.x;
            key[j] = 0;
            ok[j] = (i < count) && load(i, &key[j]);
        }
#pragma unroll
        for (int j = 0; j < LPT; ++j) {
            const bool hit = ok[j] && (key[j] & pmask) == prefix;
            const uint32_t bin = (key[j] >> shift) & (uint32_t)(nb - 1);
            if (GLOBAL) hist_add_warp(rs.hist, bin, hit);
            else if (hit) atomicAdd(&rs.hist[bin], 1u);
        }
    }
    __syncthreads();
}

// The bucket holding the need-th largest item of the histogram rs.hist[0, nb)
// (counted from the top): *bucket, *above = items in higher buckets, *cnt =
// items in the bucket.  Every thread must call it; ends synchronised, with
// rs.hist intact.
template <int NT>
__device__ void radix_pick(RadixSmem& rs, int nb, uint32_t need, uint32_t* bucket, uint32_t* above, uint32_t* cnt) {
    static_assert(NT >= 32 && NT <= 512 && NT % 32 == 0, "2048 / NT buckets per thread, at least one");
    const int w = nb / NT;  // thread t owns buckets [hi - w, hi) counted from the top
    const int hi = nb - (int)threadIdx.x * w;
    uint32_t mine = 0;
    for (int b = hi - 1; b >= hi - w; --b) mine += rs.hist[b];
    uint64_t tot;
    uint32_t ab = (uint32_t)block_exclusive_scan<NT>(mine, rs.scan, &tot);
    for (int b = hi - 1; b >= hi - w; --b) {
        const uint32_t h = rs.hist[b];
        if (ab < need && need <= ab + h) {
            rs.sel[0] = (uint32_t)b;
            rs.sel[1] = ab;
            rs.sel[2] = h;
        }
        ab += h;
    }
    __syncthreads();
    *bucket = rs.sel[0];
    *above = rs.sel[1];
    *cnt = rs.sel[2];
    __syncthreads();
}

// The rank-th largest of `count` 31-bit keys (1 <= rank <= count), by radix
// digits [30:20], [19:9] and [8:0] with shared-memory histograms.  After the
// first digit the keys of the chosen bucket are copied to cbuf when they
// fit, so the later digits look at those few keys only.  `load(i, &key)`
// returns false for items to skip.  With hist_ready the caller has already
// added every key's first digit into rs.hist (radix_hist_clear, then
// radix_hist_add per key, then a barrier).  PASSES = 3 is exact; PASSES = 2
// returns the rank-th largest key with its low 9 bits cleared (greater and
// ties then refer to the truncated keys).  GLOBAL: `load` reads global
// memory (see radix_count).  cbuf/ccap: where the chosen bucket's keys are
// compacted (shared memory; default rs.cand, kCandMax keys).  Every thread
// must call it.
template <int NT, int PASSES, bool GLOBAL = false, class Load>
__device__ SelectResult radix_select_desc(Load load, uint64_t count, uint32_t rank, RadixSmem& rs, bool hist_ready,
                                          uint32_t* cbuf = nullptr, uint32_t ccap = 0) {
    if (!cbuf) {
        cbuf = rs.cand;
        ccap = kCandMax;
    }
    static_assert(PASSES == 2 || PASSES == 3, "two or three digits");
    constexpr int LPT = GLOBAL ? 8 : 4;
    const int lane = threadIdx.x & 31;
    if (!hist_ready) radix_count<NT, GLOBAL>(rs, load, count, 0u, 0u, 20, 2048);
    uint32_t b, ab, c1;
    radix_pick<NT>(rs, 2048, rank, &b, &ab, &c1);
    uint32_t prefix = b << 20, pmask = 0x7ffu << 20, need = rank - ab, greater = ab;
    const bool compact = c1 <= ccap;
    if (compact) {
        if (threadIdx.x == 0) rs.sel[3] = 0;
        __syncthreads();
        for (uint64_t base = 0; base < count; base += LPT * (uint64_t)NT) {
            uint32_t key[LPT];
            bool ok[LPT];
#pragma unroll
            for (int j = 0; j < LPT; ++j) {
                const uint64_t i = base + (uint64_t)j * NT + threadIdx.x;
                key[j] = 0;
                ok[j] = (i < count) && load(i, &key[j]);
            }
#pragma unroll
            for (int j = 0; j < LPT; ++j) {
                const bool hit = ok[j] && (key[j] & pmask) == prefix;
                const unsigned m = __ballot_sync(kFull, hit);
                if (m) {
                    uint32_t at = 0;
                    if (lane == 0) at = atomicAdd(&rs.sel[3], (uint32_t)__popc(m));
                    at = __shfl_sync(kFull, at, 0);
                    if (hit) cbuf[at + __popc(m & ((1u << lane) - 1u))] = key[j];
                }
            }
        }
        __syncthreads();
    }
    auto cand = [&](uint64_t i, uint32_t* key) { *key = cbuf[i]; return true; };
#pragma unroll 1
    for (int pass = 1; pass < PASSES; ++pass) {
        const int shift = pass == 1 ? 9 : 0;
        const int nb = pass == 1 ? 2048 : 512;
        if (compact) radix_count<NT, false>(rs, cand, c1, pmask, prefix, shift, nb);
        else radix_count<NT, GLOBAL>(rs, load, count, pmask, prefix, shift, nb);
        uint32_t cb;
        radix_pick<NT>(rs, nb, need, &b, &ab, &cb);
        prefix |= b << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        greater += ab;
        need -= ab;
    }
    SelectResult r;
    r.thresh = prefix;
    r.greater = greater;
    r.ties = need;
    return r;
}

// ------------------------------------------------ selection of a small top
//
// For a small rank (at most 48) among keys spread over the threads of a
// block: every lane keeps its three largest keys (top3_insert); three rounds
// of warp max give every warp's third-largest key; the smallest of those, L,
// is matched or exceeded by at least three keys of every warp that holds
// three keys, so at least 48 keys are >= L (or L = 0 and every key is).  The
// keys >= L, usually a few dozen, are appended to rs.cand (cand_append) and
// ranked exactly (rank_select).  No histogram is built: keys of similar
// magnitude crowd into a few radix bins, which serialises shared atomics.

// Inserts key into the lane's three largest (a multiset; 0 = empty).
__device__ __forceinline__ void top3_insert(uint32_t key, uint32_t& t1, uint32_t& t2, uint32_t& t3) {
    if (key > t3) {
        if (key > t2) {
            t3 = t2;
            if (key > t1) {
                t2 = t1;
                t1 = key;
            } else {
                t2 = key;
            }
        } else {
            t3 = key;
        }
    }
}

// L = the smallest of the warps' third-largest keys, on every thread; also
// empties rs.cand (rs.sel[3] = 0).  Every thread must call it.
template <int NT>
__device__ uint32_t top3_bound(uint32_t t1, uint32_t t2, uint32_t t3, RadixSmem& rs) {
    static_assert(NT / 32 <= 2048, "one word per warp");
    uint32_t w3 = 0;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        w3 = __reduce_max_sync(kFull, t1);
        const unsigned own = __ballot_sync(kFull, t1 == w3);
        if ((threadIdx.x & 31) == (unsigned)__ffs(own) - 1u) {
            t1 = t2;
            t2 = t3;
            t3 = 0;
        }
    }
    if ((threadIdx.x & 31) == 0) rs.hist[threadIdx.x >> 5] = w3;
    if (threadIdx.x == 0) rs.sel[3] = 0;
    __syncthreads();
    uint32_t L = 0xffffffffu;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) L = min(L, rs.hist[w]);
    __syncthreads();  // rs.hist is free again
    return L;
}

// Appends `key` to rs.cand where `hit` (slots past kCandMax are counted in
// rs.sel[3], not written).  The whole warp calls it.
__device__ __forceinline__ void cand_append(RadixSmem& rs, uint32_t key, bool hit) {
    const unsigned m = __ballot_sync(kFull, hit);
    if (m) {
        const int lane = threadIdx.x & 31;
        uint32_t at = 0;
        if (lane == 0) at = atomicAdd(&rs.sel[3], (uint32_t)__popc(m));
        at = __shfl_sync(kFull, at, 0);
        const uint32_t slot = at + __popc(m & ((1u << lane) - 1u));
        if (hit && slot < (uint32_t)kCandMax) rs.cand[slot] = key;
    }
}

// The rank-th largest (1 <= rank <= c) of the c <= NT keys in rs.cand,
// exactly: key j's rank is the keys above it plus the equal keys before it.
// Returns the key, how many keys are above it, and rank - that (the equal
// keys to take).  Every thread must call it.
template <int NT>
__device__ SelectResult rank_select(RadixSmem& rs, uint32_t c, uint32_t rank) {
    if (threadIdx.x < c) {
        const uint32_t mine = rs.cand[threadIdx.x];
        uint32_t above = 0, r = 0;
        for (uint32_t i = 0; i < c; ++i) {
            const uint32_t o = rs.cand[i];
            above += o > mine;
            r += o > mine || (o == mine && i < threadIdx.x);
        }
        if (r == rank - 1) {
            rs.sel[0] = mine;
            rs.sel[1] = above;
        }
    }
    __syncthreads();
    SelectResult res;
    res.thresh = rs.sel[0];
    res.greater = rs.sel[1];
    res.ties = rank - rs.sel[1];
    __syncthreads();
    return res;
}

// The rank-th largest of `count` keys that all lie in [base, base + 2^bits)
// (1 <= rank <= count, bits <= 31): the selection of radix_select_desc on
// d = key - base, with digits cut from the top of d's own bit range (11
// bits, then 11, then the rest).  Keys crowded into a narrow range -- the
// candidates above a threshold hint all share their leading bits -- then
// spread over the first histogram's bins instead of piling into a few,
// which would serialise the shared-memory atomics.  After the first digit
// the chosen bucket's keys are copied to cbuf (ccap keys) when they fit.
// `load(i, &key)` reads key i (every item counts).  Every thread must call
// it; ends synchronised.
template <int NT, class Load>
__device__ SelectResult radix_select_span(Load load, uint32_t count, uint32_t rank, uint32_t base, int bits,
                                          RadixSmem& rs, uint32_t* cbuf, uint32_t ccap) {
    static_assert(NT == 512, "radix_pick needs at least NT buckets: digits are padded to 512 bins");
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0, pmask = 0, need = rank, greater = 0;
    bool compact = false;
    uint32_t ncand = 0;
    int shift = bits;
#pragma unroll 1
    for (int pass = 0; shift > 0 || pass == 0; ++pass) {
        const int nshift = shift > 11 ? shift - 11 : 0;
        const uint32_t dmask = (1u << (shift - nshift)) - 1u;  // this digit's width
        const int nb = (int)(dmask + 1) > NT ? (int)(dmask + 1) : NT;
        for (int b = threadIdx.x; b < nb; b += NT) rs.hist[b] = 0;
        __syncthreads();
        const uint32_t n_it = compact ? ncand : count;
        for (uint32_t i0 = 0; i0 < n_it; i0 += 4u * NT) {
            uint32_t d[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t i = i0 + j * NT + threadIdx.x;
                d[j] = 0xffffffffu;
                if (i < n_it) {
                    if (compact) {
                        d[j] = cbuf[i];
                    } else {
                        uint32_t key;
                        load(i, &key);
                        d[j] = key - base;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (i0 + j * NT + threadIdx.x < n_it && (d[j] & pmask) == prefix)
                    atomicAdd(&rs.hist[(d[j] >> nshift) & dmask], 1u);
        }
        __syncthreads();
        uint32_t b, ab, cb;
        radix_pick<NT>(rs, nb, need, &b, &ab, &cb);
        prefix |= b << nshift;
        pmask |= dmask << nshift;
        greater += ab;
        need -= ab;
        if (pass == 0 && nshift > 0 && cb <= ccap) {  // keep the chosen bucket's keys for the later digits
            if (threadIdx.x == 0) rs.sel[3] = 0;
            __syncthreads();
            for (uint32_t i0 = 0; i0 < count; i0 += NT) {
                const uint32_t i = i0 + threadIdx.x;
                uint32_t dv = 0;
                bool hit = false;
                if (i < count) {
                    uint32_t key;
                    load(i, &key);
                    dv = key - base;
                    hit = (dv & pmask) == prefix;
                }
                const unsigned m = __ballot_sync(kFull, hit);
                if (m) {
                    uint32_t at = 0;
                    if (lane == 0) at = atomicAdd(&rs.sel[3], (uint32_t)__popc(m));
                    at = __shfl_sync(kFull, at, 0);
                    if (hit) cbuf[at + __popc(m & ((1u << lane) - 1u))] = dv;
                }
            }
            __syncthreads();
            ncand = rs.sel[3];
            compact = true;
            __syncthreads();
            if (ncand <= (uint32_t)NT) {
                // few keys left: rank them exactly instead of more digits.
                // Key j's rank: keys above it, plus equal keys before it.
                if (threadIdx.x < ncand) {
                    const uint32_t mine = cbuf[threadIdx.x];
                    uint32_t above = 0, rank = 0;
                    for (uint32_t i = 0; i < ncand; ++i) {
                        const uint32_t o = cbuf[i];
                        above += o > mine;
                        rank += o > mine || (o == mine && i < threadIdx.x);
                    }
                    if (rank == need - 1) {
                        rs.sel[0] = mine;
                        rs.sel[1] = above;
                    }
                }
                __syncthreads();
                SelectResult r;
                r.thresh = base + rs.sel[0];
                r.greater = greater + rs.sel[1];
                r.ties = need - rs.sel[1];
                __syncthreads();
                return r;
            }
        }
        shift = nshift;
    }
    SelectResult r;
    r.thresh = base + prefix;
    r.greater = greater;
    r.ties = need;
    return r;
}

// ---------------------------------------------------------------- host side

// Records the last error of the calling thread; returns `code`.
int set_error(int code, const char* fmt, ...);

// Launch bookkeeping: counts every kernel launch and, when tracing is on,
// records CUDA events around it on its stream.
struct LaunchScope {
    const char* name;
    cudaStream_t stream;
    int slot;
    LaunchScope(const char* name, cudaStream_t s);
    ~LaunchScope();
};

// Checks cudaGetLastError() after a launch.
int check_launch(const char* name);

// Multiprocessor count of the current device (cached per device).
int sm_count();

}  // namespace gcsgd

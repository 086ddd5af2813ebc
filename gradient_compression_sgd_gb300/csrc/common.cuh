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

// Result of an exact descending selection on 31-bit magnitude keys.
struct SelectResult {
    uint32_t thresh;   // key of the rank-th largest item
    uint32_t greater;  // items with key > thresh
    uint32_t ties;     // items with key == thresh to take (1 .. count(== thresh))
};

// Exact rank-th largest of `count` keys (1 <= rank <= count), by three
// radix passes over bits [30:20], [19:9] and [8:0] of the keys with a
// shared-memory histogram; only keys that share the digits chosen so far take
// part in the next pass.  `load(i, &key)` returns false for items to skip.
// hist: 2048 words of shared memory; scan: NT/32 + 1 words of 64-bit shared
// memory; sel: 4 words of shared memory.  Every thread must call it.
template <int NT, class Load>
__device__ SelectResult radix_select_desc(Load load, uint64_t count, uint32_t rank,
                                          uint32_t* hist, uint64_t* scan, uint32_t* sel) {
    uint32_t prefix = 0, pmask = 0, need = rank, greater = 0;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 20 : (pass == 1 ? 9 : 0);
        const int nb = pass == 2 ? 512 : 2048;
        for (int b = threadIdx.x; b < nb; b += NT) hist[b] = 0;
        if (threadIdx.x == 0) { sel[0] = 0; sel[1] = 0; }
        __syncthreads();
        for (uint64_t base = 0; base < count; base += 4 * (uint64_t)NT) {
            uint32_t key[4];
            bool ok[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // four independent loads in flight
                const uint64_t i = base + (uint64_t)j * NT + threadIdx.x;
                key[j] = 0;
                ok[j] = (i < count) && load(i, &key[j]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (ok[j] && ((key[j] & pmask) == prefix)) atomicAdd(&hist[(key[j] >> shift) & (uint32_t)(nb - 1)], 1u);
        }
        __syncthreads();
        // thread t owns buckets [hi - w, hi) counted from the top
        const int w = nb / NT;
        const int t = threadIdx.x;
        const int hi = nb - t * w;
        uint32_t mine = 0;
        for (int b = hi - 1; b >= hi - w; --b) mine += hist[b];
        uint64_t tot;
        uint32_t above = (uint32_t)block_exclusive_scan<NT>(mine, scan, &tot);
        for (int b = hi - 1; b >= hi - w; --b) {
            const uint32_t h = hist[b];
            if (above < need && need <= above + h) {
                sel[0] = (uint32_t)b;
                sel[1] = above;
            }
            above += h;
        }
        __syncthreads();
        const uint32_t b = sel[0], ab = sel[1];
        prefix |= b << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        greater += ab;
        need -= ab;
        __syncthreads();
    }
    SelectResult r;
    r.thresh = prefix;
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

// spavg.cu -- decompress and average K sparse messages into a dense vector.
//
// "AdaComp ...", Proposed method: learners exchange compressed gradients and
// average them before the weight update; "Deep Gradient Compression",
// Appendix A: the nodes' gradients are summed.
//
// One kernel.  Each CTA owns a contiguous run of 4096-element output tiles.
// A tile lives in shared memory: zeroed, then every list's entries that fall
// in it are added in list order k = 0..K-1 (entries inside one list have
// distinct indices, so the adds of one k never collide; a barrier between
// lists keeps the fp32 sum in k order, bit-identical to the definition),
// then the tile is divided by K and written to HBM with 128-bit stores.  A
// CTA first finds, for every list, the run of entries inside its whole index
// range (both ends searched in parallel, 32 probes per round trip) and copies
// those entries to shared memory in one round of loads, so its tiles need no
// further global reads.  The dense output is written exactly once and each
// entry is read once, which is the minimum traffic.
#include "common.cuh"

namespace gcsgd {
namespace spavg {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr uint32_t kTile = 4096;   // output elements per shared-memory tile
constexpr uint32_t kStage = 2048;  // list entries a CTA stages for its whole index range

// First position p in [0, cnt] with list[p].idx >= target, for a list sorted
// ascending; 32 probes per round trip.  Called by a whole warp.
__device__ uint64_t warp_lower_bound(const gcsgd_pair* list, uint64_t cnt, uint64_t target) {
    const int lane = threadIdx.x & 31;
    uint64_t lo = 0, hi = cnt;  // answer in [lo, hi]
    while (hi - lo > 32) {
        const uint64_t step = (hi - lo + 31) / 32;
        const uint64_t q = lo + (uint64_t)(lane + 1) * step - 1;
        const bool pred = q >= hi || (uint64_t)__ldg(&list[q].idx) >= target;
        const unsigned b = __ballot_sync(kFull, pred);
        const int f = b ? __ffs(b) - 1 : 32;
        const uint64_t nlo = lo + (uint64_t)f * step;
        const uint64_t qf = lo + (uint64_t)(f + 1) * step - 1;
        hi = (f < 32 && qf < hi) ? qf : hi;
        lo = nlo;
    }
    const uint64_t q = lo + lane;
    const bool pred = q >= hi || (uint64_t)__ldg(&list[q].idx) >= target;
    const unsigned b = __ballot_sync(kFull, pred);
    const uint64_t r = lo + (uint64_t)(b ? __ffs(b) - 1 : 32);
    return r < hi ? r : hi;
}

// x / K rounded once.  Most outputs are +0 (no list holds them) and 0 / K is
// +0, so only non-zeros divide; for K a power of two, x * (1/K) is the same
// correctly rounded value (both are x 2^-j rounded once), so it multiplies.
__device__ __forceinline__ float div_k(float x, float fk, float inv_k, bool pow2) {
    if (x == 0.0f) return x;
    return pow2 ? __fmul_rn(x, inv_k) : __fdiv_rn(x, fk);
}

__device__ __forceinline__ void store_tile(const float* acc, float* out, uint64_t r0, uint64_t r1, float fk) {
    const uint64_t len = r1 - r0;
    const int K = (int)fk;
    const bool pow2 = (K & (K - 1)) == 0;
    const float inv_k = 1.0f / fk;
    const bool out_aligned = ((uintptr_t)(out + r0) & 15) == 0;
    for (uint32_t j = threadIdx.x * 4; j < len; j += NT * 4) {
        float4 q = *reinterpret_cast<const float4*>(acc + j);
        if ((__float_as_uint(q.x) | __float_as_uint(q.y) | __float_as_uint(q.z) | __float_as_uint(q.w)) != 0u) {
            q.x = div_k(q.x, fk, inv_k, pow2);
            q.y = div_k(q.y, fk, inv_k, pow2);
            q.z = div_k(q.z, fk, inv_k, pow2);
            q.w = div_k(q.w, fk, inv_k, pow2);
        }
        if (out_aligned && j + 4 <= len) {
            *reinterpret_cast<float4*>(out + r0 + j) = q;
        } else {
            const float* qq = &q.x;
            for (int i = 0; i < 4 && j + i < len; ++i) out[r0 + j + i] = qq[i];
        }
    }
}

// Shared memory: acc[kTile] | stage[kStage] pairs | lo[K] hi[K] cnt[K] (u64) | soff[K+1] sptr[K] (u32)
__global__ void __launch_bounds__(NT) spavg_kernel(const gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                   const int64_t* __restrict__ counts, int K, uint64_t n,
                                                   float* __restrict__ out, uint64_t tiles, uint64_t tiles_per_cta) {
    extern __shared__ __align__(16) unsigned char smem[];
    float* acc = reinterpret_cast<float*>(smem);
    gcsgd_pair* stage = reinterpret_cast<gcsgd_pair*>(smem + kTile * sizeof(float));
    uint64_t* lo = reinterpret_cast<uint64_t*>(smem + kTile * sizeof(float) + kStage * sizeof(gcsgd_pair));
    uint64_t* hi = lo + K;
    uint64_t* cnt = hi + K;
    uint32_t* soff = reinterpret_cast<uint32_t*>(cnt + K);  // list k staged at [soff[k], soff[k+1])
    uint32_t* sptr = soff + K + 1;                           // first staged entry not yet added
    __shared__ uint32_t s_total;
    const uint64_t t0 = (uint64_t)blockIdx.x * tiles_per_cta;
    if (t0 >= tiles) return;
    const uint64_t t1 = t0 + tiles_per_cta < tiles ? t0 + tiles_per_cta : tiles;
    const uint64_t R0 = t0 * kTile, R1 = t1 * kTile < n ? t1 * kTile : n;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float fk = (float)K;

    for (int k = threadIdx.x; k < K; k += NT) {
        const int64_t c = counts[k];
        cnt[k] = c < 0 ? 0 : ((uint64_t)c > cap ? cap : (uint64_t)c);
    }
    __syncthreads();
    // each list's run inside this CTA's index range [R0, R1): both ends searched in parallel
    for (int q = warp; q < 2 * K; q += NW) {
        const int k = q < K ? q : q - K;
        const uint64_t p = warp_lower_bound(lists + (uint64_t)k * cap, cnt[k], q < K ? R0 : R1);
        if (lane == 0) (q < K ? lo : hi)[k] = p;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t run = 0;
        bool fits = true;
        for (int k = 0; k < K; ++k) {
            soff[k] = run;
            const uint64_t c = hi[k] > lo[k] ? hi[k] - lo[k] : 0;
            if (run + c > kStage) fits = false;
            run = fits ? run + (uint32_t)c : run;
        }
        soff[K] = run;
        s_total = fits ? run : 0xffffffffu;
    }
    __syncthreads();
    const uint32_t total = s_total;

    if (total != 0xffffffffu) {
        // stage every entry of the range once (four loads in flight per thread)
        for (uint32_t q0 = 0; q0 < total; q0 += 4 * NT) {
            gcsgd_pair it[4];
            int kk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t q = q0 + j * NT + threadIdx.x;
                kk[j] = -1;
                if (q < total) {
                    int k = 0, kh = K;  // last list with soff[k] <= q
                    while (kh - k > 1) {
                        const int m = (k + kh) >> 1;
                        if (soff[m] <= q) k = m; else kh = m;
                    }
                    kk[j] = k;
                    it[j] = lists[(uint64_t)k * cap + lo[k] + (q - soff[k])];
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (kk[j] >= 0) stage[q0 + j * NT + threadIdx.x] = it[j];
        }
        for (int k = threadIdx.x; k < K; k += NT) sptr[k] = soff[k];
        __syncthreads();
        for (uint64_t t = t0; t < t1; ++t) {
            const uint64_t r0 = t * kTile;
            const uint64_t r1 = r0 + kTile < n ? r0 + kTile : n;
            for (uint32_t j = threadIdx.x * 4; j < kTile; j += NT * 4)
                *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
            __syncthreads();
            if (warp == 0) {
                // warp 0 adds the lists in learner order; within a list the
                // indices are distinct, so its lanes never collide
                for (int k = 0; k < K; ++k) {
                    uint32_t a = sptr[k];
                    const uint32_t e = soff[k + 1];
                    for (;;) {
                        const uint32_t i = a + lane;
                        gcsgd_pair it;
                        it.idx = 0xffffffffu;
                        it.val = 0.f;
                        if (i < e) it = stage[i];
                        const bool in = i < e && (uint64_t)it.idx < r1;
                        if (in && (uint64_t)it.idx >= r0) {
                            float* acc_j = acc + (it.idx - r0);
                            *acc_j = __fadd_rn(*acc_j, it.val);
                        }
                        const int c = __popc(__ballot_sync(kFull, in));
                        a += c;
                        if (c < 32) break;
                    }
                    __syncwarp();  // list k's adds land before list k+1's
                    if (lane == 0) sptr[k] = a;
                }
            }
            __syncthreads();
            store_tile(acc, out, r0, r1, fk);
            __syncthreads();
        }
        return;
    }

    // More entries than fit the stage (dense lists): walk each tile's entries in global memory.
    uint64_t* ptr = lo;
    uint64_t* end = hi;
    for (uint64_t t = t0; t < t1; ++t) {
        const uint64_t r0 = t * kTile;
        const uint64_t r1 = r0 + kTile < n ? r0 + kTile : n;
        for (uint32_t j = threadIdx.x * 4; j < kTile; j += NT * 4)
            *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncthreads();  // everyone has read hi[] before it is reused as end[]
        for (int k = warp; k < K; k += NW) {
            const gcsgd_pair* L = lists + (uint64_t)k * cap;
            uint64_t e = ptr[k];
            for (;;) {
                const uint64_t q = e + lane;
                const bool in = q < cnt[k] && (uint64_t)__ldg(&L[q].idx) < r1;
                const unsigned b = __ballot_sync(kFull, in);
                const int c = __popc(b);
                e += c;
                if (c < 32) break;
            }
            if (lane == 0) end[k] = e;
        }
        __syncthreads();
        for (int k = 0; k < K; ++k) {
            const gcsgd_pair* L = lists + (uint64_t)k * cap;
            for (uint64_t p = ptr[k] + threadIdx.x; p < end[k]; p += NT) {
                const gcsgd_pair it = L[p];
                if ((uint64_t)it.idx >= r0 && (uint64_t)it.idx < r1) {
                    float* a = acc + (it.idx - r0);
                    *a = __fadd_rn(*a, it.val);
                }
            }
            __syncthreads();
        }
        store_tile(acc, out, r0, r1, fk);
        for (int k = threadIdx.x; k < K; k += NT) ptr[k] = end[k];
        __syncthreads();
    }
}

}  // namespace spavg

int spavg_launch(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int K, int64_t n, float* out,
                 cudaStream_t stream) {
    using namespace spavg;
    if (n == 0) return GCSGD_OK;
    const uint64_t tiles = ((uint64_t)n + kTile - 1) / kTile;
    uint64_t grid = (uint64_t)sm_count() * 6;
    if (grid > tiles) grid = tiles;
    const uint64_t per = (tiles + grid - 1) / grid;
    grid = (tiles + per - 1) / per;
    const size_t smem = kTile * sizeof(float) + kStage * sizeof(gcsgd_pair) + 3 * sizeof(uint64_t) * (size_t)K +
                        sizeof(uint32_t) * (2 * (size_t)K + 1);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem > 48 * 1024 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(spavg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
            return set_error(GCSGD_ERR_CUDA, "sparse_average: cannot raise the shared-memory limit");
        attr_set[dev] = true;
    }
    LaunchScope ls("spavg", stream);
    spavg_kernel<<<(unsigned)grid, NT, smem, stream>>>(lists, (uint64_t)cap, counts, K, (uint64_t)n, out, tiles, per);
    return check_launch("spavg");
}

}  // namespace gcsgd

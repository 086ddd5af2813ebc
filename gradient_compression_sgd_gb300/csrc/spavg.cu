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
// then the tile is divided by K and written to HBM with 128-bit stores.  The
// dense output is written exactly once and each entry is read once (plus a
// cached re-read to find the tile's end), which is the minimum traffic.
#include "common.cuh"

namespace gcsgd {
namespace spavg {

constexpr int NT = 256;
constexpr uint32_t kTile = 4096;

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

__global__ void __launch_bounds__(NT) spavg_kernel(const gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                   const int64_t* __restrict__ counts, int K, uint64_t n,
                                                   float* __restrict__ out, uint64_t tiles, uint64_t tiles_per_cta) {
    extern __shared__ __align__(16) unsigned char smem[];
    float* acc = reinterpret_cast<float*>(smem);
    uint64_t* ptr = reinterpret_cast<uint64_t*>(smem + kTile * sizeof(float));
    uint64_t* end = ptr + K;
    uint64_t* cnt = end + K;
    const uint64_t t0 = (uint64_t)blockIdx.x * tiles_per_cta;
    if (t0 >= tiles) return;
    const uint64_t t1 = t0 + tiles_per_cta < tiles ? t0 + tiles_per_cta : tiles;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float fk = (float)K;

    for (int k = threadIdx.x; k < K; k += NT) {
        int64_t c = counts[k];
        cnt[k] = c < 0 ? 0 : ((uint64_t)c > cap ? cap : (uint64_t)c);
    }
    __syncthreads();
    for (int k = warp; k < K; k += NT / 32) {
        const uint64_t p = warp_lower_bound(lists + (uint64_t)k * cap, cnt[k], t0 * kTile);
        if (lane == 0) ptr[k] = p;
    }
    __syncthreads();

    for (uint64_t t = t0; t < t1; ++t) {
        const uint64_t r0 = t * kTile;
        const uint64_t r1 = r0 + kTile < n ? r0 + kTile : n;
        for (uint32_t j = threadIdx.x * 4; j < kTile; j += NT * 4)
            *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        // end of each list's run inside this tile: advance 32 entries at a time
        for (int k = warp; k < K; k += NT / 32) {
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
        const uint64_t len = r1 - r0;
        for (uint32_t j = threadIdx.x * 4; j < len; j += NT * 4) {
            float4 q = *reinterpret_cast<const float4*>(acc + j);
            q.x = __fdiv_rn(q.x, fk);
            q.y = __fdiv_rn(q.y, fk);
            q.z = __fdiv_rn(q.z, fk);
            q.w = __fdiv_rn(q.w, fk);
            if (j + 4 <= len && ((uintptr_t)(out + r0 + j) & 15) == 0) {
                *reinterpret_cast<float4*>(out + r0 + j) = q;
            } else {
                const float* qq = &q.x;
                for (int i = 0; i < 4 && j + i < len; ++i) out[r0 + j + i] = qq[i];
            }
        }
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
    uint64_t grid = (uint64_t)sm_count() * 8;
    if (grid > tiles) grid = tiles;
    const uint64_t per = (tiles + grid - 1) / grid;
    grid = (tiles + per - 1) / per;
    const size_t smem = kTile * sizeof(float) + 3 * sizeof(uint64_t) * (size_t)K;
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

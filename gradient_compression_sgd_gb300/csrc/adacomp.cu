// adacomp.cu -- AdaComp for K learners.
//
// "AdaComp : Adaptive Residual Gradient Compression for Data-Parallel
// Distributed Training", Proposed method: G = R + dW per layer; the layer is
// cut into bins of L_T values and each bin's max |G| is found; entries with
// |G + dW| >= the bin max are selected (O(N), no global sort); one scale per
// layer, the mean of the bin maxima; a selected entry is sent as
// sign(G) * scale and the residue keeps what was not sent.
//
// Launch sequence (caller's stream, no host sync):
//   ada_plan      one CTA: per-segment plan (bins, tiles, emit groups), zeroes
//                 the big-bin maxima
//   [ada_bigmax]  only for segments with L_T > 4096: bin maxima via atomics
//   ada_bins_warp the bandwidth-bound pass for 4 <= L_T <= 512: a tile is one
//                 warp's chunk of whole bins (<= 512 values) in registers;
//                 G = R + dW, bin maxima, selection, R <- G stored once, the
//                 selected (index, G) written in index order into the pool
//                 slots of the chunk's own index range
//   [ada_bins]    the same pass for other bin lengths, one 4096-value tile per
//                 CTA (bin maxima in shared memory; fp64 tile sums)
//   ada_scan      one CTA per (learner, segment): output slots of the emit
//                 groups, the segment's count and its scale
//   ada_emit      one warp per group of 8 tiles: writes (index, sign(G)*scale)
//                 at its ordered slot and fixes the residue R = G - sign(G)*scale.
// Tiles hold whole bins (bins of L_T <= 4096 never straddle tiles), so a
// bin's maximum is final inside one warp or CTA and the first pass is
// single-read.  Every tile owns the pool slots of its index range, so no
// counter is shared between CTAs and the result is deterministic.
//
// Deferred residue (adacomp_compress_deferred), for the warp-chunk segments:
// ada_emit does not rewrite R at the sent indices (a scattered read-modify-
// write of a 32-byte sector per entry); ada_bins_warp keeps the chunk's
// selection bits instead (16 bits per lane, 64 bytes a chunk), and the next
// call's ada_bins_warp, which streams R anyway, subtracts the sent value
// sign(R) * scale at those bits before forming G = R + dW: the same fp32
// subtraction, of the same operands, as the eager fix-up, so every message
// and every residue is bit-identical.  Until then R holds G at the sent
// indices; ada_settle applies the pending subtraction.
#include <math.h>

#include "common.cuh"

namespace gcsgd {
namespace ada {

constexpr int NT = 256;
constexpr uint32_t kTileMax = 4096;
constexpr uint32_t kWarpChunk = 512;  // values per warp chunk (4 float4 per lane)

enum : uint32_t { kModeEmpty = 0, kModeSmall = 1, kModeBig = 2 };

struct SegPlan {
    uint32_t off, n, L, mode;
    uint32_t nbins;     // ceil(n / L)
    uint32_t tile_len;  // elements per tile (whole bins in small mode)
    uint32_t bpt;       // bins per tile (small mode)
    uint32_t ntiles;
    uint32_t tile_off;  // first tile within a learner
    uint32_t big_off;   // first big-bin slot within a learner (big mode)
    float invL;         // fp32 1/L: bin = floor((e + 0.5) * invL) is exact for e < 4096
    uint32_t bpw;       // warp chunks: bins per chunk (4 <= L <= 512; a tile is one chunk), else 0
    uint32_t grp_off;   // first emit group (kGroup consecutive tiles) within a learner
};

constexpr uint32_t kGroup = 8;  // tiles per ada_emit work item
constexpr size_t kEmitSmemMax = 200 * 1024;  // ada_emit's per-learner and per-segment tables

// Shared memory of ada_emit: each learner's total and each (learner,
// segment)'s first output slot.
inline size_t emit_smem_bytes(int K, int S) { return sizeof(uint32_t) * (size_t)K * S + sizeof(uint64_t) * (size_t)K; }

template <int MAXS>
struct SegTable {
    uint32_t off[MAXS + 1];
    uint32_t L[MAXS];
};

__host__ __device__ inline uint32_t gcd4(uint32_t L) { return (L & 3) == 0 ? 4 : ((L & 1) == 0 ? 2 : 1); }

__host__ __device__ inline void seg_fields(uint32_t n, uint32_t L, SegPlan* p) {
    p->n = n;
    p->L = L;
    p->nbins = n ? (uint32_t)(((uint64_t)n + L - 1) / L) : 0;
    p->bpt = 0;
    p->invL = 1.0f / (float)L;
    p->bpw = 0;
    if (n == 0) {
        p->mode = kModeEmpty;
        p->tile_len = 0;
        p->ntiles = 0;
    } else if (L <= kTileMax) {
        p->mode = kModeSmall;
        const uint32_t g = 4 / gcd4(L);  // keep tiles 16-byte aligned where possible
        uint32_t bpt;
        if (L >= 4 && L <= kWarpChunk) {  // warp chunks of whole bins, eight per tile
            uint32_t bpw = kWarpChunk / L;
            if (bpw >= g) bpw -= bpw % g;
            p->bpw = bpw;
            bpt = bpw;
        } else {
            bpt = kTileMax / L;
            if (bpt >= g) bpt -= bpt % g;
        }
        p->bpt = bpt;
        p->tile_len = bpt * L;
        p->ntiles = (p->nbins + bpt - 1) / bpt;
    } else {
        p->mode = kModeBig;
        p->tile_len = kTileMax;
        p->ntiles = (n + kTileMax - 1) / kTileMax;
    }
}

struct HostPlan {
    uint64_t tiles_per_learner;
    uint64_t big_per_learner;
    uint64_t groups_per_learner;
};

void host_plan(const int64_t* off, const int32_t* lt, int S, HostPlan* hp) {
    hp->tiles_per_learner = 0;
    hp->big_per_learner = 0;
    hp->groups_per_learner = 0;
    for (int s = 0; s < S; ++s) {
        SegPlan p;
        seg_fields((uint32_t)(off[s + 1] - off[s]), (uint32_t)lt[s], &p);
        hp->tiles_per_learner += p.ntiles;
        hp->groups_per_learner += (p.ntiles + kGroup - 1) / kGroup;
        if (p.mode == kModeBig || p.bpw) hp->big_per_learner += p.nbins;
    }
}

struct Workspace {
    SegPlan* plan;
    uint2* tile_tab;     // (pool slot = the tile's first index, count)
    double2* tile_sum;   // compensated sum of the tile's bin maxima
    uint32_t* grp_rel;   // first output slot of the emit group within its segment
    uint32_t* big;       // bin maxima (|G| bits) of big-mode segments
    uint2* pool;         // (index within the learner, G bits); a tile's entries sit at its own index range
    uint16_t* sent;      // deferred residue: per tile and lane, the chunk's selection bits (warp-chunk tiles)
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t layout(int S, int K, int64_t off_total, const HostPlan& hp, void* base, Workspace* w) {
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    const uint64_t T = (uint64_t)K * hp.tiles_per_learner;
    const uint64_t N = (uint64_t)off_total;
    const size_t o_plan = take(sizeof(SegPlan) * (size_t)S);
    const size_t o_tt = take(sizeof(uint2) * T);
    const size_t o_ts = take(sizeof(double2) * T);
    const size_t o_tr = take(sizeof(uint32_t) * (size_t)K * hp.groups_per_learner);
    const size_t o_big = take(sizeof(uint32_t) * (size_t)K * hp.big_per_learner);
    const size_t o_pool = take(sizeof(uint2) * (size_t)K * (size_t)N);  // one slot per element: no shared counter
    const size_t o_sent = take(sizeof(uint16_t) * 32 * T);
    if (w) {
        char* b = (char*)base;
        w->plan = (SegPlan*)(b + o_plan);
        w->tile_tab = (uint2*)(b + o_tt);
        w->tile_sum = (double2*)(b + o_ts);
        w->grp_rel = (uint32_t*)(b + o_tr);
        w->big = (uint32_t*)(b + o_big);
        w->pool = (uint2*)(b + o_pool);
        w->sent = (uint16_t*)(b + o_sent);
    }
    return o;
}

// Double-float accumulation: (hi, lo) += (x, xl) with the rounding error of
// hi + x kept exactly (TwoSum, Knuth), and renormalisation (FastTwoSum,
// valid since |hi| >= |lo| after it).  fp32 only.
__device__ __forceinline__ void df_add(float& hi, float& lo, float x, float xl) {
    const float s = __fadd_rn(hi, x);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(x, bp));
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(err, xl));
}
__device__ __forceinline__ void df_norm(float& hi, float& lo) {
    const float s = __fadd_rn(hi, lo);
    lo = __fsub_rn(lo, __fsub_rn(s, hi));
    hi = s;
}

// Neumaier step: (s, c) += x.
__device__ __forceinline__ void csum_add(double& s, double& c, double x) {
    const double t = __dadd_rn(s, x);
    c = __dadd_rn(c, fabs(s) >= fabs(x) ? __dadd_rn(__dsub_rn(s, t), x) : __dadd_rn(__dsub_rn(x, t), s));
    s = t;
}

template <int MAXS>
__global__ void __launch_bounds__(1024) ada_plan(SegTable<MAXS> st, int S, int K, uint64_t big_per_learner,
                                                 SegPlan* __restrict__ plan, uint32_t* __restrict__ big) {
    __shared__ uint64_t scan[1024 / 32 + 1];
    __shared__ uint64_t carry[3];
    __shared__ int s_nbig, s_big[64];  // the big-bin segments (all of them are scanned if more)
    if (threadIdx.x < 3) carry[threadIdx.x] = 0;
    if (threadIdx.x == 0) s_nbig = 0;
    __syncthreads();
    for (int base = 0; base < S; base += 1024) {
        const int s = base + (int)threadIdx.x;
        const bool live = s < S;
        SegPlan p;
        seg_fields(live ? st.off[s + 1] - st.off[s] : 0u, live ? st.L[s] : 1u, &p);
        p.off = live ? st.off[s] : 0u;
        uint64_t tot;
        const uint64_t ex_t = block_exclusive_scan<1024>(live ? p.ntiles : 0, scan, &tot);
        const uint64_t c0 = carry[0];
        __syncthreads();
        if (threadIdx.x == 0) carry[0] = c0 + tot;
        const uint64_t ex_b =
            block_exclusive_scan<1024>(live && (p.mode == kModeBig || p.bpw) ? p.nbins : 0, scan, &tot);
        const uint64_t c1 = carry[1];
        __syncthreads();
        if (threadIdx.x == 0) carry[1] = c1 + tot;
        const uint64_t ex_g = block_exclusive_scan<1024>(live ? (p.ntiles + kGroup - 1) / kGroup : 0, scan, &tot);
        const uint64_t c2 = carry[2];
        __syncthreads();
        if (threadIdx.x == 0) carry[2] = c2 + tot;
        if (live) {
            p.tile_off = (uint32_t)(c0 + ex_t);
            p.big_off = (uint32_t)(c1 + ex_b);
            p.grp_off = (uint32_t)(c2 + ex_g);
            plan[s] = p;
            if (p.mode == kModeBig) {
                const int q = atomicAdd(&s_nbig, 1);
                if (q < 64) s_big[q] = s;
            }
        }
        __syncthreads();
    }
    // big-bin maxima are accumulated by atomicMax and start at 0 (warp-chunk
    // bins are written once by ada_bins_warp)
    __syncthreads();
    const int nbig = s_nbig < 64 ? s_nbig : 64;
    for (int q = 0; q < (s_nbig <= 64 ? nbig : S); ++q) {
        const SegPlan p = plan[s_nbig <= 64 ? s_big[q] : q];
        if (p.mode != kModeBig) continue;
        for (int k = 0; k < K; ++k)
            for (uint32_t b = threadIdx.x; b < p.nbins; b += 1024) big[(uint64_t)k * big_per_learner + p.big_off + b] = 0;
    }
}

__device__ __forceinline__ int find_segment_by_tile(const SegPlan* plan, int S, uint32_t lt) {
    int lo = 0, hi = S;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(&plan[mid].tile_off) <= lt) lo = mid; else hi = mid;
    }
    return lo;
}

// Bits of |x| with NaN read as 0: maxima of these bit patterns are the float
// maxima of |x| over the numbers (NaN never wins, as in a `>` scan).
__device__ __forceinline__ uint32_t nan0_key(float x) { return __float_as_uint(fmaxf(fabsf(x), 0.0f)); }

// Bin maxima of segments whose bins are longer than a tile.
__global__ void __launch_bounds__(NT) ada_bigmax(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                                 uint32_t tiles_per_learner, uint64_t total_tiles,
                                                 const float* __restrict__ dW, const float* __restrict__ R,
                                                 uint32_t* __restrict__ big, uint64_t big_per_learner) {
    const int lane = threadIdx.x & 31;
    for (uint32_t t = blockIdx.x; t < (uint32_t)total_tiles; t += gridDim.x) {
        const uint32_t k = t / tiles_per_learner;
        const uint32_t lt = t - k * tiles_per_learner;
        const int s = find_segment_by_tile(plan, S, lt);
        const SegPlan p = plan[s];
        if (p.mode != kModeBig) continue;
        const uint32_t start = (lt - p.tile_off) * kTileMax;
        const uint32_t len = p.n - start < kTileMax ? p.n - start : kTileMax;
        const uint64_t base = (uint64_t)k * N + p.off + start;
        uint32_t* bm = big + (uint64_t)k * big_per_learner + p.big_off;
        for (uint32_t e0 = 0; e0 < len; e0 += NT) {
            const uint32_t e = e0 + threadIdx.x;
            const bool in = e < len;
            const float g = in ? __fadd_rn(R[base + e], __ldg(dW + base + e)) : 0.0f;
            const uint32_t bin = in ? (start + e) / p.L : 0xffffffffu;
            const unsigned am = __ballot_sync(kFull, in);
            if (in) {
                const unsigned grp = __match_any_sync(am, bin);
                const uint32_t mx = __reduce_max_sync(grp, nan0_key(g));
                if (lane == __ffs(grp) - 1) atomicMax(&bm[bin], mx);
            }
        }
    }
}

// Bin of tile element e (small mode): floor((e + 0.5) / L), exact for e < 4096.
__device__ __forceinline__ uint32_t bin_of(uint32_t e, float invL) {
    return (uint32_t)__float2int_rd(((float)e + 0.5f) * invL);
}


// Selection of one tile's entries: sent iff |G + dW| >= the bin's max |G|,
// the max > 0 and G != 0 (float compares, as the definition is written: a
// NaN is never sent).  MODE 0: bins of L >= 4 inside the tile (a float4
// spans at most two bins, split at `cut`); MODE 1: bins of L < 4; MODE 2:
// bins longer than a tile, maxima precomputed in global memory.  Bit 4r+j of
// `flags` marks element j of round r; `packed` holds the per-round counts.
template <int MODE>
__device__ __forceinline__ void select_tile(const float4 (&Gv)[4], const float4 (&Dv)[4], uint32_t len, uint32_t L,
                                            float invL, uint32_t nbt, const uint32_t* bmax, const uint32_t* bigm,
                                            uint32_t start, uint32_t& flags, uint64_t& packed) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint32_t e = 4u * (r * NT + threadIdx.x);
        if (e >= len) continue;
        const float* g4 = &Gv[r].x;
        const float* d4 = &Dv[r].x;
        float gm[4];
        if (MODE == 0) {
            const uint32_t b0 = bin_of(e, invL);
            const uint32_t cut = (b0 + 1) * L - e;
            const float m0 = __uint_as_float(bmax[b0]);
            const float m1 = cut < 4 && b0 + 1 < nbt ? __uint_as_float(bmax[b0 + 1]) : m0;
#pragma unroll
            for (int j = 0; j < 4; ++j) gm[j] = (uint32_t)j < cut ? m0 : m1;
        } else if (MODE == 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) gm[j] = e + j < len ? __uint_as_float(bmax[bin_of(e + j, invL)]) : 0.0f;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) gm[j] = e + j < len ? __uint_as_float(__ldg(&bigm[(start + e + j) / L])) : 0.0f;
        }
        uint32_t f = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool sel = fabsf(__fadd_rn(g4[j], d4[j])) >= gm[j] && gm[j] > 0.0f && g4[j] != 0.0f;
            f |= (uint32_t)sel << j;
        }
        if (e + 4 > len) f &= (1u << (len - e)) - 1u;  // a partial float4 at the tile end
        flags |= f << (4 * r);
        packed |= (uint64_t)__popc(f) << (16 * r);
    }
}

// Warp-chunk tiles (4 <= L_T <= 512): a tile is one warp's chunk of bpw
// whole bins, at most 512 values.  Warps run independently, with no block
// barrier and no shared counter.  Each warp streams its chunks through a
// ring of kRing shared-memory stages filled by cp.async (R and dW, 4 KB a
// chunk; the copies of the next kRing - 1 chunks are in flight while one is
// computed, and they hold no registers).  Two stages at six CTAs of four
// warps per SM (24 warps) measured faster than three stages at four CTAs:
// the pass is bound by its instruction latencies more than by the bytes in
// flight.  When a warp issues a chunk's copies, lanes 0 and 1 also ask L2
// for the warp's next chunk of dW and R (bulk prefetches; every lane forms
// the address, no branch), which puts more bytes in flight than the ring
// holds; asking for the chunk after that instead measured slower.
// A lane copies and later reads the
// same 16-byte pieces, so only its own cp.async groups are waited on.  Past a
// chunk's end the copies zero-fill: G = 0 never raises a maximum and is never
// sent, so the arithmetic needs no bounds test.  Per chunk the warp finds its
// bins' maxima (one bin: a warp reduction; several: shared-memory atomicMax
// per float4 part), writes them to the bins array (ada_scan averages them),
// selects, stores R <- G and writes its candidates in index order into the
// pool slots of its own index range.
constexpr int NTW = 128;   // threads of an ada_bins_warp CTA
constexpr int kRing = 2;   // stages per warp
struct ChunkMeta {         // what the computing side needs of an issued chunk
    uint32_t rel, clen, k, lt, tj, L, bpw, big_off;
    float invL;
    float pscale;          // deferred residue: the previous call's scale of the segment
    uint32_t pfix;         // the previous call's selection bits apply (its learner sent)
};
// the previous call's selection bits of a chunk: 32 lanes x 16 bits
constexpr size_t kSentBytes = 32 * sizeof(uint16_t);
constexpr size_t kBinsWarpSmem =
    sizeof(float) * (NTW / 32) * kRing * 2 * kWarpChunk + sizeof(ChunkMeta) * (NTW / 32) * kRing +
    sizeof(uint32_t) * (NTW / 32) * (kWarpChunk / 4) + kSentBytes * (NTW / 32) * kRing;

__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"((uint32_t)__cvta_generic_to_shared(sdst)),
                 "l"(gsrc), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* sdst, const void* gsrc, uint32_t bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"((uint32_t)__cvta_generic_to_shared(sdst)),
                 "l"(gsrc), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// A hint: `bytes` (a multiple of 16) from the 16-byte aligned address p into L2.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// defer: keep the selection bits in `sent` instead of having ada_emit fix R;
// pending: R holds the previous deferred call's G at its sent indices, whose
// bits are in `sent` and whose scales and totals are prev_scales, prev_totals.
__global__ void __launch_bounds__(NTW, 6) ada_bins_warp(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                                        uint32_t tiles_per_learner, uint64_t total_tiles,
                                                        const float* __restrict__ dW, float* __restrict__ R,
                                                        uint32_t* __restrict__ bins, uint64_t bins_per_learner,
                                                        uint2* __restrict__ tile_tab, uint2* __restrict__ pool,
                                                        int defer, int pending, uint16_t* __restrict__ sent,
                                                        const float* __restrict__ prev_scales,
                                                        const int64_t* __restrict__ prev_totals, uint64_t cap) {
    extern __shared__ __align__(16) unsigned char bw_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* ring = reinterpret_cast<float*>(bw_smem) + (size_t)warp * kRing * 2 * kWarpChunk;  // [kRing][dW | R]
    ChunkMeta* meta = reinterpret_cast<ChunkMeta*>(bw_smem + sizeof(float) * (NTW / 32) * kRing * 2 * kWarpChunk) +
                      warp * kRing;
    uint32_t* wb = reinterpret_cast<uint32_t*>(bw_smem + sizeof(float) * (NTW / 32) * kRing * 2 * kWarpChunk +
                                               sizeof(ChunkMeta) * (NTW / 32) * kRing) +
                   warp * (kWarpChunk / 4);  // this warp's bin maxima (bpw <= 128)
    uint16_t* sbits = reinterpret_cast<uint16_t*>(bw_smem + sizeof(float) * (NTW / 32) * kRing * 2 * kWarpChunk +
                                                  sizeof(ChunkMeta) * (NTW / 32) * kRing +
                                                  sizeof(uint32_t) * (NTW / 32) * (kWarpChunk / 4)) +
                      warp * kRing * 32;  // [kRing][32] the previous selection bits of the staged chunks
    const uint32_t nw = gridDim.x * (NTW / 32), T = (uint32_t)total_tiles;  // T < 2^32 (checked by the host)

    // issuing side: the warp's tiles t = its id + i * nw, keeping the segment's fields
    uint32_t t = blockIdx.x * (NTW / 32) + warp;
    bool done = t >= T;
    uint32_t k = 0, lt = 0;
    struct {
        uint32_t off, n, L, bpw, tile_len, tile_off, big_off, next_off, k, pfix;
        float invL, pscale;
    } p = {};
    auto load_seg = [&](uint32_t at) {
        const int s = find_segment_by_tile(plan, S, at);
        const SegPlan q = plan[s];
        p.off = q.off, p.n = q.n, p.L = q.L, p.bpw = q.mode == kModeSmall ? q.bpw : 0u;
        p.tile_len = q.tile_len, p.tile_off = q.tile_off, p.big_off = q.big_off, p.invL = q.invL;
        p.next_off = s + 1 < S ? __ldg(&plan[s + 1].tile_off) : tiles_per_learner;
        p.k = k;
        p.pfix = 0u;
        p.pscale = 0.0f;
        if (pending && p.bpw) {  // the learner's previous message was sent (not over cap)
            p.pfix = (uint64_t)prev_totals[k] <= cap ? 1u : 0u;
            p.pscale = prev_scales[(uint64_t)k * S + s];
        }
    };
    auto step = [&]() {
        if (T - t <= nw) {
            done = true;
            return;
        }
        t += nw;
        lt += nw;
        while (lt >= tiles_per_learner) {
            lt -= tiles_per_learner;
            ++k;
        }
        if (lt < p.tile_off || lt >= p.next_off || k != p.k) load_seg(lt);
    };
    if (!done) {
        k = t / tiles_per_learner;
        lt = t - k * tiles_per_learner;
        load_seg(lt);
        while (!done && !p.bpw) step();  // other tiles: ada_bins
    }
    auto issue = [&](int st) {
        ChunkMeta m = {};
        if (!done) {
            const uint32_t tj = lt - p.tile_off, start = tj * p.tile_len;
            m.rel = p.off + start;
            m.clen = p.n - start < p.tile_len ? p.n - start : p.tile_len;
            m.k = k, m.lt = lt, m.tj = tj, m.L = p.L, m.bpw = p.bpw, m.big_off = p.big_off, m.invL = p.invL;
            m.pscale = p.pscale, m.pfix = p.pfix;
            if (lane < 16) {  // the previous selection bits (zeros where none apply)
                const uint16_t* src = sent + ((uint64_t)k * tiles_per_learner + lt) * 32 + 2 * lane;
                cp_async4(sbits + st * 32 + 2 * lane, src, p.pfix ? 4u : 0u);
            }
            const uint64_t base = (uint64_t)k * N + m.rel;
            const float* dWc = dW + base;
            const float* Rc = R + base;
            float* sD = ring + st * 2 * kWarpChunk;
            float* sR = sD + kWarpChunk;
            if ((((uintptr_t)dWc | (uintptr_t)Rc) & 15) == 0) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint32_t e = 4u * (lane + 32 * r);
                    const uint32_t by = e < m.clen ? (m.clen - e < 4 ? 4 * (m.clen - e) : 16u) : 0u;
                    const uint32_t o = by ? e : 0u;  // a valid address also where nothing is read
                    cp_async16(sD + e, dWc + o, by);
                    cp_async16(sR + e, Rc + o, by);
                }
            } else {  // 4-byte copies where the chunk is not 16-byte aligned
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint32_t e = 4u * (lane + 32 * r);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t by = e + j < m.clen ? 4u : 0u;
                        cp_async4(sD + e + j, by ? dWc + e + j : dWc, by);
                        cp_async4(sR + e + j, by ? Rc + e + j : Rc, by);
                    }
                }
            }
            step();
            while (!done && !p.bpw) step();
            // the warp's next chunk into L2 now (its copies are issued a round
            // later): more bytes in flight than the shared-memory ring holds
            {
                const uint32_t s2 = (lt - p.tile_off) * p.tile_len;
                const uint32_t c2 = p.n - s2 < p.tile_len ? p.n - s2 : p.tile_len;
                const float* src = (lane ? (const float*)R : dW) + ((uint64_t)k * N + p.off + s2);
                const uint32_t by = (c2 * 4u) & ~15u;  // whole 16-byte pieces inside the chunk
                if (!done && lane < 2 && by && ((uintptr_t)src & 15) == 0) l2_prefetch(src, by);  // lane 0: dW, 1: R
            }
        }
        if (lane == 0) meta[st] = m;  // clen = 0: no chunk (every later stage is empty too)
        cp_async_commit();
    };
#pragma unroll
    for (int st = 0; st < kRing - 1; ++st) issue(st);

    for (int cs = 0;; cs = cs == kRing - 1 ? 0 : cs + 1) {
        issue(cs == 0 ? kRing - 1 : cs - 1);  // that stage's chunk was computed in the previous round
        cp_async_wait<kRing - 1>();       // this lane's copies of chunk i have landed
        __syncwarp();                     // and lane 0's meta of it is visible
        const ChunkMeta m = meta[cs];
        if (m.clen == 0) break;
        const float* sD = ring + cs * 2 * kWarpChunk;
        const float* sR = sD + kWarpChunk;
        const uint64_t base = (uint64_t)m.k * N + m.rel;
        float* Rc = R + base;
        const bool cal = ((uintptr_t)Rc & 15) == 0;
        const uint32_t clen = m.clen, bpw = m.bpw, L = m.L;
        float4 Gv[4], Dv[4];
        if (m.pfix) {  // the previous call's deferred fix-up, R -= sign(R) * scale, on this lane's staged values
            float* sRw = const_cast<float*>(sR);
            for (uint32_t pb = sbits[cs * 32 + lane]; pb; pb &= pb - 1u) {  // bit 4r+j: element j of round r
                const uint32_t b = (uint32_t)__ffs(pb) - 1u;
                const uint32_t e = 4u * (lane + 32u * (b >> 2)) + (b & 3u);
                const float g = sRw[e];
                sRw[e] = __fsub_rn(g, g > 0.0f ? m.pscale : -m.pscale);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (lane + 32 * r);
            Dv[r] = *reinterpret_cast<const float4*>(sD + e);
            Gv[r] = *reinterpret_cast<const float4*>(sR + e);
            Gv[r].x = __fadd_rn(Gv[r].x, Dv[r].x);
            Gv[r].y = __fadd_rn(Gv[r].y, Dv[r].y);
            Gv[r].z = __fadd_rn(Gv[r].z, Dv[r].z);
            Gv[r].w = __fadd_rn(Gv[r].w, Dv[r].w);
        }
        // bin maxima of |G| (fmaxf skips a NaN, so NaN reads as 0)
        uint32_t* gb = bins + (uint64_t)m.k * bins_per_learner + m.big_off + m.tj * bpw;
        float m_one = 0.0f;
        if (bpw == 1) {
            float mx = 0.0f;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(Gv[r].x), fabsf(Gv[r].y)), fmaxf(fabsf(Gv[r].z), fabsf(Gv[r].w))));
            m_one = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(mx)));
            if (lane == 0) gb[0] = __float_as_uint(m_one);
        } else {
            for (uint32_t b = lane; b < bpw; b += 32) wb[b] = 0u;
            __syncwarp();
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t e = 4u * (lane + 32 * r);
                if (e >= clen) continue;
                const uint32_t b0 = bin_of(e, m.invL), cut = (b0 + 1) * L - e;
                const float* g4 = &Gv[r].x;
                float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a = fabsf(g4[j]);
                    if ((uint32_t)j < cut) m0 = fmaxf(m0, a); else m1 = fmaxf(m1, a);
                }
                if (m0 > 0.0f) atomicMax(&wb[b0], __float_as_uint(m0));
                if (m1 > 0.0f) atomicMax(&wb[b0 + 1], __float_as_uint(m1));  // only past a bin edge
            }
            __syncwarp();
            const uint32_t nbw = bin_of(clen - 1, m.invL) + 1;
            for (uint32_t b = lane; b < nbw; b += 32) gb[b] = wb[b];
        }
        // selection (float compares, as the definition: |G + dW| >= bin max
        // and G != 0; a bin max of 0 leaves only G = 0 or NaN, never sent),
        // R <- G, candidate counts per round
        uint32_t flags = 0;
        if (bpw == 1) {  // one bin: one maximum for the whole chunk
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float* g4 = &Gv[r].x;
                const float* d4 = &Dv[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    flags |= (uint32_t)(fabsf(__fadd_rn(g4[j], d4[j])) >= m_one && g4[j] != 0.0f) << (4 * r + j);
            }
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t e = 4u * (lane + 32 * r);
                if (e >= clen) continue;  // zero-filled: nothing to send
                const float* g4 = &Gv[r].x;
                const float* d4 = &Dv[r].x;
                const uint32_t b0 = bin_of(e, m.invL), cut = (b0 + 1) * L - e;
                const float gm0 = __uint_as_float(wb[b0]);
                const float gm1 = cut < 4 && b0 + 1 < bpw ? __uint_as_float(wb[b0 + 1]) : gm0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float gm = (uint32_t)j < cut ? gm0 : gm1;
                    flags |= (uint32_t)(fabsf(__fadd_rn(g4[j], d4[j])) >= gm && g4[j] != 0.0f) << (4 * r + j);
                }
            }
        }
        if (defer) sent[((uint64_t)m.k * tiles_per_learner + m.lt) * 32 + lane] = (uint16_t)flags;
        uint32_t packed = 0;  // candidates per round, 8 bits each
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (lane + 32 * r);
            const float* g4 = &Gv[r].x;
            packed |= (uint32_t)__popc((flags >> (4 * r)) & 0xFu) << (8 * r);
            if (cal && e + 4 <= clen) {
                *reinterpret_cast<float4*>(Rc + e) = Gv[r];
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (e + j < clen) Rc[e + j] = g4[j];
            }
        }
        // rank inside the chunk: rounds in order, lanes in order (8 bits per round)
        uint32_t incl = packed;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl += y;
        }
        const uint32_t wtot = __shfl_sync(kFull, incl, 31), excl = incl - packed;
        const uint32_t W = (wtot & 0xFFu) + ((wtot >> 8) & 0xFFu) + ((wtot >> 16) & 0xFFu) + (wtot >> 24);
        // the chunk's records start at the first 128-byte boundary of its own
        // pool slots [rel, rel + clen) when they fit after it (ada_emit then
        // reads whole lines), else at rel
        const uint32_t up = (uint32_t)(((16u - (uint32_t)(base & 15u)) & 15u));
        const uint32_t at = W + up <= clen ? m.rel + up : m.rel;
        if (lane == 0) tile_tab[(uint64_t)m.k * tiles_per_learner + m.lt] = make_uint2(at, W);
        // the candidates in rank order (rounds in order, lanes in order, bits in
        // order) into this chunk's stage, which every lane has read into its
        // registers; then one coalesced copy to the pool.  The stage is next
        // written by the copies issued two rounds on, after the __syncwarp below.
        __syncwarp();  // every lane's reads of the stage are done
        uint2* cst = reinterpret_cast<uint2*>(const_cast<float*>(sD));  // kWarpChunk pairs (dW and R halves)
        {
            uint32_t rbase = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                uint32_t pos = rbase + ((excl >> (8 * r)) & 0xFFu);
                rbase += (wtot >> (8 * r)) & 0xFFu;
                const uint32_t e = 4u * (lane + 32 * r);
                const float* g4 = &Gv[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if ((flags >> (4 * r + j)) & 1u) cst[pos] = make_uint2(m.rel + e + j, __float_as_uint(g4[j]));
                    pos += (flags >> (4 * r + j)) & 1u;
                }
            }
        }
        __syncwarp();
        uint2* dst = pool + (uint64_t)m.k * N + at;
        for (uint32_t i = lane; i < W; i += 32) dst[i] = cst[i];
        __syncwarp();  // wb and the stage are rewritten later
    }
    cp_async_wait<0>();
}

__global__ void __launch_bounds__(NT, 3) ada_bins(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                                  uint32_t tiles_per_learner, uint64_t total_tiles,
                                                  const float* __restrict__ dW, float* __restrict__ R,
                                                  const uint32_t* __restrict__ big, uint64_t big_per_learner,
                                                  uint2* __restrict__ tile_tab, double2* __restrict__ tile_sum,
                                                  uint2* __restrict__ pool) {
    __shared__ __align__(16) uint32_t gk[kTileMax];  // |G| bit patterns of the tile
    __shared__ uint32_t bmax[kTileMax];               // bin maxima (|G| bits)
    __shared__ uint64_t scan[NT / 32 + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint32_t t = blockIdx.x; t < (uint32_t)total_tiles; t += gridDim.x) {
        const uint32_t k = t / tiles_per_learner;
        const uint32_t lt = t - k * tiles_per_learner;
        const int s = find_segment_by_tile(plan, S, lt);
        const SegPlan p = plan[s];
        const uint32_t tj = lt - p.tile_off;
        const uint32_t start = tj * p.tile_len;
        const uint32_t len = p.n - start < p.tile_len ? p.n - start : p.tile_len;
        const uint64_t base = (uint64_t)k * N + p.off + start;
        const bool small = p.mode == kModeSmall;
        const uint32_t L = p.L;
        const uint32_t nbt = small ? (p.nbins - tj * p.bpt < p.bpt ? p.nbins - tj * p.bpt : p.bpt) : 0;
        const uint32_t* bigm = big + (uint64_t)k * big_per_learner + p.big_off;
        const float* dWt = dW + base;
        float* Rt = R + base;
        const bool aligned = (((uintptr_t)dWt | (uintptr_t)Rt) & 15) == 0;  // 128-bit accesses

        if (small && p.bpw) continue;  // warp-chunk tiles: ada_bins_warp

        // 1. G = R + dW (registers) and |G| keys to shared memory
        float4 Gv[4], Dv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (r * NT + threadIdx.x);
            if (aligned && e + 4 <= len) {
                Dv[r] = __ldg(reinterpret_cast<const float4*>(dWt + e));
                Gv[r] = *reinterpret_cast<const float4*>(Rt + e);
            } else {
                float* d4 = &Dv[r].x;
                float* g4 = &Gv[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = e + j < len;
                    d4[j] = in ? __ldg(dWt + e + j) : 0.0f;
                    g4[j] = in ? Rt[e + j] : 0.0f;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (r * NT + threadIdx.x);
            Gv[r].x = __fadd_rn(Gv[r].x, Dv[r].x);
            Gv[r].y = __fadd_rn(Gv[r].y, Dv[r].y);
            Gv[r].z = __fadd_rn(Gv[r].z, Dv[r].z);
            Gv[r].w = __fadd_rn(Gv[r].w, Dv[r].w);
            if (small && e < kTileMax)  // |G| bits; NaN counts as 0 (it never wins a maximum)
                *reinterpret_cast<uint4*>(gk + e) = make_uint4(nan0_key(Gv[r].x), nan0_key(Gv[r].y),
                                                               nan0_key(Gv[r].z), nan0_key(Gv[r].w));
        }
        __syncthreads();
        // 2. bin maxima: a warp per bin for L >= 32, a thread per bin below
        if (small) {
            if (L >= 32) {
                for (uint32_t b = warp; b < nbt; b += NT / 32) {
                    const uint32_t lo = b * L, hi = lo + L < len ? lo + L : len;
                    uint32_t m = 0;
                    for (uint32_t i = lo + lane; i < hi; i += 32) m = max(m, gk[i]);
                    m = __reduce_max_sync(kFull, m);
                    if (lane == 0) bmax[b] = m;
                }
            } else {
                for (uint32_t b = threadIdx.x; b < nbt; b += NT) {
                    const uint32_t lo = b * L, hi = lo + L < len ? lo + L : len;
                    uint32_t m = 0;
                    for (uint32_t i = lo; i < hi; ++i) m = max(m, gk[i]);
                    bmax[b] = m;
                }
            }
        }
        __syncthreads();
        // sum of this tile's bin maxima (warp 0): each lane adds a run of
        // bins in fp64, then a fixed shuffle tree; at most 133 fp64 adds
        // per lane, so the relative error stays below 2^-45 (GB300's fp64
        // rate is a few operations per cycle per SM, so it is kept short)
        if (small && warp == 0) {
            const uint32_t per = (nbt + 31) / 32;
            double sm = 0.0;
            for (uint32_t b = lane * per; b < nbt && b < (lane + 1) * per; ++b)
                sm = __dadd_rn(sm, (double)__uint_as_float(bmax[b]));
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) sm = __dadd_rn(sm, __shfl_down_sync(kFull, sm, d));
            if (lane == 0) tile_sum[t] = make_double2(sm, 0.0);
        }
        // 3. selection, residue store, candidate flags (the mode is uniform per tile)
        uint64_t packed = 0;
        uint32_t flags = 0;
        if (small && L >= 4) select_tile<0>(Gv, Dv, len, L, p.invL, nbt, bmax, bigm, start, flags, packed);
        else if (small) select_tile<1>(Gv, Dv, len, L, p.invL, nbt, bmax, bigm, start, flags, packed);
        else select_tile<2>(Gv, Dv, len, L, p.invL, nbt, bmax, bigm, start, flags, packed);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (r * NT + threadIdx.x);
            if (aligned && e + 4 <= len) {
                *reinterpret_cast<float4*>(Rt + e) = Gv[r];
            } else {
                const float* g4 = &Gv[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (e + j < len) Rt[e + j] = g4[j];
            }
        }
        if (!__syncthreads_or(flags != 0)) {
            if (threadIdx.x == 0) tile_tab[t] = make_uint2(p.off + start, 0u);
            continue;
        }
        uint64_t total;
        const uint64_t ex = block_exclusive_scan<NT>(packed, scan, &total);
        uint32_t cnt_total = 0, round_base[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            round_base[r] = cnt_total;
            cnt_total += (uint32_t)(total >> (16 * r)) & 0xFFFFu;
        }
        // the tile's entries go to the pool slots of its own index range
        if (threadIdx.x == 0) tile_tab[t] = make_uint2(p.off + start, cnt_total);
        if (flags) {
            uint2* dst = pool + base;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t fr = (flags >> (4 * r)) & 0xFu;
                if (!fr) continue;
                uint32_t pos = round_base[r] + ((uint32_t)(ex >> (16 * r)) & 0xFFFFu);
                const uint32_t e = 4u * (r * NT + threadIdx.x);
                const float* g4 = &Gv[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if ((fr >> j) & 1u) dst[pos++] = make_uint2(p.off + start + e + j, __float_as_uint(g4[j]));
            }
        }
        __syncthreads();
    }
}

// One CTA per (learner, segment): output slots of the emit groups in index
// order, the segment's count, and its scale = mean of the bin maxima.  The
// work is a few loads per thread, so the CTA is wide (1024 threads) and every
// round issues all of its loads before using any: the largest segments
// (tens of thousands of tiles and bins) take a handful of memory latencies.
constexpr int NTS = 1024;
__global__ void __launch_bounds__(NTS) ada_scan(const SegPlan* __restrict__ plan, int S,
                                               uint32_t tiles_per_learner, const uint2* __restrict__ tile_tab,
                                               const double2* __restrict__ tile_sum, const uint32_t* __restrict__ big,
                                               uint64_t big_per_learner, uint32_t groups_per_learner,
                                               uint32_t* __restrict__ grp_rel,
                                               int64_t* __restrict__ counts, float* __restrict__ scales) {
    __shared__ uint64_t scan[NTS / 32 + 1];
    const int unit = blockIdx.x;
    const int k = unit / S, s = unit - k * S;
    const SegPlan p = plan[s];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t t0 = (uint64_t)k * tiles_per_learner + p.tile_off;
    // output slots of the emit groups (kGroup consecutive tiles; ada_emit
    // ranks the tiles inside a group): chunks of kGroup * NTS tiles whose
    // counts are read coalesced into shared memory (thread t, tiles t + r NTS),
    // then one group per thread and one block scan per chunk
    static_assert(kGroup == 8, "a group is two 16-byte reads of the staged counts");
    __shared__ __align__(16) uint32_t s_cnt[kGroup * NTS];
    uint64_t run = 0;
    const uint32_t ng = (p.ntiles + kGroup - 1) / kGroup;
    uint32_t* gr = grp_rel + (uint64_t)k * groups_per_learner + p.grp_off;
    for (uint32_t tb = 0; tb < p.ntiles; tb += kGroup * NTS) {
        uint32_t cv[kGroup];
#pragma unroll
        for (int r = 0; r < (int)kGroup; ++r) {  // every load of the chunk in flight
            const uint32_t j = tb + (uint32_t)r * NTS + threadIdx.x;
            cv[r] = j < p.ntiles ? tile_tab[t0 + j].y : 0u;
        }
#pragma unroll
        for (int r = 0; r < (int)kGroup; ++r) s_cnt[r * NTS + threadIdx.x] = cv[r];
        __syncthreads();
        const uint4 a = reinterpret_cast<const uint4*>(s_cnt)[2 * threadIdx.x];
        const uint4 b = reinterpret_cast<const uint4*>(s_cnt)[2 * threadIdx.x + 1];
        const uint32_t c = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w;  // group tb / kGroup + t
        uint64_t tot;
        const uint64_t at = run + block_exclusive_scan<NTS>(c, scan, &tot);  // ends synchronised: s_cnt is free
        const uint32_t g = tb / kGroup + threadIdx.x;
        if (g < ng) gr[g] = (uint32_t)at;
        run += tot;
    }
    // Bins kept in the bins array (big bins, warp chunks): a double-float
    // sum (an fp32 pair hi + lo kept exact by TwoSum, renormalised after
    // every 16 terms; about 2^-40 relative, far below the fp32 scale's
    // rounding) in a fixed order: strided shares per thread, a shuffle tree,
    // then the warps in order.  GB300's fp64 rate is a small fraction of its
    // fp32 rate, so fp64 is kept to the final division.
    __shared__ float s_hi[NTS / 32], s_lo[NTS / 32];
    const bool in_bins = p.mode == kModeBig || p.bpw;
    if (in_bins) {
        const uint32_t* bm = big + (uint64_t)k * big_per_learner + p.big_off;
        float hi = 0.0f, lo = 0.0f;
        for (uint32_t b0 = 0; b0 < p.nbins; b0 += 16 * NTS) {  // sixteen loads in flight, then the adds
            float v[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const uint32_t b = b0 + q * NTS + threadIdx.x;
                v[q] = b < p.nbins ? __uint_as_float(bm[b]) : 0.0f;  // + 0 is exact (maxima are >= 0)
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) df_add(hi, lo, v[q], 0.0f);
            df_norm(hi, lo);
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float oh = __shfl_down_sync(kFull, hi, d), ol = __shfl_down_sync(kFull, lo, d);
            df_add(hi, lo, oh, ol);
            df_norm(hi, lo);
        }
        if (lane == 0) {
            s_hi[warp] = hi;
            s_lo[warp] = lo;
        }
        __syncthreads();
    }
    if (in_bins) {
        if (threadIdx.x == 0) {
            float hi = 0.0f, lo = 0.0f;
            for (int q = 0; q < NTS / 32; ++q) {
                df_add(hi, lo, s_hi[q], s_lo[q]);
                df_norm(hi, lo);
            }
            counts[unit] = (int64_t)run;
            scales[unit] = p.nbins ? (float)(__dadd_rn((double)hi, (double)lo) / (double)p.nbins) : 0.0f;
        }
    } else if (warp == 0) {
        // small bins in tiles: a compensated sum of the tiles' fp64 sums in
        // tile order, 32 contiguous runs combined in lane order
        double sm = 0.0, cm = 0.0;
        const uint32_t per = (p.ntiles + 31) / 32;
        for (uint32_t j = lane * per; j < p.ntiles && j < (lane + 1) * per; ++j) {
            const double2 ts = tile_sum[t0 + j];
            csum_add(sm, cm, ts.x);
            cm = __dadd_rn(cm, ts.y);
        }
        double S0 = 0.0, C0 = 0.0;
        for (int l = 0; l < 32; ++l) {
            const double ls = __shfl_sync(kFull, sm, l);
            const double lc = __shfl_sync(kFull, cm, l);
            csum_add(S0, C0, ls);
            C0 = __dadd_rn(C0, lc);
        }
        if (lane == 0) {
            counts[unit] = (int64_t)run;
            scales[unit] = p.nbins ? (float)(__dadd_rn(S0, C0) / (double)p.nbins) : 0.0f;
        }
    }
}

// Last segment whose first emit group is <= g.
__device__ __forceinline__ int find_segment_by_group(const SegPlan* plan, int S, uint32_t g) {
    int lo = 0, hi = S;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(&plan[mid].grp_off) <= g) lo = mid; else hi = mid;
    }
    return lo;
}

// One warp per group of kGroup consecutive tiles of a segment: lanes
// 0..kGroup-1 read the tiles' (pool slot, count) and first output slots, a
// shuffle scan joins their entries into one run, and the lanes walk that run
// 32 entries at a time.  Each entry goes to (entries of the learner's earlier
// segments) + (its tile's first slot in the segment) + (rank in the tile) as
// (index, sign(G)*scale), and its residue becomes R = G - sign(G)*scale
// (with defer, only outside the warp-chunk segments: there the next call's
// bin pass subtracts it).  A learner whose total exceeds cap sends nothing;
// its residue keeps G = R + dW (already stored by the bin pass).  seg_out:
// K*S words of shared memory.
__global__ void __launch_bounds__(NT, 6) ada_emit(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                               uint32_t tiles_per_learner, uint32_t groups_per_learner,
                                               const uint2* __restrict__ tile_tab, const uint32_t* __restrict__ grp_rel,
                                               const uint2* __restrict__ pool, const int64_t* __restrict__ counts,
                                               const float* __restrict__ scales, float* __restrict__ R,
                                               gcsgd_pair* __restrict__ out, uint64_t cap, int K,
                                               int64_t* __restrict__ totals, int defer) {
    extern __shared__ __align__(8) unsigned char emit_smem[];
    uint64_t* s_total = reinterpret_cast<uint64_t*>(emit_smem);            // [K] entries of each learner
    uint32_t* seg_out = reinterpret_cast<uint32_t*>(emit_smem + 8 * K);  // [K][S] first slot of each segment
    __shared__ uint64_t scan[NT / 32 + 1];
    for (int k = 0; k < K; ++k) {
        uint64_t run = 0;
        for (int sb = 0; sb < S; sb += NT) {
            const int s = sb + (int)threadIdx.x;
            const uint64_t c = s < S ? (uint64_t)counts[(uint64_t)k * S + s] : 0;
            uint64_t tot;
            const uint64_t ex = block_exclusive_scan<NT>(c, scan, &tot);
            if (s < S) seg_out[k * S + s] = (uint32_t)(run + ex);
            run += tot;
        }
        if (threadIdx.x == 0) {
            s_total[k] = run;
            if (blockIdx.x == 0) totals[k] = (int64_t)run;
        }
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const uint32_t gw = blockIdx.x * (NT / 32) + (threadIdx.x >> 5), nw = gridDim.x * (NT / 32);
    for (int k = 0; k < K; ++k) {
        if (s_total[k] > cap) continue;  // nothing sent
        const uint2* src = pool + (uint64_t)k * N;
        const uint2* tt = tile_tab + (uint64_t)k * tiles_per_learner;
        const uint32_t* gr = grp_rel + (uint64_t)k * groups_per_learner;
        float* Rk = R + (uint64_t)k * N;
        gcsgd_pair* ok = out + (uint64_t)k * cap;
        // the current segment's group range, tiles and output base, kept while the walk stays inside it
        int s = -1;
        uint32_t g_lo = 1, g_hi = 0, s_tiles = 0, s_tile_off = 0;
        float scale = 0.0f;
        uint64_t ob = 0;
        bool fix_r = true;
        for (uint32_t g = gw; g < groups_per_learner; g += nw) {
            if (g < g_lo || g >= g_hi) {
                s = find_segment_by_group(plan, S, g);
                g_lo = __ldg(&plan[s].grp_off);
                s_tiles = __ldg(&plan[s].ntiles);
                g_hi = g_lo + (s_tiles + kGroup - 1) / kGroup;
                s_tile_off = __ldg(&plan[s].tile_off);
                scale = scales[(uint64_t)k * S + s];
                ob = seg_out[k * S + s];
                fix_r = !(defer && __ldg(&plan[s].mode) == kModeSmall && __ldg(&plan[s].bpw) != 0u);
            }
            const uint32_t j0 = (g - g_lo) * kGroup;
            const uint32_t nt = s_tiles - j0 < kGroup ? s_tiles - j0 : kGroup;
            const uint2 ent = (uint32_t)lane < nt ? tt[s_tile_off + j0 + lane] : make_uint2(0u, 0u);
            uint32_t inc = ent.y;
#pragma unroll
            for (int d = 1; d < (int)kGroup; d <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, inc, d);
                if (lane >= d) inc += y;
            }
            const uint32_t T = __shfl_sync(kFull, inc, kGroup - 1);
            if (T == 0) continue;
            uint32_t incq[kGroup];
#pragma unroll
            for (int q = 0; q < (int)kGroup; ++q) incq[q] = __shfl_sync(kFull, inc, q);
            const uint32_t exc = inc - ent.y;  // rank of the tile's first entry in the group
            const uint64_t gob = ob + gr[g];
            for (uint32_t ib = 0; ib < T; ib += 32) {
                const uint32_t i = ib + lane;
                uint32_t c = 0;  // the tile holding entry i
#pragma unroll
                for (int q = 0; q < (int)kGroup; ++q) c += i >= incq[q];
                const uint32_t cx = __shfl_sync(kFull, ent.x, c & 31);
                const uint32_t ce = __shfl_sync(kFull, exc, c & 31);
                if (i < T) {
                    const uint2 it = src[(uint64_t)cx + (i - ce)];
                    const float gv = __uint_as_float(it.y);
                    const float val = gv > 0.0f ? scale : -scale;
                    if (fix_r) Rk[it.x] = __fsub_rn(gv, val);
                    const uint64_t slot = gob + i;
                    if (slot < cap) {
                        gcsgd_pair pr;
                        pr.idx = it.x;
                        pr.val = val;
                        ok[slot] = pr;
                    }
                }
            }
        }
    }
}

// The pending fix-up of a deferred call, applied to R: for every warp-chunk
// segment of every learner that sent, R[i] -= v for each (i, v) of its part
// of the message (the same fp32 subtraction the eager ada_emit makes).  One
// CTA per (learner, segment); the segment's first slot is the sum of the
// learner's earlier counts.
__global__ void __launch_bounds__(NT) ada_settle(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                                 const int64_t* __restrict__ counts,
                                                 const int64_t* __restrict__ totals, uint64_t cap,
                                                 const gcsgd_pair* __restrict__ out, float* __restrict__ R) {
    __shared__ uint64_t red[NT / 32];
    const int unit = blockIdx.x;
    const int k = unit / S, s = unit - k * S;
    const SegPlan p = plan[s];
    if (!(p.mode == kModeSmall && p.bpw != 0u)) return;
    if ((uint64_t)totals[k] > cap) return;  // the learner sent nothing
    uint64_t part = 0;
    for (int q = threadIdx.x; q < s; q += NT) part += (uint64_t)counts[(uint64_t)k * S + q];
    for (int d = 16; d > 0; d >>= 1) part += __shfl_xor_sync(kFull, part, d);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = part;
    __syncthreads();
    uint64_t first = 0;
    for (int w = 0; w < NT / 32; ++w) first += red[w];
    const uint64_t c = (uint64_t)counts[(uint64_t)k * S + s];
    const gcsgd_pair* L = out + (uint64_t)k * cap;
    float* Rk = R + (uint64_t)k * N;
    for (uint64_t i = threadIdx.x; i < c; i += NT) {
        const uint64_t slot = first + i;
        if (slot >= cap) break;
        const gcsgd_pair e = L[slot];
        if ((uint64_t)e.idx < N) Rk[e.idx] = __fsub_rn(Rk[e.idx], e.val);
    }
}

}  // namespace ada

size_t adacomp_workspace_bytes(const int64_t* off, const int32_t* lt, int S, int K, int64_t cap) {
    ada::HostPlan hp;
    ada::host_plan(off, lt, S, &hp);
    (void)cap;  // the pool has a slot per element, whatever the capacity
    return ada::layout(S, K, off[S], hp, nullptr, nullptr);
}

static int launch_plan(const int64_t* off, int S, const int32_t* lt, int K, const ada::HostPlan& hp,
                       const ada::Workspace& w, cudaStream_t stream) {
    using namespace ada;
    LaunchScope ls("ada_plan", stream);
    if (S <= 256) {
        SegTable<256> st;
        for (int s = 0; s <= S; ++s) st.off[s] = (uint32_t)off[s];
        for (int s = 0; s < S; ++s) st.L[s] = (uint32_t)lt[s];
        ada_plan<256><<<1, 1024, 0, stream>>>(st, S, K, hp.big_per_learner, w.plan, w.big);
    } else {
        SegTable<GCSGD_MAX_SEGMENTS> st;
        for (int s = 0; s <= S; ++s) st.off[s] = (uint32_t)off[s];
        for (int s = 0; s < S; ++s) st.L[s] = (uint32_t)lt[s];
        ada_plan<GCSGD_MAX_SEGMENTS><<<1, 1024, 0, stream>>>(st, S, K, hp.big_per_learner, w.plan, w.big);
    }
    return check_launch("ada_plan");
}

int adacomp_launch(const int64_t* off, int S, const int32_t* lt, int K, const float* dW, float* R, gcsgd_pair* out,
                   int64_t cap, int64_t* counts, float* scales, int64_t* totals, void* ws, size_t ws_bytes,
                   cudaStream_t stream, int defer, int pending) {
    using namespace ada;
    HostPlan hp;
    host_plan(off, lt, S, &hp);
    Workspace w;
    const size_t need = layout(S, K, off[S], hp, ws, &w);
    if (ws_bytes < need)
        return set_error(GCSGD_ERR_WORKSPACE, "adacomp_compress: workspace of %zu bytes, %zu needed", ws_bytes, need);
    const uint64_t N = (uint64_t)off[S];
    const uint64_t T = (uint64_t)K * hp.tiles_per_learner;
    if (T >= ((uint64_t)1 << 32))
        return set_error(GCSGD_ERR_INVALID_ARG, "adacomp_compress: K * tiles = %llu exceeds 2^32", (unsigned long long)T);
    if (emit_smem_bytes(K, S) > kEmitSmemMax)  // checked before anything is enqueued
        return set_error(GCSGD_ERR_INVALID_ARG,
                         "adacomp_compress: K * (4 n_seg + 8) = %lld bytes of emit tables exceed %d",
                         (long long)emit_smem_bytes(K, S), (int)kEmitSmemMax);
    int rc;
    if ((rc = launch_plan(off, S, lt, K, hp, w, stream))) return rc;
    const uint64_t grid_cap = (uint64_t)sm_count() * 3;
    bool any_warp = false, any_other = false, any_big = false;
    for (int s = 0; s < S; ++s) {
        SegPlan sp;
        seg_fields((uint32_t)(off[s + 1] - off[s]), (uint32_t)lt[s], &sp);
        if (sp.mode == kModeEmpty) continue;
        (sp.mode == kModeSmall && sp.bpw ? any_warp : any_other) = true;
        any_big |= sp.mode == kModeBig;
    }
    if (any_big && T > 0) {
        LaunchScope ls("ada_bigmax", stream);
        ada_bigmax<<<(unsigned)(T < grid_cap ? T : grid_cap), NT, 0, stream>>>(
            w.plan, S, N, (uint32_t)hp.tiles_per_learner, T, dW, R, w.big, hp.big_per_learner);
        if ((rc = check_launch("ada_bigmax"))) return rc;
    }
    if (T > 0 && any_warp) {
        LaunchScope ls("ada_bins_warp", stream);
        static bool attr_set[64] = {};
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 64 && !attr_set[dev]) {
            if (cudaFuncSetAttribute(ada_bins_warp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBinsWarpSmem) !=
                cudaSuccess)
                return set_error(GCSGD_ERR_CUDA, "adacomp_compress: cannot raise the shared-memory limit");
            attr_set[dev] = true;
        }
        const uint64_t wgrid = (uint64_t)sm_count() * 6, need_ctas = (T + NTW / 32 - 1) / (NTW / 32);
        ada_bins_warp<<<(unsigned)(need_ctas < wgrid ? need_ctas : wgrid), NTW, kBinsWarpSmem, stream>>>(
            w.plan, S, N, (uint32_t)hp.tiles_per_learner, T, dW, R, w.big, hp.big_per_learner, w.tile_tab, w.pool,
            defer, pending, w.sent, scales, totals, (uint64_t)cap);
        if ((rc = check_launch("ada_bins_warp"))) return rc;
    }
    if (T > 0 && any_other) {
        LaunchScope ls("ada_bins", stream);
        ada_bins<<<(unsigned)(T < grid_cap ? T : grid_cap), NT, 0, stream>>>(
            w.plan, S, N, (uint32_t)hp.tiles_per_learner, T, dW, R, w.big, hp.big_per_learner, w.tile_tab,
            w.tile_sum, w.pool);
        if ((rc = check_launch("ada_bins"))) return rc;
    }
    {
        LaunchScope ls("ada_scan", stream);
        ada_scan<<<(unsigned)(K * S), NTS, 0, stream>>>(w.plan, S, (uint32_t)hp.tiles_per_learner, w.tile_tab,
                                                        w.tile_sum, w.big, hp.big_per_learner,
                                                        (uint32_t)hp.groups_per_learner, w.grp_rel, counts, scales);
        if ((rc = check_launch("ada_scan"))) return rc;
    }
    {
        LaunchScope ls("ada_emit", stream);
        const size_t smem = emit_smem_bytes(K, S);
        if (smem > 48 * 1024) {
            static bool done[64] = {};
            int dev = 0;
            cudaGetDevice(&dev);
            if (dev < 64 && !done[dev]) {
                if (cudaFuncSetAttribute(ada_emit, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kEmitSmemMax) !=
                    cudaSuccess)
                    return set_error(GCSGD_ERR_CUDA, "adacomp_compress: cannot raise the shared-memory limit");
                done[dev] = true;
            }
        }
        ada_emit<<<(unsigned)sm_count() * 6, NT, smem, stream>>>(
            w.plan, S, N, (uint32_t)hp.tiles_per_learner, (uint32_t)hp.groups_per_learner, w.tile_tab, w.grp_rel,
            w.pool, counts, scales, R, out, (uint64_t)cap, K, totals, defer);
        if ((rc = check_launch("ada_emit"))) return rc;
    }
    return GCSGD_OK;
}

int adacomp_settle_launch(const int64_t* off, int S, const int32_t* lt, int K, float* R, const gcsgd_pair* out,
                          int64_t cap, const int64_t* counts, const int64_t* totals, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
    using namespace ada;
    HostPlan hp;
    host_plan(off, lt, S, &hp);
    Workspace w;
    const size_t need = layout(S, K, off[S], hp, ws, &w);
    if (ws_bytes < need)
        return set_error(GCSGD_ERR_WORKSPACE, "adacomp_settle: workspace of %zu bytes, %zu needed", ws_bytes, need);
    if (K * S == 0 || off[S] == 0) return GCSGD_OK;
    int rc;
    if ((rc = launch_plan(off, S, lt, K, hp, w, stream))) return rc;  // the plan, whatever the workspace holds
    LaunchScope ls("ada_settle", stream);
    ada_settle<<<(unsigned)(K * S), NT, 0, stream>>>(w.plan, S, (uint64_t)off[S], counts, totals, (uint64_t)cap, out, R);
    return check_launch("ada_settle");
}

}  // namespace gcsgd

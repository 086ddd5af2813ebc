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
//   ada_plan     one CTA: per-segment plan (bins, tiles), zeroes counters
//   [ada_bigmax] only for segments with L_T > 4096: bin maxima via atomics
//   ada_bins     the bandwidth-bound pass: 128-bit loads of R and dW, G = R+dW,
//                bin maxima in shared memory (warp-aggregated atomicMax on the
//                |G| bit patterns), selection, R <- G stored once, ordered
//                compaction of the selected (index, G) into the learner's
//                pool, and a compensated fp64 sum of the tile's bin maxima
//   ada_scan     one CTA per (learner, segment): prefix of the tile counts in
//                index order, the segment's count and its scale
//   ada_emit     one warp per tile: writes (index, sign(G)*scale) at its
//                ordered slot and fixes the residue R = G - sign(G)*scale.
// Tiles hold whole bins (bins of L_T <= 4096 never straddle tiles), so a
// bin's maximum is final inside one CTA and the first pass is single-read.
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
    uint32_t bpw;       // warp chunks: bins per warp (4 <= L <= 512; a tile is 8 chunks), else 0
};

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
            bpt = (NT / 32) * bpw;
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
};

void host_plan(const int64_t* off, const int32_t* lt, int S, HostPlan* hp) {
    hp->tiles_per_learner = 0;
    hp->big_per_learner = 0;
    for (int s = 0; s < S; ++s) {
        SegPlan p;
        seg_fields((uint32_t)(off[s + 1] - off[s]), (uint32_t)lt[s], &p);
        hp->tiles_per_learner += p.ntiles;
        if (p.mode == kModeBig || p.bpw) hp->big_per_learner += p.nbins;
    }
}

struct Workspace {
    SegPlan* plan;
    uint32_t* pool_cnt;
    uint2* tile_tab;     // (pool slot, count)
    double2* tile_sum;   // compensated sum of the tile's bin maxima
    uint32_t* tile_rel;  // first output slot of the tile within its segment
    uint32_t* big;       // bin maxima (|G| bits) of big-mode segments
    uint2* pool;         // (index within the learner, G bits)
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t layout(int S, int K, int64_t cap, const HostPlan& hp, void* base, Workspace* w) {
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    const uint64_t T = (uint64_t)K * hp.tiles_per_learner;
    const size_t o_plan = take(sizeof(SegPlan) * (size_t)S);
    const size_t o_cnt = take(sizeof(uint32_t) * (size_t)K);
    const size_t o_tt = take(sizeof(uint2) * T);
    const size_t o_ts = take(sizeof(double2) * T);
    const size_t o_tr = take(sizeof(uint32_t) * T);
    const size_t o_big = take(sizeof(uint32_t) * (size_t)K * hp.big_per_learner);
    const size_t o_pool = take(sizeof(uint2) * (size_t)K * (size_t)cap);
    if (w) {
        char* b = (char*)base;
        w->plan = (SegPlan*)(b + o_plan);
        w->pool_cnt = (uint32_t*)(b + o_cnt);
        w->tile_tab = (uint2*)(b + o_tt);
        w->tile_sum = (double2*)(b + o_ts);
        w->tile_rel = (uint32_t*)(b + o_tr);
        w->big = (uint32_t*)(b + o_big);
        w->pool = (uint2*)(b + o_pool);
    }
    return o;
}

// Neumaier step: (s, c) += x.
__device__ __forceinline__ void csum_add(double& s, double& c, double x) {
    const double t = __dadd_rn(s, x);
    c = __dadd_rn(c, fabs(s) >= fabs(x) ? __dadd_rn(__dsub_rn(s, t), x) : __dadd_rn(__dsub_rn(x, t), s));
    s = t;
}

template <int MAXS>
__global__ void __launch_bounds__(1024) ada_plan(SegTable<MAXS> st, int S, int K, uint64_t big_per_learner,
                                                 SegPlan* __restrict__ plan, uint32_t* __restrict__ pool_cnt,
                                                 uint32_t* __restrict__ big) {
    __shared__ uint64_t scan[1024 / 32 + 1];
    __shared__ uint64_t carry[2];
    __shared__ int s_nbig, s_big[64];  // the big-bin segments (all of them are scanned if more)
    if (threadIdx.x < 2) carry[threadIdx.x] = 0;
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
        if (live) {
            p.tile_off = (uint32_t)(c0 + ex_t);
            p.big_off = (uint32_t)(c1 + ex_b);
            plan[s] = p;
            if (p.mode == kModeBig) {
                const int q = atomicAdd(&s_nbig, 1);
                if (q < 64) s_big[q] = s;
            }
        }
        __syncthreads();
    }
    for (int k = threadIdx.x; k < K; k += 1024) pool_cnt[k] = 0;
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

// Warp-chunk tiles (4 <= L_T <= 512): warp w of a tile owns bins
// [w bpw, (w + 1) bpw), at most 512 values, four float4 per lane.  It finds
// their maxima from its registers (one bin: a warp reduction; several:
// shared-memory atomicMax per float4 part), writes them to the bins array
// (ada_scan averages them in fp64, so this pass needs no fp64), selects,
// stores R <- G and ranks its candidates with warp scans; two block
// barriers per tile give the warps their pool offsets.  Lean enough for four
// CTAs per SM, so more loads stay in flight.
__global__ void __launch_bounds__(NT, 4) ada_bins_warp(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                                       uint32_t tiles_per_learner, uint64_t total_tiles,
                                                       const float* __restrict__ dW, float* __restrict__ R,
                                                       uint32_t* __restrict__ bins, uint64_t bins_per_learner,
                                                       uint32_t* __restrict__ pool_cnt, uint2* __restrict__ tile_tab,
                                                       uint2* __restrict__ pool, uint64_t pool_cap) {
    __shared__ uint32_t wbins[NT / 32][kWarpChunk / 4];
    __shared__ uint32_t s_base, s_total;
    __shared__ uint32_t wcnt[NT / 32], wbase[NT / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint32_t t = blockIdx.x; t < (uint32_t)total_tiles; t += gridDim.x) {
        const uint32_t k = t / tiles_per_learner;
        const uint32_t lt = t - k * tiles_per_learner;
        const int s = find_segment_by_tile(plan, S, lt);
        const SegPlan p = plan[s];
        if (p.mode != kModeSmall || !p.bpw) continue;  // other tiles: ada_bins
        const uint32_t tj = lt - p.tile_off;
        const uint32_t start = tj * p.tile_len;
        const uint32_t len = p.n - start < p.tile_len ? p.n - start : p.tile_len;
        const uint64_t base = (uint64_t)k * N + p.off + start;
        const uint32_t L = p.L;
        const float* dWt = dW + base;
        float* Rt = R + base;
        const uint32_t bpw = p.bpw, cl = bpw * L, c0 = (uint32_t)warp * cl;
        const uint32_t clen = c0 < len ? (len - c0 < cl ? len - c0 : cl) : 0u;
        uint32_t* wb = wbins[warp];  // this warp's bin maxima (bpw <= 128)
        const float* dWc = dWt + c0;
        float* Rc = Rt + c0;
        const bool cal = (((uintptr_t)dWc | (uintptr_t)Rc) & 15) == 0;
        float4 Gv[4], Dv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (lane + 32 * r);
            if (cal && e + 4 <= clen) {
                Dv[r] = __ldg(reinterpret_cast<const float4*>(dWc + e));
                Gv[r] = *reinterpret_cast<const float4*>(Rc + e);
            } else {
                float* d4 = &Dv[r].x;
                float* g4 = &Gv[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = e + j < clen;
                    d4[j] = in ? __ldg(dWc + e + j) : 0.0f;
                    g4[j] = in ? Rc[e + j] : 0.0f;
                }
            }
            Gv[r].x = __fadd_rn(Gv[r].x, Dv[r].x);
            Gv[r].y = __fadd_rn(Gv[r].y, Dv[r].y);
            Gv[r].z = __fadd_rn(Gv[r].z, Dv[r].z);
            Gv[r].w = __fadd_rn(Gv[r].w, Dv[r].w);
        }
        // bin maxima (|G|, NaN read as 0): one bin per chunk -> a warp
        // reduction; several -> shared-memory atomicMax per float4 part
        float m_one = 0.0f;
        if (bpw == 1) {
            float m = 0.0f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t e = 4u * (lane + 32 * r);
                const float* g4 = &Gv[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (e + j < clen) m = fmaxf(m, fabsf(g4[j]));
            }
            m_one = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(m)));
        } else {
            for (uint32_t b = lane; b < bpw; b += 32) wb[b] = 0u;
            __syncwarp();
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t e = 4u * (lane + 32 * r);
                if (e >= clen) continue;
                const uint32_t b0 = bin_of(e, p.invL), cut = (b0 + 1) * L - e;
                const float* g4 = &Gv[r].x;
                float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a = e + j < clen ? fabsf(g4[j]) : 0.0f;
                    if ((uint32_t)j < cut) m0 = fmaxf(m0, a); else m1 = fmaxf(m1, a);
                }
                if (m0 > 0.0f) atomicMax(&wb[b0], __float_as_uint(m0));
                if (cut < 4 && m1 > 0.0f) atomicMax(&wb[b0 + 1], __float_as_uint(m1));
            }
            __syncwarp();
        }
        // this chunk's bin maxima to the bins array (ada_scan averages them)
        const uint32_t nbw = clen ? (clen + L - 1) / L : 0u;
        uint32_t* gb = bins + (uint64_t)k * bins_per_learner + p.big_off + tj * p.bpt + (uint32_t)warp * bpw;
        if (bpw == 1) {
            if (lane == 0 && nbw) gb[0] = __float_as_uint(m_one);
        } else {
            for (uint32_t b = lane; b < nbw; b += 32) gb[b] = wb[b];
        }
        // selection (float compares, as the definition), R <- G, candidate counts per round
        uint32_t flags = 0, packed = 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (lane + 32 * r);
            const float* g4 = &Gv[r].x;
            const float* d4 = &Dv[r].x;
            if (e < clen) {
                float gm0 = m_one, gm1 = m_one;
                uint32_t cut = 4;
                if (bpw != 1) {
                    const uint32_t b0 = bin_of(e, p.invL);
                    cut = (b0 + 1) * L - e;
                    gm0 = __uint_as_float(wb[b0]);
                    gm1 = cut < 4 && b0 + 1 < bpw ? __uint_as_float(wb[b0 + 1]) : gm0;
                }
                uint32_t f = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float gm = (uint32_t)j < cut ? gm0 : gm1;
                    const bool sel = e + j < clen && fabsf(__fadd_rn(g4[j], d4[j])) >= gm && gm > 0.0f &&
                                     g4[j] != 0.0f;
                    f |= (uint32_t)sel << j;
                }
                flags |= f << (4 * r);
                packed |= (uint32_t)__popc(f) << (8 * r);
            }
            if (cal && e + 4 <= clen) {
                *reinterpret_cast<float4*>(Rc + e) = Gv[r];
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (e + j < clen) Rc[e + j] = g4[j];
            }
        }
        // rank inside the warp: rounds in order, lanes in order (8 bits per round)
        uint32_t incl = packed;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl += y;
        }
        const uint32_t wtot = __shfl_sync(kFull, incl, 31), excl = incl - packed;
        const uint32_t W = (wtot & 0xFFu) + ((wtot >> 8) & 0xFFu) + ((wtot >> 16) & 0xFFu) + (wtot >> 24);
        if (lane == 0) wcnt[warp] = W;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t tot = 0;
            for (int q = 0; q < NT / 32; ++q) {
                wbase[q] = tot;
                tot += wcnt[q];
            }
            uint32_t b = 0;
            if (tot) b = atomicAdd(&pool_cnt[k], tot);
            s_base = b;
            s_total = tot;
            tile_tab[t] = make_uint2(tot ? b : 0u, tot);
        }
        __syncthreads();
        const uint32_t pb = s_base;
        if (flags && (uint64_t)pb + s_total <= pool_cap) {
            uint2* dst = pool + (uint64_t)k * pool_cap + pb + wbase[warp];
            uint32_t rb = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t fr = (flags >> (4 * r)) & 0xFu;
                uint32_t pos = rb + ((excl >> (8 * r)) & 0xFFu);
                rb += (wtot >> (8 * r)) & 0xFFu;
                if (!fr) continue;
                const uint32_t e = 4u * (lane + 32 * r);
                const float* g4 = &Gv[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if ((fr >> j) & 1u) dst[pos++] = make_uint2(p.off + start + c0 + e + j, __float_as_uint(g4[j]));
            }
        }

    }
}

__global__ void __launch_bounds__(NT, 3) ada_bins(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                                  uint32_t tiles_per_learner, uint64_t total_tiles,
                                                  const float* __restrict__ dW, float* __restrict__ R,
                                                  const uint32_t* __restrict__ big, uint64_t big_per_learner,
                                                  uint32_t* __restrict__ pool_cnt, uint2* __restrict__ tile_tab,
                                                  double2* __restrict__ tile_sum, uint2* __restrict__ pool,
                                                  uint64_t pool_cap) {
    __shared__ __align__(16) uint32_t gk[kTileMax];  // |G| bit patterns of the tile
    __shared__ uint32_t bmax[kTileMax];               // bin maxima (|G| bits)
    __shared__ uint64_t scan[NT / 32 + 1];
    __shared__ uint32_t s_base;
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
            if (threadIdx.x == 0) tile_tab[t] = make_uint2(0u, 0u);
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
        if (threadIdx.x == 0) {
            const uint32_t b = atomicAdd(&pool_cnt[k], cnt_total);
            s_base = b;
            tile_tab[t] = make_uint2(b, cnt_total);
        }
        __syncthreads();
        const uint32_t pb = s_base;
        if ((uint64_t)pb + cnt_total <= pool_cap && flags) {
            uint2* dst = pool + (uint64_t)k * pool_cap + pb;
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

// One CTA per (learner, segment): output slots of the tiles in index order,
// the segment's count, and its scale = mean of the bin maxima.
__global__ void __launch_bounds__(NT) ada_scan(const SegPlan* __restrict__ plan, int S,
                                               uint32_t tiles_per_learner, const uint2* __restrict__ tile_tab,
                                               const double2* __restrict__ tile_sum, const uint32_t* __restrict__ big,
                                               uint64_t big_per_learner, uint32_t* __restrict__ tile_rel,
                                               int64_t* __restrict__ counts, float* __restrict__ scales) {
    __shared__ uint64_t scan[NT / 32 + 1];
    const int unit = blockIdx.x;
    const int k = unit / S, s = unit - k * S;
    const SegPlan p = plan[s];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t t0 = (uint64_t)k * tiles_per_learner + p.tile_off;
    uint64_t run = 0;
    for (uint32_t jb = 0; jb < p.ntiles; jb += NT) {
        const uint32_t j = jb + threadIdx.x;
        const uint32_t c = j < p.ntiles ? tile_tab[t0 + j].y : 0u;
        uint64_t tot;
        const uint64_t ex = block_exclusive_scan<NT>(c, scan, &tot);
        if (j < p.ntiles) tile_rel[t0 + j] = (uint32_t)(run + ex);
        run += tot;
    }
    // bins kept in the bins array (big bins, warp chunks): every thread adds
    // a strided share in fp64 (plain adds: at most nbins / 256 per thread),
    // then a fixed tree; the error stays far below the fp32 scale's rounding
    __shared__ double s_wsum[NT / 32];
    double bins_sum = 0.0;
    const bool in_bins = p.mode == kModeBig || p.bpw;
    if (in_bins) {
        const uint32_t* bm = big + (uint64_t)k * big_per_learner + p.big_off;
        double su = 0.0;
        for (uint32_t b = threadIdx.x; b < p.nbins; b += NT) su = __dadd_rn(su, (double)__uint_as_float(bm[b]));
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) su = __dadd_rn(su, __shfl_down_sync(kFull, su, d));
        if (lane == 0) s_wsum[warp] = su;
        __syncthreads();
        for (int q = 0; q < NT / 32; ++q) bins_sum = __dadd_rn(bins_sum, s_wsum[q]);
    }
    if (warp == 0) {
        // compensated sum of the tiles' sums of bin maxima in bin order, 32 contiguous runs
        double sm = 0.0, cm = 0.0;
        if (p.mode == kModeSmall && !p.bpw) {
            const uint32_t per = (p.ntiles + 31) / 32;
            for (uint32_t j = lane * per; j < p.ntiles && j < (lane + 1) * per; ++j) {
                const double2 ts = tile_sum[t0 + j];
                csum_add(sm, cm, ts.x);
                cm = __dadd_rn(cm, ts.y);
            }
        } else if (in_bins && lane == 0) {
            sm = bins_sum;
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

// Last segment whose first element is <= idx.
__device__ __forceinline__ int find_segment_by_index(const SegPlan* plan, int S, uint32_t idx) {
    int lo = 0, hi = S;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(&plan[mid].off) <= idx) lo = mid; else hi = mid;
    }
    return lo;
}

// One thread per pool entry: the entry's index gives its segment and tile,
// and its distance from the tile's pool base gives its rank inside the tile,
// so its output slot is (entries of the learner's earlier segments) + (the
// tile's first slot in its segment) + rank.  It writes (index,
// sign(G)*scale) there and fixes the residue R = G - sign(G)*scale.  A
// learner whose total exceeds cap sends nothing; its residue keeps G = R + dW
// (already stored by ada_bins).  seg_out: K*S words of shared memory.
__global__ void __launch_bounds__(NT) ada_emit(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                               uint32_t tiles_per_learner, const uint2* __restrict__ tile_tab,
                                               const uint32_t* __restrict__ tile_rel, const uint2* __restrict__ pool,
                                               const uint32_t* __restrict__ pool_cnt, uint64_t pool_cap,
                                               const int64_t* __restrict__ counts, const float* __restrict__ scales,
                                               float* __restrict__ R, gcsgd_pair* __restrict__ out, uint64_t cap,
                                               int K, int64_t* __restrict__ totals) {
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
    const uint64_t stride = (uint64_t)gridDim.x * NT;
    for (int k = 0; k < K; ++k) {
        if (s_total[k] > cap) continue;  // nothing sent
        const uint32_t pc = pool_cnt[k];
        const uint2* src = pool + (uint64_t)k * pool_cap;
        const uint2* tt = tile_tab + (uint64_t)k * tiles_per_learner;
        const uint32_t* tr = tile_rel + (uint64_t)k * tiles_per_learner;
        float* Rk = R + (uint64_t)k * N;
        gcsgd_pair* ok = out + (uint64_t)k * cap;
        for (uint64_t q = (uint64_t)blockIdx.x * NT + threadIdx.x; q < pc; q += stride) {
            const uint2 it = src[q];
            const int s = find_segment_by_index(plan, S, it.x);
            const SegPlan p = plan[s];
            const uint32_t t = p.tile_off + (it.x - p.off) / p.tile_len;
            const uint2 ent = tt[t];
            const uint64_t slot = (uint64_t)seg_out[k * S + s] + tr[t] + ((uint32_t)q - ent.x);
            const float g = __uint_as_float(it.y);
            const float scale = scales[(uint64_t)k * S + s];
            const float val = g > 0.0f ? scale : -scale;
            Rk[it.x] = __fsub_rn(g, val);
            if (slot < cap) {
                gcsgd_pair pr;
                pr.idx = it.x;
                pr.val = val;
                ok[slot] = pr;
            }
        }
    }
}

}  // namespace ada

size_t adacomp_workspace_bytes(const int64_t* off, const int32_t* lt, int S, int K, int64_t cap) {
    ada::HostPlan hp;
    ada::host_plan(off, lt, S, &hp);
    return ada::layout(S, K, cap, hp, nullptr, nullptr);
}

int adacomp_launch(const int64_t* off, int S, const int32_t* lt, int K, const float* dW, float* R, gcsgd_pair* out,
                   int64_t cap, int64_t* counts, float* scales, int64_t* totals, void* ws, size_t ws_bytes,
                   cudaStream_t stream) {
    using namespace ada;
    HostPlan hp;
    host_plan(off, lt, S, &hp);
    Workspace w;
    const size_t need = layout(S, K, cap, hp, ws, &w);
    if (ws_bytes < need)
        return set_error(GCSGD_ERR_WORKSPACE, "adacomp_compress: workspace of %zu bytes, %zu needed", ws_bytes, need);
    const uint64_t N = (uint64_t)off[S];
    const uint64_t T = (uint64_t)K * hp.tiles_per_learner;
    if (T >= ((uint64_t)1 << 32))
        return set_error(GCSGD_ERR_INVALID_ARG, "adacomp_compress: K * tiles = %llu exceeds 2^32", (unsigned long long)T);
    int rc;
    {
        LaunchScope ls("ada_plan", stream);
        if (S <= 256) {
            SegTable<256> st;
            for (int s = 0; s <= S; ++s) st.off[s] = (uint32_t)off[s];
            for (int s = 0; s < S; ++s) st.L[s] = (uint32_t)lt[s];
            ada_plan<256><<<1, 1024, 0, stream>>>(st, S, K, hp.big_per_learner, w.plan, w.pool_cnt, w.big);
        } else {
            SegTable<GCSGD_MAX_SEGMENTS> st;
            for (int s = 0; s <= S; ++s) st.off[s] = (uint32_t)off[s];
            for (int s = 0; s < S; ++s) st.L[s] = (uint32_t)lt[s];
            ada_plan<GCSGD_MAX_SEGMENTS><<<1, 1024, 0, stream>>>(st, S, K, hp.big_per_learner, w.plan, w.pool_cnt,
                                                                w.big);
        }
        if ((rc = check_launch("ada_plan"))) return rc;
    }
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
        const uint64_t wgrid = (uint64_t)sm_count() * 4;
        ada_bins_warp<<<(unsigned)(T < wgrid ? T : wgrid), NT, 0, stream>>>(
            w.plan, S, N, (uint32_t)hp.tiles_per_learner, T, dW, R, w.big, hp.big_per_learner, w.pool_cnt,
            w.tile_tab, w.pool, (uint64_t)cap);
        if ((rc = check_launch("ada_bins_warp"))) return rc;
    }
    if (T > 0 && any_other) {
        LaunchScope ls("ada_bins", stream);
        ada_bins<<<(unsigned)(T < grid_cap ? T : grid_cap), NT, 0, stream>>>(
            w.plan, S, N, (uint32_t)hp.tiles_per_learner, T, dW, R, w.big, hp.big_per_learner, w.pool_cnt,
            w.tile_tab, w.tile_sum, w.pool, (uint64_t)cap);
        if ((rc = check_launch("ada_bins"))) return rc;
    }
    {
        LaunchScope ls("ada_scan", stream);
        ada_scan<<<(unsigned)(K * S), NT, 0, stream>>>(w.plan, S, (uint32_t)hp.tiles_per_learner, w.tile_tab,
                                                        w.tile_sum, w.big, hp.big_per_learner, w.tile_rel, counts,
                                                        scales);
        if ((rc = check_launch("ada_scan"))) return rc;
    }
    {
        LaunchScope ls("ada_emit", stream);
        const size_t smem = sizeof(uint32_t) * (size_t)K * S + sizeof(uint64_t) * (size_t)K;
        if (smem > 200 * 1024)
            return set_error(GCSGD_ERR_INVALID_ARG, "adacomp_compress: K * n_seg = %d too large (at most ~51000)",
                             K * S);
        if (smem > 48 * 1024) {
            static bool done[64] = {};
            int dev = 0;
            cudaGetDevice(&dev);
            if (dev < 64 && !done[dev]) {
                if (cudaFuncSetAttribute(ada_emit, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
                    cudaSuccess)
                    return set_error(GCSGD_ERR_CUDA, "adacomp_compress: cannot raise the shared-memory limit");
                done[dev] = true;
            }
        }
        ada_emit<<<(unsigned)sm_count() * 4, NT, smem, stream>>>(w.plan, S, N, (uint32_t)hp.tiles_per_learner,
                                                                 w.tile_tab, w.tile_rel, w.pool, w.pool_cnt,
                                                                 (uint64_t)cap, counts, scales, R, out,
                                                                 (uint64_t)cap, K, totals);
        if ((rc = check_launch("ada_emit"))) return rc;
    }
    return GCSGD_OK;
}

}  // namespace gcsgd

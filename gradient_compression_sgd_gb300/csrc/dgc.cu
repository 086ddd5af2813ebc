// dgc.cu -- Deep Gradient Compression for K learners in one pass over HBM.
//
// "Deep Gradient Compression: Reducing the Communication Bandwidth for
// Distributed Training": local gradient clipping (Appendix C), momentum
// correction (section 3.2), exact top-k sparsification with local
// accumulation (section 3.1) and momentum factor masking (section 3.3), in
// the order of the vanilla-momentum algorithm of Appendix D.
//
// Launch sequence of one call (all on the caller's stream, no host sync):
//   [dgc_sumsq]   per-learner sum of squares, only when clipping is on
//   dgc_prepare   one CTA per (learner, segment) plus one: the extra CTA
//                 writes the per-segment plan (k_s, tiles, pool sizes and
//                 offsets) and each learner's clip scale; the others read a
//                 strided sample of the updated |v| of their segment and take
//                 a threshold hint safely below the k-th largest value
//   dgc_update    the bandwidth-bound pass: reads g, u, v once (128-bit
//                 loads), writes u', v' once, and appends every |v'| >= hint
//                 to a small per-(learner, segment) candidate pool, keeping
//                 index order inside each 4096-element tile
//   dgc_select    one CTA per (learner, segment): stages the candidates (in
//                 index order, through the tile table) or, for small segments
//                 and when the hint failed, the segment's v' in shared memory,
//                 finds the k-th largest |v'| exactly by radix select, then
//                 emits (index, v') in index order with ties to the lower
//                 index and masks u = v = 0 at the sent indices; a pool too
//                 large to stage is selected and emitted from global memory
//   [dgc_pack]    sampled threshold only: packs each learner's per-tensor
//                 regions into one list
// The answer never depends on the hint: a pool is used only when it provably
// contains every entry of the top k (at least k candidates, no overflow).
// Nesterov momentum (Appendix B, as read) is the same sequence with the
// update of dgc_prepare's samples and of dgc_update templated on it.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include <cooperative_groups.h>

#include "common.cuh"
#include "dgc.cuh"

namespace gcsgd {
namespace dgc {

constexpr int NT = 256;                  // threads per CTA of dgc_update and dgc_sumsq
constexpr int NTS = 512;                 // threads per CTA of dgc_select
constexpr int NTP = 512;                 // threads per CTA of dgc_prepare
constexpr uint32_t kSmallK = 32;         // raw segments with k <= 32 ...
constexpr uint32_t kSmallN = 8192;       // ... and at most 8192 values use the register top-k
constexpr int kTile = 4096;              // elements per dgc_update tile (NT x 4 float4)
constexpr uint32_t kRawMax = 8192;       // segments up to this size select from v' directly
constexpr uint32_t kSampleMax = 16384;   // largest hint sample (keys held in shared memory)
constexpr uint32_t kSampleAbove = 48;    // sampled entries expected above the hint
constexpr uint32_t kSampleBlock = 64;    // consecutive values per sample block
constexpr uint32_t kPoolFloor = 512;     // smallest expected candidate count
constexpr uint32_t kStageItems = 10240;  // candidates dgc_select stages in shared memory (80 KB)
constexpr int kChunkTiles = 2 * NTS;     // tile-table entries dgc_select scans per round
static_assert(kChunkTiles <= kCandMax, "the crowded-tile list lives in the radix scratch");
constexpr size_t kStageBytes = kStageItems * sizeof(uint2);  // also holds kRawMax floats
static_assert(kStageBytes >= kRawMax * sizeof(float), "the stage must hold a raw segment");
constexpr int kSumsqBlocks = 512;        // CTAs per learner in dgc_sumsq

// Plan of one segment.  sample_frac = 0: the exact step (the hint only
// steers the candidate pool).  sample_frac > 0: the sampled threshold (the
// system-analysis reading: m = floor(sample_frac n) rounded down to whole
// 64-value blocks; a tensor with no whole block is selected exactly; tau is
// the round(k m / n)-th largest sampled |v| and is the selection threshold
// itself).  Sampled tensors of at most kRawMax values take tau from the
// staged v' in dgc_select; larger ones get it from dgc_prepare as the hint.
__host__ __device__ __forceinline__ void seg_fields(uint32_t n, double density, double sample_frac, SegPlan* p) {
    p->n = n;
    p->k = dgc_k_of(density, n);
    p->ntiles = (n + kTile - 1) / kTile;
    p->cap = 0;
    p->m = 0;
    p->a = 0;
    p->sampled = 0;
    uint64_t ms = 0;  // sampled threshold: whole blocks in floor(sample_frac n) values
    if (sample_frac > 0.0) {
        ms = (uint64_t)(sample_frac * (double)n);
        ms -= ms % kSampleBlock;
    }
    if (n == 0) {
        p->kind = kKindEmpty;
    } else if (ms > 0) {
        p->sampled = 1;
        p->m = (uint32_t)ms;
        const uint64_t a = ((uint64_t)p->k * ms + n / 2) / n;
        p->a = (uint32_t)(a < 1 ? 1 : (a > ms ? ms : a));
        if (n <= kRawMax) {
            p->kind = kKindRaw;
        } else {
            p->kind = kKindPool;
            const uint64_t R = p->k > kPoolFloor ? p->k : kPoolFloor;  // expected candidates ~ k
            const uint64_t cap = 4 * R + 256;
            p->cap = (uint32_t)(cap < n ? cap : n);
        }
    } else if (n <= kRawMax || 5ull * p->k > n) {
        p->kind = kKindRaw;
    } else {
        p->kind = kKindPool;
        const uint64_t R = 5ull * p->k / 2 > kPoolFloor ? 5ull * p->k / 2 : kPoolFloor;  // expected candidates
        const uint64_t cap = 4 * R + 256;
        p->cap = (uint32_t)(cap < n ? cap : n);
        uint64_t m = (uint64_t)kSampleAbove * n / R;
        if (m > kSampleMax) m = kSampleMax;
        m &= ~(uint64_t)(kSampleBlock - 1);
        if (m < kSampleBlock) m = kSampleBlock;
        p->m = (uint32_t)m;
        uint64_t a = (R * m + n / 2) / n;
        p->a = (uint32_t)(a < 1 ? 1 : (a > m ? m : a));
    }
}

// Sample keys of a pool segment that do not fit dgc_prepare's shared memory
// go to the workspace (sampled threshold only).
__host__ __device__ __forceinline__ bool sample_spills(const SegPlan& p) {
    return p.kind == kKindPool && p.sampled && p.m > kSampleMax;
}

// Host mirror of the plan's totals (workspace sizing and argument checks).
int host_plan(const int64_t* off, int S, double density, double sample_frac, HostPlan* hp) {
    hp->tiles_per_learner = 0;
    hp->pool_per_learner = 0;
    hp->out_per_learner = 0;
    hp->pool_segments = 0;
    hp->skeys_per_learner = 0;
    for (int s = 0; s < S; ++s) {
        SegPlan p;
        seg_fields((uint32_t)(off[s + 1] - off[s]), density, sample_frac, &p);
        hp->tiles_per_learner += p.ntiles;
        hp->pool_per_learner += p.cap;
        hp->out_per_learner += p.k;
        hp->pool_segments += p.kind == kKindPool;
        if (sample_spills(p)) hp->skeys_per_learner += p.m;
    }
    return 0;
}

// ---------------------------------------------------------------- kernels

// Sum of squares of learner blockIdx.y's gradient over a fixed slice.  Each
// square is split exactly into x*x = p + e (p rounded, e = fma(x, x, -p));
// the terms are summed as double-float (an fp32 pair kept exact by TwoSum,
// renormalised every 8 elements; ~2^-40 relative), reduced in a fixed tree
// and stored as fp64: deterministic, and no per-element fp64 arithmetic,
// whose rate on GB300 is a small fraction of fp32's.
__device__ __forceinline__ void dsq_add(float& hi, float& lo, float x) {
    const float p = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -p);
    const float s = __fadd_rn(hi, p);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(err, e));
}
__device__ __forceinline__ void dsq_merge(float& hi, float& lo, float oh, float ol) {
    const float s = __fadd_rn(hi, oh);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(oh, bp));
    lo = __fadd_rn(lo, __fadd_rn(err, ol));
    hi = s;
}
__device__ __forceinline__ void dsq_norm(float& hi, float& lo) {
    const float s = __fadd_rn(hi, lo);
    lo = __fsub_rn(lo, __fsub_rn(s, hi));
    hi = s;
}

__global__ void __launch_bounds__(NT) dgc_sumsq(const float* __restrict__ grad, uint64_t N,
                                                 double* __restrict__ part) {
    __shared__ float red_hi[NT / 32], red_lo[NT / 32];
    const uint64_t k = blockIdx.y;
    const uint64_t chunk = (N + gridDim.x - 1) / gridDim.x;
    const uint64_t lo_i = (uint64_t)blockIdx.x * chunk;
    const uint64_t hi_i = lo_i + chunk < N ? lo_i + chunk : N;
    const float* g = grad + k * N;
    float hi = 0.0f, lo = 0.0f;
    for (uint64_t i0 = lo_i; i0 < hi_i; i0 += 8 * (uint64_t)NT) {
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // eight loads in flight
            const uint64_t i = i0 + (uint64_t)j * NT + threadIdx.x;
            x[j] = i < hi_i ? __ldg(g + i) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) dsq_add(hi, lo, x[j]);
        dsq_norm(hi, lo);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float oh = __shfl_down_sync(kFull, hi, d), ol = __shfl_down_sync(kFull, lo, d);
        dsq_merge(hi, lo, oh, ol);
        dsq_norm(hi, lo);
    }
    if ((threadIdx.x & 31) == 0) {
        red_hi[threadIdx.x >> 5] = hi;
        red_lo[threadIdx.x >> 5] = lo;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float h = 0.0f, l = 0.0f;
        for (int w = 0; w < NT / 32; ++w) {
            dsq_merge(h, l, red_hi[w], red_lo[w]);
            dsq_norm(h, l);
        }
        part[k * gridDim.x + blockIdx.x] = __dadd_rn((double)h, (double)l);
    }
}

// Local gradient clipping scale (Appendix C): thr_k = thr / sqrt(N_nodes),
// c = thr_k / ||G|| when ||G|| > thr_k.  Called by a whole warp: lane l adds
// partial sums 16l .. 16l+15 as a pairwise tree, then a butterfly over the
// lanes adds the lane sums in a fixed tree (a + b and b + a are the same
// bits), so every lane of every CTA that evaluates this gets the same c.
// The partials are non-negative, so the tree sum needs no compensation
// (relative error below 9 * 2^-53).  Callers test clip_thr > 0 first and
// call it only then: kept out of line so that its fp64 square root and
// division, slow on GB300's few FP64 units, never run when clipping is off
// (inlined, the unclipped path paid ~4 us per CTA for them).
__device__ __noinline__ float clip_scale_warp(const double* __restrict__ part, int k, float clip_thr,
                                              int clip_nodes) {
    static_assert(kSumsqBlocks == 16 * 32, "16 partial sums per lane");
    const double* pk = part + (uint64_t)k * kSumsqBlocks + 16 * (threadIdx.x & 31);
    double x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = pk[i];
#pragma unroll
    for (int w = 1; w < 16; w <<= 1)
#pragma unroll
        for (int i = 0; i < 16; i += 2 * w) x[i] = x[i] + x[i + w];
    double s = x[0];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) s = s + __shfl_xor_sync(kFull, s, d);
    const double norm = sqrt(s);
    const double thr_k = (double)clip_thr / sqrt((double)clip_nodes);
    return norm > thr_k ? (float)(thr_k / norm) : 1.0f;
}

// The update of one element: u' = m*u + c*g, v' = v + u' (vanilla momentum,
// Appendix D), or with NEST (Nesterov momentum, Appendix B, as read: the
// accumulated state takes the look-ahead step) v' = v + (m*u' + c*g).
template <bool NEST>
__device__ __forceinline__ void dgc_elem(float g, float& u, float& v, float m, float c) {
    const float gc = __fmul_rn(g, c);
    u = __fadd_rn(__fmul_rn(m, u), gc);
    v = __fadd_rn(v, NEST ? __fadd_rn(__fmul_rn(m, u), gc) : u);
}

// The last CTA writes the per-segment plan, the clip scales and the order in
// which dgc_select takes the segments (largest first).  The other CTAs walk
// the (learner, segment) units that have a candidate pool, one per CTA when
// there are enough CTAs: each samples m of the segment's values in
// 32-element blocks spread evenly over it and computes the updated |v|
// there exactly as dgc_update will.  The
// hint is the a-th largest sampled key (a = R m / n <= 48 for R =
// max(2.5k, 512) expected candidates), found exactly by radix select over the
// sampled keys held in shared memory.
// Being a rank estimate, it keeps the candidate count near R whatever the
// distribution of
// |v| -- including the pile-up of entries just below the send threshold that
// accumulation builds.  The hint only steers speed: dgc_select checks that
// the pool holds the top k.
template <int MAXS, bool NEST>
__global__ void __launch_bounds__(NTP, 2) dgc_prepare(SegOffsets<MAXS> so, PoolList<MAXS> pl, int S, int K,
                                                     double density, double sample_frac,
                                                     float clip_thr, int clip_nodes, const double* __restrict__ part,
                                                     SegPlan* __restrict__ plan, float* __restrict__ clip_c,
                                                     uint16_t* __restrict__ order, uint64_t N,
                                                     const float* __restrict__ grad, const float* __restrict__ u,
                                                     const float* __restrict__ v, float momentum,
                                                     uint32_t* __restrict__ hint, uint32_t* __restrict__ pool_cnt,
                                                     uint32_t* __restrict__ skeys, uint64_t skeys_per_learner) {
    extern __shared__ __align__(16) uint32_t keys[];  // kSampleMax
    __shared__ RadixSmem rs;
    __shared__ uint64_t carry[3];
    __shared__ float s_c;
    __shared__ SegPlan s_plan;
    if (blockIdx.x == gridDim.x - 1) {  // the extra CTA: plan, order, clip scales
        if (threadIdx.x < 3) carry[threadIdx.x] = 0;
        __syncthreads();
        for (int base = 0; base < S; base += NTP) {
            const int s = base + (int)threadIdx.x;
            SegPlan p;
            const bool live = s < S;
            seg_fields(live ? so.off[s + 1] - so.off[s] : 0u, density, sample_frac, &p);
            p.off = live ? so.off[s] : 0u;
            uint64_t tot;
            const uint64_t ex_pool = block_exclusive_scan<NTP>(live ? p.cap : 0, rs.scan, &tot);
            const uint64_t c0 = carry[0];
            __syncthreads();
            if (threadIdx.x == 0) carry[0] = c0 + tot;
            const uint64_t ex_tile = block_exclusive_scan<NTP>(live ? p.ntiles : 0, rs.scan, &tot);
            const uint64_t c1 = carry[1];
            __syncthreads();
            if (threadIdx.x == 0) carry[1] = c1 + tot;
            const uint64_t ex_out = block_exclusive_scan<NTP>(live ? p.k : 0, rs.scan, &tot);
            const uint64_t c2 = carry[2];
            __syncthreads();
            if (threadIdx.x == 0) carry[2] = c2 + tot;
            if (live) {
                p.pool_off = (uint32_t)(c0 + ex_pool);
                p.tile_off = (uint32_t)(c1 + ex_tile);
                p.out_off = (uint32_t)(c2 + ex_out);
                plan[s] = p;
                order[s] = pl.order[s];  // segments by size, largest first (from the host)
            }
            __syncthreads();
        }
        if (clip_thr > 0.0f) {
            for (int k = (int)threadIdx.x >> 5; k < K; k += NTP / 32) {  // one warp per learner
                const float c = clip_scale_warp(part, k, clip_thr, clip_nodes);
                if ((threadIdx.x & 31) == 0) clip_c[k] = c;
            }
        } else {
            for (int k = (int)threadIdx.x; k < K; k += NTP) clip_c[k] = 1.0f;
        }
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int P = (int)pl.n_pool;
    const int samplers = (int)gridDim.x - 1;
    for (int pj = blockIdx.x; pj < K * P; pj += samplers) {  // only segments with a candidate pool
        const int k = pj / P, q = pj - k * P;
        const int s = pl.seg[q];
        const int unit = k * S + s;
        if (warp == 0) {
            const float c = clip_thr > 0.0f ? clip_scale_warp(part, k, clip_thr, clip_nodes) : 1.0f;
            if (lane == 0) {
                s_c = c;
                pool_cnt[unit] = 0;
            }
        }
        if (threadIdx.x == 32) {  // one thread evaluates the plan (fp64; GB300 has few FP64 units)
            SegPlan sp;
            seg_fields(so.off[s + 1] - so.off[s], density, sample_frac, &sp);
            sp.off = so.off[s];
            s_plan = sp;
        }
        __syncthreads();
        const SegPlan p = s_plan;
        const float c = s_c;
        const uint32_t nblk = p.m / kSampleBlock;
        const uint32_t stride = p.n / nblk;  // >= 64 since m <= n: blocks never overlap
        // keys of a sample larger than the shared array go to the learner's spill region
        const bool spill = sample_spills(p);
        uint32_t* kdst = spill ? skeys + (uint64_t)k * skeys_per_learner + pl.koff[q] : keys;
        const uint64_t base = (uint64_t)k * N + p.off;
        const float* gs = grad + base;
        const float* us = u + base;
        const float* vs = v + base;
        const bool hint_mode = !p.sampled;  // the hint: a <= 48 (see below), no histogram while sampling
        uint32_t t1 = 0, t2 = 0, t3 = 0;     // hint mode: the lane's three largest keys (a multiset)
        radix_hist_clear<NTP>(rs);
        __syncthreads();
        // sample element j of block b sits at b * stride + j; a warp issues
        // the loads of kB blocks (two values per lane each) before using any
        constexpr int kB = 4, kH = kSampleBlock / 32;
        for (uint32_t b0 = warp; b0 < nblk; b0 += kB * (NTP / 32)) {
            float gg[kB][kH], uu[kB][kH], vv[kB][kH];
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                const uint32_t b = b0 + j * (NTP / 32);
#pragma unroll
                for (int h = 0; h < kH; ++h) {
                    gg[j][h] = uu[j][h] = vv[j][h] = 0.0f;
                    if (b < nblk) {
                        const uint32_t i = b * stride + 32 * h + lane;
                        gg[j][h] = __ldg(gs + i);
                        uu[j][h] = __ldg(us + i);
                        vv[j][h] = __ldg(vs + i);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                const uint32_t b = b0 + j * (NTP / 32);
                if (b < nblk) {
#pragma unroll
                    for (int h = 0; h < kH; ++h) {
                        dgc_elem<NEST>(gg[j][h], uu[j][h], vv[j][h], momentum, c);
                        const uint32_t key = mag_key(vv[j][h]);
                        kdst[b * kSampleBlock + 32 * h + lane] = key;
                        if (hint_mode) {
                            top3_insert(key, t1, t2, t3);
                        } else {
                            radix_hist_add(rs, key);
                        }
                    }
                }
            }
        }
        __syncthreads();
        if (spill) {
            // the sampled threshold over spilled keys (written by this CTA before
            // the barrier above; plain loads, not the read-only path): the shared
            // array is free and takes the first digit's bucket
            const SelectResult sr = radix_select_desc<NTP, 3, true>(
                [&](uint64_t i, uint32_t* key) { *key = kdst[i]; return true; }, p.m, p.a, rs, true, keys,
                kSampleMax);
            if (threadIdx.x == 0) hint[unit] = sr.thresh;
        } else if (p.sampled) {
            // the sampled threshold: the a-th largest sampled key, exactly
            const SelectResult sr = radix_select_desc<NTP, 3>(
                [&](uint64_t i, uint32_t* key) { *key = keys[i]; return true; }, p.m, p.a, rs, true);
            if (threadIdx.x == 0) hint[unit] = sr.thresh;
        } else {
            // The hint: the a-th largest sampled key, a <= 48, among the
            // keys at or above the per-warp top-3 bound (top3_bound).
            const uint32_t L = top3_bound<NTP>(t1, t2, t3, rs);
            // warp-uniform trip count (the ballots need every lane); a lane's
            // four keys are all in range or all out (m is a multiple of 64)
            for (uint32_t w0 = 128u * warp; w0 < p.m; w0 += 128u * (NTP / 32)) {
                const uint32_t i0 = w0 + 4u * lane;
                const bool in = i0 < p.m;
                const uint4 q4 = in ? *reinterpret_cast<const uint4*>(keys + i0) : make_uint4(0u, 0u, 0u, 0u);
                cand_append(rs, q4.x, in && q4.x >= L);
                cand_append(rs, q4.y, in && q4.y >= L);
                cand_append(rs, q4.z, in && q4.z >= L);
                cand_append(rs, q4.w, in && q4.w >= L);
            }
            __syncthreads();
            const uint32_t c = rs.sel[3];
            uint32_t h = 0;
            if (c <= (uint32_t)NTP) {
                h = rank_select<NTP>(rs, c, p.a).thresh;
            } else if (c <= (uint32_t)kCandMax) {
                h = radix_select_desc<NTP, 3>([&](uint64_t i, uint32_t* key) { *key = rs.cand[i]; return true; },
                                              c, p.a, rs, false, keys + p.m, kSampleMax - p.m)
                        .thresh;
            } else {
                h = radix_select_desc<NTP, 3>([&](uint64_t i, uint32_t* key) { *key = keys[i]; return true; },
                                              p.m, p.a, rs, false)
                        .thresh;
            }
            if (threadIdx.x == 0) hint[unit] = h > 1u ? h : 1u;
        }
        __syncthreads();
    }
}

__device__ __forceinline__ int find_segment_by_tile(const SegPlan* plan, int S, uint32_t lt) {
    int lo = 0, hi = S;  // last s with tile_off <= lt and ntiles > 0
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(&plan[mid].tile_off) <= lt) lo = mid; else hi = mid;
    }
    return lo;
}

// The bandwidth-bound pass.  Persistent CTAs walk (learner, segment, tile)
// work items.  Per tile: 128-bit loads of g, u, v (4 per array per thread,
// all issued before use), fused momentum-corrected update, 128-bit stores of
// u', v', then an ordered block compaction of the candidates |v'| >= hint
// into the segment's pool; the tile's (pool offset, count) goes to tile_tab.
template <bool NEST>
__global__ void __launch_bounds__(NT, 3) dgc_update(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                                    uint32_t tiles_per_learner, uint64_t total_tiles,
                                                    const float* __restrict__ grad, float* __restrict__ u,
                                                    float* __restrict__ v, float momentum,
                                                    const float* __restrict__ clip_c,
                                                    const uint32_t* __restrict__ hint,
                                                    uint32_t* __restrict__ pool_cnt, uint2* __restrict__ tile_tab,
                                                    uint2* __restrict__ pool, uint64_t pool_per_learner) {
    __shared__ uint64_t scan[NT / 32 + 1];
    __shared__ uint32_t s_base;
    for (uint32_t t = blockIdx.x; t < (uint32_t)total_tiles; t += gridDim.x) {
        const uint32_t k = t / tiles_per_learner;
        const uint32_t lt = t - k * tiles_per_learner;
        const int s = find_segment_by_tile(plan, S, lt);
        const SegPlan p = plan[s];
        const uint32_t start = (lt - p.tile_off) * (uint32_t)kTile;
        const uint32_t len = p.n - start < (uint32_t)kTile ? p.n - start : (uint32_t)kTile;
        const uint64_t base = (uint64_t)k * N + p.off + start;
        const uint32_t unit = k * S + s;
        const uint32_t h = p.kind == kKindPool ? __ldg(&hint[unit]) : 0xffffffffu;  // no candidates
        const float c = __ldg(&clip_c[k]);
        const bool aligned =  // 128-bit accesses need 16-byte addresses
            (((uintptr_t)(grad + base) | (uintptr_t)(u + base) | (uintptr_t)(v + base)) & 15) == 0;

        float4 G[4], U[4], V[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (r * NT + threadIdx.x);
            if (aligned && e + 4 <= len) {
                G[r] = __ldg(reinterpret_cast<const float4*>(grad + base + e));
                U[r] = *reinterpret_cast<const float4*>(u + base + e);
                V[r] = *reinterpret_cast<const float4*>(v + base + e);
            } else {
                float* g4 = &G[r].x;
                float* u4 = &U[r].x;
                float* v4 = &V[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = e + j < len;
                    g4[j] = in ? __ldg(grad + base + e + j) : 0.0f;
                    u4[j] = in ? u[base + e + j] : 0.0f;
                    v4[j] = in ? v[base + e + j] : 0.0f;
                }
            }
        }
        uint64_t packed = 0;  // candidate count of round r in bits [16r, 16r+16)
        uint32_t flags = 0;   // bit 4r+j: element j of round r is a candidate
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t e = 4u * (r * NT + threadIdx.x);
            float* g4 = &G[r].x;
            float* u4 = &U[r].x;
            float* v4 = &V[r].x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                dgc_elem<NEST>(g4[j], u4[j], v4[j], momentum, c);
                const bool cand = (e + j < len) && mag_key(v4[j]) >= h;
                flags |= (uint32_t)cand << (4 * r + j);
            }
            packed |= (uint64_t)__popc((flags >> (4 * r)) & 0xFu) << (16 * r);
            if (aligned && e + 4 <= len) {
                *reinterpret_cast<float4*>(u + base + e) = U[r];
                *reinterpret_cast<float4*>(v + base + e) = V[r];
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (e + j < len) {
                        u[base + e + j] = u4[j];
                        v[base + e + j] = v4[j];
                    }
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
            const uint32_t b = atomicAdd(&pool_cnt[unit], cnt_total);
            s_base = b;
            tile_tab[t] = make_uint2(b, cnt_total);
        }
        __syncthreads();
        const uint32_t pb = s_base;
        if ((uint64_t)pb + cnt_total <= p.cap) {
            uint2* dst = pool + (uint64_t)k * pool_per_learner + p.pool_off + pb;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                uint32_t pos = round_base[r] + ((uint32_t)(ex >> (16 * r)) & 0xFFFFu);
                const uint32_t e = 4u * (r * NT + threadIdx.x);
                const float* v4 = &V[r].x;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if ((flags >> (4 * r + j)) & 1u) dst[pos++] = make_uint2(start + e + j, __float_as_uint(v4[j]));
            }
        }
        __syncthreads();  // s_base and scan are reused by the next tile
    }
}

// Ordered emission over `count` items given in ascending index order: an
// item is sent if its key > T, or == T and fewer than `ties` equal keys
// precede it; its slot is slot0 + (#greater before it) + min(#equal before
// it, ties).
// Sent items are written to dst and u = v = 0 at their indices (momentum
// factor masking).  Warp w owns one contiguous run of the items: a first
// sweep counts its greater and equal keys (warp ballots), one barrier shares
// the 16 warp counts, and a second sweep writes, ranking each item by ballots
// inside its warp.  wsum: NTS / 32 words of shared memory.  R: rounds of 32
// items whose loads are issued together (items read from global memory).
template <int R = 1, class Get>
__device__ void emit_in_order(Get get, uint32_t count, uint32_t T, uint32_t ties, const SegPlan& p,
                              gcsgd_pair* __restrict__ dst, float* __restrict__ u, float* __restrict__ v,
                              uint64_t ebase, uint2* wsum, uint32_t slot0 = 0) {
    constexpr uint32_t NW = NTS / 32;
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t per = (count + NW * 32 - 1) / (NW * 32) * 32;  // items per warp, a multiple of 32
    const uint32_t lo = warp * per < count ? warp * per : count;
    const uint32_t hi = lo + per < count ? lo + per : count;
    const unsigned below = (1u << lane) - 1u;
    uint32_t ngt = 0, neq = 0;
    for (uint32_t b = lo; b < hi; b += 32 * R) {
        uint32_t bits[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {  // every load of the R rounds in flight before the first ballot
            const uint32_t i = b + 32 * r + lane;
            uint32_t loc = 0;
            bits[r] = 0;
            if (i < hi) get(i, &loc, &bits[r]);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t i = b + 32 * r + lane;
            const uint32_t key = bits[r] & 0x7fffffffu;
            ngt += __popc(__ballot_sync(kFull, i < hi && key > T));
            neq += __popc(__ballot_sync(kFull, i < hi && key == T));
        }
    }
    if (lane == 0) wsum[warp] = make_uint2(ngt, neq);
    __syncthreads();
    uint32_t gb = 0, eb = 0;
    for (uint32_t w = 0; w < warp; ++w) {
        const uint2 c = wsum[w];
        gb += c.x;
        eb += c.y;
    }
    if (ngt > 0 || (neq > 0 && eb < ties)) {
        for (uint32_t b = lo; b < hi; b += 32 * R) {
            uint32_t locs[R], bits[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t i = b + 32 * r + lane;
                locs[r] = 0;
                bits[r] = 0;
                if (i < hi) get(i, &locs[r], &bits[r]);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t i = b + 32 * r + lane;
                const uint32_t key = bits[r] & 0x7fffffffu;
                const bool gt = i < hi && key > T, eq = i < hi && key == T;
                const unsigned mg = __ballot_sync(kFull, gt), me = __ballot_sync(kFull, eq);
                const uint32_t g_before = gb + __popc(mg & below), e_before = eb + __popc(me & below);
                const uint32_t slot = slot0 + g_before + (e_before < ties ? e_before : ties);
                if ((gt || (eq && e_before < ties)) && slot < p.k && locs[r] < p.n) {
                    gcsgd_pair pr;
                    pr.idx = p.off + locs[r];
                    pr.val = __uint_as_float(bits[r]);
                    dst[slot] = pr;
                    u[ebase + locs[r]] = 0.0f;
                    v[ebase + locs[r]] = 0.0f;
                }
                gb += __popc(mg);
                eb += __popc(me);
            }
        }
    }
    __syncthreads();  // wsum is reused
}

// Largest 64-bit value across a warp.
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const uint64_t y = __shfl_xor_sync(kFull, x, d);
        x = y > x ? y : x;
    }
    return x;
}

// Exact top-k for a segment of n <= kSmallN values and k <= kSmallK, held in
// registers (thread t owns elements t + j NTS).  The order key packs
// (|v| bits, ~index) into 64 bits, so the largest key is the largest
// magnitude with ties to the lower index and all keys are distinct.  Each
// warp takes its own top k by k rounds of warp max (only the winning thread
// rescans its elements); warp 0 merges the 16 warps' candidates the same
// way; the k winners go out in index order and u = v = 0 there.
__device__ void small_topk(const SegPlan& p, const float* __restrict__ vseg, float* __restrict__ u,
                           float* __restrict__ v, uint64_t ebase, gcsgd_pair* __restrict__ dst, uint64_t* cand,
                           uint64_t* win) {
    constexpr int J = kSmallN / NTS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t jn = (p.n + NTS - 1) / NTS;  // elements per thread in use (uniform)
    uint32_t mag[J];
    uint32_t live = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        mag[j] = 0;
        const uint32_t i = threadIdx.x + j * NTS;
        if ((uint32_t)j < jn && i < p.n) {
            mag[j] = mag_key(vseg[i]);
            live |= 1u << j;
        }
    }
    auto best_of = [&]() {
        uint64_t b = 0;
#pragma unroll
        for (int j = 0; j < J; ++j)
            if ((live >> j) & 1u) {
                const uint64_t key = ((uint64_t)mag[j] << 32) | (uint32_t)~(threadIdx.x + j * NTS);
                b = key > b ? key : b;
            }
        return b;
    };
    uint64_t tb = best_of();
    uint32_t r = 0;
    for (; r < p.k; ++r) {
        const uint64_t wb = warp_max_u64(tb);
        if (wb == 0) break;  // this warp has no elements left
        if (tb == wb) {      // the owner drops its winner and rescans
            const uint32_t idx = ~(uint32_t)wb;
            live &= ~(1u << ((idx - threadIdx.x) / NTS));
            tb = best_of();
        }
        if (lane == 0) cand[warp * kSmallK + r] = wb;
    }
    for (uint32_t q = r + lane; q < kSmallK; q += 32) cand[warp * kSmallK + q] = 0;
    __syncthreads();
    if (warp == 0) {
        constexpr int C = (NTS / 32) * kSmallK / 32;  // candidates per lane
        uint64_t c[C];
        uint32_t cl = 0;
#pragma unroll
        for (int i = 0; i < C; ++i) {
            c[i] = cand[lane + 32 * i];
            if (c[i]) cl |= 1u << i;
        }
        auto best_c = [&]() {
            uint64_t b = 0;
#pragma unroll
            for (int i = 0; i < C; ++i)
                if ((cl >> i) & 1u) b = c[i] > b ? c[i] : b;
            return b;
        };
        uint64_t cb = best_c();
        for (uint32_t q = 0; q < p.k; ++q) {
            const uint64_t wb = warp_max_u64(cb);
            if (cb == wb && wb != 0) {
#pragma unroll
                for (int i = 0; i < C; ++i)
                    if (c[i] == wb) cl &= ~(1u << i);
                cb = best_c();
            }
            if (lane == 0) win[q] = wb;
        }
    }
    __syncthreads();
    if (threadIdx.x < p.k) {
        const uint32_t idx = ~(uint32_t)win[threadIdx.x];
        uint32_t rank = 0;
        for (uint32_t q = 0; q < p.k; ++q) rank += ~(uint32_t)win[q] < idx;
        if (idx < p.n) {
            gcsgd_pair pr;
            pr.idx = p.off + idx;
            pr.val = vseg[idx];
            dst[rank] = pr;
            u[ebase + idx] = 0.0f;
            v[ebase + idx] = 0.0f;
        }
    }
}

// Stages the candidates of tiles [t_begin, t_end) of a pool in index order
// (tiles in order, items of a tile in order) at stage[0 ..), noting the range
// of their keys in kmin/kmax (this thread's share).  Per chunk of tiles: a
// block scan of the tile counts gives each tile's stage offset; every tile
// writes its own (chunk-local) index into the stage slots it owns (a warp
// per tile holding more than 16); then every thread gathers its slots'
// items, eight loads in flight, reading the tile from the slot.  The caller
// guarantees at most kStageItems items.  Returns the items staged.  Every
// thread must call it; ends synchronised.
__device__ uint32_t stage_tiles(const uint2* __restrict__ tt, uint32_t t_begin, uint32_t t_end,
                                const uint2* __restrict__ items, uint2* stage, uint32_t* toff, uint32_t* tbase,
                                RadixSmem& rs, uint32_t& kmin, uint32_t& kmax) {
    uint32_t run = 0;
    for (uint32_t tb = t_begin; tb < t_end; tb += kChunkTiles) {
        constexpr int TPT = kChunkTiles / NTS;  // tiles per thread
        uint2 ent[TPT];
        uint32_t c = 0;
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
            const uint32_t jt = tb + TPT * threadIdx.x + j;
            ent[j] = jt < t_end ? tt[jt] : make_uint2(0u, 0u);
            c += ent[j].y;
        }
        if (threadIdx.x == 0) rs.sel[3] = 0;  // tiles with many candidates, tagged by warps below
        uint64_t tot;
        uint32_t ex = (uint32_t)block_exclusive_scan<NTS>(c, rs.scan, &tot);
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
            const uint32_t lt = TPT * threadIdx.x + j;
            toff[lt] = ex;
            tbase[lt] = ent[j].x;
            if (ent[j].y <= 16) {
                for (uint32_t i = 0; i < ent[j].y && run + ex + i < kStageItems; ++i) stage[run + ex + i].x = lt;
            } else {
                rs.cand[atomicAdd(&rs.sel[3], 1u)] = lt;  // kChunkTiles <= kCandMax slots
            }
            ex += ent[j].y;
        }
        __syncthreads();
        {  // a warp per crowded tile tags its slots
            const uint32_t nbig = rs.sel[3], lane = threadIdx.x & 31;
            for (uint32_t b = threadIdx.x >> 5; b < nbig; b += NTS / 32) {
                const uint32_t lt = rs.cand[b], o = toff[lt];
                const uint32_t cnt = (lt + 1 < (uint32_t)kChunkTiles ? toff[lt + 1] : (uint32_t)tot) - o;
                for (uint32_t i = lane; i < cnt && run + o + i < kStageItems; i += 32) stage[run + o + i].x = lt;
            }
        }
        __syncthreads();
        const uint32_t total = (uint32_t)tot;
        constexpr int IPT = 8;
        for (uint32_t q0 = 0; q0 < total; q0 += IPT * NTS) {
            uint2 it[IPT];
#pragma unroll
            for (int jj = 0; jj < IPT; ++jj) {
                const uint32_t q = q0 + jj * NTS + threadIdx.x;
                it[jj] = make_uint2(0u, 0u);
                if (q < total && run + q < kStageItems) {
                    const uint32_t lt = stage[run + q].x;
                    it[jj] = items[tbase[lt] + (q - toff[lt])];
                }
            }
#pragma unroll
            for (int jj = 0; jj < IPT; ++jj) {
                const uint32_t q = q0 + jj * NTS + threadIdx.x;
                if (q < total && run + q < kStageItems) {
                    stage[run + q] = it[jj];
                    const uint32_t key = it[jj].y & 0x7fffffffu;
                    kmin = min(kmin, key);
                    kmax = max(kmax, key);
                }
            }
        }
        run += total;
        __syncthreads();
    }
    return run;
}

// Arguments of dgc_select and dgc_select_big.
struct SelectArgs {
    const SegPlan* plan;
    int S;
    uint64_t N;
    uint32_t tiles_per_learner;
    float* u;
    float* v;
    const uint32_t* pool_cnt;
    const uint2* tile_tab;
    const uint2* pool;
    uint64_t pool_per_learner;
    gcsgd_pair* out;
    uint64_t cap;
    int64_t* counts;
    int64_t* totals;
    uint32_t out_per_learner;
    const uint16_t* order;
    int K;
    int sampled;
};

// Shared memory of one selecting CTA.
struct SelectSmem {
    unsigned char* stage_raw;  // kStageBytes, dynamic
    RadixSmem* rs;
    uint32_t* toff;  // [kChunkTiles]
    uint32_t* tbase;  // [kChunkTiles]
    uint2* wsum;  // [NTS / 32]
};

// Pools whose expected candidate count (about cap / 4) is too large for one
// CTA's stage go to dgc_select_big; a smaller pool that happens to outgrow
// the stage is read from global memory by select_unit.
__host__ __device__ __forceinline__ bool big_pool(const SegPlan& p) {
    return p.kind == kKindPool && p.cap > 4 * kStageItems;
}

// The exact top-k and ordered emission of unit (learner k, segment s) by
// one CTA.  Sources, fastest first:
//   pool, staged  -- the candidates (k <= count <= pool capacity, so they hold
//                    the whole top k), copied tile by tile in index order into
//                    shared memory when they fit (kStageItems);
//   raw, small k  -- segments of at most kSmallN values with k <= 32: top k
//                    kept in registers (small_topk);
//   raw, staged   -- other segments of at most kRawMax values: v' copied to
//                    shared memory;
//   global        -- anything else (a failed hint, or more candidates than
//                    fit): the same selection read from global memory.
__device__ void select_unit(const SelectArgs& A, const SelectSmem& M, int k, int s) {
    const SegPlan* __restrict__ plan = A.plan;
    const int S = A.S;
    const uint64_t N = A.N;
    const uint32_t tiles_per_learner = A.tiles_per_learner;
    float* __restrict__ u = A.u;
    float* __restrict__ v = A.v;
    const uint32_t* __restrict__ pool_cnt = A.pool_cnt;
    const uint2* __restrict__ tile_tab = A.tile_tab;
    const uint2* __restrict__ pool = A.pool;
    const uint64_t pool_per_learner = A.pool_per_learner;
    gcsgd_pair* __restrict__ out = A.out;
    const uint64_t cap = A.cap;
    int64_t* __restrict__ counts = A.counts;
    unsigned char* stage_raw = M.stage_raw;
    uint2* stage = reinterpret_cast<uint2*>(stage_raw);
    float* stagef = reinterpret_cast<float*>(stage_raw);
    RadixSmem& rs = *M.rs;
    uint32_t* toff = M.toff;
    uint32_t* tbase = M.tbase;
    uint2* wsum = M.wsum;
    const int unit = k * S + s;
    const SegPlan p = plan[s];
    const uint32_t pc = p.kind == kKindPool ? pool_cnt[unit] : 0;
    // sampled threshold, fewer than k above it: every candidate is sent
    const bool take_all = p.kind == kKindPool && p.sampled && pc < p.k;
    const bool raw_sampled = p.kind == kKindRaw && p.sampled;  // counted once tau is known
    if (threadIdx.x == 0 && !raw_sampled) counts[unit] = take_all ? pc : p.k;
    if (p.k == 0) return;
    const uint64_t ebase = (uint64_t)k * N + p.off;
    const bool pool_ok = p.kind == kKindPool && (pc >= p.k || take_all) && pc <= p.cap;
    const uint2* items = pool + (uint64_t)k * pool_per_learner + p.pool_off;
    const uint2* tt = tile_tab + (uint64_t)k * tiles_per_learner + p.tile_off;
    const float* vseg = v + ebase;
    gcsgd_pair* dst = out + (uint64_t)k * cap + p.out_off;

    if (pool_ok && pc <= kStageItems) {
        uint32_t kmin = 0xffffffffu, kmax = 0;
        stage_tiles(tt, 0, p.ntiles, items, stage, toff, tbase, rs, kmin, kmax);
        uint32_t T = 0, ties = pc;  // take_all: every key >= 0 goes, in index order
        if (!take_all) {
            // the candidates share their leading bits (all sit just above the
            // hint): select over their own key range [kmin, kmax]
            kmin = __reduce_min_sync(kFull, kmin);
            kmax = __reduce_max_sync(kFull, kmax);
            if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = make_uint2(kmin, kmax);
            __syncthreads();
#pragma unroll
            for (int w = 0; w < NTS / 32; ++w) {
                kmin = min(kmin, wsum[w].x);
                kmax = max(kmax, wsum[w].y);
            }
            __syncthreads();  // wsum is reused by the emission
            const int bits = kmax > kmin ? 32 - __clz(kmax - kmin) : 0;
            const SelectResult r = radix_select_span<NTS>(
                [&](uint32_t i, uint32_t* key) { *key = stage[i].y & 0x7fffffffu; }, pc, p.k, kmin, bits, rs,
                rs.cand, (uint32_t)kCandMax);
            T = r.thresh;
            ties = r.ties;
        }
        emit_in_order(
            [&](uint32_t i, uint32_t* loc, uint32_t* bits) {
                const uint2 it = stage[i];
                *loc = it.x;
                *bits = it.y;
            },
            pc, T, ties, p, dst, u, v, ebase, wsum);
        return;
    }
    if (!pool_ok && p.n <= kSmallN && p.k <= kSmallK && !raw_sampled) {
        small_topk(p, vseg, u, v, ebase, dst, reinterpret_cast<uint64_t*>(stage_raw),
                   reinterpret_cast<uint64_t*>(stage_raw) + (NTS / 32) * kSmallK);
        return;
    }
    if (raw_sampled) {
        // the sampled threshold on a segment of at most kRawMax values: v' is
        // staged, tau = the a-th largest |v'| of the sample blocks (block b at
        // b * stride), and either every |v'| >= tau is sent (fewer than k) or,
        // the hierarchical second step, the exact top k
        for (uint32_t i = threadIdx.x; i < p.n; i += NTS) stagef[i] = vseg[i];
        __syncthreads();
        const uint32_t stride = p.n / (p.m / kSampleBlock);
        const SelectResult st = radix_select_desc<NTS, 3>(
            [&](uint64_t i, uint32_t* key) {
                *key = mag_key(stagef[(uint32_t)i / kSampleBlock * stride + ((uint32_t)i & (kSampleBlock - 1))]);
                return true;
            },
            p.m, p.a, rs, false);
        const uint32_t tau = st.thresh;
        uint32_t above = 0;
        for (uint32_t i = threadIdx.x; i < p.n; i += NTS) above += mag_key(stagef[i]) >= tau;
        uint64_t tot;
        block_exclusive_scan<NTS>(above, rs.scan, &tot);
        uint32_t T = tau, ties = p.n;  // fewer than k at or above tau: all of them
        if (tot >= p.k) {
            const SelectResult r = radix_select_desc<NTS, 3>(
                [&](uint64_t i, uint32_t* key) { *key = mag_key(stagef[i]); return true; }, p.n, p.k, rs, false);
            T = r.thresh;
            ties = r.ties;
        }
        if (threadIdx.x == 0) counts[unit] = tot >= p.k ? (int64_t)p.k : (int64_t)tot;
        emit_in_order(
            [&](uint32_t i, uint32_t* loc, uint32_t* bits) {
                *loc = i;
                *bits = __float_as_uint(stagef[i]);
            },
            p.n, T, ties, p, dst, u, v, ebase, wsum);
        return;
    }
    if (!pool_ok && p.n <= kRawMax) {
        // kRawMax = 4 float4 per thread: issue every load before the first store
        const bool aligned = ((uintptr_t)vseg & 15) == 0;
        float4 q[kRawMax / (4 * NTS)];
#pragma unroll
        for (int r = 0; r < (int)(kRawMax / (4 * NTS)); ++r) {
            const uint32_t e0 = 4 * (r * NTS + threadIdx.x);
            if (aligned && e0 + 4 <= p.n) {
                q[r] = *reinterpret_cast<const float4*>(vseg + e0);
            } else {
                q[r].x = e0 < p.n ? vseg[e0] : 0.f;
                q[r].y = e0 + 1 < p.n ? vseg[e0 + 1] : 0.f;
                q[r].z = e0 + 2 < p.n ? vseg[e0 + 2] : 0.f;
                q[r].w = e0 + 3 < p.n ? vseg[e0 + 3] : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < (int)(kRawMax / (4 * NTS)); ++r) {
            const uint32_t e0 = 4 * (r * NTS + threadIdx.x);
            if (e0 + 4 <= p.n) {
                *reinterpret_cast<float4*>(stagef + e0) = q[r];
            } else {
                if (e0 < p.n) stagef[e0] = q[r].x;
                if (e0 + 1 < p.n) stagef[e0 + 1] = q[r].y;
                if (e0 + 2 < p.n) stagef[e0 + 2] = q[r].z;
            }
        }
        __syncthreads();
        auto emit_stage = [&](uint32_t T, uint32_t ties) {
            emit_in_order(
                [&](uint32_t i, uint32_t* loc, uint32_t* bits) {
                    *loc = i;
                    *bits = __float_as_uint(stagef[i]);
                },
                p.n, T, ties, p, dst, u, v, ebase, wsum);
        };
        if (p.k <= 48) {  // a small top: the top-3 bound and an exact rank, no histogram
            // rolled loops over the staged keys: a CTA runs each phase once, and
            // unrolled it would be long straight-line code fetched line by line
            uint32_t t1 = 0, t2 = 0, t3 = 0;
#pragma unroll 1
            for (uint32_t i = threadIdx.x; i < p.n; i += NTS) top3_insert(mag_key(stagef[i]), t1, t2, t3);
            const uint32_t L = top3_bound<NTS>(t1, t2, t3, rs);
#pragma unroll 1
            for (uint32_t i0 = 0; i0 < p.n; i0 += NTS) {  // CTA-uniform trip count (cand_append is warp-wide)
                const uint32_t i = i0 + threadIdx.x;
                const uint32_t key = i < p.n ? mag_key(stagef[i]) : 0u;
                cand_append(rs, key, i < p.n && key >= L);
            }
            __syncthreads();
            const uint32_t c = rs.sel[3];
            if (c <= (uint32_t)NTS) {
                const SelectResult r = rank_select<NTS>(rs, c, p.k);
                emit_stage(r.thresh, r.ties);
                return;
            }
        }
        radix_hist_clear<NTS>(rs);
        __syncthreads();  // the histogram is clear everywhere before any count
#pragma unroll
        for (int r = 0; r < (int)(kRawMax / (4 * NTS)); ++r) {
            const uint32_t e0 = 4 * (r * NTS + threadIdx.x);
            if (e0 < p.n) radix_hist_add(rs, mag_key(q[r].x));
            if (e0 + 1 < p.n) radix_hist_add(rs, mag_key(q[r].y));
            if (e0 + 2 < p.n) radix_hist_add(rs, mag_key(q[r].z));
            if (e0 + 3 < p.n) radix_hist_add(rs, mag_key(q[r].w));
        }
        __syncthreads();
        const SelectResult r = radix_select_desc<NTS, 3>(
            [&](uint64_t i, uint32_t* key) { *key = mag_key(stagef[i]); return true; }, p.n, p.k, rs, true);
        emit_stage(r.thresh, r.ties);
        return;
    }
    if (!pool_ok) {
        // the hint failed: select among all of the segment's v' in global memory
        const SelectResult r = radix_select_desc<NTS, 3, true>(
            [&](uint64_t i, uint32_t* key) { *key = mag_key(vseg[i]); return true; }, p.n, p.k, rs, false,
            reinterpret_cast<uint32_t*>(stage_raw), (uint32_t)(kStageBytes / sizeof(uint32_t)));
        emit_in_order<8>(
            [&](uint32_t i, uint32_t* loc, uint32_t* bits) {
                *loc = i;
                *bits = __float_as_uint(vseg[i]);
            },
            p.n, r.thresh, r.ties, p, dst, u, v, ebase, wsum);
        return;
    }
    // a valid pool too large to stage: select from global memory, emit through the tile table
    uint32_t T = 0, ties = pc;  // take_all: every candidate goes
    if (!take_all) {
        // the stage is free on this path: it takes the threshold bucket's keys
        const SelectResult r = radix_select_desc<NTS, 3, true>(
            [&](uint64_t i, uint32_t* key) { *key = __ldg(&items[i].y) & 0x7fffffffu; return true; }, pc, p.k, rs,
            false, reinterpret_cast<uint32_t*>(stage_raw), (uint32_t)(kStageBytes / sizeof(uint32_t)));
        T = r.thresh;
        ties = r.ties;
    }
    uint32_t run_gt = 0, run_eq = 0;
    for (uint32_t tb = 0; tb < p.ntiles; tb += kChunkTiles) {  // kChunkTiles tiles a round, TPT per thread
        constexpr int TPT = kChunkTiles / NTS;
        uint2 ent[TPT];
        uint32_t c = 0;
#pragma unroll
        for (int jj = 0; jj < TPT; ++jj) {
            const uint32_t j = tb + TPT * threadIdx.x + jj;
            ent[jj] = j < p.ntiles ? tt[j] : make_uint2(0u, 0u);
            c += ent[jj].y;
        }
        uint64_t tot;
        uint32_t ex = (uint32_t)block_exclusive_scan<NTS>(c, rs.scan, &tot);
#pragma unroll
        for (int jj = 0; jj < TPT; ++jj) {
            toff[TPT * threadIdx.x + jj] = ex;
            tbase[TPT * threadIdx.x + jj] = ent[jj].x;
            ex += ent[jj].y;
        }
        __syncthreads();
        const uint32_t chunk_items = (uint32_t)tot;
        constexpr int IPT = 8;  // consecutive items per thread per round: eight loads in flight
        for (uint32_t ib = 0; ib < chunk_items; ib += IPT * NTS) {
            const uint32_t q0 = ib + IPT * threadIdx.x;
            uint32_t local[IPT], bits[IPT];
            uint32_t ngt = 0, neq = 0;
            int lo = 0;  // last tile with toff <= q0, then walked forward item by item
            if (q0 < chunk_items) {
                int hi = kChunkTiles;
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (toff[mid] <= q0) lo = mid; else hi = mid;
                }
            }
#pragma unroll
            for (int j = 0; j < IPT; ++j) {
                const uint32_t q = q0 + j;
                local[j] = 0xffffffffu;
                bits[j] = 0u;
                if (q < chunk_items) {
                    while (lo + 1 < kChunkTiles && toff[lo + 1] <= q) ++lo;
                    const uint2 it = items[tbase[lo] + (q - toff[lo])];
                    local[j] = it.x;
                    bits[j] = it.y;
                }
            }
#pragma unroll
            for (int j = 0; j < IPT; ++j) {
                const uint32_t key = bits[j] & 0x7fffffffu;
                const bool live = q0 + j < chunk_items;
                ngt += live && key > T;
                neq += live && key == T;
            }
            const uint64_t ex2 = block_exclusive_scan<NTS>((uint64_t)ngt | ((uint64_t)neq << 32), rs.scan, &tot);
            uint32_t gb = run_gt + (uint32_t)ex2, eb = run_eq + (uint32_t)(ex2 >> 32);
#pragma unroll
            for (int j = 0; j < IPT; ++j) {
                const uint32_t key = bits[j] & 0x7fffffffu;
                const bool live = q0 + j < chunk_items;
                const bool gt = live && key > T, eq = live && key == T;
                const uint32_t slot = gb + (eb < ties ? eb : ties);
                if ((gt || (eq && eb < ties)) && slot < p.k && local[j] < p.n) {
                    gcsgd_pair pr;
                    pr.idx = p.off + local[j];
                    pr.val = __uint_as_float(bits[j]);
                    dst[slot] = pr;
                    u[ebase + local[j]] = 0.0f;
                    v[ebase + local[j]] = 0.0f;
                }
                gb += gt;
                eb += eq;
            }
            run_gt += (uint32_t)tot;
            run_eq += (uint32_t)(tot >> 32);
        }
        __syncthreads();  // toff/tbase reused by the next chunk
    }
}

// One CTA per (learner, segment), largest segments first, every learner's
// copy of a segment together; pools too large for the stage are left to
// dgc_select_big.
__global__ void __launch_bounds__(NTS, 2) dgc_select(SelectArgs A) {
    extern __shared__ __align__(16) unsigned char stage_raw[];  // kStageBytes
    __shared__ RadixSmem rs;
    __shared__ uint32_t toff[kChunkTiles];
    __shared__ uint32_t tbase[kChunkTiles];
    __shared__ uint2 wsum[NTS / 32];
    const int k = (int)blockIdx.x % A.K;
    const int s = A.order[(int)blockIdx.x / A.K];
    if (threadIdx.x == 0 && s == 0 && A.totals && !A.sampled) A.totals[k] = A.out_per_learner;
    if (big_pool(A.plan[s])) return;
    const SelectSmem M = {stage_raw, &rs, toff, tbase, wsum};
    select_unit(A, M, k, s);
}

// ------------------------------------------------------- large pools
//
// Pools whose capacity exceeds one CTA's stage (more than kStageItems
// candidates possible) are selected by a thread-block cluster of
// kClusterCTAs CTAs, one cluster per (learner, segment).  CTA r stages the
// candidates of its share of the tiles (index order, so the cluster holds
// the pool in index order across its ranks), and the cluster then runs the
// range-adaptive radix select of select_unit with distributed shared memory:
// every rank histograms its own keys, rank 0 adds the kClusterCTAs
// histograms and picks the bucket, every rank appends that bucket's keys to
// rank 0's candidate buffer, and rank 0 finishes the selection (exact rank or
// more digits).  Each rank then emits its own items at slots offset by the
// greater and tied items of the ranks before it.  A pool the cluster cannot
// stage (a rank's share above kStageItems, a failed hint, an overflow) is
// selected by rank 0 alone through select_unit's global paths.
namespace cg = cooperative_groups;
constexpr int kClusterCTAs = 8;

template <int MAXS>
struct BigList {
    uint32_t n;
    uint16_t seg[MAXS];  // segments whose pools go to dgc_select_big
};

// Per-rank words of the cluster exchange (each rank's own shared memory,
// read by the others through distributed shared memory).
struct ClusterXch {
    uint32_t cnt, kmin, kmax, ngt, neq;  // this rank's items, key range, emission counts
    uint32_t bucket, above, bcnt;        // rank 0: the pass's pick
    uint32_t T, ties;                    // rank 0: the selection's result
};

template <int MAXS>
__global__ void __cluster_dims__(kClusterCTAs, 1, 1) __launch_bounds__(NTS, 2)
    dgc_select_big(SelectArgs A, BigList<MAXS> big) {
    extern __shared__ __align__(16) unsigned char stage_raw[];  // kStageBytes
    __shared__ RadixSmem rs;
    __shared__ uint32_t toff[kChunkTiles];
    __shared__ uint32_t tbase[kChunkTiles];
    __shared__ uint2 wsum[NTS / 32];
    __shared__ ClusterXch xch;
    __shared__ uint32_t red[NTS / 32][2];
    cg::cluster_group cl = cg::this_cluster();
    const uint32_t r = cl.block_rank();
    const int c = (int)(blockIdx.x / kClusterCTAs);
    const int k = c % A.K;
    const int s = big.seg[c / A.K];
    const SegPlan p = A.plan[s];
    const SelectSmem M = {stage_raw, &rs, toff, tbase, wsum};
    uint2* stage = reinterpret_cast<uint2*>(stage_raw);
    const int unit = k * A.S + s;
    const uint32_t pc = A.pool_cnt[unit];
    const bool take_all = p.sampled && pc < p.k;
    const bool pool_ok = (pc >= p.k || take_all) && pc <= p.cap;
    const uint2* tt = A.tile_tab + (uint64_t)k * A.tiles_per_learner + p.tile_off;
    const uint2* items = A.pool + (uint64_t)k * A.pool_per_learner + p.pool_off;
    const uint32_t t0 = (uint32_t)((uint64_t)r * p.ntiles / kClusterCTAs);
    const uint32_t t1 = (uint32_t)((uint64_t)(r + 1) * p.ntiles / kClusterCTAs);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // block sums of two words (warp shuffles, then one word per warp)
    auto block_sum2 = [&](uint32_t a, uint32_t b, uint32_t* ta, uint32_t* tb) {
        a = __reduce_add_sync(kFull, a);
        b = __reduce_add_sync(kFull, b);
        if (lane == 0) {
            red[warp][0] = a;
            red[warp][1] = b;
        }
        __syncthreads();
        uint32_t sa = 0, sb = 0;
#pragma unroll
        for (int w = 0; w < NTS / 32; ++w) {
            sa += red[w][0];
            sb += red[w][1];
        }
        *ta = sa;
        *tb = sb;
        __syncthreads();
    };

    // this rank's share of the candidates
    uint32_t mine = 0;
    if (pool_ok)
        for (uint32_t t = t0 + threadIdx.x; t < t1; t += NTS) mine += tt[t].y;
    uint32_t my_cnt, unused;
    block_sum2(mine, 0u, &my_cnt, &unused);
    if (threadIdx.x == 0) xch.cnt = my_cnt;
    cl.sync();
    bool fits = pool_ok;
    for (int q = 0; q < kClusterCTAs; ++q) fits = fits && cl.map_shared_rank(&xch, q)->cnt <= kStageItems;
    cl.sync();  // every rank has read the counts before any rank leaves
    if (!fits) {
        if (r == 0) select_unit(A, M, k, s);
        return;
    }
    if (r == 0 && threadIdx.x == 0) A.counts[unit] = take_all ? pc : p.k;
    if (p.k == 0) return;  // uniform: every rank leaves (no later cluster barrier)

    // stage this rank's items; the cluster's key range
    uint32_t kmin = 0xffffffffu, kmax = 0;
    const uint32_t cnt = stage_tiles(tt, t0, t1, items, stage, toff, tbase, rs, kmin, kmax);
    kmin = __reduce_min_sync(kFull, kmin);
    kmax = __reduce_max_sync(kFull, kmax);
    if (lane == 0) {
        red[warp][0] = kmin;
        red[warp][1] = kmax;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t a = 0xffffffffu, b = 0;
        for (int w = 0; w < NTS / 32; ++w) {
            a = min(a, red[w][0]);
            b = max(b, red[w][1]);
        }
        xch.kmin = a;
        xch.kmax = b;
    }
    cl.sync();
    kmin = 0xffffffffu;
    kmax = 0;
    for (int q = 0; q < kClusterCTAs; ++q) {
        const ClusterXch* o = cl.map_shared_rank(&xch, q);
        kmin = min(kmin, o->kmin);
        kmax = max(kmax, o->kmax);
    }

    uint32_t T = 0, ties = pc;  // take_all: every candidate goes
    if (!take_all) {
        // the range-adaptive radix select, distributed over the ranks
        const uint32_t base = kmin;
        int shift = kmax > kmin ? 32 - __clz(kmax - kmin) : 0;
        uint32_t prefix = 0, pmask = 0, need = p.k, greater = 0;
        bool done = false;
#pragma unroll 1
        for (int pass = 0; !done; ++pass) {
            const int nshift = shift > 11 ? shift - 11 : 0;
            const uint32_t dmask = (1u << (shift - nshift)) - 1u;
            const int nb = (int)(dmask + 1) > NTS ? (int)(dmask + 1) : NTS;
            for (int b = threadIdx.x; b < nb; b += NTS) rs.hist[b] = 0;
            __syncthreads();
#pragma unroll 1
            for (uint32_t i = threadIdx.x; i < cnt; i += NTS) {
                const uint32_t d = (stage[i].y & 0x7fffffffu) - base;
                if ((d & pmask) == prefix) atomicAdd(&rs.hist[(d >> nshift) & dmask], 1u);
            }
            cl.sync();  // every rank's histogram is complete
            if (r == 0) {
                // totals into rs.cand (free until the compaction), then back into rs.hist
                for (int b = threadIdx.x; b < nb; b += NTS) {
                    uint32_t t = 0;
                    for (int q = 0; q < kClusterCTAs; ++q) t += cl.map_shared_rank(rs.hist, q)[b];
                    rs.cand[b] = t;
                }
            }
            cl.sync();  // the other ranks' histograms have been read
            if (r == 0) {
                for (int b = threadIdx.x; b < nb; b += NTS) rs.hist[b] = rs.cand[b];
                __syncthreads();
                uint32_t b, ab, cb;
                radix_pick<NTS>(rs, nb, need, &b, &ab, &cb);
                if (threadIdx.x == 0) {
                    xch.bucket = b;
                    xch.above = ab;
                    xch.bcnt = cb;
                    rs.sel[3] = 0;  // the candidate buffer, empty
                }
            }
            cl.sync();
            {
                const ClusterXch* o = cl.map_shared_rank(&xch, 0);
                prefix |= o->bucket << nshift;
                pmask |= dmask << nshift;
                greater += o->above;
                need -= o->above;
                const uint32_t cb = o->bcnt;
                shift = nshift;
                if (shift == 0) {  // every digit taken: the bucket is the threshold
                    T = base + prefix;
                    ties = need;
                    done = true;
                } else if (cb <= (uint32_t)kCandMax) {
                    // the bucket's keys (offsets from base) to rank 0, which finishes
                    RadixSmem* rs0 = cl.map_shared_rank(&rs, 0);
#pragma unroll 1
                    for (uint32_t i0 = 0; i0 < cnt; i0 += NTS) {  // CTA-uniform trip count
                        const uint32_t i = i0 + threadIdx.x;
                        const uint32_t d = i < cnt ? (stage[i].y & 0x7fffffffu) - base : 0u;
                        const bool hit = i < cnt && (d & pmask) == prefix;
                        const unsigned m = __ballot_sync(kFull, hit);
                        if (m) {
                            uint32_t at = 0;
                            if (lane == 0) at = atomicAdd(&rs0->sel[3], (uint32_t)__popc(m));
                            at = __shfl_sync(kFull, at, 0);
                            const uint32_t slot = at + __popc(m & ((1u << lane) - 1u));
                            if (hit && slot < (uint32_t)kCandMax) rs0->cand[slot] = d;
                        }
                    }
                    cl.sync();  // rank 0 holds the bucket's cb keys
                    if (r == 0) {
                        SelectResult sr;
                        if (cb <= (uint32_t)NTS) {
                            sr = rank_select<NTS>(rs, cb, need);  // offsets rank like keys
                        } else {
                            // keys in [base + prefix, base + prefix + 2^shift)
                            sr = radix_select_span<NTS>(
                                [&](uint32_t i, uint32_t* key) { *key = rs.cand[i] - prefix; }, cb, need, 0u, shift,
                                rs, toff, (uint32_t)kChunkTiles);
                            sr.thresh += prefix;
                        }
                        if (threadIdx.x == 0) {
                            xch.T = base + sr.thresh;
                            xch.ties = sr.ties;
                        }
                    }
                    cl.sync();
                    const ClusterXch* o0 = cl.map_shared_rank(&xch, 0);
                    T = o0->T;
                    ties = o0->ties;
                    done = true;
                }
                // else another digit over the staged keys
            }
            cl.sync();  // rank 0's words have been read before the next pass rewrites them
        }
    }

    // emission: this rank's items at slots after the ranks before it
    uint32_t ngt = 0, neq = 0;
#pragma unroll 1
    for (uint32_t i = threadIdx.x; i < cnt; i += NTS) {
        const uint32_t key = stage[i].y & 0x7fffffffu;
        ngt += key > T;
        neq += key == T;
    }
    uint32_t tg, te;
    block_sum2(ngt, neq, &tg, &te);
    if (threadIdx.x == 0) {
        xch.ngt = tg;
        xch.neq = te;
    }
    cl.sync();
    uint32_t gb = 0, eb = 0;
    for (uint32_t q = 0; q < r; ++q) {
        const ClusterXch* o = cl.map_shared_rank(&xch, q);
        gb += o->ngt;
        eb += o->neq;
    }
    const uint32_t mine_ties = eb >= ties ? 0u : (ties - eb < te ? ties - eb : te);
    const uint32_t slot0 = gb + (eb < ties ? eb : ties);
    const uint64_t ebase = (uint64_t)k * A.N + p.off;
    gcsgd_pair* dst = A.out + (uint64_t)k * A.cap + p.out_off;
    emit_in_order(
        [&](uint32_t i, uint32_t* loc, uint32_t* bits) {
            const uint2 it = stage[i];
            *loc = it.x;
            *bits = it.y;
        },
        cnt, T, mine_ties, p, dst, A.u, A.v, ebase, wsum, slot0);
    cl.sync();  // no rank leaves while another may still read its words
}

// Sampled threshold: the selection wrote tensor s's entries at its k_s-slot
// region of the scratch list; each learner's list is packed to be contiguous
// (tensors in order, a warp per tensor) and its total written.
__global__ void __launch_bounds__(NTS) dgc_pack(const SegPlan* __restrict__ plan, int S,
                                               const int64_t* __restrict__ counts, const gcsgd_pair* __restrict__ msg,
                                               uint32_t out_per_learner, gcsgd_pair* __restrict__ out, uint64_t cap,
                                               int64_t* __restrict__ totals) {
    constexpr int NW = NTS / 32;
    __shared__ uint64_t scan[NW + 1];
    __shared__ uint64_t pre[NTS];
    __shared__ uint32_t cnt[NTS];
    __shared__ uint64_t s_carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int k = blockIdx.x;
    const gcsgd_pair* src = msg + (uint64_t)k * out_per_learner;
    gcsgd_pair* dst = out + (uint64_t)k * cap;
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (int base = 0; base < S; base += NTS) {
        const int s = base + (int)threadIdx.x;
        const uint32_t c = s < S ? (uint32_t)counts[(int64_t)k * S + s] : 0u;
        uint64_t tot;
        const uint64_t ex = block_exclusive_scan<NTS>(c, scan, &tot);
        pre[threadIdx.x] = s_carry + ex;
        cnt[threadIdx.x] = c;
        __syncthreads();
        for (int q = warp; q < NTS && base + q < S; q += NW) {
            const uint64_t at = pre[q];
            const uint32_t from = __ldg(&plan[base + q].out_off);
            for (uint32_t i = lane; i < cnt[q]; i += 32) dst[at + i] = src[from + i];
        }
        __syncthreads();
        if (threadIdx.x == 0) s_carry += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0 && totals) totals[k] = (int64_t)s_carry;
}

}  // namespace dgc

// ------------------------------------------------------------- host launch

// Opt in to more than 48 KB of dynamic shared memory, once per device.
static int dgc_set_smem_limits() {
    using namespace dgc;
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return set_error(GCSGD_ERR_CUDA, "dgc_compress: no current device");
    if (done[dev]) return GCSGD_OK;
    const int ks = (int)(kSampleMax * sizeof(uint32_t));
    if (cudaFuncSetAttribute(dgc_prepare<256, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, ks) != cudaSuccess ||
        cudaFuncSetAttribute(dgc_prepare<GCSGD_MAX_SEGMENTS, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, ks) !=
            cudaSuccess ||
        cudaFuncSetAttribute(dgc_prepare<256, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, ks) != cudaSuccess ||
        cudaFuncSetAttribute(dgc_prepare<GCSGD_MAX_SEGMENTS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, ks) !=
            cudaSuccess ||
        cudaFuncSetAttribute(dgc_select, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStageBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(dgc_select_big<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStageBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(dgc_select_big<GCSGD_MAX_SEGMENTS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStageBytes) != cudaSuccess)
        return set_error(GCSGD_ERR_CUDA, "dgc_compress: cannot raise the shared-memory limit");
    done[dev] = true;
    return GCSGD_OK;
}

int dgc_launch(const int64_t* off, int S, int K, const float* grad, float* u, float* v, double density,
               double sample_frac, float momentum, bool nesterov, float clip_thr, int clip_nodes, gcsgd_pair* out,
               int64_t cap, int64_t* counts, int64_t* totals, void* ws, size_t ws_bytes, cudaStream_t stream) {
    using namespace dgc;
    HostPlan hp;
    host_plan(off, S, density, sample_frac, &hp);
    const uint64_t N = (uint64_t)off[S];
    const bool sampled = sample_frac > 0.0;
    DgcWorkspace w;
    const size_t need = dgc_workspace_layout(S, K, hp, sampled, ws, &w);
    if (ws_bytes < need)
        return set_error(GCSGD_ERR_WORKSPACE, "dgc_compress: workspace of %zu bytes, %zu needed", ws_bytes, need);
    if ((uint64_t)cap < hp.out_per_learner)
        return set_error(GCSGD_ERR_CAPACITY, "dgc_compress: cap %lld below the %llu entries per learner",
                         (long long)cap, (unsigned long long)hp.out_per_learner);
    const uint64_t total_tiles = (uint64_t)K * hp.tiles_per_learner;
    if (total_tiles >= ((uint64_t)1 << 32))
        return set_error(GCSGD_ERR_INVALID_ARG, "dgc_compress: K * tiles = %llu exceeds 2^32",
                         (unsigned long long)total_tiles);
    const bool clip = clip_thr > 0.0f;
    int rc;
    if (clip) {
        LaunchScope ls("dgc_sumsq", stream);
        dgc_sumsq<<<dim3(kSumsqBlocks, K), NT, 0, stream>>>(grad, N, w.clip_part);
        if ((rc = check_launch("dgc_sumsq"))) return rc;
    }
    const unsigned units = (unsigned)K * (unsigned)S;
    if ((rc = dgc_set_smem_limits())) return rc;
    {
        LaunchScope ls("dgc_prepare", stream);
        const size_t smem = kSampleMax * sizeof(uint32_t);
        auto fill = [&](auto& so, auto& pl) {
            pl.n_pool = 0;
            uint32_t koff = 0;
            for (int s = 0; s <= S; ++s) so.off[s] = (uint32_t)off[s];
            // segments by size, largest first, ties to the lower index (a stable sort)
            for (int s = 0; s < S; ++s) pl.order[s] = (uint16_t)s;
            std::stable_sort(pl.order, pl.order + S,
                             [&](uint16_t a, uint16_t b) { return off[a + 1] - off[a] > off[b + 1] - off[b]; });
            for (int s = 0; s < S; ++s) {
                SegPlan sp;
                seg_fields((uint32_t)(off[s + 1] - off[s]), density, sample_frac, &sp);
                if (sp.kind != kKindPool) continue;
                pl.seg[pl.n_pool] = (uint16_t)s;
                pl.koff[pl.n_pool] = koff;
                if (sample_spills(sp)) koff += sp.m;
                ++pl.n_pool;
            }
        };
        const unsigned pool_units = (unsigned)K * (unsigned)hp.pool_segments;
        const unsigned slots = (unsigned)sm_count() * 2 - 1;  // two CTAs of NTP threads per SM
        const unsigned prep_grid = (pool_units < slots ? pool_units : slots) + 1;  // + the plan CTA
        if (S <= 256) {
            SegOffsets<256> so;
            PoolList<256> pl;
            fill(so, pl);
            (nesterov ? dgc_prepare<256, true> : dgc_prepare<256, false>)<<<prep_grid, NTP, smem, stream>>>(
                so, pl, S, K, density, sample_frac, clip_thr, clip_nodes, w.clip_part, w.plan, w.clip_c, w.order, N,
                grad, u, v, momentum, w.hint, w.pool_cnt, w.skeys, hp.skeys_per_learner);
        } else {
            SegOffsets<GCSGD_MAX_SEGMENTS> so;
            PoolList<GCSGD_MAX_SEGMENTS> pl;
            fill(so, pl);
            (nesterov ? dgc_prepare<GCSGD_MAX_SEGMENTS, true> : dgc_prepare<GCSGD_MAX_SEGMENTS, false>)
                <<<prep_grid, NTP, smem, stream>>>(so, pl, S, K, density, sample_frac, clip_thr, clip_nodes,
                                                   w.clip_part, w.plan, w.clip_c, w.order, N, grad, u, v, momentum,
                                                   w.hint, w.pool_cnt, w.skeys, hp.skeys_per_learner);
        }
        if ((rc = check_launch("dgc_prepare"))) return rc;
    }
    if (total_tiles > 0) {
        LaunchScope ls("dgc_update", stream);
        uint64_t grid = (uint64_t)sm_count() * 3;
        if (grid > total_tiles) grid = total_tiles;
        (nesterov ? dgc_update<true> : dgc_update<false>)<<<(unsigned)grid, NT, 0, stream>>>(
            w.plan, S, N, (uint32_t)hp.tiles_per_learner, total_tiles, grad, u, v, momentum, w.clip_c, w.hint,
            w.pool_cnt, w.tile_tab, w.pool, hp.pool_per_learner);
        if ((rc = check_launch("dgc_update"))) return rc;
    }
    {
        LaunchScope ls("dgc_select", stream);
        // the sampled threshold writes each tensor's entries into its k_s-slot region of the scratch list
        gcsgd_pair* dst = sampled ? w.msg : out;
        const uint64_t dst_stride = sampled ? hp.out_per_learner : (uint64_t)cap;
        SelectArgs A = {w.plan, S, N, (uint32_t)hp.tiles_per_learner, u, v, w.pool_cnt, w.tile_tab, w.pool,
                        hp.pool_per_learner, dst, dst_stride, counts, totals, (uint32_t)hp.out_per_learner,
                        w.order, K, sampled ? 1 : 0};
        dgc_select<<<units, NTS, kStageBytes, stream>>>(A);
        if ((rc = check_launch("dgc_select"))) return rc;
    }
    {
        // pools too large for one CTA's stage: a cluster per (learner, segment)
        gcsgd_pair* dst = sampled ? w.msg : out;
        const uint64_t dst_stride = sampled ? hp.out_per_learner : (uint64_t)cap;
        SelectArgs A = {w.plan, S, N, (uint32_t)hp.tiles_per_learner, u, v, w.pool_cnt, w.tile_tab, w.pool,
                        hp.pool_per_learner, dst, dst_stride, counts, totals, (uint32_t)hp.out_per_learner,
                        w.order, K, sampled ? 1 : 0};
        auto launch_big = [&](auto& bl, auto kernel) {
            bl.n = 0;
            for (int s = 0; s < S; ++s) {
                SegPlan sp;
                seg_fields((uint32_t)(off[s + 1] - off[s]), density, sample_frac, &sp);
                if (big_pool(sp)) bl.seg[bl.n++] = (uint16_t)s;
            }
            if (bl.n == 0) return GCSGD_OK;
            LaunchScope lb("dgc_select_big", stream);
            kernel<<<(unsigned)K * bl.n * kClusterCTAs, NTS, kStageBytes, stream>>>(A, bl);
            return check_launch("dgc_select_big");
        };
        if (S <= 256) {
            BigList<256> bl;
            if ((rc = launch_big(bl, dgc_select_big<256>))) return rc;
        } else {
            BigList<GCSGD_MAX_SEGMENTS> bl;
            if ((rc = launch_big(bl, dgc_select_big<GCSGD_MAX_SEGMENTS>))) return rc;
        }
    }
    if (sampled) {
        LaunchScope ls("dgc_pack", stream);
        dgc_pack<<<(unsigned)K, NTS, 0, stream>>>(w.plan, S, counts, w.msg, (uint32_t)hp.out_per_learner, out,
                                                 (uint64_t)cap, totals);
        if ((rc = check_launch("dgc_pack"))) return rc;
    }
    return GCSGD_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int dgc_collect_stats(const int64_t* off, int S, int K, double density, const void* ws, cudaStream_t stream,
                      gcsgd_dgc_stats_t* st) {
    using namespace dgc;
    HostPlan hp;
    host_plan(off, S, density, 0.0, &hp);
    DgcWorkspace w;
    dgc_workspace_layout(S, K, hp, false, const_cast<void*>(ws), &w);
    std::vector<uint32_t> cnt((size_t)K * S);
    cudaError_t e = cudaMemcpyAsync(cnt.data(), w.pool_cnt, sizeof(uint32_t) * cnt.size(), cudaMemcpyDeviceToHost,
                                    stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return set_error(GCSGD_ERR_CUDA, "gcsgd_dgc_stats: %s", cudaGetErrorString(e));
    memset(st, 0, sizeof(*st));
    st->units = (int64_t)K * S;
    for (int k = 0; k < K; ++k)
        for (int s = 0; s < S; ++s) {
            SegPlan p;
            seg_fields((uint32_t)(off[s + 1] - off[s]), density, 0.0, &p);
            const uint32_t c = cnt[(size_t)k * S + s];
            if (p.kind == kKindEmpty) ++st->empty;
            else if (p.kind == kKindRaw) (p.n <= kRawMax ? st->raw : st->raw_global)++;
            else if (c < p.k || c > p.cap) ++st->hint_failed;
            else (c <= kStageItems || (big_pool(p) && c <= (uint32_t)kClusterCTAs * kStageItems) ? st->pool
                                                                                                  : st->pool_global)++;
        }
    return GCSGD_OK;
}

size_t dgc_workspace_layout(int S, int K, const dgc::HostPlan& hp, bool sampled, void* base,
                            dgc::DgcWorkspace* w) {
    using namespace dgc;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    const size_t o_plan = take(sizeof(SegPlan) * (size_t)S);
    const size_t o_cc = take(sizeof(float) * (size_t)K);
    const size_t o_part = take(sizeof(double) * (size_t)K * kSumsqBlocks);
    const size_t o_order = take(sizeof(uint16_t) * (size_t)S);
    const size_t o_hint = take(sizeof(uint32_t) * (size_t)K * S);
    const size_t o_cnt = take(sizeof(uint32_t) * (size_t)K * S);
    const size_t o_tt = take(sizeof(uint2) * (size_t)K * hp.tiles_per_learner);
    const size_t o_pool = take(sizeof(uint2) * (size_t)K * hp.pool_per_learner);
    const size_t o_msg = take(sampled ? sizeof(gcsgd_pair) * (size_t)K * hp.out_per_learner : 0);
    const size_t o_skeys = take(sampled ? sizeof(uint32_t) * (size_t)K * hp.skeys_per_learner : 0);
    if (w) {
        char* b = (char*)base;
        w->plan = (SegPlan*)(b + o_plan);
        w->clip_c = (float*)(b + o_cc);
        w->clip_part = (double*)(b + o_part);
        w->order = (uint16_t*)(b + o_order);
        w->hint = (uint32_t*)(b + o_hint);
        w->pool_cnt = (uint32_t*)(b + o_cnt);
        w->tile_tab = (uint2*)(b + o_tt);
        w->pool = (uint2*)(b + o_pool);
        w->msg = sampled ? (gcsgd_pair*)(b + o_msg) : nullptr;
        w->skeys = sampled ? (uint32_t*)(b + o_skeys) : nullptr;
    }
    return o;
}

}  // namespace gcsgd

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
//   dgc_plan      one CTA: per-segment plan (k_s, tiles, pool sizes, offsets)
//                 and, when clipping is on, the clip scale of each learner
//   dgc_hint      one CTA per (learner, segment): a strided sample of the
//                 updated |v| gives a threshold hint safely below the k-th
//                 largest value
//   dgc_update    the bandwidth-bound pass: reads g, u, v once (128-bit
//                 loads), writes u', v' once, and appends every |v'| >= hint
//                 to a small per-(learner, segment) candidate pool, keeping
//                 index order inside each 4096-element tile
//   dgc_select    one CTA per (learner, segment): exact radix select of the
//                 k-th largest |v'| among the candidates (or, if the hint
//                 failed, among all of the segment's v'), then the ordered
//                 emission of (index, v') with ties to the lower index, and
//                 the masking u = v = 0 at the sent indices.
// The answer never depends on the hint: a pool is used only when it provably
// contains every entry of the top k (at least k candidates, no overflow).
#include <math.h>

#include "common.cuh"
#include "dgc.cuh"

namespace gcsgd {
namespace dgc {

constexpr int NT = 256;                 // threads per CTA in every DGC kernel
constexpr int kTile = 4096;             // elements per dgc_update tile (NT x 4 float4)
constexpr uint32_t kRawMax = 32768;     // segments up to this size select from v' directly
constexpr uint32_t kSampleMax = 8192;   // largest hint sample (keys held in shared memory)
constexpr uint32_t kSampleAbove = 32;   // sampled entries expected above the hint
constexpr uint32_t kPoolFloor = 512;    // smallest expected candidate count
constexpr int kSumsqBlocks = 128;       // CTAs per learner in dgc_sumsq

__host__ __device__ inline void seg_fields(uint32_t n, double density, SegPlan* p) {
    p->n = n;
    p->k = dgc_k_of(density, n);
    p->ntiles = (n + kTile - 1) / kTile;
    p->cap = 0;
    p->m = 0;
    p->a = 0;
    if (n == 0) {
        p->kind = kKindEmpty;
    } else if (n <= kRawMax || 3ull * p->k > n / 2) {
        p->kind = kKindRaw;
    } else {
        p->kind = kKindPool;
        const uint64_t R = 3ull * p->k > kPoolFloor ? 3ull * p->k : kPoolFloor;  // expected candidates
        const uint64_t cap = 4 * R + 256;
        p->cap = (uint32_t)(cap < n ? cap : n);
        uint64_t m = (uint64_t)kSampleAbove * n / R;
        if (m > kSampleMax) m = kSampleMax;
        m &= ~(uint64_t)31;
        if (m < 32) m = 32;
        p->m = (uint32_t)m;
        uint64_t a = (R * m + n / 2) / n;
        p->a = (uint32_t)(a < 1 ? 1 : (a > m ? m : a));
    }
}

// Host mirror of dgc_plan's totals (workspace sizing and argument checks).
int host_plan(const int64_t* off, int S, double density, HostPlan* hp) {
    hp->tiles_per_learner = 0;
    hp->pool_per_learner = 0;
    hp->out_per_learner = 0;
    for (int s = 0; s < S; ++s) {
        SegPlan p;
        seg_fields((uint32_t)(off[s + 1] - off[s]), density, &p);
        hp->tiles_per_learner += p.ntiles;
        hp->pool_per_learner += p.cap;
        hp->out_per_learner += p.k;
    }
    return 0;
}

// ---------------------------------------------------------------- kernels

// Sum of squares of learner blockIdx.y's gradient over a fixed slice, fp64
// with exact products (fma), reduced in a fixed tree: deterministic.
__global__ void __launch_bounds__(NT) dgc_sumsq(const float* __restrict__ grad, uint64_t N,
                                                 double* __restrict__ part) {
    __shared__ double red[NT / 32];
    const uint64_t k = blockIdx.y;
    const uint64_t chunk = (N + gridDim.x - 1) / gridDim.x;
    const uint64_t lo = (uint64_t)blockIdx.x * chunk;
    const uint64_t hi = lo + chunk < N ? lo + chunk : N;
    const float* g = grad + k * N;
    double acc = 0.0;
    for (uint64_t i = lo + threadIdx.x; i < hi; i += NT) {
        const double x = (double)__ldg(g + i);
        acc = __fma_rn(x, x, acc);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) acc = __dadd_rn(acc, __shfl_down_sync(kFull, acc, d));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int w = 0; w < NT / 32; ++w) s = __dadd_rn(s, red[w]);
        part[k * gridDim.x + blockIdx.x] = s;
    }
}

// One CTA: the per-segment plan (prefix sums of pool sizes, tiles and
// message lengths) and each learner's clip scale.
template <int MAXS>
__global__ void __launch_bounds__(1024) dgc_plan(SegOffsets<MAXS> so, int S, int K, double density,
                                                 float clip_thr, int clip_nodes, int nparts,
                                                 const double* __restrict__ part, SegPlan* __restrict__ plan,
                                                 float* __restrict__ clip_c) {
    __shared__ uint64_t scan[1024 / 32 + 1];
    __shared__ uint64_t carry[3];
    if (threadIdx.x < 3) carry[threadIdx.x] = 0;
    __syncthreads();
    for (int base = 0; base < S; base += 1024) {
        const int s = base + (int)threadIdx.x;
        SegPlan p;
        const bool live = s < S;
        seg_fields(live ? so.off[s + 1] - so.off[s] : 0u, density, &p);
        p.off = live ? so.off[s] : 0u;
        uint64_t tot;
        const uint64_t ex_pool = block_exclusive_scan<1024>(live ? p.cap : 0, scan, &tot);
        const uint64_t c0 = carry[0];
        __syncthreads();
        if (threadIdx.x == 0) carry[0] = c0 + tot;
        const uint64_t ex_tile = block_exclusive_scan<1024>(live ? p.ntiles : 0, scan, &tot);
        const uint64_t c1 = carry[1];
        __syncthreads();
        if (threadIdx.x == 0) carry[1] = c1 + tot;
        const uint64_t ex_out = block_exclusive_scan<1024>(live ? p.k : 0, scan, &tot);
        const uint64_t c2 = carry[2];
        __syncthreads();
        if (threadIdx.x == 0) carry[2] = c2 + tot;
        if (live) {
            p.pool_off = (uint32_t)(c0 + ex_pool);
            p.tile_off = (uint32_t)(c1 + ex_tile);
            p.out_off = (uint32_t)(c2 + ex_out);
            p.pad = 0;
            plan[s] = p;
        }
        __syncthreads();
    }
    // local gradient clipping scale (Appendix C): thr_k = thr / sqrt(N_nodes);
    // c = thr_k / ||G|| when ||G|| > thr_k.  Partial sums are combined in a
    // fixed order with compensated summation.
    for (int k = threadIdx.x; k < K; k += 1024) {
        float c = 1.0f;
        if (clip_thr > 0.0f) {
            double s = 0.0, comp = 0.0;
            for (int i = 0; i < nparts; ++i) {
                const double x = part[(uint64_t)k * nparts + i];
                const double t = s + x;
                comp += fabs(s) >= fabs(x) ? (s - t) + x : (x - t) + s;
                s = t;
            }
            const double norm = sqrt(s + comp);
            const double thr_k = (double)clip_thr / sqrt((double)clip_nodes);
            if (norm > thr_k) c = (float)(thr_k / norm);
        }
        clip_c[k] = c;
    }
}

// The update of one element: u' = m*u + c*g, v' = v + u'.
__device__ __forceinline__ void dgc_elem(float g, float& u, float& v, float m, float c) {
    u = __fadd_rn(__fmul_rn(m, u), __fmul_rn(g, c));
    v = __fadd_rn(v, u);
}

// One CTA per (learner, segment).  Samples kSampleAbove/R of the segment in
// 32-element blocks, computes the updated |v| there exactly as dgc_update
// will, and takes the a-th largest sampled key as the candidate threshold.
__global__ void __launch_bounds__(NT) dgc_hint(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                               const float* __restrict__ grad, const float* __restrict__ u,
                                               const float* __restrict__ v, float momentum,
                                               const float* __restrict__ clip_c, uint32_t* __restrict__ hint,
                                               uint32_t* __restrict__ pool_cnt) {
    __shared__ uint32_t keys[kSampleMax];
    __shared__ uint32_t hist[2048];
    __shared__ uint64_t scan[NT / 32 + 1];
    __shared__ uint32_t sel[4];
    const int unit = blockIdx.x;
    const int k = unit / S, s = unit - k * S;
    const SegPlan p = plan[s];
    if (threadIdx.x == 0) pool_cnt[unit] = 0;
    if (p.kind != kKindPool) {
        if (threadIdx.x == 0) hint[unit] = 0xffffffffu;  // no candidates
        return;
    }
    const float c = clip_c[k];
    const uint32_t nblk = p.m / 32;
    const uint32_t stride = p.n / nblk;  // >= 512 since m <= n / 16
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t base = (uint64_t)k * N + p.off;
    for (uint32_t b = warp; b < nblk; b += NT / 32) {
        const uint64_t i = base + (uint64_t)b * stride + lane;
        float uu = __ldg(u + i), vv = __ldg(v + i);
        dgc_elem(__ldg(grad + i), uu, vv, momentum, c);
        keys[b * 32 + lane] = mag_key(vv);
    }
    __syncthreads();
    const SelectResult r = radix_select_desc<NT>(
        [&](uint64_t i, uint32_t* key) { *key = keys[i]; return true; }, p.m, p.a, hist, scan, sel);
    if (threadIdx.x == 0) hint[unit] = r.thresh > 1u ? r.thresh : 1u;
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
    for (uint64_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
        const uint32_t k = (uint32_t)(t / tiles_per_learner);
        const uint32_t lt = (uint32_t)(t - (uint64_t)k * tiles_per_learner);
        const int s = find_segment_by_tile(plan, S, lt);
        const SegPlan p = plan[s];
        const uint32_t start = (lt - p.tile_off) * (uint32_t)kTile;
        const uint32_t len = p.n - start < (uint32_t)kTile ? p.n - start : (uint32_t)kTile;
        const uint64_t base = (uint64_t)k * N + p.off + start;
        const uint32_t unit = k * S + s;
        const uint32_t h = __ldg(&hint[unit]);
        const float c = __ldg(&clip_c[k]);
        const bool aligned = (base & 3) == 0;

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
                dgc_elem(g4[j], u4[j], v4[j], momentum, c);
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

// One CTA per (learner, segment): exact top-k and ordered emission.
__global__ void __launch_bounds__(NT) dgc_select(const SegPlan* __restrict__ plan, int S, uint64_t N,
                                                 uint32_t tiles_per_learner, float* __restrict__ u,
                                                 float* __restrict__ v, const uint32_t* __restrict__ pool_cnt,
                                                 const uint2* __restrict__ tile_tab, const uint2* __restrict__ pool,
                                                 uint64_t pool_per_learner, gcsgd_pair* __restrict__ out, uint64_t cap,
                                                 int64_t* __restrict__ counts, int64_t* __restrict__ totals,
                                                 uint32_t out_per_learner) {
    __shared__ uint32_t hist[2048];
    __shared__ uint64_t scan[NT / 32 + 1];
    __shared__ uint32_t sel[4];
    __shared__ uint32_t toff[NT + 1];
    __shared__ uint32_t tbase[NT];
    const int unit = blockIdx.x;
    const int k = unit / S, s = unit - k * S;
    const SegPlan p = plan[s];
    if (threadIdx.x == 0) {
        counts[unit] = p.k;
        if (s == 0 && totals) totals[k] = out_per_learner;
    }
    if (p.k == 0) return;
    const uint64_t ebase = (uint64_t)k * N + p.off;
    const uint32_t pc = p.kind == kKindPool ? pool_cnt[unit] : 0;
    const bool use_pool = p.kind == kKindPool && pc >= p.k && pc <= p.cap;
    const uint2* items = pool + (uint64_t)k * pool_per_learner + p.pool_off;
    const float* vseg = v + ebase;

    SelectResult r;
    if (use_pool) {
        r = radix_select_desc<NT>(
            [&](uint64_t i, uint32_t* key) { *key = __ldg(&items[i].y) & 0x7fffffffu; return true; }, pc, p.k, hist,
            scan, sel);
    } else {
        r = radix_select_desc<NT>([&](uint64_t i, uint32_t* key) { *key = mag_key(vseg[i]); return true; }, p.n, p.k,
                                  hist, scan, sel);
    }
    const uint32_t T = r.thresh, ties = r.ties, greater = r.greater;
    gcsgd_pair* dst = out + (uint64_t)k * cap + p.out_off;

    // Ordered emission: an element is sent if its key > T, or == T and fewer
    // than `ties` equal keys precede it.  Its slot is (#greater before it) +
    // min(#equal before it, ties).
    uint32_t run_gt = 0, run_eq = 0;

    if (!use_pool) {
        const bool aligned = (ebase & 3) == 0;
        for (uint32_t cb = 0; cb < p.n; cb += 4 * NT) {
            const uint32_t e = cb + 4 * threadIdx.x;
            float x[4];
            if (aligned && e + 4 <= p.n) {
                const float4 q = *reinterpret_cast<const float4*>(vseg + e);
                x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) x[j] = e + j < p.n ? vseg[e + j] : 0.0f;
            }
            uint32_t ngt = 0, neq = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (e + j < p.n) {
                    const uint32_t key = mag_key(x[j]);
                    ngt += key > T;
                    neq += key == T;
                }
            }
            uint64_t tot;
            const uint64_t ex = block_exclusive_scan<NT>((uint64_t)ngt | ((uint64_t)neq << 32), scan, &tot);
            uint32_t gb = run_gt + (uint32_t)ex, eb = run_eq + (uint32_t)(ex >> 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (e + j >= p.n) break;
                const uint32_t key = mag_key(x[j]);
                const bool gt = key > T, eq = key == T;
                const uint32_t slot = gb + (eb < ties ? eb : ties);
                if ((gt || (eq && eb < ties)) && slot < p.k) {
                    dst[slot].idx = p.off + e + j;
                    dst[slot].val = x[j];
                    u[ebase + e + j] = 0.0f;
                    v[ebase + e + j] = 0.0f;
                }
                gb += gt;
                eb += eq;
            }
            run_gt += (uint32_t)tot;
            run_eq += (uint32_t)(tot >> 32);
            if (run_gt >= greater && run_eq >= ties) break;  // everything sent
        }
    } else {
        const uint2* tt = tile_tab + (uint64_t)k * tiles_per_learner + p.tile_off;
        for (uint32_t tb = 0; tb < p.ntiles; tb += NT) {
            const uint32_t j = tb + threadIdx.x;
            uint2 ent = make_uint2(0u, 0u);
            if (j < p.ntiles) ent = tt[j];
            uint64_t tot;
            const uint32_t ex = (uint32_t)block_exclusive_scan<NT>(ent.y, scan, &tot);
            toff[threadIdx.x] = ex;
            tbase[threadIdx.x] = ent.x;
            if (threadIdx.x == 0) toff[NT] = (uint32_t)tot;
            __syncthreads();
            const uint32_t chunk_items = (uint32_t)tot;
            for (uint32_t ib = 0; ib < chunk_items; ib += NT) {
                const uint32_t q = ib + threadIdx.x;
                uint32_t local = 0, bits = 0;
                bool live = q < chunk_items;
                if (live) {
                    int lo = 0, hi = NT;  // last tile with toff <= q
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (toff[mid] <= q) lo = mid; else hi = mid;
                    }
                    const uint2 it = items[tbase[lo] + (q - toff[lo])];
                    local = it.x;
                    bits = it.y;
                }
                const uint32_t key = bits & 0x7fffffffu;
                const bool gt = live && key > T, eq = live && key == T;
                const uint64_t ex2 = block_exclusive_scan<NT>((uint64_t)gt | ((uint64_t)eq << 32), scan, &tot);
                const uint32_t gb = run_gt + (uint32_t)ex2, eb = run_eq + (uint32_t)(ex2 >> 32);
                const uint32_t slot = gb + (eb < ties ? eb : ties);
                if ((gt || (eq && eb < ties)) && slot < p.k && local < p.n) {
                    dst[slot].idx = p.off + local;
                    dst[slot].val = __uint_as_float(bits);
                    u[ebase + local] = 0.0f;
                    v[ebase + local] = 0.0f;
                }
                run_gt += (uint32_t)tot;
                run_eq += (uint32_t)(tot >> 32);
            }
            __syncthreads();  // toff/tbase reused by the next chunk
        }
    }
}

}  // namespace dgc

// ------------------------------------------------------------- host launch

int dgc_launch(const int64_t* off, int S, int K, const float* grad, float* u, float* v, double density,
               float momentum, float clip_thr, int clip_nodes, gcsgd_pair* out, int64_t cap, int64_t* counts,
               int64_t* totals, void* ws, size_t ws_bytes, cudaStream_t stream) {
    using namespace dgc;
    HostPlan hp;
    host_plan(off, S, density, &hp);
    const uint64_t N = (uint64_t)off[S];
    DgcWorkspace w;
    const size_t need = dgc_workspace_layout(S, K, hp, ws, &w);
    if (ws_bytes < need)
        return set_error(GCSGD_ERR_WORKSPACE, "dgc_compress: workspace of %zu bytes, %zu needed", ws_bytes, need);
    if ((uint64_t)cap < hp.out_per_learner)
        return set_error(GCSGD_ERR_CAPACITY, "dgc_compress: cap %lld below the %llu entries per learner",
                         (long long)cap, (unsigned long long)hp.out_per_learner);
    const bool clip = clip_thr > 0.0f;
    int rc;
    if (clip) {
        LaunchScope ls("dgc_sumsq", stream);
        dgc_sumsq<<<dim3(kSumsqBlocks, K), NT, 0, stream>>>(grad, N, w.clip_part);
        if ((rc = check_launch("dgc_sumsq"))) return rc;
    }
    {
        LaunchScope ls("dgc_plan", stream);
        if (S <= 256) {
            SegOffsets<256> so;
            for (int s = 0; s <= S; ++s) so.off[s] = (uint32_t)off[s];
            dgc_plan<256><<<1, 1024, 0, stream>>>(so, S, K, density, clip_thr, clip_nodes, kSumsqBlocks,
                                                  w.clip_part, w.plan, w.clip_c);
        } else {
            SegOffsets<GCSGD_MAX_SEGMENTS> so;
            for (int s = 0; s <= S; ++s) so.off[s] = (uint32_t)off[s];
            dgc_plan<GCSGD_MAX_SEGMENTS><<<1, 1024, 0, stream>>>(so, S, K, density, clip_thr, clip_nodes,
                                                                 kSumsqBlocks, w.clip_part, w.plan, w.clip_c);
        }
        if ((rc = check_launch("dgc_plan"))) return rc;
    }
    const unsigned units = (unsigned)K * (unsigned)S;
    {
        LaunchScope ls("dgc_hint", stream);
        dgc_hint<<<units, NT, 0, stream>>>(w.plan, S, N, grad, u, v, momentum, w.clip_c, w.hint, w.pool_cnt);
        if ((rc = check_launch("dgc_hint"))) return rc;
    }
    const uint64_t total_tiles = (uint64_t)K * hp.tiles_per_learner;
    if (total_tiles > 0) {
        LaunchScope ls("dgc_update", stream);
        uint64_t grid = (uint64_t)sm_count() * 3;
        if (grid > total_tiles) grid = total_tiles;
        dgc_update<<<(unsigned)grid, NT, 0, stream>>>(w.plan, S, N, (uint32_t)hp.tiles_per_learner, total_tiles,
                                                      grad, u, v, momentum, w.clip_c, w.hint, w.pool_cnt,
                                                      w.tile_tab, w.pool, hp.pool_per_learner);
        if ((rc = check_launch("dgc_update"))) return rc;
    }
    {
        LaunchScope ls("dgc_select", stream);
        dgc_select<<<units, NT, 0, stream>>>(w.plan, S, N, (uint32_t)hp.tiles_per_learner, u, v, w.pool_cnt,
                                             w.tile_tab, w.pool, hp.pool_per_learner, out, (uint64_t)cap, counts,
                                             totals, (uint32_t)hp.out_per_learner);
        if ((rc = check_launch("dgc_select"))) return rc;
    }
    return GCSGD_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t dgc_workspace_layout(int S, int K, const dgc::HostPlan& hp, void* base, dgc::DgcWorkspace* w) {
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
    const size_t o_hint = take(sizeof(uint32_t) * (size_t)K * S);
    const size_t o_cnt = take(sizeof(uint32_t) * (size_t)K * S);
    const size_t o_tt = take(sizeof(uint2) * (size_t)K * hp.tiles_per_learner);
    const size_t o_pool = take(sizeof(uint2) * (size_t)K * hp.pool_per_learner);
    if (w) {
        char* b = (char*)base;
        w->plan = (SegPlan*)(b + o_plan);
        w->clip_c = (float*)(b + o_cc);
        w->clip_part = (double*)(b + o_part);
        w->hint = (uint32_t*)(b + o_hint);
        w->pool_cnt = (uint32_t*)(b + o_cnt);
        w->tile_tab = (uint2*)(b + o_tt);
        w->pool = (uint2*)(b + o_pool);
    }
    return o;
}

}  // namespace gcsgd

// spavg.cu -- decompress and average K sparse messages into a dense vector.
//
// "AdaComp ...", Proposed method: learners exchange compressed gradients and
// average them before the weight update; "Deep Gradient Compression",
// Appendix A: the nodes' gradients are summed.
//
// Two kernels for the dense average (the choice is made on the capacity:
// K * cap >= n / 4 counts as dense lists) and the tile kernel for the update.
// Tile kernel: each CTA owns a contiguous run of 4096-element output tiles.
// A tile lives in shared memory: zeroed, then every list's entries that fall
// in it are added in list order k = 0..K-1 (entries inside one list have
// distinct indices, so the adds of one k never collide; a barrier between
// lists keeps the fp32 sum in k order, bit-identical to the definition),
// then the tile is divided by K and written to HBM with 128-bit stores.  Each
// list keeps a window of its next entries staged in shared memory, refilled
// (one round of loads) only when it no longer reaches past the current tile,
// so most tiles need no global reads.  Each warp owns 512 output indices of
// the tile and adds, for its indices, list 0, then list 1, ..., so the
// learner order holds with warp-level synchronisation only.  The dense output
// is written exactly once and each entry is read once (a list denser than its
// window in some tile is read in place for that tile), which is the minimum
// traffic.
//
// Update mode (sparse_average_update): the same sums, but instead of a dense
// average the weights are stepped, w[j] -= lr * avg[j], at the carried
// indices only.  When a CTA's entries fit its stage and K <= 32, each warp
// merges the staged runs and updates 32 weights at a time (merge_update: the
// work follows the entries, no dense pass); otherwise the tile path marks the
// carried positions in a bitmap and read-modify-writes only those
// (update_tile).
#include "common.cuh"

namespace gcsgd {
namespace spavg {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr uint32_t kTile = 4096;   // output elements per shared-memory tile
constexpr uint32_t kStage = 4096;  // list entries a CTA keeps staged (split evenly among the K lists)

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

// Writes acc / K for the output range [r0, r1) and leaves acc zeroed for the
// next tile.
__device__ __forceinline__ void store_tile(float* acc, float* out, uint64_t r0, uint64_t r1, float fk) {
    const uint64_t len = r1 - r0;
    const int K = (int)fk;
    const bool pow2 = (K & (K - 1)) == 0;
    const float inv_k = 1.0f / fk;
    const bool out_aligned = ((uintptr_t)(out + r0) & 15) == 0;
    for (uint32_t j = threadIdx.x * 4; j < kTile; j += NT * 4) {
        float4 q = *reinterpret_cast<const float4*>(acc + j);
        *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j >= len) continue;
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

// Update mode: w[j] <- w[j] - lr * (acc[j] / K) at the positions of the tile
// that some list carries (`touched` bits), with 128-bit read-modify-writes
// where aligned; leaves acc zeroed.  Also clears `next_touched`, the bitmap
// of the tile after this one (its last readers finished before this tile
// began).
__device__ __forceinline__ void update_tile(float* acc, const uint32_t* touched, uint32_t* next_touched, float* w,
                                            uint64_t r0, uint64_t r1, float fk, float lr) {
    constexpr int kRounds = kTile / (4 * NT);
    const uint64_t len = r1 - r0;
    const int K = (int)fk;
    const bool pow2 = (K & (K - 1)) == 0;
    const float inv_k = 1.0f / fk;
    const bool w_aligned = ((uintptr_t)(w + r0) & 15) == 0;
    float4 q[kRounds], x[kRounds];
    uint32_t bits[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {  // every weight load in flight before the first use
        const uint32_t j = 4 * (r * NT + threadIdx.x);
        q[r] = *reinterpret_cast<const float4*>(acc + j);
        *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        bits[r] = j < len ? (touched[j >> 5] >> (j & 31)) & 0xFu : 0u;
        if (bits[r] && w_aligned && j + 4 <= len) x[r] = *reinterpret_cast<const float4*>(w + r0 + j);
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        if (!bits[r]) continue;
        const uint32_t j = 4 * (r * NT + threadIdx.x);
        const float* qq = &q[r].x;
        float* wj = w + r0 + j;
        if (w_aligned && j + 4 <= len) {
            float* xx = &x[r].x;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if ((bits[r] >> c) & 1u) xx[c] = __fsub_rn(xx[c], __fmul_rn(lr, div_k(qq[c], fk, inv_k, pow2)));
            *reinterpret_cast<float4*>(wj) = x[r];
        } else {
            for (int c = 0; c < 4 && j + c < len; ++c)
                if ((bits[r] >> c) & 1u) wj[c] = __fsub_rn(wj[c], __fmul_rn(lr, div_k(qq[c], fk, inv_k, pow2)));
        }
    }
    for (uint32_t t = threadIdx.x; t < kTile / 32; t += NT) next_touched[t] = 0u;
}

// First position in [a, b) of a sorted run whose index is >= target.
__device__ __forceinline__ uint32_t lower_in(const gcsgd_pair* st, uint32_t a, uint32_t b, uint64_t target) {
    while (a < b) {
        const uint32_t m = (a + b) >> 1;
        if ((uint64_t)st[m].idx < target) a = m + 1; else b = m;
    }
    return a;
}

// First position in [a, b) of a sorted list in global memory whose index is >= target.
__device__ __forceinline__ uint64_t lower_global(const gcsgd_pair* L, uint64_t a, uint64_t b, uint64_t target) {
    while (a < b) {
        const uint64_t m = (a + b) >> 1;
        if ((uint64_t)__ldg(&L[m].idx) < target) a = m + 1; else b = m;
    }
    return a;
}

// Update mode over a staged range with K <= 32 lists: warp w merges the K
// sorted runs over its part of [R0, R1), lane k holding list k's next entry.
// At the smallest head index the heads there are summed in learner order
// from +0 (the definition's fp32 sum, bit for bit); lane b of the warp keeps
// the b-th such (index, sum), and every 32 of them the lanes update their
// weights together (independent loads, one latency per 32 updates).  No
// dense pass: the work follows the entries.
__device__ void merge_update(const gcsgd_pair* stage, const uint32_t* soff, int K, uint64_t R0, uint64_t R1, float fk,
                             float lr, float* w) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t per_w = (R1 - R0 + NW - 1) / NW;
    const uint64_t P0 = R0 + (uint64_t)warp * per_w < R1 ? R0 + (uint64_t)warp * per_w : R1;
    const uint64_t P1 = P0 + per_w < R1 ? P0 + per_w : R1;
    const bool pow2 = (K & (K - 1)) == 0;
    const float inv_k = 1.0f / fk;
    uint32_t c = 0, e = 0, hidx = 0xffffffffu;  // head of list `lane` (valid when `has`)
    float hval = 0.0f;
    bool has = false;
    auto load_head = [&]() {
        has = false;
        if (c < e) {
            const gcsgd_pair it = stage[c];
            if ((uint64_t)it.idx < P1) {
                hidx = it.idx;
                hval = it.val;
                has = true;
            }
        }
    };
    if (lane < K) {
        e = soff[lane + 1];
        c = lower_in(stage, soff[lane], e, P0);
        load_head();
    }
    uint32_t my_idx = 0, nb = 0;
    float my_sum = 0.0f;
    auto flush = [&]() {
        if ((uint32_t)lane < nb) w[my_idx] = __fsub_rn(w[my_idx], __fmul_rn(lr, div_k(my_sum, fk, inv_k, pow2)));
        nb = 0;
    };
    for (;;) {  // every round advances at least one lane: at most `total` rounds
        if (!__any_sync(kFull, has)) break;
        const uint32_t m = __reduce_min_sync(kFull, has ? hidx : 0xffffffffu);
        const unsigned at = __ballot_sync(kFull, has && hidx == m);
        float sum = 0.0f;
        for (unsigned mm = at; mm; mm &= mm - 1u) sum = __fadd_rn(sum, __shfl_sync(kFull, hval, __ffs(mm) - 1));
        if ((uint64_t)m >= P0 && (uint32_t)lane == nb) {  // (m < P0 only for unsorted input)
            my_idx = m;
            my_sum = sum;
        }
        nb += (uint64_t)m >= P0 ? 1u : 0u;
        if (has && hidx == m) {
            ++c;
            load_head();
        }
        if (nb == 32) flush();
    }
    flush();
}

// Shared memory: acc[kTile] | stage[kStage] pairs | per list (u64): cnt, ptr, wbeg |
// (u32): wlen, flag, soff[K+1] | bnd[K][NW+1] (u32)
template <bool UPDATE>
__global__ void __launch_bounds__(NT) spavg_kernel(const gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                   const int64_t* __restrict__ counts, int K, uint64_t n,
                                                   float* __restrict__ out, uint64_t tiles, uint64_t tiles_per_cta,
                                                   uint32_t C, float lr) {
    extern __shared__ __align__(16) unsigned char smem[];
    float* acc = reinterpret_cast<float*>(smem);
    gcsgd_pair* stage = reinterpret_cast<gcsgd_pair*>(smem + kTile * sizeof(float));
    const size_t stage_items = (size_t)K * C > kStage ? (size_t)K * C : kStage;  // as sized by the host
    uint64_t* cnt = reinterpret_cast<uint64_t*>(smem + kTile * sizeof(float) + stage_items * sizeof(gcsgd_pair));
    uint64_t* ptr = cnt + K;   // first entry of list k not yet added (global position)
    uint64_t* wbeg = ptr + K;  // global position of the first staged entry of list k
    uint32_t* wlen = reinterpret_cast<uint32_t*>(wbeg + K);  // staged entries of list k
    uint32_t* flag = wlen + K;                               // window k refills / list k is dense in this tile
    uint32_t* soff = flag + K;                               // range staging: list k at [soff[k], soff[k+1])
    uint32_t* bnd = soff + K + 1;                            // [K][NW+1] slice bounds within the windows
    __shared__ int s_any;
    __shared__ uint32_t s_total;
    __shared__ uint32_t touched2[2][kTile / 32];  // update mode: positions some list carries, by tile parity
    if (UPDATE)
        for (uint32_t q = threadIdx.x; q < 2 * (kTile / 32); q += NT) (&touched2[0][0])[q] = 0u;
    const uint64_t t0 = (uint64_t)blockIdx.x * tiles_per_cta;
    if (t0 >= tiles) return;
    const uint64_t t1 = t0 + tiles_per_cta < tiles ? t0 + tiles_per_cta : tiles;
    const uint64_t R0 = t0 * kTile, R1 = t1 * kTile < n ? t1 * kTile : n;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float fk = (float)K;
    constexpr uint32_t kSpan = kTile / NW;  // output indices owned by one warp within a tile

    for (int k = threadIdx.x; k < K; k += NT) {
        const int64_t c = counts[k];
        cnt[k] = c < 0 ? 0 : ((uint64_t)c > cap ? cap : (uint64_t)c);
        wlen[k] = 0;
    }
    __syncthreads();
    // each list's run inside this CTA's index range [R0, R1): both ends searched in parallel
    for (int q = warp; q < 2 * K; q += NW) {
        const int k = q < K ? q : q - K;
        const uint64_t p = warp_lower_bound(lists + (uint64_t)k * cap, cnt[k], q < K ? R0 : R1);
        if (lane == 0) {
            if (q < K) ptr[k] = p;
            else wbeg[k] = p;  // temporarily: the run's end
        }
        __syncwarp();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint64_t run = 0;
        for (int k = 0; k < K; ++k) {
            soff[k] = (uint32_t)(run < kStage ? run : kStage);
            run += wbeg[k] > ptr[k] ? wbeg[k] - ptr[k] : 0;
        }
        soff[K] = (uint32_t)(run < kStage ? run : kStage);
        s_total = run <= kStage ? (uint32_t)run : 0xffffffffu;
    }
    for (uint32_t j = threadIdx.x * 4; j < kTile; j += NT * 4)
        *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    const uint32_t total = s_total;

    if (total != 0xffffffffu) {
        // The whole range's entries fit: stage them once (four loads in
        // flight per thread); warp 0 adds them tile by tile in learner order.
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
                    it[j] = lists[(uint64_t)k * cap + ptr[k] + (q - soff[k])];
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (kk[j] >= 0) stage[q0 + j * NT + threadIdx.x] = it[j];
        }
        for (int k = threadIdx.x; k < K; k += NT) wlen[k] = soff[k];  // reuse: next staged entry of list k
        __syncthreads();
        if (UPDATE && K <= 32) {
            merge_update(stage, soff, K, R0, R1, fk, lr, out);
            return;
        }
        for (uint64_t t = t0; t < t1; ++t) {
            const uint64_t r0 = t * kTile;
            const uint64_t r1 = r0 + kTile < n ? r0 + kTile : n;
            if (warp == 0) {
                for (int k = 0; k < K; ++k) {
                    uint32_t a = wlen[k];
                    const uint32_t e = soff[k + 1];
                    for (;;) {
                        const uint32_t i = a + lane;
                        gcsgd_pair it;
                        it.idx = 0xffffffffu;
                        it.val = 0.f;
                        if (i < e) it = stage[i];
                        const bool in = i < e && (uint64_t)it.idx < r1;
                        if (in && (uint64_t)it.idx >= r0) {
                            const uint32_t pos = (uint32_t)(it.idx - r0);
                            acc[pos] = __fadd_rn(acc[pos], it.val);
                            if (UPDATE) atomicOr(&touched2[t & 1][pos >> 5], 1u << (pos & 31));
                        }
                        const int c = __popc(__ballot_sync(kFull, in));
                        a += c;
                        if (c < 32) break;
                    }
                    __syncwarp();  // list k's adds land before list k+1's
                    if (lane == 0) wlen[k] = a;
                }
            }
            __syncthreads();
            if (UPDATE) update_tile(acc, touched2[t & 1], touched2[(t + 1) & 1], out, r0, r1, fk, lr);
            else store_tile(acc, out, r0, r1, fk);  // also re-zeroes acc
            __syncthreads();
        }
        return;
    }

    // Too many entries for one staging: each list keeps a window of C of its
    // next entries, refilled when it no longer reaches past the tile; each
    // warp owns kSpan output indices of the tile and adds the lists in order.
    for (int k = threadIdx.x; k < K; k += NT) wbeg[k] = ptr[k];
    __syncthreads();
    for (uint64_t t = t0; t < t1; ++t) {
        const uint64_t r0 = t * kTile;
        const uint64_t r1 = r0 + kTile < n ? r0 + kTile : n;
        if (threadIdx.x == 0) s_any = 0;
        __syncthreads();
        for (int k = threadIdx.x; k < K; k += NT) {
            const gcsgd_pair* st = stage + (size_t)k * C;
            const bool covers = wbeg[k] + wlen[k] == cnt[k] || (wlen[k] > 0 && (uint64_t)st[wlen[k] - 1].idx >= r1);
            flag[k] = 0;
            if (!covers) {
                wbeg[k] = ptr[k];
                const uint64_t left = cnt[k] - ptr[k];
                wlen[k] = (uint32_t)(left < C ? left : C);
                flag[k] = 1;
                s_any = 1;
            }
        }
        __syncthreads();
        if (s_any) {
            for (int k = 0; k < K; ++k) {  // refill windows (four loads in flight per thread)
                if (!flag[k] || wlen[k] == 0) continue;
                const gcsgd_pair* L = lists + (uint64_t)k * cap + wbeg[k];
                gcsgd_pair* st = stage + (size_t)k * C;
                const uint32_t wl = wlen[k];
                for (uint32_t q0 = 0; q0 < wl; q0 += 4 * NT) {
                    gcsgd_pair it[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint32_t q = q0 + jj * NT + threadIdx.x;
                        if (q < wl) it[jj] = L[q];
                    }
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint32_t q = q0 + jj * NT + threadIdx.x;
                        if (q < wl) st[q] = it[jj];
                    }
                }
            }
            __syncthreads();
        }
        // slice bounds: one thread per (list, warp slice edge), all searched at once
        for (int q = threadIdx.x; q < K * (NW + 1); q += NT) {
            const int k = q / (NW + 1), w = q - k * (NW + 1);
            const gcsgd_pair* st = stage + (size_t)k * C;
            const bool covers = wbeg[k] + wlen[k] == cnt[k] || (wlen[k] > 0 && (uint64_t)st[wlen[k] - 1].idx >= r1);
            if (w == 0) flag[k] = !covers;  // dense in this tile: read in place
            const uint64_t edge = r0 + (uint64_t)w * kSpan < r1 ? r0 + (uint64_t)w * kSpan : r1;
            bnd[q] = covers ? lower_in(st, (uint32_t)(ptr[k] - wbeg[k]), wlen[k], edge) : 0u;
        }
        __syncthreads();
        const uint64_t s0 = r0 + (uint64_t)warp * kSpan;
        const uint64_t s1 = s0 + kSpan < r1 ? s0 + kSpan : r1;
        if (s0 < r1) {
            for (int k = 0; k < K; ++k) {
                if (!flag[k]) {
                    const gcsgd_pair* st = stage + (size_t)k * C;
                    const uint32_t a = bnd[k * (NW + 1) + warp], b = bnd[k * (NW + 1) + warp + 1];
                    for (uint32_t i = a + lane; i < b; i += 32) {
                        const gcsgd_pair it = st[i];
                        if ((uint64_t)it.idx >= s0 && (uint64_t)it.idx < s1) {  // always, for sorted lists
                            const uint32_t pos = (uint32_t)(it.idx - r0);
                            acc[pos] = __fadd_rn(acc[pos], it.val);
                            if (UPDATE) atomicOr(&touched2[t & 1][pos >> 5], 1u << (pos & 31));
                        }
                    }
                } else {
                    const gcsgd_pair* L = lists + (uint64_t)k * cap;
                    const uint64_t a = lower_global(L, ptr[k], cnt[k], s0);
                    const uint64_t b = lower_global(L, a, cnt[k], s1);
                    for (uint64_t i = a + lane; i < b; i += 32) {
                        const gcsgd_pair it = L[i];
                        if ((uint64_t)it.idx >= s0 && (uint64_t)it.idx < s1) {
                            const uint32_t pos = (uint32_t)(it.idx - r0);
                            acc[pos] = __fadd_rn(acc[pos], it.val);
                            if (UPDATE) atomicOr(&touched2[t & 1][pos >> 5], 1u << (pos & 31));
                        }
                    }
                }
                __syncwarp();  // list k's adds land before list k+1's
            }
        }
        __syncthreads();
        for (int k = threadIdx.x; k < K; k += NT)
            ptr[k] = flag[k] ? lower_global(lists + (uint64_t)k * cap, ptr[k], cnt[k], r1)
                             : wbeg[k] + bnd[k * (NW + 1) + NW];
        if (UPDATE) update_tile(acc, touched2[t & 1], touched2[(t + 1) & 1], out, r0, r1, fk, lr);
        else store_tile(acc, out, r0, r1, fk);
        __syncthreads();
    }
}


// ---------------------------------------------------------------- warp spans
// The dense average for dense lists, without CTA barriers: every warp owns a
// contiguous run of 512-index output spans and keeps, per list, a cursor at
// the first entry it has not consumed (found once, at the run's start, by a
// 32-ary search of eight lists at a time).  For each span the warp loads the
// next 64 entries of eight lists at once (sixteen loads in flight per lane),
// then adds them in learner order into its 2 KB accumulator (a list's
// indices are distinct, so one list's adds never collide; __syncwarp orders
// the lists), loads more of a list only when all 64 fell inside the span,
// and writes the span once with 128-bit stores.  Lists sorted ascending make
// every entry read once (plus the look-ahead) and every output written once.
// A span costs one load latency, so sparse lists (a few entries per span)
// go to the tile kernel instead, which pays its latencies per 4096-index
// tile and stages whole ranges of entries.
constexpr uint32_t kWSpan = 512;  // output indices per warp span
constexpr int kBatch = 8;         // lists loaded together

__device__ __forceinline__ gcsgd_pair load_entry(const gcsgd_pair* L, uint32_t i, uint32_t cnt) {
    gcsgd_pair it;
    it.idx = 0u;
    it.val = 0.0f;
    if (i < cnt) it = L[i];
    return it;
}

// First position p in [0, cnt_k] with list_k[p].idx >= target, for the lists
// k0 .. k0+nb-1 at once (nb <= kBatch); results to cur[k].  Called by a warp.
__device__ void batch_lower_bound(const gcsgd_pair* lists, uint64_t cap, const uint32_t* cnt, int k0, int nb,
                                  uint64_t target, uint32_t* cur) {
    const int lane = threadIdx.x & 31;
    uint32_t lo[kBatch], hi[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
        lo[q] = 0;
        hi[q] = q < nb ? cnt[k0 + q] : 0u;
    }
    for (;;) {
        bool wide = false;
#pragma unroll
        for (int q = 0; q < kBatch; ++q) wide |= hi[q] - lo[q] > 32;
        if (!wide) break;
        bool pr[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {  // every probe of the round in flight together
            pr[q] = true;
            if (hi[q] - lo[q] > 32) {
                const uint32_t step = (hi[q] - lo[q] + 31) / 32;
                const uint64_t p = (uint64_t)lo[q] + (uint64_t)(lane + 1) * step - 1;
                if (p < hi[q]) pr[q] = (uint64_t)__ldg(&lists[(uint64_t)(k0 + q) * cap + p].idx) >= target;
            }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            if (hi[q] - lo[q] <= 32) continue;  // uniform across the warp
            const uint32_t step = (hi[q] - lo[q] + 31) / 32;
            const unsigned b = __ballot_sync(kFull, pr[q]);
            const int f = b ? __ffs(b) - 1 : 32;
            const uint64_t nlo = (uint64_t)lo[q] + (uint64_t)f * step;
            const uint64_t qf = (uint64_t)lo[q] + (uint64_t)(f + 1) * step - 1;
            hi[q] = (f < 32 && qf < hi[q]) ? (uint32_t)qf : hi[q];
            lo[q] = (uint32_t)(nlo < hi[q] ? nlo : hi[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
        if (q >= nb) break;
        const uint32_t p = lo[q] + lane;
        const bool pred = p >= hi[q] || (uint64_t)__ldg(&lists[(uint64_t)(k0 + q) * cap + p].idx) >= target;
        const unsigned b = __ballot_sync(kFull, pred);
        const uint32_t r = lo[q] + (b ? __ffs(b) - 1 : 32);
        if (lane == 0) cur[k0 + q] = r < hi[q] ? r : hi[q];
    }
}

// Shared memory: acc[NW][kWSpan] floats | cnt[K] | cur[NW][K] (u32).
// REG (K <= kBatch): counts and cursors live in registers instead.
template <bool REG>
__global__ void __launch_bounds__(NT, 4) spavg_warp(const gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                    const int64_t* __restrict__ counts, int K, uint64_t n,
                                                    float* __restrict__ out, uint64_t spans, uint64_t per_warp) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* acc = reinterpret_cast<float*>(smem) + (size_t)warp * kWSpan;
    uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + sizeof(float) * NW * kWSpan);
    uint32_t* cur = cnt + K + (size_t)warp * K;
    for (int k = threadIdx.x; k < K; k += NT) {
        const int64_t c = counts[k];
        const uint64_t cc = c < 0 ? 0 : ((uint64_t)c > cap ? cap : (uint64_t)c);
        cnt[k] = (uint32_t)(cc < 0xffffffffu - 64 ? cc : 0xffffffffu - 64);
    }
    for (uint32_t j = lane * 4; j < kWSpan; j += 128) *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    const uint64_t sp0 = ((uint64_t)blockIdx.x * NW + warp) * per_warp;
    if (sp0 >= spans) return;
    const uint64_t sp1 = sp0 + per_warp < spans ? sp0 + per_warp : spans;
    for (int kb = 0; kb < K; kb += kBatch)
        batch_lower_bound(lists, cap, cnt, kb, K - kb < kBatch ? K - kb : kBatch, sp0 * kWSpan, cur);
    __syncwarp();
    uint32_t rcur[kBatch], rcnt[kBatch];  // REG: list q's cursor and count (the same in every lane)
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
        rcur[q] = REG && q < K ? cur[q] : 0u;
        rcnt[q] = REG && q < K ? cnt[q] : 0u;
    }
    const float fk = (float)K, inv_k = 1.0f / fk;
    const bool pow2 = (K & (K - 1)) == 0;
    for (uint64_t sp = sp0; sp < sp1; ++sp) {
        // span [s0, s0 + len): an entry is inside iff idx - s0 < len in 32 bits (s0 < 2^32)
        const uint32_t s0 = (uint32_t)(sp * kWSpan);
        const uint32_t len = (uint32_t)((sp + 1) * kWSpan < n ? kWSpan : n - sp * kWSpan);
        for (int kb = 0; kb < (REG ? 1 : K); kb += kBatch) {
            const int nb = K - kb < kBatch ? K - kb : kBatch;
            gcsgd_pair e[kBatch], f[kBatch];  // the next 64 entries of each list (two per lane)
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                e[q].idx = f[q].idx = 0u;
                e[q].val = f[q].val = 0.0f;
                if (q < nb) {
                    const gcsgd_pair* L = lists + (uint64_t)(kb + q) * cap;
                    const uint32_t c0 = REG ? rcur[q] : cur[kb + q], c = REG ? rcnt[q] : cnt[kb + q];
                    e[q] = load_entry(L, c0 + lane, c);
                    f[q] = load_entry(L, c0 + 32 + lane, c);
                }
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                if (q >= nb) break;
                const int k = kb + q;
                const uint32_t ck = REG ? rcnt[q] : cnt[k];
                uint32_t c0 = REG ? rcur[q] : cur[k];
                gcsgd_pair it = e[q];
                for (int round = 0;; ++round) {
                    // entries of this span form a prefix of the 32 (lists sorted ascending); an
                    // entry below the span (an unsorted list) ends the prefix and stays unread
                    const uint32_t d = it.idx - s0;
                    const bool in = c0 + lane < ck && d < len;
                    const unsigned b = __ballot_sync(kFull, !in);
                    const uint32_t c = b ? (uint32_t)__ffs(b) - 1 : 32u;
                    if ((uint32_t)lane < c) acc[d] = __fadd_rn(acc[d], it.val);
                    c0 += c;
                    if (c < 32) break;
                    it = round == 0 ? f[q] : load_entry(lists + (uint64_t)k * cap, c0 + lane, ck);
                }
                __syncwarp();  // list k's adds land before list k+1's, and every lane has read cur[k]
                if (REG) {
                    rcur[q] = c0;
                } else {
                    if (lane == 0) cur[k] = c0;
                    __syncwarp();
                }
            }
        }
        // the span's average, written once; acc re-zeroed for the next span
        const bool al = ((uintptr_t)(out + s0) & 15) == 0;
#pragma unroll
        for (int r = 0; r < (int)(kWSpan / 128); ++r) {
            const uint32_t j = 4u * (lane + 32 * r);
            float4 q = *reinterpret_cast<const float4*>(acc + j);
            *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j >= len) continue;
            if (pow2) {  // x * 2^-j is x / 2^j rounded once
                q.x = __fmul_rn(q.x, inv_k);
                q.y = __fmul_rn(q.y, inv_k);
                q.z = __fmul_rn(q.z, inv_k);
                q.w = __fmul_rn(q.w, inv_k);
            } else {
                q.x = div_k(q.x, fk, inv_k, false);
                q.y = div_k(q.y, fk, inv_k, false);
                q.z = div_k(q.z, fk, inv_k, false);
                q.w = div_k(q.w, fk, inv_k, false);
            }
            if (al && j + 4 <= len) {
                *reinterpret_cast<float4*>(out + s0 + j) = q;
            } else {
                const float* qq = &q.x;
                for (uint32_t i = 0; i < 4 && j + i < len; ++i) out[s0 + j + i] = qq[i];
            }
        }
        __syncwarp();
    }
}


// ---------------------------------------------------------------- regions
// The dense average with a workspace (sparse_average_ws), in two kernels.
//
// spavg_checkpoints reads every 128th entry of every list and writes a
// cursor table: lo[k][g] = 128 j for the last checkpoint j of list k whose
// index is below g * kRegion (0 if none).  The first entry of list k at or
// after region g then lies in [lo[k][g], lo[k][g] + 128], and every entry of
// region g in [lo[k][g], lo[k][g+1] + 128).  (A 32-byte read brings in the
// whole 128-byte line, so a denser table would cost far more list bytes.)
//
// spavg_region: CTA c takes the 4096-output regions c, c + grid, ... (every
// CTA gets dense and sparse parts of the output alike).  One producer warp
// plans each region (the list ranges from the table, their stage slots)
// and copies the ranges into shared memory with TMA bulk copies (one per
// list, 16-byte aligned; a first or last pair off that boundary by
// cp.async), completing on an mbarrier, into one of two stage buffers: the
// copies for the next region fly while the consumers add the current one.
// Eight consumer warps add each list's staged entries into a shared
// accumulator in learner order (a named barrier among them between lists;
// a list's indices are distinct, so its adds never collide; entries outside
// the region are skipped), release the buffer and write the region once.
// A region whose ranges exceed a stage buffer is added straight from global
// memory instead.
constexpr uint32_t kRegion = 4096;        // outputs per region
constexpr uint32_t kRStage = 6048;        // list entries per stage buffer
constexpr uint32_t kCheck = 128;          // checkpoint stride of the cursor table
constexpr uint32_t kSlow = 0xffffffffu;   // stage total of a region added from global memory
constexpr uint32_t kSuspendNs = 20000;    // longest sleep of one barrier try
constexpr uint64_t kWaitNs = 1000000000;  // a barrier phase not complete after 1 s counts as lost
constexpr uint32_t kWaitLimit = 1u << 26; // tries, should the global timer not advance

__device__ __forceinline__ uint32_t clamp_count(int64_t c, uint64_t cap) {
    const uint64_t cc = c < 0 ? 0 : ((uint64_t)c > cap ? cap : (uint64_t)c);
    return (uint32_t)(cc < 0xffffffffu ? cc : 0xffffffffu);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// True once the phase with `parity` has completed; the warp sleeps (up to
// kSuspendNs) while it has not, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "n"(kSuspendNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Waits until the phase with `parity` completes; false once kWaitNs have
// passed (or kWaitLimit tries, should the clock not advance).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
    return false;
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned), counted on `bar`.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// Cursor table lo[K][G+1] (G regions; lo[k][G] closes the last one).  Block
// row y = list; blocks along x stride over the list's checkpoints.  For a
// sorted list every lo[k][g] is written exactly once: checkpoint j (index a)
// owns the regions g with a < g * kRegion <= the next checkpoint's index
// (all regions up to G for the last checkpoint, from 0 for the first).
// Block (0, 0) also clears the status word.
__global__ void __launch_bounds__(NT) spavg_checkpoints(const gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                        const int64_t* __restrict__ counts, uint64_t G,
                                                        uint32_t* __restrict__ lo, uint32_t* __restrict__ status) {
    const int k = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const uint32_t cnt = clamp_count(counts[k], cap);
    const uint64_t J = (cnt + kCheck - 1) / kCheck;
    uint32_t* row = lo + (uint64_t)k * (G + 1);
    if (k == 0 && blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
    if (J == 0) {  // an empty list: every region starts at position 0
        for (uint64_t g = (uint64_t)blockIdx.x * NT + threadIdx.x; g <= G; g += (uint64_t)gridDim.x * NT) row[g] = 0u;
        return;
    }
    const gcsgd_pair* L = lists + (uint64_t)k * cap;
    for (uint64_t j0 = (uint64_t)blockIdx.x * NT; j0 < J; j0 += (uint64_t)gridDim.x * NT) {  // uniform per block
        const uint64_t j = j0 + threadIdx.x;
        uint64_t g0 = 0, g1 = 0;  // this checkpoint's regions [g0, g1)
        if (j < J) {
            const uint64_t a = __ldg(&L[j * kCheck].idx);
            g0 = j == 0 ? 0 : a / kRegion + 1;
            g1 = j + 1 < J ? (uint64_t)__ldg(&L[(j + 1) * kCheck].idx) / kRegion + 1 : G + 1;
            g0 = g0 < G + 1 ? g0 : G + 1;
            g1 = g1 < G + 1 ? g1 : G + 1;
            g1 = g1 > g0 ? g1 : g0;  // a checkpoint out of order (a malformed list) owns none
        }
        const uint32_t val = (uint32_t)(j * kCheck);
        const bool many = g1 - g0 > 4;
        if (!many)
            for (uint64_t g = g0; g < g1; ++g) row[g] = val;
        for (unsigned pend = __ballot_sync(kFull, many); pend; pend &= pend - 1u) {  // long runs: the warp writes them
            const int src = __ffs(pend) - 1;
            const uint64_t s0 = __shfl_sync(kFull, g0, src), s1 = __shfl_sync(kFull, g1, src);
            const uint32_t v = __shfl_sync(kFull, val, src);
            for (uint64_t g = s0 + lane; g < s1; g += 32) row[g] = v;
        }
    }
}

// Shared memory (dynamic): acc[kRegion] floats | stage[kNBuf][kRStage] pairs |
// per buffer b: pa[K] (first list position of the range), pl[K] (its
// length), pm[K] (staged slots, even, | 1 when the first pair is copied
// alone), st[K] (stage slot of the first entry) | cnt[K].  Lists must be
// 8-byte aligned.
//
// Warp kCW is the producer: for its CTA's regions in turn it waits until
// the consumers have released the stage buffer (empty[b]), plans the
// region's ranges and stage slots, and issues the copies, which complete
// on full[b] (kFullArrivals arrivals: its expect-tx arrive plus one
// cp.async arrive per lane, and the bulk-copied bytes).  Warps 0..kCW-1 are
// the consumers: wait for full[b], add list by list (a named barrier among
// them between lists), release the buffer, and store the region.  Every
// wait is bounded; a wait that runs out sets the status word, and the
// consumers leave together (their decision is reduced over all of them).
constexpr int kCW = 8;                      // consumer warps
constexpr int kProducer = kCW;
constexpr int NTR = (kCW + 1) * 32;         // threads per CTA: consumers and one producer warp
constexpr int kNBuf = 2;                    // stage buffers
constexpr int kPer = 2;                     // entries per consumer thread and list read ahead
constexpr int kRegK = 8;                    // lists whose staged ranges the consumers keep in registers
constexpr uint32_t kFullArrivals = 33;      // producer lane 0's expect-tx arrive + 32 cp.async arrives

__device__ __forceinline__ void mbar_init_n(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

// One arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kCW * 32) : "memory"); }

// True iff p holds in every consumer thread (a named barrier among them).
__device__ __forceinline__ bool consumers_all(bool p) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred q, a;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred a, 1, %2, q;\n selp.u32 %0, 1, 0, a;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)p), "n"(kCW * 32)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    return v;
}

// A list's range for a region from its table entries t_a = lo[k][g] and
// t_b = lo[k][g+1]: the first position a, the length, whether the first
// pair is copied alone (it sits 8 bytes off the 16-byte boundary), the
// bulk-copied pairs and the staged slots (even; the first and last pairs
// copied alone take slots of their own beside the bulk part).
struct Range {
    uint32_t a, len, head, body, slots;
};

__device__ __forceinline__ Range range_of(const gcsgd_pair* lists, uint64_t cap, uint32_t c, int k, uint32_t t_a,
                                          uint32_t t_b) {
    Range R;
    R.a = t_a < c ? t_a : c;
    const uint64_t e64 = (uint64_t)t_b + kCheck;
    const uint32_t e0 = e64 < c ? (uint32_t)e64 : c;
    R.len = e0 > R.a ? e0 - R.a : 0u;
    const uintptr_t s = (uintptr_t)(lists + (uint64_t)k * cap + R.a);
    R.head = R.len > 0 && (s & 8) ? 1u : 0u;
    const uintptr_t bs = s + 8 * R.head, be = (s + 8 * (uintptr_t)R.len) & ~(uintptr_t)15;
    R.body = be > bs ? (uint32_t)((be - bs) / 8) : 0u;
    R.slots = (2 * R.head + R.body + (R.len - R.head - R.body) + 1) & ~1u;
    return R;
}

// UPDATE: instead of writing the average, step the weights in `out` at the
// carried indices, w <- w - lr * avg (one rounding each; every other weight
// keeps its bits): the consumers mark the carried positions in a bitmap (two,
// by region parity, so the next region's is cleared while this one is read)
// and read the region's weights while the lists are added.
template <bool UPDATE>
__global__ void __launch_bounds__(NTR, 2) spavg_region(const gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                    const int64_t* __restrict__ counts, int K, uint64_t n,
                                                    float* __restrict__ out, const uint32_t* __restrict__ lo,
                                                    uint64_t G, uint32_t* __restrict__ status, float lr) {
    extern __shared__ __align__(16) unsigned char smem[];
    float* acc = reinterpret_cast<float*>(smem);
    gcsgd_pair* stage = reinterpret_cast<gcsgd_pair*>(smem + kRegion * sizeof(float));
    uint32_t* arr = reinterpret_cast<uint32_t*>(stage + kNBuf * kRStage);
    uint32_t* cnt = arr + 4 * kNBuf * K;
    __shared__ __align__(8) uint64_t full[kNBuf], empty[kNBuf];
    __shared__ uint32_t s_total[kNBuf];
    __shared__ uint32_t touched[UPDATE ? 2 : 1][UPDATE ? kRegion / 32 : 1];
    auto PA = [&](int b) { return arr + (4 * b + 0) * K; };
    auto PL = [&](int b) { return arr + (4 * b + 1) * K; };
    auto PM = [&](int b) { return arr + (4 * b + 2) * K; };
    auto ST = [&](int b) { return arr + (4 * b + 3) * K; };
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t g0 = blockIdx.x, grid = gridDim.x;
    if (g0 >= G) return;
    for (int k = threadIdx.x; k < K; k += NTR) cnt[k] = clamp_count(counts[k], cap);
    for (uint32_t j = threadIdx.x * 4; j < kRegion; j += NTR * 4)
        *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (UPDATE)
        for (uint32_t q = threadIdx.x; q < 2 * (kRegion / 32); q += NTR) (&touched[0][0])[q] = 0u;
    if (threadIdx.x == 0) {
        for (int b = 0; b < kNBuf; ++b) {
            mbar_init_n(&full[b], kFullArrivals);
            mbar_init_n(&empty[b], kCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        fence_proxy_async();
    }
    __syncthreads();

    if (warp == kProducer) {
        // ------------------------------------------------------ producer
        uint32_t pre_a = 0, pre_b = 0;  // K <= 32: list `lane`'s table entries for the next region
        auto prefetch = [&](uint64_t gr) {
            if (K <= 32 && gr < G && lane < K) {
                pre_a = __ldg(&lo[(uint64_t)lane * (G + 1) + gr]);
                pre_b = __ldg(&lo[(uint64_t)lane * (G + 1) + gr + 1]);
            }
        };
        prefetch(g0);
        int i = 0;
        bool aborted = false;
        for (uint64_t g = g0; g < G; g += grid, ++i) {
            const int b = i % kNBuf;
            if (i >= kNBuf && !mbar_wait_bounded(&empty[b], (uint32_t)((i / kNBuf - 1) & 1))) {
                aborted = true;
                break;
            }
            uint32_t* pa = PA(b);
            uint32_t* pl = PL(b);
            uint32_t* pm = PM(b);
            uint32_t* st = ST(b);
            gcsgd_pair* buf = stage + (size_t)b * kRStage;
            // ranges (chunks of 32 lists), the stage total and the bulk bytes
            uint32_t total = 0, bytes = 0;
            for (int c0 = 0; c0 < K; c0 += 32) {
                const int k = c0 + lane;
                uint32_t slots = 0, body = 0;
                if (k < K) {
                    const uint32_t ta_ = K <= 32 ? pre_a : __ldg(&lo[(uint64_t)k * (G + 1) + g]);
                    const uint32_t tb_ = K <= 32 ? pre_b : __ldg(&lo[(uint64_t)k * (G + 1) + g + 1]);
                    const Range R = range_of(lists, cap, cnt[k], k, ta_, tb_);
                    pa[k] = R.a;
                    pl[k] = R.len;
                    pm[k] = R.slots | R.head;
                    slots = R.slots;
                    body = R.body;
                }
                total += warp_sum(slots);
                bytes += warp_sum(body * 8u);
            }
            prefetch(g + grid);
            const bool fits = total <= kRStage;
            // stage slots; the single first and last pairs by cp.async
            uint32_t carry = 0;
            for (int c0 = 0; c0 < K; c0 += 32) {
                const int k = c0 + lane;
                const uint32_t m = k < K ? pm[k] : 0u, slots = m & ~1u, head = m & 1u;
                uint32_t incl = slots;
                for (int d = 1; d < 32; d <<= 1) {
                    const uint32_t v = __shfl_up_sync(kFull, incl, d);
                    if (lane >= d) incl += v;
                }
                if (k < K) {
                    const uint32_t slot = carry + incl - slots + head;
                    st[k] = slot;
                    const uint32_t len = pl[k];
                    if (fits && len > 0) {
                        const gcsgd_pair* L = lists + (uint64_t)k * cap + pa[k];
                        const uintptr_t s = (uintptr_t)L;
                        const uintptr_t bs = s + 8 * head, be = (s + 8 * (uintptr_t)len) & ~(uintptr_t)15;
                        const uint32_t body = be > bs ? (uint32_t)((be - bs) / 8) : 0u;
                        if (head) cp_async8(&buf[slot], &L[0]);
                        if (head + body < len) cp_async8(&buf[slot + len - 1], &L[len - 1]);
                    }
                }
                carry += __shfl_sync(kFull, incl, 31);
            }
            __syncwarp();  // every lane's plan written before lane 0 publishes it
            if (lane == 0) {
                s_total[b] = fits ? total : kSlow;
                mbar_arrive_expect(&full[b], fits ? bytes : 0u);
            }
            __syncwarp();
            if (fits)
                for (int k = lane; k < K; k += 32) {
                    const uint32_t len = pl[k], head = pm[k] & 1u;
                    if (len == 0) continue;
                    const gcsgd_pair* L = lists + (uint64_t)k * cap + pa[k];
                    const uintptr_t s = (uintptr_t)L;
                    const uintptr_t bs = s + 8 * head, be = (s + 8 * (uintptr_t)len) & ~(uintptr_t)15;
                    const uint32_t body = be > bs ? (uint32_t)((be - bs) / 8) : 0u;
                    if (body) bulk_copy(&buf[st[k] + head], L + head, body * 8u, &full[b]);
                }
            cp_async_arrive(&full[b]);
        }
        if (aborted) {
            atomicOr(status, 1u);
            // the copies of the buffers still armed land before the CTA may end
            for (int q = 1; q <= kNBuf && i - q >= 0; ++q)
                (void)mbar_wait_bounded(&full[(i - q) % kNBuf], (uint32_t)(((i - q) / kNBuf) & 1));
        }
        cp_async_wait<0>();
        return;
    }

    // ---------------------------------------------------------- consumers
    // Every consumer thread takes entries ct, ct + 256, ... of each list's
    // staged range, list after list in learner order (a named barrier among
    // the consumers between lists; a list's indices are distinct, so its adds
    // never collide; entries outside the region are skipped), then the
    // consumers release the buffer and store the region.  The first two
    // entries per thread of list k+1 are read while list k is added.  A list
    // step is a dependent chain (accumulator read, add, write, barrier), so
    // for K <= 8 the ranges sit in registers and the next list's entries are
    // read after this list's accumulator reads are issued: nothing of the
    // read-ahead waits in front of the chain.
    const int ct = threadIdx.x;
    constexpr int NC = kCW * 32;
    const float fk = (float)K, inv_k = 1.0f / fk;
    const bool pow2 = (K & (K - 1)) == 0;
    const bool al = ((uintptr_t)out & 15) == 0;
    int i = 0;
    for (uint64_t g = g0; g < G; g += grid, ++i) {
        const int b = i % kNBuf;
        const bool ok = mbar_wait_bounded(&full[b], (uint32_t)((i / kNBuf) & 1));
        if (!consumers_all(ok)) {
            if (ct == 0) atomicOr(status, 1u);
            return;
        }
        const uint32_t R0 = (uint32_t)(g * kRegion);
        const uint32_t rlen = (uint32_t)((uint64_t)R0 + kRegion < n ? kRegion : n - R0);
        const uint32_t* pl = PL(b);
        uint32_t* tb = touched[UPDATE ? (i & 1) : 0];
        constexpr int kW = UPDATE ? (int)(kRegion / (4 * NC)) : 1;
        float4 wv[kW];  // UPDATE: the region's weights of this thread, read while the lists are added
        if (UPDATE) {
#pragma unroll
            for (int r = 0; r < kW; ++r) {
                const uint32_t j = 4u * (ct + r * NC);
                const float* wj = out + R0 + j;
                wv[r] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (al && j + 4 <= rlen) {
                    wv[r] = *reinterpret_cast<const float4*>(wj);
                } else {
                    float* ww = &wv[r].x;
                    for (uint32_t t = 0; t < 4 && j + t < rlen; ++t) ww[t] = wj[t];
                }
            }
        }
        if (s_total[b] != kSlow && K <= kRegK) {
            // every list's staged range (length, first slot) in registers
            const gcsgd_pair* buf = stage + (size_t)b * kRStage;
            const uint32_t* st = ST(b);
            uint32_t rl[kRegK], rs[kRegK];
#pragma unroll
            for (int k = 0; k < kRegK; ++k) {
                rl[k] = k < K ? pl[k] : 0u;
                rs[k] = k < K ? st[k] : 0u;
            }
            const gcsgd_pair none = {0xffffffffu, 0.0f};
            gcsgd_pair nx[kPer];
            auto read_ahead = [&](int k) {  // this thread's first kPer entries of list k
#pragma unroll
                for (int r = 0; r < kPer; ++r)
                    nx[r] = (uint32_t)(ct + r * NC) < rl[k] ? buf[rs[k] + ct + r * NC] : none;
            };
            read_ahead(0);
#pragma unroll
            for (int k = 0; k < kRegK; ++k) {
                if (k >= K) break;
                const uint32_t len = rl[k];
                gcsgd_pair e[kPer];
#pragma unroll
                for (int r = 0; r < kPer; ++r) e[r] = nx[r];
                if (len != 0) {  // uniform: an empty range needs no barrier
                    uint32_t d[kPer];
                    bool in[kPer];
                    float a[kPer];
#pragma unroll
                    for (int r = 0; r < kPer; ++r) {
                        d[r] = e[r].idx - R0;
                        in[r] = (uint32_t)(ct + r * NC) < len && d[r] < rlen;
                        a[r] = in[r] ? acc[d[r]] : 0.0f;
                    }
                    if (k + 1 < kRegK && k + 1 < K) read_ahead(k + 1);  // after this list's reads
#pragma unroll
                    for (int r = 0; r < kPer; ++r)
                        if (in[r]) {
                            acc[d[r]] = __fadd_rn(a[r], e[r].val);
                            if (UPDATE) atomicOr(&tb[d[r] >> 5], 1u << (d[r] & 31));
                        }
                    for (uint32_t q = ct + kPer * NC; q < len; q += NC) {  // longer ranges
                        const gcsgd_pair ee = buf[rs[k] + q];
                        const uint32_t dd = ee.idx - R0;
                        if (dd < rlen) {
                            acc[dd] = __fadd_rn(acc[dd], ee.val);
                            if (UPDATE) atomicOr(&tb[dd >> 5], 1u << (dd & 31));
                        }
                    }
                    consumer_sync();  // list k's adds land before list k+1's
                } else if (k + 1 < kRegK && k + 1 < K) {
                    read_ahead(k + 1);
                }
            }
        } else if (s_total[b] != kSlow) {
            const gcsgd_pair* buf = stage + (size_t)b * kRStage;
            const uint32_t* st = ST(b);
            const gcsgd_pair none = {0xffffffffu, 0.0f};
            uint32_t lenN = pl[0];
            const gcsgd_pair* SN = buf + st[0];
            gcsgd_pair nx[kPer];
#pragma unroll
            for (int r = 0; r < kPer; ++r) nx[r] = (uint32_t)(ct + r * NC) < lenN ? SN[ct + r * NC] : none;
            for (int k = 0; k < K; ++k) {
                const uint32_t len = lenN;
                const gcsgd_pair* S = SN;
                gcsgd_pair e[kPer];
#pragma unroll
                for (int r = 0; r < kPer; ++r) e[r] = nx[r];
                if (k + 1 < K) {
                    lenN = pl[k + 1];
                    SN = buf + st[k + 1];
#pragma unroll
                    for (int r = 0; r < kPer; ++r) nx[r] = (uint32_t)(ct + r * NC) < lenN ? SN[ct + r * NC] : none;
                }
                if (len == 0) continue;  // uniform: an empty range needs no barrier
                {
                    // a list's indices are distinct, so these adds touch different outputs:
                    // every read of acc before any write
                    uint32_t d[kPer];
                    bool in[kPer];
                    float a[kPer];
#pragma unroll
                    for (int r = 0; r < kPer; ++r) {
                        d[r] = e[r].idx - R0;  // inside iff d < rlen (R0 + rlen <= 2^32)
                        in[r] = (uint32_t)(ct + r * NC) < len && d[r] < rlen;
                        a[r] = in[r] ? acc[d[r]] : 0.0f;
                    }
#pragma unroll
                    for (int r = 0; r < kPer; ++r)
                        if (in[r]) {
                            acc[d[r]] = __fadd_rn(a[r], e[r].val);
                            if (UPDATE) atomicOr(&tb[d[r] >> 5], 1u << (d[r] & 31));
                        }
                }
                for (uint32_t q = ct + kPer * NC; q < len; q += NC) {  // longer ranges
                    const gcsgd_pair e = S[q];
                    const uint32_t d = e.idx - R0;
                    if (d < rlen) {
                        acc[d] = __fadd_rn(acc[d], e.val);
                        if (UPDATE) atomicOr(&tb[d >> 5], 1u << (d & 31));
                    }
                }
                consumer_sync();  // list k's adds land before list k+1's
            }
        } else {
            const uint32_t* pa = PA(b);
            for (int k = 0; k < K; ++k) {
                const uint32_t len = pl[k];
                if (len == 0) continue;
                const gcsgd_pair* S = lists + (uint64_t)k * cap + pa[k];
                for (uint32_t q = ct; q < len; q += NC) {
                    const gcsgd_pair e = S[q];
                    const uint32_t d = e.idx - R0;
                    if (d < rlen) {
                        acc[d] = __fadd_rn(acc[d], e.val);
                        if (UPDATE) atomicOr(&tb[d >> 5], 1u << (d & 31));
                    }
                }
                consumer_sync();
            }
        }
        // the buffer is free: its reads done before the bulk copies that refill it
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
        float* o = out + R0;
        if (UPDATE) {  // the carried weights stepped, each float4 written only where one of its values is carried
            uint32_t* tn = touched[(i + 1) & 1];  // the next region's bitmap, last read a region ago
            for (int q = ct; q < (int)(kRegion / 32); q += NC) tn[q] = 0u;
#pragma unroll
            for (int r = 0; r < kW; ++r) {
                const uint32_t j = 4u * (ct + r * NC);
                const float4 q = *reinterpret_cast<const float4*>(acc + j);
                *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
                const uint32_t bits = j < rlen ? (tb[j >> 5] >> (j & 31)) & 0xFu : 0u;
                if (!bits) continue;
                const float* qq = &q.x;
                float* xx = &wv[r].x;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if ((bits >> c) & 1u) xx[c] = __fsub_rn(xx[c], __fmul_rn(lr, div_k(qq[c], fk, inv_k, pow2)));
                if (al && j + 4 <= rlen) {
                    *reinterpret_cast<float4*>(o + j) = wv[r];
                } else {
                    for (uint32_t t = 0; t < 4 && j + t < rlen; ++t)
                        if ((bits >> t) & 1u) o[j + t] = xx[t];
                }
            }
            consumer_sync();  // acc zeroed and the bitmaps read before the next region's adds
            continue;
        }
        // the region's average, written once; acc re-zeroed for the next region
#pragma unroll
        for (int r = 0; r < (int)(kRegion / (4 * NC)); ++r) {
            const uint32_t j = 4u * (ct + r * NC);
            float4 q = *reinterpret_cast<const float4*>(acc + j);
            *reinterpret_cast<float4*>(acc + j) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j >= rlen) continue;
            if (pow2) {  // x * 2^-j is x / 2^j rounded once
                q.x = __fmul_rn(q.x, inv_k);
                q.y = __fmul_rn(q.y, inv_k);
                q.z = __fmul_rn(q.z, inv_k);
                q.w = __fmul_rn(q.w, inv_k);
            } else {
                q.x = div_k(q.x, fk, inv_k, false);
                q.y = div_k(q.y, fk, inv_k, false);
                q.z = div_k(q.z, fk, inv_k, false);
                q.w = div_k(q.w, fk, inv_k, false);
            }
            if (al && j + 4 <= rlen) {
                *reinterpret_cast<float4*>(o + j) = q;
            } else {
                const float* qq = &q.x;
                for (uint32_t t = 0; t < 4 && j + t < rlen; ++t) o[j + t] = qq[t];
            }
        }
        consumer_sync();  // acc zeroed before the next region's adds
    }
}

}  // namespace spavg

int spavg_launch(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int K, int64_t n, float* out,
                 cudaStream_t stream, bool update, float lr) {
    using namespace spavg;
    if (n == 0) return GCSGD_OK;
    // dense lists (by capacity: K * cap >= n / 4, a quarter entry per output
    // or more) take the warp spans, sparse ones the tile kernel
    if (!update && (uint64_t)K * (uint64_t)cap >= (uint64_t)n / 4) {  // at most 34 KB of shared memory (K = 512)
        const uint64_t spans = ((uint64_t)n + kWSpan - 1) / kWSpan;
        uint64_t ctas = (uint64_t)sm_count() * 4;  // resident CTAs per SM
        const uint64_t need = (spans + NW - 1) / NW;
        if (ctas > need) ctas = need;
        const uint64_t per_warp = (spans + ctas * NW - 1) / (ctas * NW);
        ctas = (spans + per_warp * NW - 1) / (per_warp * NW);
        const size_t wsmem = sizeof(float) * NW * kWSpan + sizeof(uint32_t) * (size_t)K * (NW + 1);
        LaunchScope ls("spavg", stream);
        if (K <= kBatch)
            spavg_warp<true><<<(unsigned)ctas, NT, wsmem, stream>>>(lists, (uint64_t)cap, counts, K, (uint64_t)n, out,
                                                                    spans, per_warp);
        else
            spavg_warp<false><<<(unsigned)ctas, NT, wsmem, stream>>>(lists, (uint64_t)cap, counts, K, (uint64_t)n,
                                                                     out, spans, per_warp);
        return check_launch("spavg");
    }
    const uint64_t tiles = ((uint64_t)n + kTile - 1) / kTile;
    uint64_t grid = (uint64_t)sm_count() * 4;
    if (grid > tiles) grid = tiles;
    const uint64_t per = (tiles + grid - 1) / grid;
    grid = (tiles + per - 1) / per;
    uint32_t C = kStage / (uint32_t)K;  // window per list when the range does not fit the stage
    if (C < 32) C = 32;
    const size_t stage_items = (size_t)K * C > kStage ? (size_t)K * C : kStage;
    const size_t smem = kTile * sizeof(float) + stage_items * sizeof(gcsgd_pair) + 3 * sizeof(uint64_t) * (size_t)K +
                        sizeof(uint32_t) * (3 * (size_t)K + 1 + (size_t)K * (NW + 1));
    const char* fn = update ? "sparse_average_update" : "sparse_average";
    if (smem > 200 * 1024) return set_error(GCSGD_ERR_INVALID_ARG, "%s: K = %d too large", fn, K);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem > 48 * 1024 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(spavg_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
                cudaSuccess ||
            cudaFuncSetAttribute(spavg_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
                cudaSuccess)
            return set_error(GCSGD_ERR_CUDA, "%s: cannot raise the shared-memory limit", fn);
        attr_set[dev] = true;
    }
    LaunchScope ls(update ? "spavg_update" : "spavg", stream);
    if (update)
        spavg_kernel<true><<<(unsigned)grid, NT, smem, stream>>>(lists, (uint64_t)cap, counts, K, (uint64_t)n, out,
                                                                 tiles, per, C, lr);
    else
        spavg_kernel<false><<<(unsigned)grid, NT, smem, stream>>>(lists, (uint64_t)cap, counts, K, (uint64_t)n, out,
                                                                  tiles, per, C, 0.0f);
    return check_launch(update ? "spavg_update" : "spavg");
}

}  // namespace gcsgd

namespace gcsgd {

static size_t spavg_table_bytes(int K, int64_t n) {
    const uint64_t G = ((uint64_t)(n > 0 ? n : 0) + spavg::kRegion - 1) / spavg::kRegion;
    return ((size_t)K * (size_t)(G + 1) * sizeof(uint32_t) + 255) / 256 * 256;
}

size_t spavg_ws_bytes(int K, int64_t n) { return spavg_table_bytes(K, n) + 256; }  // the table, then the status word

// update: step the weights in `out` (w -= lr * avg at the carried indices)
// instead of writing the dense average.
int spavg_ws_launch(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int K, int64_t n, float* out,
                    void* ws, cudaStream_t stream, bool update, float lr) {
    const char* fn = update ? "sparse_average_update_ws" : "sparse_average_ws";
    using namespace spavg;
    if (n == 0) return GCSGD_OK;
    // sparse lists (K * cap < n / 4) stay on the tile kernel, and lists off
    // the 8-byte boundary (which bulk copies cannot fetch) on sparse_average's
    // kernels; the status word still reads 0
    if ((uint64_t)K * (uint64_t)cap < (uint64_t)n / 4 || ((uintptr_t)lists & 7) != 0) {
        const cudaError_t e =
            cudaMemsetAsync(static_cast<unsigned char*>(ws) + spavg_table_bytes(K, n), 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess)
            return set_error(GCSGD_ERR_CUDA, "%s: status clear failed: %s", fn, cudaGetErrorString(e));
        return spavg_launch(lists, cap, counts, K, n, out, stream, update, lr);
    }
    const uint64_t G = ((uint64_t)n + kRegion - 1) / kRegion;
    uint32_t* lo = static_cast<uint32_t*>(ws);
    uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(ws) + spavg_table_bytes(K, n));
    const int sms = sm_count();
    const uint64_t checks = ((uint64_t)cap + kCheck - 1) / kCheck;
    uint64_t bx = (checks + NT - 1) / NT;
    const uint64_t bx_max = ((uint64_t)sms * 8 + K - 1) / K;
    if (bx > bx_max) bx = bx_max;
    if (bx < 1) bx = 1;
    const size_t smem =
        kRegion * sizeof(float) + kNBuf * kRStage * sizeof(gcsgd_pair) + sizeof(uint32_t) * (4 * kNBuf + 1) * (size_t)K;
    constexpr size_t kMaxSmem =
        kRegion * sizeof(float) + kNBuf * kRStage * sizeof(gcsgd_pair) + sizeof(uint32_t) * (4 * kNBuf + 1) * 512;
    static int occ_of[64][2][2] = {};  // per device and mode: resident CTAs for K <= 64 and for larger K
    int dev = 0;
    cudaGetDevice(&dev);
    const int kc = K <= 64 ? 0 : 1, um = update ? 1 : 0;
    if (dev >= 64) return set_error(GCSGD_ERR_CUDA, "%s: device ordinal %d >= 64", fn, dev);
    if (!occ_of[dev][um][kc]) {
        int occ = 0;
        const void* kern = update ? (const void*)spavg_region<true> : (const void*)spavg_region<false>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NTR, kc ? kMaxSmem : smem) != cudaSuccess)
            return set_error(GCSGD_ERR_CUDA, "%s: cannot set up the region kernel", fn);
        occ_of[dev][um][kc] = occ > 0 ? occ : 1;
    }
    uint64_t grid = (uint64_t)sms * (uint64_t)occ_of[dev][um][kc];
    if (grid > G) grid = G;
    {
        LaunchScope ls("spavg_checkpoints", stream);
        spavg_checkpoints<<<dim3((unsigned)bx, (unsigned)K), NT, 0, stream>>>(lists, (uint64_t)cap, counts, G, lo,
                                                                             status);
        const int rc = check_launch("spavg_checkpoints");
        if (rc) return rc;
    }
    LaunchScope ls(update ? "spavg_update" : "spavg", stream);
    if (update)
        spavg_region<true><<<(unsigned)grid, NTR, smem, stream>>>(lists, (uint64_t)cap, counts, K, (uint64_t)n, out,
                                                                  lo, G, status, lr);
    else
        spavg_region<false><<<(unsigned)grid, NTR, smem, stream>>>(lists, (uint64_t)cap, counts, K, (uint64_t)n, out,
                                                                   lo, G, status, 0.0f);
    return check_launch("spavg_region");
}

int spavg_ws_status(const void* ws, int K, int64_t n, cudaStream_t stream, int32_t* status) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, static_cast<const unsigned char*>(ws) + spavg_table_bytes(K, n), sizeof(v),
                                    cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return set_error(GCSGD_ERR_CUDA, "gcsgd_sparse_average_status: %s", cudaGetErrorString(e));
    *status = (int32_t)v;
    return GCSGD_OK;
}

}  // namespace gcsgd

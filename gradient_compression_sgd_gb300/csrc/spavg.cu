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

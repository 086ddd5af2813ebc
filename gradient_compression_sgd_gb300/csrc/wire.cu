// wire.cu -- the messages as byte streams, and back.
//
// "Deep Gradient Compression", section 3.1: a sent value travels as 32 bits
// and the unsent positions before it as a 16-bit count.  Reading: one 6-byte
// record per sent entry, little-endian [uint16 unsent positions since the
// previous entry][fp32 value]; a gap of 65536 or more is split by escape
// records (65535, +0.0f), each covering 65535 zeros and one explicit zero.
//
// "AdaComp ...", Proposed method: one scale per layer (the mean |g_max|) and
// each sent entry as sign + scale.  Reading: per layer a header [uint32
// count][fp32 scale], then one uint32 per entry, (local index << 1) | sign.
//
// One CTA per learner (a message is a few hundred KB); record and layer
// offsets come from block scans, and every record is written with 16- or
// 32-bit stores at its own offset.
#include "common.cuh"

namespace gcsgd {
namespace wire {

constexpr int NT = 1024;
constexpr int IPT = 4;  // entries per thread per round
constexpr uint32_t kEscapeRun = 65535u;

// Layer offsets within a learner, passed by value (no host-to-device copy).
struct WireOffsets {
    uint32_t off[GCSGD_MAX_SEGMENTS + 1];
};

__device__ __forceinline__ void put16(uint8_t* b, uint64_t at, uint32_t x) {
    *reinterpret_cast<uint16_t*>(b + at) = (uint16_t)x;
}

// records of one DGC entry: its escapes and itself
__device__ __forceinline__ uint64_t dgc_records(uint64_t gap) { return 1 + gap / 65536; }

__global__ void __launch_bounds__(NT) dgc_encode_kernel(const gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                        const int64_t* __restrict__ totals,
                                                        uint8_t* __restrict__ streams, uint64_t stream_cap,
                                                        int64_t* __restrict__ nbytes) {
    __shared__ uint64_t scan[NT / 32 + 1];
    __shared__ uint64_t s_carry;
    __shared__ int s_bad;
    const int k = blockIdx.x;
    const gcsgd_pair* L = lists + (uint64_t)k * cap;
    uint8_t* out = streams + (uint64_t)k * stream_cap;
    int64_t c = totals[k];
    c = c < 0 ? 0 : ((uint64_t)c > cap ? (int64_t)cap : c);
    if (threadIdx.x == 0) {
        s_carry = 0;
        s_bad = 0;
    }
    __syncthreads();
    // the size first (one pass), so an over-long stream writes nothing
    for (uint64_t base = 0; base < (uint64_t)c; base += (uint64_t)NT * IPT) {
        uint64_t recs = 0;
        int bad = 0;
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const uint64_t i = base + (uint64_t)threadIdx.x * IPT + j;
            if (i < (uint64_t)c) {
                const int64_t prev = i ? (int64_t)L[i - 1].idx : -1;
                const int64_t cur = (int64_t)L[i].idx;
                if (cur <= prev) bad = 1;
                else recs += dgc_records((uint64_t)(cur - prev - 1));
            }
        }
        uint64_t tot;
        block_exclusive_scan<NT>(recs, scan, &tot);
        if (bad) s_bad = 1;
        if (threadIdx.x == 0) s_carry += tot;
        __syncthreads();
    }
    const uint64_t bytes = 6 * s_carry;
    if (s_bad || bytes > stream_cap) {
        if (threadIdx.x == 0) nbytes[k] = -1;
        return;
    }
    __syncthreads();
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (uint64_t base = 0; base < (uint64_t)c; base += (uint64_t)NT * IPT) {
        uint64_t gap[IPT], recs = 0;
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const uint64_t i = base + (uint64_t)threadIdx.x * IPT + j;
            gap[j] = 0;
            if (i < (uint64_t)c) {
                const int64_t prev = i ? (int64_t)L[i - 1].idx : -1;
                gap[j] = (uint64_t)((int64_t)L[i].idx - prev - 1);
                recs += dgc_records(gap[j]);
            }
        }
        uint64_t tot;
        uint64_t r = s_carry + block_exclusive_scan<NT>(recs, scan, &tot);
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const uint64_t i = base + (uint64_t)threadIdx.x * IPT + j;
            if (i >= (uint64_t)c) break;
            uint64_t g = gap[j];
            for (; g >= 65536; g -= 65536, ++r) {
                put16(out, 6 * r, kEscapeRun);
                put16(out, 6 * r + 2, 0u);
                put16(out, 6 * r + 4, 0u);
            }
            const uint32_t vb = __float_as_uint(L[i].val);
            put16(out, 6 * r, (uint32_t)g);
            put16(out, 6 * r + 2, vb & 0xffffu);
            put16(out, 6 * r + 4, vb >> 16);
            ++r;
        }
        __syncthreads();
        if (threadIdx.x == 0) s_carry += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) nbytes[k] = (int64_t)bytes;
}

__global__ void __launch_bounds__(NT) dgc_decode_kernel(const uint8_t* __restrict__ streams, uint64_t stream_cap,
                                                        const int64_t* __restrict__ nbytes,
                                                        gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                        int64_t* __restrict__ totals) {
    __shared__ uint64_t scan[NT / 32 + 1];
    __shared__ uint64_t s_pos, s_cnt;
    const int k = blockIdx.x;
    const uint8_t* in = streams + (uint64_t)k * stream_cap;
    gcsgd_pair* L = lists + (uint64_t)k * cap;
    int64_t nb = nbytes[k];
    nb = nb < 0 ? 0 : ((uint64_t)nb > stream_cap ? (int64_t)stream_cap : nb);
    const uint64_t R = (uint64_t)nb / 6;
    if (threadIdx.x == 0) {
        s_pos = 0;  // position after the last record
        s_cnt = 0;
    }
    __syncthreads();
    for (uint64_t base = 0; base < R; base += (uint64_t)NT * IPT) {
        uint32_t run[IPT], vb[IPT];
        uint64_t adv = 0, keep = 0;
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const uint64_t r = base + (uint64_t)threadIdx.x * IPT + j;
            run[j] = 0;
            vb[j] = 0;
            if (r < R) {
                const uint16_t* p = reinterpret_cast<const uint16_t*>(in + 6 * r);
                run[j] = p[0];
                vb[j] = (uint32_t)p[1] | ((uint32_t)p[2] << 16);
                adv += run[j] + 1;
                keep += !(run[j] == kEscapeRun && vb[j] == 0u);
            }
        }
        uint64_t tot;
        const uint64_t ex = block_exclusive_scan<NT>(adv | (keep << 40), scan, &tot);
        uint64_t pos = s_pos + (ex & ((1ull << 40) - 1)), slot = s_cnt + (ex >> 40);
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const uint64_t r = base + (uint64_t)threadIdx.x * IPT + j;
            if (r >= R) break;
            pos += run[j];
            if (!(run[j] == kEscapeRun && vb[j] == 0u)) {
                if (slot < cap) {
                    gcsgd_pair pr;
                    pr.idx = (uint32_t)pos;
                    pr.val = __uint_as_float(vb[j]);
                    L[slot] = pr;
                }
                ++slot;
            }
            ++pos;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            s_pos += tot & ((1ull << 40) - 1);
            s_cnt += tot >> 40;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) totals[k] = s_cnt <= cap ? (int64_t)s_cnt : -1;
}

// AdaComp: layer s of learner k holds counts[k][s] entries of the list,
// the layers one after another.  Grid (chunks, K): every CTA computes the
// layer offsets (entries and bytes before each layer, a block scan), then
// writes the words of its share of the entries, each finding its layer by
// binary search; chunk 0 writes the headers and the length.
constexpr int kAdaChunks = 64;
__global__ void __launch_bounds__(NT) ada_encode_kernel(const WireOffsets so, int S,
                                                        const gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                        const int64_t* __restrict__ counts,
                                                        const float* __restrict__ scales,
                                                        uint8_t* __restrict__ streams, uint64_t stream_cap,
                                                        int64_t* __restrict__ nbytes) {
    __shared__ uint64_t scan[NT / 32 + 1];
    __shared__ uint64_t s_ent, s_bytes;
    __shared__ uint32_t ent_at[GCSGD_MAX_SEGMENTS + 1];  // entries before layer s (list positions < 2^32)
    const int k = blockIdx.y;
    const gcsgd_pair* L = lists + (uint64_t)k * cap;
    uint8_t* out = streams + (uint64_t)k * stream_cap;
    if (threadIdx.x == 0) {
        s_ent = 0;
        s_bytes = 0;
    }
    __syncthreads();
    for (int base = 0; base < S; base += NT) {
        const int s = base + (int)threadIdx.x;
        const uint64_t c = s < S ? (uint64_t)counts[(int64_t)k * S + s] : 0;
        uint64_t tot_b, tot_e;
        block_exclusive_scan<NT>(s < S ? 8 + 4 * c : 0, scan, &tot_b);
        const uint64_t ee = block_exclusive_scan<NT>(c, scan, &tot_e);
        if (s < S) ent_at[s] = (uint32_t)(s_ent + ee);
        __syncthreads();
        if (threadIdx.x == 0) {
            s_bytes += tot_b;
            s_ent += tot_e;
        }
        __syncthreads();
    }
    const uint64_t total_bytes = s_bytes, total_ent = s_ent;
    // every CTA sees the same totals: an over-long stream (or counts beyond
    // the list, as after a capacity overflow) writes nothing
    if (total_bytes > stream_cap || total_ent > cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) nbytes[k] = -1;
        return;
    }
    if (threadIdx.x == 0) ent_at[S] = (uint32_t)total_ent;
    __syncthreads();
    // layer s starts at byte 8 s + 4 ent_at[s]
    if (blockIdx.x == 0)
        for (int s = threadIdx.x; s < S; s += NT) {
            uint8_t* o = out + 8ull * s + 4ull * ent_at[s];
            *reinterpret_cast<uint32_t*>(o) = ent_at[s + 1] - ent_at[s];
            *reinterpret_cast<uint32_t*>(o + 4) = __float_as_uint(scales[(int64_t)k * S + s]);
        }
    const uint64_t per = (total_ent + gridDim.x - 1) / gridDim.x;
    const uint64_t j0 = (uint64_t)blockIdx.x * per, j1 = j0 + per < total_ent ? j0 + per : total_ent;
    for (uint64_t j = j0 + threadIdx.x; j < j1; j += NT) {
        int lo = 0, hi = S;  // last layer with ent_at <= j
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (ent_at[mid] <= j) lo = mid; else hi = mid;
        }
        const gcsgd_pair pr = L[j];
        const uint32_t local = pr.idx - so.off[lo];
        *reinterpret_cast<uint32_t*>(out + 8ull * (lo + 1) + 4ull * j) = (local << 1) | (pr.val < 0.0f ? 1u : 0u);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) nbytes[k] = (int64_t)total_bytes;
}

__global__ void __launch_bounds__(NT) ada_decode_kernel(const WireOffsets so, int S,
                                                        const uint8_t* __restrict__ streams, uint64_t stream_cap,
                                                        const int64_t* __restrict__ nbytes,
                                                        gcsgd_pair* __restrict__ lists, uint64_t cap,
                                                        int64_t* __restrict__ totals) {
    __shared__ uint64_t s_at, s_ent;
    __shared__ int s_bad;
    const int k = blockIdx.x;
    const uint8_t* in = streams + (uint64_t)k * stream_cap;
    gcsgd_pair* L = lists + (uint64_t)k * cap;
    int64_t nb = nbytes[k];
    nb = nb < 0 ? 0 : ((uint64_t)nb > stream_cap ? (int64_t)stream_cap : nb);
    if (threadIdx.x == 0) {
        s_at = 0;
        s_ent = 0;
        s_bad = 0;
    }
    __syncthreads();
    // headers are sequential (each layer's size is in its header): warp 0
    // walks them, then the warps decode the layer's words in parallel
    for (int s = 0; s < S; ++s) {
        const uint64_t at = s_at;
        if (at + 8 > (uint64_t)nb) {
            if (threadIdx.x == 0) s_bad = 1;
            break;
        }
        const uint32_t c = *reinterpret_cast<const uint32_t*>(in + at);
        const float scale = __uint_as_float(*reinterpret_cast<const uint32_t*>(in + at + 4));
        if (at + 8 + 4ull * c > (uint64_t)nb || s_ent + c > cap) {
            if (threadIdx.x == 0) s_bad = 1;
            break;
        }
        const uint32_t* words = reinterpret_cast<const uint32_t*>(in + at + 8);
        const uint32_t n_s = so.off[s + 1] - so.off[s];
        for (uint32_t i = threadIdx.x; i < c; i += NT) {
            const uint32_t w = words[i];
            gcsgd_pair pr;
            pr.idx = so.off[s] + ((w >> 1) < n_s ? (w >> 1) : n_s - 1);
            pr.val = (w & 1u) ? -scale : scale;
            L[s_ent + i] = pr;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            s_at = at + 8 + 4ull * c;
            s_ent += c;
        }
        __syncthreads();
    }
    __syncthreads();
    if (threadIdx.x == 0) totals[k] = s_bad ? -1 : (int64_t)s_ent;
}

}  // namespace wire

int wire_dgc_encode(const gcsgd_pair* lists, int64_t cap, const int64_t* totals, int K, uint8_t* streams,
                    int64_t stream_cap, int64_t* nbytes, cudaStream_t stream) {
    LaunchScope ls("dgc_encode", stream);
    wire::dgc_encode_kernel<<<K, wire::NT, 0, stream>>>(lists, (uint64_t)cap, totals, streams, (uint64_t)stream_cap,
                                                        nbytes);
    return check_launch("dgc_encode");
}

int wire_dgc_decode(const uint8_t* streams, int64_t stream_cap, const int64_t* nbytes, int K, gcsgd_pair* lists,
                    int64_t cap, int64_t* totals, cudaStream_t stream) {
    LaunchScope ls("dgc_decode", stream);
    wire::dgc_decode_kernel<<<K, wire::NT, 0, stream>>>(streams, (uint64_t)stream_cap, nbytes, lists, (uint64_t)cap,
                                                        totals);
    return check_launch("dgc_decode");
}

int wire_ada_encode(const int64_t* off, int S, const gcsgd_pair* lists, int64_t cap, const int64_t* counts,
                    const float* scales, int K, uint8_t* streams, int64_t stream_cap, int64_t* nbytes,
                    cudaStream_t stream) {
    wire::WireOffsets so;
    for (int s = 0; s <= S; ++s) so.off[s] = (uint32_t)off[s];
    LaunchScope ls("adacomp_encode", stream);
    wire::ada_encode_kernel<<<dim3(wire::kAdaChunks, K), wire::NT, 0, stream>>>(so, S, lists, (uint64_t)cap, counts,
                                                                              scales, streams, (uint64_t)stream_cap,
                                                                              nbytes);
    return check_launch("adacomp_encode");
}

int wire_ada_decode(const int64_t* off, int S, const uint8_t* streams, int64_t stream_cap, const int64_t* nbytes,
                    int K, gcsgd_pair* lists, int64_t cap, int64_t* totals, cudaStream_t stream) {
    wire::WireOffsets so;
    for (int s = 0; s <= S; ++s) so.off[s] = (uint32_t)off[s];
    LaunchScope ls("adacomp_decode", stream);
    wire::ada_decode_kernel<<<K, wire::NT, 0, stream>>>(so, S, streams, (uint64_t)stream_cap, nbytes, lists,
                                                        (uint64_t)cap, totals);
    return check_launch("adacomp_decode");
}

}  // namespace gcsgd

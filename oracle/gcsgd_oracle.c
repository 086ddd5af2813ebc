/*
 * gcsgd_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of the per-worker
 * gradient-compression step, written to check the CUDA library against.
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it; the product path never calls it and shares no code with it.
 *
 * Precision.  The DGC page fixes 32-bit gradient values on the wire
 * ("Deep Gradient Compression", section 3.1, its description of the
 * message encoding), and the workloads are fp32 tensors, so every
 * element-wise update here is fp32 with one IEEE round-to-nearest per
 * operation and no fused multiply-add (compile with -ffp-contract=off).
 * Reductions that feed a single scalar (the clipping norm, the AdaComp scale)
 * are taken in fp64 with compensated summation, so they sit within an ulp of
 * the exact sum whatever order a faster implementation adds them in.
 *
 * Every function cites the passage it follows.  Where a page only describes
 * a step in words, the plainest reading is taken and named at that step.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ECAP (-2)
#define ORACLE_ENOMEM (-3)

/* ---------------------------------------------------------------- helpers */

static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* Magnitude key: the bit pattern of |x|.  For finite floats, unsigned order of
 * these keys is the order of |x|, and +0 and -0 share key 0. */
static uint32_t mag_key(float f) { return bits_of(f) & 0x7fffffffu; }

/* Neumaier's compensated summation in fp64. */
typedef struct { double s, c; } csum_t;
static void csum_add(csum_t* a, double x) {
    double t = a->s + x;
    if (fabs(a->s) >= fabs(x)) a->c += (a->s - t) + x;
    else a->c += (x - t) + a->s;
    a->s = t;
}
static double csum_value(const csum_t* a) { return a->s + a->c; }

/* Number of entries DGC sends from a tensor of n values at the given density
 * ("Deep Gradient Compression", section 3.1: only the largest-magnitude
 * fraction is sent).  Reading: k = ceil(density * n) in fp64, at least one
 * entry for a non-empty tensor and at most n. */
int64_t oracle_dgc_k(double density, int64_t n) {
    if (n <= 0) return 0;
    double kd = ceil(density * (double)n);
    int64_t k = (int64_t)kd;
    if (k < 1) k = 1;
    if (k > n) k = n;
    return k;
}

/* ------------------------------------------------------------ DGC (step) */

typedef struct { uint32_t key; uint32_t idx; } keyed_t;

/* Larger magnitude first; equal magnitudes: lower index first. */
static int keyed_cmp(const void* a, const void* b) {
    const keyed_t* x = (const keyed_t*)a;
    const keyed_t* y = (const keyed_t*)b;
    if (x->key != y->key) return x->key > y->key ? -1 : 1;
    if (x->idx != y->idx) return x->idx < y->idx ? -1 : 1;
    return 0;
}

/*
 * One DGC step of K learners that share a layout of S tensors
 * ("Deep Gradient Compression", Appendix D, the algorithm with vanilla
 * momentum, on node k):
 *
 *  1. local gradient clipping (Appendix C; section 3.2): when clip_thr > 0
 *     and the L2 norm s of the learner's gradient exceeds
 *     thr_k = clip_thr / sqrt(clip_nodes), the gradient is rescaled by
 *     c = thr_k / s before it is added to the accumulation.  Reading: the norm
 *     is over the learner's whole gradient in this call; c is rounded to fp32
 *     once and applied as one fp32 multiply.
 *  2. momentum correction (section 3.2): u <- m*u + G, then v <- v + u, i.e.
 *     the momentum-adjusted gradient is accumulated locally before
 *     sparsification.  The page states this in words only; this is the reading.
 *  3. sparsification with local accumulation (section 3.1): per tensor, the
 *     k_s entries of largest |v| are sent; ties are broken by the lower index
 *     (a sort key, so the result is unique).
 *  4. momentum factor masking (section 3.3): at every sent coordinate both v
 *     (its mass has left the accumulator) and u are set to zero.
 *
 * grad, u, v : [K][N] fp32, N = seg_off[S].  u, v are updated in place.
 * out_idx/out_val : [K][cap]; learner k's list starts at k*cap and holds its
 *     tensors' selections one after another, each in ascending index order;
 *     indices are global within the learner (seg_off[s] + local index).
 * counts : [K][S] entries sent per tensor.  clip_scale : [K] the c applied
 *     (1 when not clipped), may be NULL.
 */
/*
 * The sampled threshold ("Deep Gradient Compression", section 5, system
 * analysis: a sample of 0.1 % to 1 % of the gradients is enough to estimate
 * the threshold of the whole population; section 6: hierarchical threshold
 * selection).  The pages give the idea, not the procedure.  Reading, per
 * tensor of n values with k_s to send and the caller's sample fraction f:
 *   - the sample is m = floor(f * n) values rounded down to whole blocks of
 *     64 consecutive values (how the sample is drawn is not on the page:
 *     evenly spaced blocks keep it deterministic), block b starting at
 *     b * floor(n / (m / 64));
 *   - a tensor whose sample holds no whole block (f * n < 64) has nothing to
 *     estimate from and is selected exactly (the second, exact step alone);
 *   - the threshold tau is the a-th largest sampled |v| (bit pattern order),
 *     a = round(k_s * m / n) clamped to [1, m]: the sample's share of k_s;
 *   - every entry with |v| >= tau is selected; when that is more than k_s
 *     (the hierarchical second step) the k_s largest of them are kept, which
 *     is the exact top-k, otherwise all of them are sent (fewer than k_s).
 * Nothing else limits the sample: every tensor size and every density is
 * sampled the same way.  Learner k's list holds its tensors' selections one
 * after another, so its length is the sum of the per-tensor counts.
 */
#define ORACLE_SAMPLE_BLOCK 64

/* Values sampled from a tensor of n values at fraction f (0: not sampled). */
static int64_t dgc_sample_size(int64_t n, double sample_frac) {
    if (!(sample_frac > 0.0)) return 0;
    int64_t m = (int64_t)(sample_frac * (double)n);
    return m - m % ORACLE_SAMPLE_BLOCK;
}

static int dgc_step_impl(int K, int S, const int64_t* seg_off,
                         const float* grad, float* u, float* v,
                         double density, double sample_frac, float momentum, int nesterov, float clip_thr,
                         int clip_nodes, uint32_t* out_idx, float* out_val, int64_t cap,
                         int64_t* counts, float* clip_scale) {
    if (K < 1 || S < 1 || !(density > 0.0 && density <= 1.0) || clip_nodes < 1) return ORACLE_EINVAL;
    if (!(sample_frac >= 0.0 && sample_frac <= 1.0)) return ORACLE_EINVAL;
    const int64_t N = seg_off[S];
    int64_t total = 0;
    for (int s = 0; s < S; ++s) total += oracle_dgc_k(density, seg_off[s + 1] - seg_off[s]);
    if (total > cap) return ORACLE_ECAP;

    int64_t max_len = 0;
    for (int s = 0; s < S; ++s)
        if (seg_off[s + 1] - seg_off[s] > max_len) max_len = seg_off[s + 1] - seg_off[s];
    keyed_t* order = (keyed_t*)malloc(sizeof(keyed_t) * (size_t)(max_len > 0 ? max_len : 1));
    unsigned char* sent = (unsigned char*)malloc((size_t)(max_len > 0 ? max_len : 1));
    if (!order || !sent) { free(order); free(sent); return ORACLE_ENOMEM; }

    for (int k = 0; k < K; ++k) {
        const float* G = grad + (int64_t)k * N;
        float* uk = u + (int64_t)k * N;
        float* vk = v + (int64_t)k * N;

        /* 1. local gradient clipping */
        int clipped = 0;
        float c = 1.0f;
        if (clip_thr > 0.0f) {
            csum_t acc = {0.0, 0.0};
            for (int64_t i = 0; i < N; ++i) csum_add(&acc, (double)G[i] * (double)G[i]);
            double norm = sqrt(csum_value(&acc));
            double thr_k = (double)clip_thr / sqrt((double)clip_nodes);
            if (norm > thr_k) { c = (float)(thr_k / norm); clipped = 1; }
        }
        if (clip_scale) clip_scale[k] = c;

        /* 2. momentum correction: accumulate the momentum-adjusted gradient
         * (Nesterov: the accumulated state takes the look-ahead step m*u + g) */
        for (int64_t i = 0; i < N; ++i) {
            float g = clipped ? G[i] * c : G[i];
            float mu = momentum * uk[i];
            uk[i] = mu + g;
            if (nesterov) {
                float step = momentum * uk[i];
                step = step + g;
                vk[i] = vk[i] + step;
            } else {
                vk[i] = vk[i] + uk[i];
            }
        }

        /* 3 + 4. per-tensor top-k of |v|, send, then mask u and v */
        int64_t pos = (int64_t)k * cap;
        for (int s = 0; s < S; ++s) {
            const int64_t off = seg_off[s];
            const int64_t n = seg_off[s + 1] - off;
            const int64_t ks = oracle_dgc_k(density, n);
            for (int64_t i = 0; i < n; ++i) {
                order[i].key = mag_key(vk[off + i]);
                order[i].idx = (uint32_t)i;
                sent[i] = 0;
            }
            int64_t take = ks;
            const int64_t m = dgc_sample_size(n, sample_frac);
            if (m > 0) {
                /* the sample and its a-th largest |v| */
                const int64_t nblk = m / ORACLE_SAMPLE_BLOCK, stride = n / nblk;
                keyed_t* smp = (keyed_t*)malloc(sizeof(keyed_t) * (size_t)m);
                if (!smp) { free(order); free(sent); return ORACLE_ENOMEM; }
                for (int64_t b = 0; b < nblk; ++b)
                    for (int64_t j = 0; j < ORACLE_SAMPLE_BLOCK; ++j) {
                        smp[b * ORACLE_SAMPLE_BLOCK + j].key = mag_key(vk[off + b * stride + j]);
                        smp[b * ORACLE_SAMPLE_BLOCK + j].idx = 0;
                    }
                qsort(smp, (size_t)m, sizeof(keyed_t), keyed_cmp);
                int64_t a = (ks * m + n / 2) / n;
                if (a < 1) a = 1;
                if (a > m) a = m;
                const uint32_t tau = smp[a - 1].key;
                free(smp);
                int64_t c = 0;
                for (int64_t i = 0; i < n; ++i) c += order[i].key >= tau;
                if (c < ks) take = c;  /* all of |v| >= tau; else the k_s largest of them */
            }
            if (n > 1) qsort(order, (size_t)n, sizeof(keyed_t), keyed_cmp);
            for (int64_t j = 0; j < take; ++j) sent[order[j].idx] = 1;
            for (int64_t i = 0; i < n; ++i) {
                if (!sent[i]) continue;
                out_idx[pos] = (uint32_t)(off + i);
                out_val[pos] = vk[off + i];
                ++pos;
                vk[off + i] = 0.0f;
                uk[off + i] = 0.0f;
            }
            counts[(int64_t)k * S + s] = take;
        }
    }
    free(order);
    free(sent);
    return ORACLE_OK;
}

int oracle_dgc_step(int K, int S, const int64_t* seg_off,
                    const float* grad, float* u, float* v,
                    double density, float momentum, float clip_thr, int clip_nodes,
                    uint32_t* out_idx, float* out_val, int64_t cap,
                    int64_t* counts, float* clip_scale) {
    return dgc_step_impl(K, S, seg_off, grad, u, v, density, 0.0, momentum, 0, clip_thr, clip_nodes, out_idx,
                         out_val, cap, counts, clip_scale);
}

/*
 * The DGC step with Nesterov momentum ("Deep Gradient Compression",
 * Appendix B, gradient sparsification with Nesterov momentum correction).
 * The page states the shape of the update, not its equations: after the
 * correction the update keeps the local momentum and an accumulated state,
 * and conventional Nesterov momentum steps by the look-ahead m*u + g.
 * Reading (parity unpinned by the page): per element, in fp32 with one
 * rounding per operation,
 *   u <- m*u + g        (local momentum, as in the vanilla step)
 *   v <- v + (m*u + g)  (the accumulated state takes the Nesterov step,
 *                        with the u just updated)
 * then the same clipping, per-tensor top-k of |v|, sending and masking of u
 * and v as oracle_dgc_step.  With m = 0 it is the vanilla step.
 */
int oracle_dgc_step_nesterov(int K, int S, const int64_t* seg_off,
                             const float* grad, float* u, float* v,
                             double density, float momentum, float clip_thr, int clip_nodes,
                             uint32_t* out_idx, float* out_val, int64_t cap,
                             int64_t* counts, float* clip_scale) {
    return dgc_step_impl(K, S, seg_off, grad, u, v, density, 0.0, momentum, 1, clip_thr, clip_nodes, out_idx,
                         out_val, cap, counts, clip_scale);
}

/* The DGC step with the sampled threshold (see dgc_sample_size above). */
int oracle_dgc_step_sampled(int K, int S, const int64_t* seg_off,
                            const float* grad, float* u, float* v,
                            double density, double sample_frac, float momentum, float clip_thr, int clip_nodes,
                            uint32_t* out_idx, float* out_val, int64_t cap,
                            int64_t* counts, float* clip_scale) {
    if (!(sample_frac > 0.0)) return ORACLE_EINVAL;
    return dgc_step_impl(K, S, seg_off, grad, u, v, density, sample_frac, momentum, 0, clip_thr, clip_nodes,
                         out_idx, out_val, cap, counts, clip_scale);
}

/* --------------------------------------------------------- AdaComp (step) */

/*
 * One AdaComp step of K learners ("AdaComp : Adaptive Residual Gradient
 * Compression for Data-Parallel Distributed Training", Proposed method):
 *
 *  1. the residue is added to the new gradient: G = R + dW, per layer;
 *  2. the layer vector is cut into bins of L_T values (lt[s] for tensor s)
 *     and each bin's maximum |G| is found.  Reading: a last partial bin is a
 *     bin of its own;
 *  3. in each bin, entries are selected where |H| >= the bin maximum, with
 *     H = G + dW -- the residue plus a doubled ("about 2x") copy of the new
 *     gradient.  Reading: >= so the maximum itself may qualify; a bin whose
 *     maximum is zero selects nothing;
 *  4. one scale per layer, the mean of the bin maxima over every bin of the
 *     layer (fp64 sum, divided by the bin count, rounded to fp32 once);
 *  5. a selected entry is sent as sign(G)*scale (the sign of the value being
 *     transmitted; an entry with G == 0 has sign 0 and is not sent); the
 *     residue keeps what was not sent: R = G - sign(G)*scale for a sent
 *     entry, R = G otherwise.
 *
 * dW, R : [K][N] fp32 (R updated in place); lt : [S] bin lengths >= 1.
 * out_idx/out_val : [K][cap], learner k's tensors one after another, each in
 * ascending index order.  counts : [K][S].  scales : [K][S].
 * totals : [K] entries of each learner, reported even when they exceed cap;
 * such a learner sends nothing (its residue becomes G) and the call returns
 * ORACLE_ECAP.
 */
int oracle_adacomp_step(int K, int S, const int64_t* seg_off, const int32_t* lt,
                        const float* dW, float* R,
                        uint32_t* out_idx, float* out_val, int64_t cap,
                        int64_t* counts, float* scales, int64_t* totals) {
    if (K < 1 || S < 1) return ORACLE_EINVAL;
    for (int s = 0; s < S; ++s) if (lt[s] < 1) return ORACLE_EINVAL;
    const int64_t N = seg_off[S];
    float* G = (float*)malloc(sizeof(float) * (size_t)(N > 0 ? N : 1));
    float* Q = (float*)malloc(sizeof(float) * (size_t)(N > 0 ? N : 1));
    unsigned char* sel = (unsigned char*)malloc((size_t)(N > 0 ? N : 1));
    float* bmax = (float*)malloc(sizeof(float) * (size_t)(N > 0 ? N : 1));
    if (!G || !Q || !sel || !bmax) { free(G); free(Q); free(sel); free(bmax); return ORACLE_ENOMEM; }
    int rc = ORACLE_OK;

    for (int k = 0; k < K; ++k) {
        const float* dWk = dW + (int64_t)k * N;
        float* Rk = R + (int64_t)k * N;
        int64_t total = 0;
        for (int s = 0; s < S; ++s) {
            const int64_t off = seg_off[s];
            const int64_t n = seg_off[s + 1] - off;
            const int64_t L = lt[s];
            const int64_t nb = (n + L - 1) / L;
            int64_t sent = 0;
            if (n == 0) {
                counts[(int64_t)k * S + s] = 0;
                scales[(int64_t)k * S + s] = 0.0f;
                continue;
            }
            /* 1. G = R + dW */
            for (int64_t i = 0; i < n; ++i) G[off + i] = Rk[off + i] + dWk[off + i];
            /* 2. per-bin maximum of |G|;  4. mean of the maxima */
            csum_t acc = {0.0, 0.0};
            for (int64_t b = 0; b < nb; ++b) {
                int64_t lo = b * L, hi = lo + L < n ? lo + L : n;
                float m = 0.0f;
                for (int64_t i = lo; i < hi; ++i) {
                    float a = fabsf(G[off + i]);
                    if (a > m) m = a;
                }
                bmax[b] = m;
                csum_add(&acc, (double)m);
            }
            const float scale = (float)(csum_value(&acc) / (double)nb);
            /* 3. select |G + dW| >= bin max;  5. the value sent */
            for (int64_t i = 0; i < n; ++i) {
                const float m = bmax[i / L];
                const float h = G[off + i] + dWk[off + i];
                sel[off + i] = (fabsf(h) >= m) && (m > 0.0f) && (G[off + i] != 0.0f);
                Q[off + i] = G[off + i] > 0.0f ? scale : -scale;
                sent += sel[off + i];
            }
            counts[(int64_t)k * S + s] = sent;
            scales[(int64_t)k * S + s] = scale;
            total += sent;
        }
        totals[k] = total;
        /* Reading (capacity is not on the page): a learner whose message does
         * not fit in cap entries sends nothing this step; its residue keeps
         * all of G, so no gradient mass is lost. */
        const int fits = total <= cap;
        if (!fits) rc = ORACLE_ECAP;
        int64_t pos = 0;
        for (int64_t i = 0; i < N; ++i) {
            if (fits && sel[i]) {
                out_idx[(int64_t)k * cap + pos] = (uint32_t)i;
                out_val[(int64_t)k * cap + pos] = Q[i];
                ++pos;
                Rk[i] = G[i] - Q[i];
            } else {
                Rk[i] = G[i];
            }
        }
    }
    free(G);
    free(Q);
    free(sel);
    free(bmax);
    return rc;
}

/* --------------------------------------------------------- sparse average */

/*
 * Decompress and average K learners' sparse messages
 * ("AdaComp ...", Proposed method: learners exchange compressed gradients and
 * average them before the weight update; "Deep Gradient Compression",
 * Appendix A: the nodes' gradients are summed).
 *
 * out[j] = (sum over lists k = 0..K-1 that hold j, in that order, of their
 * value) / K, with fp32 adds starting from +0 and one fp32 divide; 0 where no
 * list holds j.  lists: idx/val [K][cap], counts [K].  Every index must be < n.
 */
int oracle_sparse_average(int K, const uint32_t* idx, const float* val, int64_t cap,
                          const int64_t* counts, int64_t n, float* out) {
    if (K < 1 || n < 0) return ORACLE_EINVAL;
    for (int64_t j = 0; j < n; ++j) out[j] = 0.0f;
    for (int k = 0; k < K; ++k) {
        if (counts[k] < 0 || counts[k] > cap) return ORACLE_EINVAL;
        for (int64_t p = 0; p < counts[k]; ++p) {
            uint32_t j = idx[(int64_t)k * cap + p];
            if ((int64_t)j >= n) return ORACLE_EINVAL;
            out[j] = out[j] + val[(int64_t)k * cap + p];
        }
    }
    const float fk = (float)K;
    for (int64_t j = 0; j < n; ++j) out[j] = out[j] / fk;
    return ORACLE_OK;
}

/*
 * Averaged sparse update of the weights: the learners' messages are averaged
 * as above and the weights step against the average, w[j] <- w[j] - lr * avg[j]
 * ("AdaComp ...", Proposed method: learners exchange compressed gradients and
 * average them to update the weights; "Deep Gradient Compression", Appendix A:
 * the summed gradients optimise the model).  Reading: only the indices that
 * some message carries are updated (every other weight keeps its exact bits);
 * lr * avg and the subtraction are one fp32 rounding each.
 */
int oracle_sparse_average_update(int K, const uint32_t* idx, const float* val, int64_t cap,
                                 const int64_t* counts, int64_t n, float lr, float* w) {
    if (K < 1 || n < 0) return ORACLE_EINVAL;
    float* avg = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    unsigned char* carried = (unsigned char*)calloc((size_t)(n > 0 ? n : 1), 1);
    if (!avg || !carried) {
        free(avg);
        free(carried);
        return ORACLE_ENOMEM;
    }
    int rc = oracle_sparse_average(K, idx, val, cap, counts, n, avg);
    if (rc == ORACLE_OK) {
        for (int k = 0; k < K; ++k)
            for (int64_t p = 0; p < counts[k]; ++p) carried[idx[(int64_t)k * cap + p]] = 1;
        for (int64_t j = 0; j < n; ++j)
            if (carried[j]) {
                const float step = lr * avg[j];
                w[j] = w[j] - step;
            }
    }
    free(avg);
    free(carried);
    return rc;
}

/* ------------------------------------------------------- Philox4x32-10 */

/*
 * Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11): each round multiplies words 0 and 2
 * by the two round constants, swaps the high halves across with the odd
 * words and the key, and the key is bumped by the two Weyl constants
 * between rounds.
 */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Random word of element e of node i at iteration t: counter (e/4, i, t, 0),
 * key (low, high halves of seed), word e mod 4 of the block. */
static uint32_t dcd_word(uint64_t seed, uint32_t node, uint32_t t, uint64_t e) {
    uint32_t ctr[4] = {(uint32_t)(e >> 2), node, t, (uint32_t)(e >> 34)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    oracle_philox4x32_10(ctr, key, o);
    return o[e & 3];
}

/* Keep threshold of the random sparsification: keep when word < thr,
 * thr = round(p * 2^32) (all kept for p >= 1).  Returned as uint64 so that
 * "keep everything" is representable. */
uint64_t oracle_keep_threshold(double p) {
    if (p >= 1.0) return (uint64_t)1 << 32;
    if (p <= 0.0) return 0;
    return (uint64_t)llround(p * 4294967296.0);
}

/* C(z) = z * (1/p) where kept, 0 elsewhere (random sparsification, unbiased). */
static float dcd_compress(float z, uint32_t word, uint64_t thr, float inv_p) {
    return ((uint64_t)word < thr) ? z * inv_p : 0.0f;
}

/*
 * One DCD-PSGD iteration of n nodes on a ring ("Communication Compression for
 * Decentralized Training", DCD-PSGD, steps 1-3), with the replicas held once:
 *
 *  step 1: x_half_i = sum_j W_ij xhat_j - gamma * g_i, with W on the ring:
 *          w[0] on node i-1, w[1] on node i, w[2] on node i+1 (indices mod n),
 *          added in that order;
 *  step 2: z_i = x_half_i - x_i;  x_i <- x_i + C(z_i);
 *  step 3: every neighbour's replica of x_i receives the same C(z_i).
 *
 * Reading: every holder of a replica of node i applies the same C(z_i) to it,
 * so, starting equal, all replicas of x_i stay bit-identical to x_i; one array
 * xhat [n][d] then stands for every model and every replica
 * (oracle_dcd_step_replicas below checks this).  All nodes read the models of
 * iteration t.  C is random sparsification ("... any other operators", the
 * paragraph that defines alpha): keep an entry with probability p, scaled by
 * 1/p; the keep draw is Philox4x32-10 word (seed, node, t, e).
 *
 * oracle_dcd_step_window computes the columns [e_base, e_base + d) of a
 * longer model (the same arithmetic; e_base only enters the counter), so a
 * sampled window of a full-size run can be checked; xhat and g are then the
 * [n][d] window.
 */
int oracle_dcd_step_window(int n, int64_t d, int64_t e_base, const float w[3], float* xhat, const float* g,
                           float gamma, double p, uint64_t seed, uint32_t t) {
    if (n < 1 || d < 0 || e_base < 0 || !(p > 0.0 && p <= 1.0)) return ORACLE_EINVAL;
    float* xn = (float*)malloc(sizeof(float) * (size_t)(n * d > 0 ? n * d : 1));
    if (!xn) return ORACLE_ENOMEM;
    const uint64_t thr = oracle_keep_threshold(p);
    const float inv_p = (float)(1.0 / p);
    for (int i = 0; i < n; ++i) {
        const int l = (i + n - 1) % n, r = (i + 1) % n;
        const float* xl = xhat + (int64_t)l * d;
        const float* xi = xhat + (int64_t)i * d;
        const float* xr = xhat + (int64_t)r * d;
        const float* gi = g + (int64_t)i * d;
        for (int64_t e = 0; e < d; ++e) {
            float acc = w[0] * xl[e];
            acc = acc + w[1] * xi[e];
            acc = acc + w[2] * xr[e];
            const float xh = acc - gamma * gi[e];
            const float z = xh - xi[e];
            const uint32_t word = dcd_word(seed, (uint32_t)i, t, (uint64_t)(e_base + e));
            const float cz = dcd_compress(z, word, thr, inv_p);
            xn[(int64_t)i * d + e] = xi[e] + cz;
        }
    }
    memcpy(xhat, xn, sizeof(float) * (size_t)(n * d));
    free(xn);
    return ORACLE_OK;
}

int oracle_dcd_step(int n, int64_t d, const float w[3], float* xhat, const float* g,
                    float gamma, double p, uint64_t seed, uint32_t t) {
    return oracle_dcd_step_window(n, d, 0, w, xhat, g, gamma, p, seed, t);
}

/*
 * The same iteration for the nodes one rank of several holds, with copies of
 * its two ring neighbours beside them (DCD-PSGD step 3 across processes: the
 * neighbours' C(z) reach the copies by a message).  xhat is [rows][d]: row 0
 * is the copy of node first_node - 1, rows 1 .. rows-2 the own nodes
 * first_node .. first_node + rows - 3, row rows-1 the copy of the node after
 * them (ring indices taken by the caller).  Own row r mixes rows r-1, r and
 * r+1 exactly as oracle_dcd_step mixes its ring neighbours, with the keep
 * draw of node first_node + r - 1; the copies are read, not updated.
 * g is [rows-2][d].  c_first and c_last ([d] each) receive the C(z) the first
 * and the last own node added to themselves, which their neighbours' holders
 * add to their copies.
 */
int oracle_dcd_step_rows(int rows, int64_t d, int64_t first_node, const float w[3], float* xhat, const float* g,
                         float gamma, double p, uint64_t seed, uint32_t t, float* c_first, float* c_last) {
    if (rows < 3 || d < 0 || first_node < 0 || !(p > 0.0 && p <= 1.0)) return ORACLE_EINVAL;
    const int own = rows - 2;
    float* xn = (float*)malloc(sizeof(float) * (size_t)(own * d > 0 ? own * d : 1));
    if (!xn) return ORACLE_ENOMEM;
    const uint64_t thr = oracle_keep_threshold(p);
    const float inv_p = (float)(1.0 / p);
    for (int r = 1; r <= own; ++r) {
        const float* xl = xhat + (int64_t)(r - 1) * d;
        const float* xi = xhat + (int64_t)r * d;
        const float* xr = xhat + (int64_t)(r + 1) * d;
        const float* gi = g + (int64_t)(r - 1) * d;
        const uint32_t node = (uint32_t)(first_node + r - 1);
        for (int64_t e = 0; e < d; ++e) {
            float acc = w[0] * xl[e];
            acc = acc + w[1] * xi[e];
            acc = acc + w[2] * xr[e];
            const float xh = acc - gamma * gi[e];
            const float z = xh - xi[e];
            const float cz = dcd_compress(z, dcd_word(seed, node, t, (uint64_t)e), thr, inv_p);
            xn[(int64_t)(r - 1) * d + e] = xi[e] + cz;
            if (r == 1) c_first[e] = cz;
            if (r == own) c_last[e] = cz;
        }
    }
    memcpy(xhat + d, xn, sizeof(float) * (size_t)(own * d));
    free(xn);
    return ORACLE_OK;
}

/*
 * The same iteration with every replica stored explicitly, for the replica
 * identity check: rep[i][j] is node i's copy of node j's model ([n][n][d];
 * rep[i][i] is node i's own model).  Node i mixes its own copies of its ring
 * neighbours, compresses its own difference, and then every node that keeps a
 * copy of node j (j itself and j's two ring neighbours) adds C(z_j) to it
 * (DCD-PSGD step 3).
 */
int oracle_dcd_step_replicas(int n, int64_t d, const float w[3], float* rep, const float* g,
                             float gamma, double p, uint64_t seed, uint32_t t) {
    if (n < 1 || d < 0 || !(p > 0.0 && p <= 1.0)) return ORACLE_EINVAL;
    float* cz = (float*)malloc(sizeof(float) * (size_t)(n * d > 0 ? n * d : 1));
    if (!cz) return ORACLE_ENOMEM;
    const uint64_t thr = oracle_keep_threshold(p);
    const float inv_p = (float)(1.0 / p);
#define REP(i, j) (rep + ((int64_t)(i) * n + (j)) * d)
    for (int i = 0; i < n; ++i) {
        const int l = (i + n - 1) % n, r = (i + 1) % n;
        for (int64_t e = 0; e < d; ++e) {
            float acc = w[0] * REP(i, l)[e];
            acc = acc + w[1] * REP(i, i)[e];
            acc = acc + w[2] * REP(i, r)[e];
            const float xh = acc - gamma * g[(int64_t)i * d + e];
            const float z = xh - REP(i, i)[e];
            cz[(int64_t)i * d + e] = dcd_compress(z, dcd_word(seed, (uint32_t)i, t, (uint64_t)e), thr, inv_p);
        }
    }
    for (int j = 0; j < n; ++j) {
        /* holders of a copy of node j: j itself and its two ring neighbours */
        int holders[3] = {j, (j + n - 1) % n, (j + 1) % n};
        int nh = n >= 3 ? 3 : n;  /* n=1: only j; n=2: j and the other node */
        for (int h = 0; h < nh; ++h) {
            float* x = REP(holders[h], j);
            for (int64_t e = 0; e < d; ++e) x[e] = x[e] + cz[(int64_t)j * d + e];
        }
    }
#undef REP
    free(cz);
    return ORACLE_OK;
}

/* ------------------------------------------------------------- ECD-PSGD */

/*
 * One ECD-PSGD iteration t >= 1 of n nodes on a ring ("Communication
 * Compression for Decentralized Training", ECD-PSGD, equations (3) and (4)):
 * each node j extrapolates
 *     z_j = (1 - t/2) x_{t-1}^(j) + (t/2) x_t^(j)                     (3)
 * and its neighbours update their estimate of its model from C(z_j)
 *     xt_j <- (1 - 2/t) xt_j + (2/t) C(z_j).                          (4)
 * Reading (the equivalent update form is not printed): ECD-PSGD keeps the
 * D-PSGD step with the neighbours' models replaced by these estimates,
 *     x_{t+1}^(i) = w[0] xt_{i-1} + w[1] x_t^(i) + w[2] xt_{i+1} - gamma g_i,
 * a node using its own model exactly.  Every holder of an estimate of x^(j)
 * applies the same C(z_j), so one array xt[n][d] stands for all of them.  C is
 * the random sparsification of the DCD-PSGD step (Philox4x32-10, keep with
 * probability p, scale 1/p).  The coefficients are rounded to fp32 once from
 * fp64: a = 1 - t/2, b = t/2, c = 1 - 2/t, e2 = 2/t.
 * x [n][d] holds x_t (read), x_prev [n][d] holds x_{t-1} and receives x_{t+1},
 * xt [n][d] the estimates (updated in place), g [n][d] the gradients.
 */
int oracle_ecd_step(int n, int64_t d, const float w[3], const float* x, float* x_prev, float* xt, const float* g,
                    float gamma, double p, uint64_t seed, uint32_t t) {
    if (n < 1 || d < 0 || !(p > 0.0 && p <= 1.0) || t < 1) return ORACLE_EINVAL;
    const uint64_t thr = oracle_keep_threshold(p);
    const float inv_p = (float)(1.0 / p);
    const float a = (float)(1.0 - 0.5 * (double)t), b = (float)(0.5 * (double)t);
    const float c = (float)(1.0 - 2.0 / (double)t), e2 = (float)(2.0 / (double)t);
    /* (3), (4): the new estimates of every node */
    for (int j = 0; j < n; ++j)
        for (int64_t e = 0; e < d; ++e) {
            const int64_t q = (int64_t)j * d + e;
            const float z = a * x_prev[q] + b * x[q];
            const float cz = dcd_compress(z, dcd_word(seed, (uint32_t)j, t, (uint64_t)e), thr, inv_p);
            xt[q] = c * xt[q] + e2 * cz;
        }
    /* the D-PSGD step on the estimates */
    for (int i = 0; i < n; ++i) {
        const int l = (i + n - 1) % n, r = (i + 1) % n;
        for (int64_t e = 0; e < d; ++e) {
            float acc = w[0] * xt[(int64_t)l * d + e];
            acc = acc + w[1] * x[(int64_t)i * d + e];
            acc = acc + w[2] * xt[(int64_t)r * d + e];
            x_prev[(int64_t)i * d + e] = acc - gamma * g[(int64_t)i * d + e];
        }
    }
    return ORACLE_OK;
}

/* -------------------------------------------------------- wire encodings */

static void put_u16(unsigned char* b, uint16_t x) { b[0] = (unsigned char)(x & 0xff); b[1] = (unsigned char)(x >> 8); }
static void put_u32(unsigned char* b, uint32_t x) {
    for (int i = 0; i < 4; ++i) b[i] = (unsigned char)((x >> (8 * i)) & 0xff);
}
static uint16_t get_u16(const unsigned char* b) { return (uint16_t)(b[0] | (b[1] << 8)); }
static uint32_t get_u32(const unsigned char* b) {
    return (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);
}

/*
 * DGC's message as a byte stream ("Deep Gradient Compression", section 3.1:
 * each sent value travels as 32 bits, and the unsent positions before it as
 * a 16-bit count).  Reading: one 6-byte record per sent entry, little-endian
 * [uint16 number of unsent positions since the previous entry (or the
 * start)][fp32 value]; a gap of 65536 or more is split by escape records
 * (65535, +0.0f), each standing for 65535 zeros and one explicit zero.
 * idx ascending.  Writes at most 6 * (count + escapes) bytes; returns the
 * byte count, or -1 if out_cap is too small or the indices do not ascend.
 */
int64_t oracle_dgc_encode(const uint32_t* idx, const float* val, int64_t count, unsigned char* out, int64_t out_cap) {
    int64_t at = 0, next = 0; /* next: first position not yet covered */
    for (int64_t j = 0; j < count; ++j) {
        if ((int64_t)idx[j] < next) return -1;
        int64_t gap = (int64_t)idx[j] - next;
        while (gap >= 65536) {
            if (at + 6 > out_cap) return -1;
            put_u16(out + at, 65535);
            put_u32(out + at + 2, 0u);
            at += 6;
            gap -= 65536;
        }
        if (at + 6 > out_cap) return -1;
        put_u16(out + at, (uint16_t)gap);
        put_u32(out + at + 2, bits_of(val[j]));
        at += 6;
        next = (int64_t)idx[j] + 1;
    }
    return at;
}

/* Decodes a DGC byte stream into dense[n] (zeros elsewhere); -1 if it runs past n. */
int oracle_dgc_decode(const unsigned char* in, int64_t nbytes, int64_t n, float* dense) {
    for (int64_t j = 0; j < n; ++j) dense[j] = 0.0f;
    int64_t pos = 0;
    for (int64_t at = 0; at + 6 <= nbytes; at += 6) {
        pos += get_u16(in + at);
        if (pos >= n) return -1;
        uint32_t b = get_u32(in + at + 2);
        memcpy(&dense[pos], &b, 4);
        ++pos;
    }
    return 0;
}

/*
 * AdaComp's message as a byte stream ("AdaComp ...", Proposed method: one
 * scale per layer, the mean of |g_max|, with each sent entry as sign +
 * scale).  Reading: per layer, in order, a header [uint32 count][fp32 scale]
 * and then count uint32 words (local index << 1 | sign bit, sign = 1 for a
 * negative value), little-endian.  idx/val: the learner's list (layers one
 * after another, ascending); counts/scales: [S].  Returns the byte count or
 * -1 if out_cap is too small.
 */
int64_t oracle_adacomp_encode(const int64_t* seg_off, int S, const uint32_t* idx, const float* val,
                              const int64_t* counts, const float* scales, unsigned char* out, int64_t out_cap) {
    int64_t at = 0, j = 0;
    for (int s = 0; s < S; ++s) {
        if (at + 8 + 4 * counts[s] > out_cap) return -1;
        put_u32(out + at, (uint32_t)counts[s]);
        put_u32(out + at + 4, bits_of(scales[s]));
        at += 8;
        for (int64_t q = 0; q < counts[s]; ++q, ++j) {
            const uint32_t local = (uint32_t)((int64_t)idx[j] - seg_off[s]);
            const uint32_t sign = val[j] < 0.0f ? 1u : 0u;
            put_u32(out + at, (local << 1) | sign);
            at += 4;
        }
    }
    return at;
}

/* Decodes an AdaComp byte stream into dense[n]: +-scale at the sent entries. */
int oracle_adacomp_decode(const unsigned char* in, int64_t nbytes, const int64_t* seg_off, int S, float* dense) {
    const int64_t n = seg_off[S];
    for (int64_t j = 0; j < n; ++j) dense[j] = 0.0f;
    int64_t at = 0;
    for (int s = 0; s < S; ++s) {
        if (at + 8 > nbytes) return -1;
        const uint32_t c = get_u32(in + at);
        const uint32_t sb = get_u32(in + at + 4);
        float scale;
        memcpy(&scale, &sb, 4);
        at += 8;
        for (uint32_t q = 0; q < c; ++q, at += 4) {
            if (at + 4 > nbytes) return -1;
            const uint32_t w = get_u32(in + at);
            const int64_t local = (int64_t)(w >> 1);
            if (seg_off[s] + local >= seg_off[s + 1]) return -1;
            dense[seg_off[s] + local] = (w & 1u) ? -scale : scale;
        }
    }
    return 0;
}

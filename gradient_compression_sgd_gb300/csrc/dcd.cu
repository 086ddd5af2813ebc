// dcd.cu -- one DCD-PSGD iteration of n ring nodes in one pass.
//
// "Communication Compression for Decentralized Training", DCD-PSGD steps
// 1-3: mix the neighbours' replicas with W and take the SGD step
// (x_half), compress the difference z = x_half - x, and add C(z) to the model
// and to every replica of it.  Every holder of a replica of node i applies
// the same C(z_i), so one array xhat[n][d] stands for all models and
// replicas.  C is random sparsification: keep z_e with probability p and
// scale it by 1/p, the keep draw taken from Philox4x32-10 (Salmon et al.,
// SC'11) at counter (e/4, node, t, e/2^34) under key (seed).
//
// Each thread owns four consecutive elements of every node: it loads the
// n models' and gradients' float4s, computes all n new values from the old
// ones held in registers, and stores them, so the update is in place with no
// second buffer and every element is read and written exactly once.  One
// Philox call yields the keep words of the thread's four elements of a node.
#include "common.cuh"

namespace gcsgd {
namespace dcd {

constexpr int NT = 256;

struct Params {
    float w0, w1, w2, gamma, inv_p;
    uint64_t thr;  // keep when word < thr (2^32 keeps everything)
    uint32_t key0, key1, t;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
        const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

__device__ __forceinline__ float mix_step(const Params& P, float xl, float xi, float xr, float g, uint32_t word) {
    float acc = __fmul_rn(P.w0, xl);
    acc = __fadd_rn(acc, __fmul_rn(P.w1, xi));
    acc = __fadd_rn(acc, __fmul_rn(P.w2, xr));
    const float xh = __fsub_rn(acc, __fmul_rn(P.gamma, g));
    const float z = __fsub_rn(xh, xi);
    const float cz = ((uint64_t)word < P.thr) ? __fmul_rn(z, P.inv_p) : 0.0f;
    return __fadd_rn(xi, cz);
}

__device__ __forceinline__ float4 node_update(const Params& P, const float4& L, const float4& X, const float4& Rr,
                                              const float4& G, uint64_t q, uint32_t node) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)q, node, P.t, (uint32_t)(q >> 32)), P.key0, P.key1);
    float4 o;
    o.x = mix_step(P, L.x, X.x, Rr.x, G.x, w.x);
    o.y = mix_step(P, L.y, X.y, Rr.y, G.y, w.y);
    o.z = mix_step(P, L.z, X.z, Rr.z, G.z, w.z);
    o.w = mix_step(P, L.w, X.w, Rr.w, G.w, w.w);
    return o;
}

__device__ __forceinline__ float4 ld4(const float* p, uint64_t e, uint64_t d, bool vec) {
    if (vec) return *reinterpret_cast<const float4*>(p + e);
    float4 r;
    r.x = e < d ? p[e] : 0.f;
    r.y = e + 1 < d ? p[e + 1] : 0.f;
    r.z = e + 2 < d ? p[e + 2] : 0.f;
    r.w = e + 3 < d ? p[e + 3] : 0.f;
    return r;
}

__device__ __forceinline__ void st4(float* p, uint64_t e, uint64_t d, bool vec, const float4& v) {
    if (vec) {
        *reinterpret_cast<float4*>(p + e) = v;
        return;
    }
    if (e < d) p[e] = v.x;
    if (e + 1 < d) p[e + 1] = v.y;
    if (e + 2 < d) p[e + 2] = v.z;
    if (e + 3 < d) p[e + 3] = v.w;
}

// NN > 0: node count known at compile time, every load issued up front.
template <int NN>
__global__ void __launch_bounds__(NT, 2) dcd_fixed(Params P, uint64_t d, float* __restrict__ xhat,
                                                const float* __restrict__ grad, bool rows_aligned) {
    const uint64_t nq = (d + 3) / 4;
    for (uint64_t q = (uint64_t)blockIdx.x * NT + threadIdx.x; q < nq; q += (uint64_t)gridDim.x * NT) {
        const uint64_t e = 4 * q;
        const bool vec = rows_aligned && e + 4 <= d;
        float4 X[NN], G[NN];
#pragma unroll
        for (int i = 0; i < NN; ++i) {
            X[i] = ld4(xhat + (uint64_t)i * d, e, d, vec);
            G[i] = ld4(grad + (uint64_t)i * d, e, d, vec);
        }
#pragma unroll
        for (int i = 0; i < NN; ++i) {
            const int l = (i + NN - 1) % NN, r = (i + 1) % NN;
            const float4 o = node_update(P, X[l], X[i], X[r], G[i], q, (uint32_t)i);
            st4(xhat + (uint64_t)i * d, e, d, vec, o);
        }
    }
}

// Any node count: a rolling window keeps the old left neighbour and node 0.
__global__ void __launch_bounds__(NT) dcd_rolling(Params P, int n, uint64_t d, float* __restrict__ xhat,
                                                  const float* __restrict__ grad, bool rows_aligned) {
    const uint64_t nq = (d + 3) / 4;
    for (uint64_t q = (uint64_t)blockIdx.x * NT + threadIdx.x; q < nq; q += (uint64_t)gridDim.x * NT) {
        const uint64_t e = 4 * q;
        const bool vec = rows_aligned && e + 4 <= d;
        const float4 x0 = ld4(xhat, e, d, vec);
        float4 left = ld4(xhat + (uint64_t)(n - 1) * d, e, d, vec);
        float4 cur = x0;
        for (int i = 0; i < n; ++i) {
            const float4 right = (i == n - 1) ? x0 : ld4(xhat + (uint64_t)(i + 1) * d, e, d, vec);
            const float4 g = ld4(grad + (uint64_t)i * d, e, d, vec);
            const float4 o = node_update(P, left, cur, right, g, q, (uint32_t)i);
            st4(xhat + (uint64_t)i * d, e, d, vec, o);
            left = cur;
            cur = right;
        }
    }
}

// ------------------------------------------------ DCD-PSGD across ranks
//
// The nodes one rank of several holds, with copies of its two ring
// neighbours beside them: rows 0 and R-1 of xhat are the copies (read only),
// rows 1..R-2 the own nodes first_node.. .  Each own row mixes its row
// neighbours as dcd_fixed mixes its ring neighbours; the C(z) the first and
// the last own node add to themselves is what the neighbouring ranks add to
// their copies (DCD-PSGD step 3), so every kept entry of those two rows goes
// out as an (index, value) pair: per CTA and round, a block scan of the
// threads' kept counts and one atomic per list reserve the slots (the lists
// are not in index order; their indices are unique).

// mix_step, also returning C(z) and whether the entry was kept.
__device__ __forceinline__ float mix_step_c(const Params& P, float xl, float xi, float xr, float g, uint32_t word,
                                            float* cz, bool* kept) {
    float acc = __fmul_rn(P.w0, xl);
    acc = __fadd_rn(acc, __fmul_rn(P.w1, xi));
    acc = __fadd_rn(acc, __fmul_rn(P.w2, xr));
    const float xh = __fsub_rn(acc, __fmul_rn(P.gamma, g));
    const float z = __fsub_rn(xh, xi);
    *kept = (uint64_t)word < P.thr;
    *cz = *kept ? __fmul_rn(z, P.inv_p) : 0.0f;
    return __fadd_rn(xi, *cz);
}

__global__ void __launch_bounds__(NT) dcd_rows(Params P, int R, uint64_t d, uint32_t first_node,
                                               float* __restrict__ xhat, const float* __restrict__ grad,
                                               bool rows_aligned, gcsgd_pair* __restrict__ c_first,
                                               gcsgd_pair* __restrict__ c_last, uint64_t cap,
                                               unsigned long long* __restrict__ counts) {
    __shared__ uint64_t scan[NT / 32 + 1];
    __shared__ unsigned long long s_base[2];
    const uint64_t nq = (d + 3) / 4;
    const int own = R - 2;
    for (uint64_t q0 = (uint64_t)blockIdx.x * NT; q0 < nq; q0 += (uint64_t)gridDim.x * NT) {  // CTA-uniform
        const uint64_t q = q0 + threadIdx.x;
        const bool live = q < nq;
        const uint64_t e = 4 * q;
        const bool vec = rows_aligned && e + 4 <= d;
        float cf[4] = {0.f, 0.f, 0.f, 0.f}, cl[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t kf = 0, kl = 0;  // kept masks of the first and last own row's four entries
        if (live) {
            float4 left = ld4(xhat, e, d, vec);
            float4 cur = ld4(xhat + d, e, d, vec);
            for (int r = 1; r <= own; ++r) {
                const float4 right = ld4(xhat + (uint64_t)(r + 1) * d, e, d, vec);
                const float4 g = ld4(grad + (uint64_t)(r - 1) * d, e, d, vec);
                const uint4 w = philox4x32_10(make_uint4((uint32_t)q, first_node + (uint32_t)(r - 1), P.t,
                                                         (uint32_t)(q >> 32)), P.key0, P.key1);
                const float* L = &left.x;
                const float* X = &cur.x;
                const float* Rr = &right.x;
                const float* G = &g.x;
                const uint32_t* W = &w.x;
                float4 o;
                float* oo = &o.x;
                float cz[4];
                uint32_t km = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    bool kept;
                    oo[j] = mix_step_c(P, L[j], X[j], Rr[j], G[j], W[j], &cz[j], &kept);
                    km |= (uint32_t)(kept && e + j < d) << j;
                }
                st4(xhat + (uint64_t)r * d, e, d, vec, o);
                if (r == 1) {
                    kf = km;
#pragma unroll
                    for (int j = 0; j < 4; ++j) cf[j] = cz[j];
                }
                if (r == own) {
                    kl = km;
#pragma unroll
                    for (int j = 0; j < 4; ++j) cl[j] = cz[j];
                }
                left = cur;
                cur = right;
            }
        }
        uint64_t tot;
        const uint64_t ex = block_exclusive_scan<NT>((uint64_t)__popc(kf) | ((uint64_t)__popc(kl) << 32), scan, &tot);
        if (threadIdx.x == 0) {
            s_base[0] = atomicAdd(&counts[0], (unsigned long long)(tot & 0xffffffffu));
            s_base[1] = atomicAdd(&counts[1], (unsigned long long)(tot >> 32));
        }
        __syncthreads();
        uint64_t at_f = s_base[0] + (ex & 0xffffffffu), at_l = s_base[1] + (ex >> 32);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if ((kf >> j) & 1u) {
                if (at_f < cap) {
                    gcsgd_pair pr;
                    pr.idx = (uint32_t)(e + j);
                    pr.val = cf[j];
                    c_first[at_f] = pr;
                }
                ++at_f;
            }
            if ((kl >> j) & 1u) {
                if (at_l < cap) {
                    gcsgd_pair pr;
                    pr.idx = (uint32_t)(e + j);
                    pr.val = cl[j];
                    c_last[at_l] = pr;
                }
                ++at_l;
            }
        }
        __syncthreads();  // s_base and scan are reused by the next round
    }
}

// A neighbour's copy takes the C(z) its owner added: x[idx] += val at every
// pair (the indices of a list are unique, so the adds do not race).
__global__ void __launch_bounds__(NT) dcd_copy_scatter(float* __restrict__ x, uint64_t d,
                                                       const gcsgd_pair* __restrict__ pairs,
                                                       const int64_t* __restrict__ count, uint64_t cap) {
    const int64_t c = *count;
    const uint64_t n = c < 0 ? 0 : ((uint64_t)c < cap ? (uint64_t)c : cap);
    for (uint64_t i = (uint64_t)blockIdx.x * NT + threadIdx.x; i < n; i += (uint64_t)gridDim.x * NT) {
        const gcsgd_pair pr = pairs[i];
        if (pr.idx < d) x[pr.idx] = __fadd_rn(x[pr.idx], pr.val);
    }
}

// x <- x + 0 everywhere: the owner adds C(z) = +0 to every entry it did not
// keep, which turns a -0 into +0; a copy that starts with -0 entries takes
// this once so that its later adds stay bit-equal to the owner's.
__global__ void __launch_bounds__(NT) dcd_copy_zero_pass(float* __restrict__ x, uint64_t d) {
    for (uint64_t i = (uint64_t)blockIdx.x * NT + threadIdx.x; i < d; i += (uint64_t)gridDim.x * NT)
        x[i] = __fadd_rn(x[i], 0.0f);
}

// ---------------------------------------------------------------- ECD-PSGD
//
// "Communication Compression for Decentralized Training", ECD-PSGD,
// equations (3) and (4): node j extrapolates z_j = (1 - t/2) x_{t-1} +
// (t/2) x_t, its neighbours' estimate of it becomes xt_j <- (1 - 2/t) xt_j +
// (2/t) C(z_j), and the D-PSGD step runs on the estimates (a node uses its own
// model): x_{t+1}^(i) = w0 xt_{i-1} + w1 x_t^(i) + w2 xt_{i+1} - gamma g_i.
// One estimate array stands for every holder (they all apply the same
// C(z_j)).  Per thread: four consecutive elements of every node; the new
// estimates are computed first, then each node's step; x_{t+1} goes into the
// x_{t-1} buffer once that node's x_{t-1} has been read.

struct EcdParams {
    float w0, w1, w2, gamma, inv_p;
    float a, b, c, e2;  // 1 - t/2, t/2, 1 - 2/t, 2/t (rounded once to fp32)
    uint64_t thr;
    uint32_t key0, key1, t;
};

__device__ __forceinline__ float4 ecd_estimate(const EcdParams& P, const float4& X, const float4& XP,
                                               const float4& XT, uint64_t q, uint32_t node) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)q, node, P.t, (uint32_t)(q >> 32)), P.key0, P.key1);
    const float* x = &X.x;
    const float* xp = &XP.x;
    const float* xt = &XT.x;
    const uint32_t* wd = &w.x;
    float4 o;
    float* oo = &o.x;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float z = __fadd_rn(__fmul_rn(P.a, xp[j]), __fmul_rn(P.b, x[j]));
        const float cz = ((uint64_t)wd[j] < P.thr) ? __fmul_rn(z, P.inv_p) : 0.0f;
        oo[j] = __fadd_rn(__fmul_rn(P.c, xt[j]), __fmul_rn(P.e2, cz));
    }
    return o;
}

__device__ __forceinline__ float4 ecd_mix(const EcdParams& P, const float4& L, const float4& X, const float4& R,
                                          const float4& G) {
    const float* l = &L.x;
    const float* x = &X.x;
    const float* r = &R.x;
    const float* g = &G.x;
    float4 o;
    float* oo = &o.x;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float acc = __fmul_rn(P.w0, l[j]);
        acc = __fadd_rn(acc, __fmul_rn(P.w1, x[j]));
        acc = __fadd_rn(acc, __fmul_rn(P.w2, r[j]));
        oo[j] = __fsub_rn(acc, __fmul_rn(P.gamma, g[j]));
    }
    return o;
}

// NN <= 4: every node's float4s in registers (larger rings take the rolling
// window, which keeps the register count low enough for two CTAs per SM).
template <int NN>
__global__ void __launch_bounds__(NT, 2) ecd_fixed(EcdParams P, uint64_t d, const float* __restrict__ x,
                                                float* __restrict__ x_prev, float* __restrict__ xt,
                                                const float* __restrict__ grad, bool rows_aligned) {
    const uint64_t nq = (d + 3) / 4;
    for (uint64_t q = (uint64_t)blockIdx.x * NT + threadIdx.x; q < nq; q += (uint64_t)gridDim.x * NT) {
        const uint64_t e = 4 * q;
        const bool vec = rows_aligned && e + 4 <= d;
        float4 X[NN], T[NN];
#pragma unroll
        for (int i = 0; i < NN; ++i) {
            X[i] = ld4(x + (uint64_t)i * d, e, d, vec);
            const float4 xp = ld4(x_prev + (uint64_t)i * d, e, d, vec);
            const float4 xo = ld4(xt + (uint64_t)i * d, e, d, vec);
            T[i] = ecd_estimate(P, X[i], xp, xo, q, (uint32_t)i);
        }
#pragma unroll
        for (int i = 0; i < NN; ++i) {
            const int l = (i + NN - 1) % NN, r = (i + 1) % NN;
            const float4 g = ld4(grad + (uint64_t)i * d, e, d, vec);
            st4(x_prev + (uint64_t)i * d, e, d, vec, ecd_mix(P, T[l], X[i], T[r], g));
            st4(xt + (uint64_t)i * d, e, d, vec, T[i]);
        }
    }
}

// Any node count: estimates computed along a rolling window (node 0's and
// node n-1's are kept for the wrap-around).
__global__ void __launch_bounds__(NT) ecd_rolling(EcdParams P, int n, uint64_t d, const float* __restrict__ x,
                                                  float* __restrict__ x_prev, float* __restrict__ xt,
                                                  const float* __restrict__ grad, bool rows_aligned) {
    const uint64_t nq = (d + 3) / 4;
    for (uint64_t q = (uint64_t)blockIdx.x * NT + threadIdx.x; q < nq; q += (uint64_t)gridDim.x * NT) {
        const uint64_t e = 4 * q;
        const bool vec = rows_aligned && e + 4 <= d;
        auto est = [&](int i) {
            return ecd_estimate(P, ld4(x + (uint64_t)i * d, e, d, vec), ld4(x_prev + (uint64_t)i * d, e, d, vec),
                                ld4(xt + (uint64_t)i * d, e, d, vec), q, (uint32_t)i);
        };
        const float4 t0 = est(0);
        float4 left = est(n - 1);
        float4 cur = t0;
        for (int i = 0; i < n; ++i) {
            const float4 right = (i == n - 1) ? t0 : est(i + 1);
            const float4 xi = ld4(x + (uint64_t)i * d, e, d, vec);
            const float4 g = ld4(grad + (uint64_t)i * d, e, d, vec);
            st4(x_prev + (uint64_t)i * d, e, d, vec, ecd_mix(P, left, xi, right, g));
            st4(xt + (uint64_t)i * d, e, d, vec, cur);
            left = cur;
            cur = right;
        }
    }
}

}  // namespace dcd

int dcd_launch(int n, int64_t d, const float* w, float* xhat, const float* grad, float gamma, double p,
               uint64_t seed, uint32_t t, cudaStream_t stream) {
    using namespace dcd;
    if (d == 0) return GCSGD_OK;
    Params P;
    P.w0 = w[0];
    P.w1 = w[1];
    P.w2 = w[2];
    P.gamma = gamma;
    P.inv_p = (float)(1.0 / p);
    P.thr = p >= 1.0 ? (1ull << 32) : (uint64_t)llround(p * 4294967296.0);
    P.key0 = (uint32_t)seed;
    P.key1 = (uint32_t)(seed >> 32);
    P.t = t;
    const bool rows_aligned = ((d & 3) == 0) && (((uintptr_t)xhat & 15) == 0) && (((uintptr_t)grad & 15) == 0);
    const uint64_t nq = ((uint64_t)d + 3) / 4;
    uint64_t grid = (uint64_t)sm_count() * (n <= 4 ? 8 : 4);
    const uint64_t need = (nq + NT - 1) / NT;
    if (grid > need) grid = need;
    LaunchScope ls("dcd_step", stream);
    switch (n) {
#define DCD_CASE(NNV) \
    case NNV: dcd_fixed<NNV><<<(unsigned)grid, NT, 0, stream>>>(P, (uint64_t)d, xhat, grad, rows_aligned); break;
        DCD_CASE(1)
        DCD_CASE(2)
        DCD_CASE(3)
        DCD_CASE(4)
        DCD_CASE(5)
        DCD_CASE(6)
        DCD_CASE(7)
        DCD_CASE(8)
#undef DCD_CASE
        default:
            dcd_rolling<<<(unsigned)grid, NT, 0, stream>>>(P, n, (uint64_t)d, xhat, grad, rows_aligned);
    }
    return check_launch("dcd_step");
}

int dcd_rows_launch(int rows, int64_t d, int64_t first_node, const float* w, float* xhat, const float* grad,
                    float gamma, double p, uint64_t seed, uint32_t t, gcsgd_pair* c_first, gcsgd_pair* c_last,
                    int64_t cap, int64_t* counts, cudaStream_t stream) {
    using namespace dcd;
    if (cudaMemsetAsync(counts, 0, 2 * sizeof(int64_t), stream) != cudaSuccess)
        return set_error(GCSGD_ERR_CUDA, "dcd_step_rows: clearing counts failed");
    if (d == 0) return GCSGD_OK;
    Params P;
    P.w0 = w[0];
    P.w1 = w[1];
    P.w2 = w[2];
    P.gamma = gamma;
    P.inv_p = (float)(1.0 / p);
    P.thr = p >= 1.0 ? (1ull << 32) : (uint64_t)llround(p * 4294967296.0);
    P.key0 = (uint32_t)seed;
    P.key1 = (uint32_t)(seed >> 32);
    P.t = t;
    const bool rows_aligned = ((d & 3) == 0) && (((uintptr_t)xhat & 15) == 0) && (((uintptr_t)grad & 15) == 0);
    const uint64_t nq = ((uint64_t)d + 3) / 4;
    uint64_t grid = (uint64_t)sm_count() * 4;
    const uint64_t need = (nq + NT - 1) / NT;
    if (grid > need) grid = need;
    LaunchScope ls("dcd_step_rows", stream);
    dcd_rows<<<(unsigned)grid, NT, 0, stream>>>(P, rows, (uint64_t)d, (uint32_t)first_node, xhat, grad, rows_aligned,
                                                c_first, c_last, (uint64_t)cap,
                                                reinterpret_cast<unsigned long long*>(counts));
    return check_launch("dcd_step_rows");
}

int dcd_copy_add_launch(float* x, int64_t d, const gcsgd_pair* pairs, const int64_t* count, int64_t cap,
                        bool zero_pass, cudaStream_t stream) {
    using namespace dcd;
    if (d == 0) return GCSGD_OK;
    int rc;
    if (zero_pass) {
        uint64_t grid = (uint64_t)sm_count() * 4, need = ((uint64_t)d + NT - 1) / NT;
        if (grid > need) grid = need;
        LaunchScope ls("dcd_copy_zero_pass", stream);
        dcd_copy_zero_pass<<<(unsigned)grid, NT, 0, stream>>>(x, (uint64_t)d);
        if ((rc = check_launch("dcd_copy_zero_pass"))) return rc;
    }
    if (cap == 0) return GCSGD_OK;
    uint64_t grid = (uint64_t)sm_count() * 2, need = ((uint64_t)cap + NT - 1) / NT;
    if (grid > need) grid = need;
    LaunchScope ls("dcd_copy_add", stream);
    dcd_copy_scatter<<<(unsigned)grid, NT, 0, stream>>>(x, (uint64_t)d, pairs, count, (uint64_t)cap);
    return check_launch("dcd_copy_add");
}

int ecd_launch(int n, int64_t d, const float* w, const float* x, float* x_prev, float* xt, const float* grad,
               float gamma, double p, uint64_t seed, uint32_t t, cudaStream_t stream) {
    using namespace dcd;
    if (d == 0) return GCSGD_OK;
    EcdParams P;
    P.w0 = w[0];
    P.w1 = w[1];
    P.w2 = w[2];
    P.gamma = gamma;
    P.inv_p = (float)(1.0 / p);
    P.a = (float)(1.0 - 0.5 * (double)t);
    P.b = (float)(0.5 * (double)t);
    P.c = (float)(1.0 - 2.0 / (double)t);
    P.e2 = (float)(2.0 / (double)t);
    P.thr = p >= 1.0 ? (1ull << 32) : (uint64_t)llround(p * 4294967296.0);
    P.key0 = (uint32_t)seed;
    P.key1 = (uint32_t)(seed >> 32);
    P.t = t;
    const bool rows_aligned = ((d & 3) == 0) && ((((uintptr_t)x | (uintptr_t)x_prev | (uintptr_t)xt |
                                                   (uintptr_t)grad) & 15) == 0);
    const uint64_t nq = ((uint64_t)d + 3) / 4;
    uint64_t grid = (uint64_t)sm_count() * (n <= 4 ? 8 : 4);
    const uint64_t need = (nq + NT - 1) / NT;
    if (grid > need) grid = need;
    LaunchScope ls("ecd_step", stream);
    switch (n) {
#define ECD_CASE(NNV)                                                                                        \
    case NNV:                                                                                                \
        ecd_fixed<NNV><<<(unsigned)grid, NT, 0, stream>>>(P, (uint64_t)d, x, x_prev, xt, grad, rows_aligned); \
        break;
        ECD_CASE(1)
        ECD_CASE(2)
        ECD_CASE(3)
        ECD_CASE(4)
#undef ECD_CASE
        default:
            ecd_rolling<<<(unsigned)grid, NT, 0, stream>>>(P, n, (uint64_t)d, x, x_prev, xt, grad, rows_aligned);
    }
    return check_launch("ecd_step");
}

}  // namespace gcsgd

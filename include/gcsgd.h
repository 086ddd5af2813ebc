/*
 * gcsgd.h -- C ABI of the GB300 gradient-compression library (libgcsgd.so).
 *
 * The per-worker hot path of communication-efficient data-parallel SGD:
 * Deep Gradient Compression, AdaComp, the decompress-and-average of K
 * learners' sparse messages, and the DCD-PSGD replica update.  K learners
 * (or n ring nodes) are batched in one call on one GPU.
 *
 * Conventions for every entry point
 *  - Pointers are device pointers unless the comment says "host".  The
 *    caller owns every buffer; the library allocates no memory in these
 *    calls and never synchronises the stream.  Work is enqueued on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream) and runs
 *    asynchronously.
 *  - Tensors are flat, contiguous, row-major fp32.  A "layout" is a host
 *    array seg_offsets[n_seg + 1] of int64 with seg_offsets[0] = 0 and
 *    non-decreasing entries: segment (tensor) s is the element range
 *    [seg_offsets[s], seg_offsets[s+1]) of each learner's N =
 *    seg_offsets[n_seg] elements.  Empty segments are allowed.  N must be
 *    below 2^32 (indices are uint32), n_seg at most GCSGD_MAX_SEGMENTS.
 *  - A learner's sparse message is a list of gcsgd_pair with global
 *    (within the learner) indices: segments one after another, each in
 *    ascending index order, so the whole list is ascending.  Lists of K
 *    learners sit at out + k*cap.
 *  - Inputs must be finite; NaN/Inf give unspecified (but memory-safe)
 *    results.
 *  - Return value: GCSGD_OK, or a negative GCSGD_ERR_*; nothing was enqueued
 *    when an argument check fails.  gcsgd_last_error() describes the last
 *    failure of the calling thread.
 */
#ifndef GCSGD_H
#define GCSGD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GCSGD_OK 0
#define GCSGD_ERR_INVALID_ARG (-1)  /* null pointer, bad size, bad layout, bad scalar */
#define GCSGD_ERR_CAPACITY (-2)     /* output capacity too small for a known count   */
#define GCSGD_ERR_WORKSPACE (-3)    /* workspace smaller than *_workspace_size says  */
#define GCSGD_ERR_CUDA (-4)         /* a CUDA runtime call failed (launch, device)   */

#define GCSGD_MAX_SEGMENTS 2048

/* One entry of a sparse message: 8 bytes, index then fp32 value. */
typedef struct {
    uint32_t idx;
    float val;
} gcsgd_pair;

/* ------------------------------------------------------------------ DGC */

/* Entries DGC sends from a segment of n values: max(1, ceil(density*n))
 * computed in fp64, capped at n; 0 for an empty segment.  ("Deep Gradient
 * Compression", section 3.1: only the largest-magnitude fraction of the
 * accumulated gradient is sent.)  Host function. */
int64_t gcsgd_dgc_k(double density, int64_t n);

/* Bytes of device workspace dgc_compress needs for this layout, K and
 * density (written to *bytes).  Host function. */
int gcsgd_dgc_workspace_size(const int64_t* seg_offsets, int32_t n_seg, int32_t K,
                             double density, size_t* bytes);

/*
 * One Deep Gradient Compression step for K learners ("Deep Gradient
 * Compression: Reducing the Communication Bandwidth for Distributed
 * Training", Appendix D with vanilla momentum; sections 3.1-3.3 and
 * Appendix C):
 *   1. local gradient clipping, when clip_thr > 0: if the L2 norm s of a
 *      learner's gradient exceeds thr_k = clip_thr / sqrt(clip_nodes), the
 *      gradient is scaled by c = (float)(thr_k / s) before accumulation;
 *   2. momentum correction: u <- m*u + c*G, then v <- v + u (fp32, one
 *      rounding per operation, no FMA);
 *   3. exact per-segment top-k of |v| with k_s = gcsgd_dgc_k(density, n_s);
 *      ties go to the lower index;
 *   4. the selected (index, v) are written out and momentum factor masking
 *      zeroes u and v at those indices.
 *
 * seg_offsets   host [n_seg+1] layout (see above).
 * grad          [K][N] fp32 gradients, read only.
 * u, v          [K][N] fp32 momentum and accumulated velocity, updated in
 *               place (caller-owned state; zero them before the first step).
 * density       in (0, 1];  momentum any finite value;  clip_thr <= 0 turns
 *               clipping off;  clip_nodes >= 1 (the N of thr*N^-1/2).
 * out           [K][cap] pairs; learner k's list at out + k*cap holds
 *               sum_s k_s entries; cap must be at least that sum
 *               (GCSGD_ERR_CAPACITY otherwise).
 * counts        [K][n_seg] int64, entries per segment (always k_s).
 * totals        [K] int64 entries per learner, or NULL.
 * workspace     device scratch of at least gcsgd_dgc_workspace_size bytes,
 *               256-byte aligned; its contents need not be initialised and
 *               are not kept between calls.  Calls that share a workspace
 *               must be ordered on the GPU.
 */
int dgc_compress(const int64_t* seg_offsets, int32_t n_seg, int32_t K,
                 const float* grad, float* u, float* v,
                 double density, float momentum, float clip_thr, int32_t clip_nodes,
                 gcsgd_pair* out, int64_t cap, int64_t* counts, int64_t* totals,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same step with Nesterov momentum ("Deep Gradient Compression",
 * Appendix B, gradient sparsification with Nesterov momentum correction).
 * The page gives the shape of the corrected update (local momentum plus an
 * accumulated state) but not its equations; read as
 *   u <- m*u + c*G,  then  v <- v + (m*u + c*G)   (fp32, one rounding per
 *   operation, no FMA; the u just updated),
 * i.e. the accumulated state takes the look-ahead step of conventional
 * Nesterov momentum.  Everything else, arguments, workspace and errors, as
 * dgc_compress.  With momentum 0 it equals dgc_compress.
 */
int dgc_compress_nesterov(const int64_t* seg_offsets, int32_t n_seg, int32_t K,
                          const float* grad, float* u, float* v,
                          double density, float momentum, float clip_thr, int32_t clip_nodes,
                          gcsgd_pair* out, int64_t cap, int64_t* counts, int64_t* totals,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * The DGC step with the sampled threshold ("Deep Gradient Compression",
 * section 5: a 0.1 % to 1 % sample of the gradients estimates the population
 * threshold; section 6: hierarchical threshold selection).  Steps 1, 2 and 4
 * as dgc_compress; step 3, per tensor of n values:
 *   m   = floor(sample_frac * n) rounded down to a multiple of 64; the
 *         sample is m / 64 blocks of 64 consecutive updated |v| starting at
 *         b * floor(n / (m / 64)).  A tensor with m = 0 (fewer than 64
 *         values in its sample) is selected exactly, as dgc_compress does;
 *         no other size or density is exempt and the sample is not capped;
 *   tau = the a-th largest sampled |v| (bit-pattern order),
 *         a = round(k_s * m / n) clamped to [1, m];
 *   every entry with |v| >= tau is selected; past k_s the k_s largest of
 *   them are kept (ties to the lower index: the exact top-k), otherwise all
 *   of them are sent, fewer than k_s.
 * counts[k][s] is the number sent for tensor s (at most k_s) and learner k's
 * list in out holds the tensors' entries back to back, totals[k] of them.
 * sample_frac in (0, 1]; the workspace comes from
 * gcsgd_dgc_sampled_workspace_size.  Other arguments and errors: as
 * dgc_compress.
 */
int dgc_compress_sampled(const int64_t* seg_offsets, int32_t n_seg, int32_t K,
                         const float* grad, float* u, float* v,
                         double density, double sample_frac, float momentum, float clip_thr, int32_t clip_nodes,
                         gcsgd_pair* out, int64_t cap, int64_t* counts, int64_t* totals,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of dgc_compress_sampled for this layout, K and sample_frac.  Host. */
int gcsgd_dgc_sampled_workspace_size(const int64_t* seg_offsets, int32_t n_seg, int32_t K, double density,
                                     double sample_frac, size_t* bytes);

/* Diagnostics of the last dgc_compress call made with `workspace`: how each
 * (learner, segment) found its top k.  The answer is exact on every path;
 * only the speed differs.  Host function; it copies a few counters from
 * the workspace and synchronises `stream`. */
typedef struct {
    int64_t units;        /* K * n_seg */
    int64_t empty;        /* empty segments */
    int64_t raw;          /* small segment: its v' staged in shared memory */
    int64_t pool;         /* candidate pool held the top k and was staged in shared memory */
    int64_t pool_global;  /* candidate pool held the top k but was read from global memory */
    int64_t raw_global;   /* large segment at high density: the whole v' read from global memory */
    int64_t hint_failed;  /* candidate pool missed (too few or overflow): the whole v' read */
} gcsgd_dgc_stats_t;
int gcsgd_dgc_stats(const int64_t* seg_offsets, int32_t n_seg, int32_t K, double density,
                    const void* workspace, void* stream, gcsgd_dgc_stats_t* out);

/*
 * dgc_compress without a workspace argument, for callers that cannot
 * allocate device memory (for example a plugin whose host framework's caching
 * allocator owns the device-memory budget, or a loop that must not enter the
 * driver's allocator, which can block or synchronise, in the middle of a
 * step).  The pages have no counterpart: this is a deployment variant of the
 * same DGC step, with the same arguments and results as dgc_compress.
 *
 * Its scratch is a fixed array of GCSGD_NOALLOC_SCRATCH_BYTES built into the
 * library, held on a device from the first call there until the process
 * exits.  A layout and K that need more scratch than that
 * (gcsgd_dgc_workspace_size) are rejected with GCSGD_ERR_WORKSPACE before any
 * GPU work.  The first call on a device looks up the array's device address
 * (once per device, with that device current).  Under CUDA's default lazy
 * module loading that first lookup is also when the driver places the array
 * on the device, committing its bytes: if the device is already full it fails
 * with GCSGD_ERR_CUDA and a message saying so.  Make one warm-up call per
 * device before the caller's allocator reserves the device's memory, and
 * before any stream capture.  Later calls allocate nothing (no cudaMalloc, no
 * cudaFree, no driver allocation).  The address is looked up in the device's
 * primary context: do not call this after cudaDeviceReset or from another
 * driver context on the same device.  All calls share the one array and leave their contents in it;
 * nothing in it needs clearing between calls, but calls that overlap on the
 * GPU (unordered streams, several host threads) race on it and must not be
 * made.
 */
#define GCSGD_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int dgc_compress_noalloc(const int64_t* seg_offsets, int32_t n_seg, int32_t K,
                         const float* grad, float* u, float* v,
                         double density, float momentum, float clip_thr, int32_t clip_nodes,
                         gcsgd_pair* out, int64_t cap, int64_t* counts, int64_t* totals,
                         void* stream);

/* -------------------------------------------------------------- AdaComp */

/* Bytes of device workspace adacomp_compress needs.  lt: host [n_seg] bin
 * lengths L_T >= 1.  Dominated by the candidate pool, 8 B per element per
 * learner (every tile writes its candidates into the slots of its own index
 * range, so no counter is shared); cap does not change it.  Host function. */
int gcsgd_adacomp_workspace_size(const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt,
                                 int32_t K, int64_t cap, size_t* bytes);

/*
 * One AdaComp step for K learners ("AdaComp : Adaptive Residual Gradient
 * Compression for Data-Parallel Distributed Training", Proposed method):
 *   G = R + dW; per bin of L_T values (a last partial bin is a bin of its
 *   own) gmax = max |G|; an entry is selected when |G + dW| >= gmax of its
 *   bin, gmax > 0 and G != 0; scale_s = mean of gmax over every bin of the
 *   segment (the sum accurate to 2^-40 relative or better, divided in fp64
 *   and rounded to fp32 once); a selected entry is sent as
 *   sign(G)*scale_s and the residue keeps R = G - sign(G)*scale_s; an
 *   unselected entry keeps R = G.
 *
 * seg_offsets host layout;  lt host [n_seg] L_T per segment (>= 1).
 * dW          [K][N] new gradients, read only.
 * residue     [K][N] R, updated in place (zero it before the first step).
 * out         [K][cap] pairs, lists as described above.
 * counts      [K][n_seg] int64 entries per segment.
 * scales      [K][n_seg] fp32 scale of each segment.
 * totals      [K] int64 entries per learner (required).  The number of
 *             selected entries is only known on the GPU: when totals[k] >
 *             cap, learner k sends nothing this step (its list is not
 *             written; counts and totals hold the would-be numbers) and its
 *             residue becomes G = R + dW, so no gradient mass is lost; a
 *             larger cap lets the next step send.
 * workspace   at least gcsgd_adacomp_workspace_size bytes, 256-byte aligned.
 * Limit: K * (4 * n_seg + 8) <= 204800 (K <= 24 at 2048 tensors, K <= 198 at
 * 256); a larger call returns GCSGD_ERR_INVALID_ARG before anything is
 * enqueued.
 */
int adacomp_compress(const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt, int32_t K,
                     const float* dW, float* residue,
                     gcsgd_pair* out, int64_t cap, int64_t* counts, float* scales, int64_t* totals,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same step with the residue fix-up deferred to the next call
 * ("AdaComp ...", Proposed method: the residue keeps what was not sent; the
 * order of the fp32 operations is unchanged, so every list, count, scale and
 * residue is bit-identical to adacomp_compress over the same calls).  In the
 * segments with 4 <= L_T <= 512 the sent entries' R = G - sign(G)*scale is
 * not written at the end of the call: R keeps G there, the workspace keeps
 * the call's selection bits, and the next deferred call subtracts sign(R) *
 * scale at those bits while it reads R to form G = R + dW, which saves the
 * scattered read-modify-write of R per sent entry.  Other segments are fixed
 * at once, as in adacomp_compress.
 * pending     0: R is a settled residue (the first call, or after
 *             adacomp_settle); 1: the previous call on this R was deferred,
 *             and out, counts, scales, totals and the workspace still hold
 *             what it wrote.
 * Everything else as for adacomp_compress.  Before R is read as a residue,
 * call adacomp_settle.
 */
int adacomp_compress_deferred(const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt, int32_t K,
                              const float* dW, float* residue, gcsgd_pair* out, int64_t cap, int64_t* counts,
                              float* scales, int64_t* totals, int32_t pending, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Applies the fix-up a deferred call left pending: R[i] -= v for every
 * (i, v) of the message in out, in the 4 <= L_T <= 512 segments of every
 * learner that sent (totals[k] <= cap), one fp32 subtraction each.  out,
 * counts and totals: the deferred call's; workspace: any workspace of the
 * layout's size (the plan is rebuilt).  Errors as for adacomp_compress.
 */
int adacomp_settle(const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt, int32_t K, float* residue,
                   const gcsgd_pair* out, int64_t cap, const int64_t* counts, const int64_t* totals,
                   void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------- sparse average */

/*
 * Decompress and average K learners' sparse messages ("AdaComp ...",
 * Proposed method: learners exchange compressed gradients and average them
 * before the weight update; "Deep Gradient Compression", Appendix A: the
 * nodes' gradients are summed):
 *   out[j] = (sum over the lists k = 0..K-1 that contain j, added in that
 *             order in fp32 starting from +0) / K   (one fp32 divide),
 *   out[j] = 0 where no list contains j.
 * lists   [K][cap] pairs (K at most 512); list k is lists[k*cap .. k*cap + counts[k]),
 *         strictly ascending indices below n.  Entries that break this are
 *         skipped or misplaced but never cause an out-of-range access.
 * counts  [K] int64 device array (0 <= counts[k] <= cap).
 * out     [n] fp32, fully overwritten.
 */
int sparse_average(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K,
                   int64_t n, float* out, void* stream);

/* Bytes of device workspace sparse_average_ws needs for K lists over n
 * outputs: 4 K (ceil(n / 4096) + 1) rounded up to a multiple of 256, plus
 * 256 for a status word.  Host call; GCSGD_ERR_INVALID_ARG for K outside
 * [1, 512], n outside [0, 2^32] or bytes NULL. */
int gcsgd_sparse_average_workspace_size(int32_t K, int64_t n, size_t* bytes);

/*
 * sparse_average with device scratch: the same out, bit for bit (learner
 * order, one fp32 divide by K).  For dense lists (K * cap >= n / 4) with
 * 8-byte aligned records it runs two kernels: the first reads every 128th
 * entry of every list and writes a cursor table into the workspace (per
 * list and 4096-output region, a position at most 128 entries before the
 * region's first entry); the second copies each region's list ranges into
 * shared memory with TMA bulk copies, the next region's copies in flight
 * while the current one is added, and writes every region's average once.
 * Other lists take sparse_average's kernels (the workspace then only holds
 * the status word).
 * lists, cap, counts, K, n, out: as for sparse_average.
 * workspace   device scratch of at least gcsgd_sparse_average_workspace_size
 *             bytes, 256-byte aligned, contents ignored and overwritten; one
 *             call at a time per workspace (calls that share one must be
 *             ordered, e.g. on one stream).
 * Errors: as for sparse_average; GCSGD_ERR_WORKSPACE when workspace_bytes is
 * too small, GCSGD_ERR_INVALID_ARG when workspace is NULL or misaligned
 * (n = 0 writes nothing and needs no workspace).  Every wait in the kernel
 * is bounded: a copy that has not completed after 1 s ends the kernel early
 * with part of out unwritten and sets the status word, which
 * gcsgd_sparse_average_status reads.
 */
int sparse_average_ws(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K,
                      int64_t n, float* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * sparse_average_update with device scratch: the same weights, bit for bit
 * (the learner-order average, one fp32 divide by K, then w <- w - lr * avg
 * with one rounding for the product and one for the difference, at every
 * index some list carries; every other weight keeps its bits).  Dense,
 * 8-byte aligned lists take the cursor table and region kernel of
 * sparse_average_ws, in update mode: the carried positions are marked in a
 * bitmap while the lists are added, the region's weights are read
 * meanwhile, and only the 16-byte groups holding a carried weight are
 * written back.  Other lists take sparse_average_update's kernels.
 * lists, cap, counts, K, n, lr, w: as for sparse_average_update;
 * workspace, workspace_bytes, errors, the status word: as for
 * sparse_average_ws.
 */
int sparse_average_update_ws(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K,
                             int64_t n, float lr, float* w, void* workspace, size_t workspace_bytes, void* stream);

/* The status word of the last sparse_average_ws or sparse_average_update_ws
 * call made with `workspace` for this K and n (0: every copy completed; 1: a copy timed out).  Waits for
 * `stream`, then reads 4 bytes.  Errors: GCSGD_ERR_INVALID_ARG for K outside
 * [1, 512], n outside [1, 2^32] or a NULL pointer; GCSGD_ERR_CUDA when the
 * copy or the wait fails. */
int gcsgd_sparse_average_status(const void* workspace, int32_t K, int64_t n, void* stream, int32_t* status);

/*
 * The averaged sparse weight update: the K messages are averaged exactly as
 * sparse_average does (learner order, one fp32 divide by K) and the weights
 * step against the average, w[j] <- w[j] - lr * avg_j (one fp32 rounding for
 * the product and one for the difference), at every index j that at least
 * one message carries; every other weight keeps its bits.  Learners
 * exchange compressed gradients and average them to update the weights
 * ("AdaComp ...", Proposed method; "Deep Gradient Compression", Appendix A:
 * the summed gradients optimise the model).  Unlike sparse_average, no dense
 * average is written: only the carried weights are read and rewritten.
 * lists, cap, counts, K, n: as for sparse_average.
 * lr      learning rate (finite; the caller folds any 1/K or sum convention in).
 * w       [n] fp32 weights, updated in place; any alignment.
 * Errors: as for sparse_average.
 */
int sparse_average_update(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K,
                          int64_t n, float lr, float* w, void* stream);

/* ------------------------------------------------------------- DCD-PSGD */

/*
 * One DCD-PSGD iteration of n_nodes nodes on a ring ("Communication
 * Compression for Decentralized Training", DCD-PSGD steps 1-3), every node
 * and every replica held once in xhat (each holder of a replica of node i
 * applies the same C(z_i), so all replicas of x_i equal x_i):
 *   x_half_i = w[0]*xhat_{i-1} + w[1]*xhat_i + w[2]*xhat_{i+1} - gamma*g_i
 *              (indices mod n_nodes, products and sums in that order, fp32);
 *   z_i      = x_half_i - xhat_i;
 *   C(z)_e   = z_e * (float)(1/keep_p) if word < round(keep_p * 2^32), else 0,
 *              word = Philox4x32-10(counter (e/4, i, t, e/2^34),
 *                                   key (seed low, seed high))[e mod 4];
 *   xhat_i  <- xhat_i + C(z_i).
 * All nodes read the models of iteration t.
 * w_ring  host [3] weights of the left neighbour, self and right neighbour.
 * xhat    [n_nodes][d] fp32 models, updated in place.
 * grad    [n_nodes][d] fp32 stochastic gradients, read only.
 * keep_p  in (0, 1];  t the iteration number (part of the counter).
 */
int dcd_step(int32_t n_nodes, int64_t d, const float* w_ring, float* xhat, const float* grad,
             float gamma, double keep_p, uint64_t seed, uint32_t t, void* stream);

/*
 * dcd_step for the nodes one process of several holds ("Communication
 * Compression for Decentralized Training", DCD-PSGD steps 1-3, with step 3's
 * message to the neighbours made explicit).  xhat is [rows][d]: row 0 is this
 * process's copy of node first_node - 1, rows 1 .. rows-2 its own nodes
 * first_node .. first_node + rows - 3, row rows-1 its copy of the node after
 * them (ring indices mod n are the caller's).  Every own row takes dcd_step's
 * update with its row neighbours (the copies are read, not written) and the
 * keep draw of its own node index; the result equals the own rows of a
 * dcd_step over the whole ring, bit for bit.
 * c_first / c_last  [cap] gcsgd_pair: every kept entry (C(z) bits and
 *         column index) of the first and of the last own row -- what the
 *         holders of copies of those nodes must add (dcd_copy_add).  The
 *         pairs of a list are not in index order; their indices are unique.
 * counts  device [2] int64: set by the call to the number of kept entries of
 *         each list; entries past cap are counted, not written (size cap to d
 *         to never drop one).
 * rows >= 3; d <= 2^32 (32-bit pair indices); other arguments as dcd_step.
 */
int dcd_step_rows(int32_t rows, int64_t d, int64_t first_node, const float* w_ring, float* xhat, const float* grad,
                  float gamma, double keep_p, uint64_t seed, uint32_t t, gcsgd_pair* c_first, gcsgd_pair* c_last,
                  int64_t cap, int64_t* counts, void* stream);

/*
 * A neighbour's copy of node j takes the C(z_j) the node added to itself
 * (DCD-PSGD step 3): x_row[idx] += val (fp32) for the first min(*count, cap)
 * pairs, whose indices are unique.  The owner adds +0 to every entry it did
 * not keep, which only changes a -0 into +0: with zero_pass != 0 the call
 * first adds +0 to every entry of x_row, which a copy needs once, before its
 * first update, if its starting model may hold -0 (after one iteration no
 * own row holds -0).  x_row [d] fp32, updated in place; count is a device
 * pointer (for example dcd_step_rows's counts, after the transfer).
 */
int dcd_copy_add(float* x_row, int64_t d, const gcsgd_pair* pairs, const int64_t* count, int64_t cap,
                 int32_t zero_pass, void* stream);

/*
 * One ECD-PSGD iteration t >= 1 of n_nodes nodes on a ring ("Communication
 * Compression for Decentralized Training", ECD-PSGD, equations (3)-(4)):
 *   z_j   = (1 - t/2) x_{t-1}^(j) + (t/2) x_t^(j)          (extrapolation)
 *   xt_j <- (1 - 2/t) xt_j + (2/t) C(z_j)                   (neighbours' estimate)
 *   x_{t+1}^(i) = w[0] xt_{i-1} + w[1] x_t^(i) + w[2] xt_{i+1} - gamma g_i
 * (reading: the D-PSGD step on the estimates, a node using its own model;
 * every holder of an estimate applies the same C(z_j), so xtilde holds one
 * estimate per node).  The coefficients are rounded once to fp32; products
 * and sums in the order written, fp32.  C is dcd_step's random
 * sparsification (same Philox counter, node and t).
 * x       [n_nodes][d] x_t, read only.
 * x_prev  [n_nodes][d] x_{t-1} on entry, x_{t+1} on return (the caller swaps
 *         x and x_prev for the next iteration).
 * xtilde  [n_nodes][d] the estimates, updated in place (start: the initial model).
 * t >= 1; other arguments as dcd_step.
 */
int ecd_step(int32_t n_nodes, int64_t d, const float* w_ring, const float* x, float* x_prev, float* xtilde,
             const float* grad, float gamma, double keep_p, uint64_t seed, uint32_t t, void* stream);

/* -------------------------------------------------------- wire formats */

/*
 * DGC's messages as byte streams ("Deep Gradient Compression", section 3.1:
 * a sent value travels as 32 bits and the unsent positions before it as a
 * 16-bit count).  Learner k's list (lists[k*cap ..], totals[k] entries, indices
 * strictly ascending) becomes streams[k*stream_cap ..]: one 6-byte record
 * per entry, little-endian [uint16 unsent positions since the previous
 * entry (or index 0)][fp32 value]; a gap of 65536 or more is split by escape
 * records (65535, +0.0f), each standing for 65535 zeros and one zero.
 * nbytes[k] = the stream's length, or -1 if it would exceed stream_cap or the
 * indices do not ascend (then nothing is written).  streams: 16-byte
 * aligned, stream_cap a multiple of 16.  Device arrays; one CTA per learner.
 */
int dgc_encode(const gcsgd_pair* lists, int64_t cap, const int64_t* totals, int32_t K, uint8_t* streams,
               int64_t stream_cap, int64_t* nbytes, void* stream);

/* The inverse: records back to (index, value) pairs, escapes dropped;
 * totals[k] = entries, or -1 if more than cap. */
int dgc_decode(const uint8_t* streams, int64_t stream_cap, const int64_t* nbytes, int32_t K, gcsgd_pair* lists,
               int64_t cap, int64_t* totals, void* stream);

/*
 * AdaComp's messages as byte streams ("AdaComp ...", Proposed method: one
 * scale per layer, the mean |g_max|, and each sent entry as sign + scale).
 * Per layer s, in order: [uint32 counts[k][s]][fp32 scales[k][s]], then one
 * uint32 (local index << 1 | sign bit, 1 = negative) per entry; the list
 * holds the layers one after another (as adacomp_compress writes it).
 * nbytes[k] = the length, or -1 if over stream_cap or if the counts add up
 * to more than cap (a learner that overflowed sends nothing).  Same
 * alignment rules.
 */
int adacomp_encode(const int64_t* seg_offsets, int32_t n_seg, const gcsgd_pair* lists, int64_t cap,
                   const int64_t* counts, const float* scales, int32_t K, uint8_t* streams, int64_t stream_cap,
                   int64_t* nbytes, void* stream);

/* The inverse: (global index, +-scale) pairs; totals[k] = entries, or -1 if
 * the stream is malformed or holds more than cap. */
int adacomp_decode(const int64_t* seg_offsets, int32_t n_seg, const uint8_t* streams, int64_t stream_cap,
                   const int64_t* nbytes, int32_t K, gcsgd_pair* lists, int64_t cap, int64_t* totals, void* stream);

/* ----------------------------------------------------- errors, tracing */

/* Message of the calling thread's last failure ("" if none).  Host. */
const char* gcsgd_last_error(void);

/* Library version: major*10000 + minor*100 + patch.  Host. */
int32_t gcsgd_version(void);

/* Number of kernels this process has launched through the library since
 * load or the last gcsgd_launch_count_reset().  Host. */
int64_t gcsgd_launch_count(void);
void gcsgd_launch_count_reset(void);

/* Per-kernel timing.  While enabled, every kernel launch is bracketed by
 * two CUDA events recorded on its own stream (a small extra cost).  Under
 * stream capture the events become external event nodes of the graph: each
 * replay records them again, and a read after the replays returns the last
 * replay's times.  The read hands the events back to the library, so a
 * graph replayed after it records into events that later launches may
 * reuse: read once, after the last replay.
 * gcsgd_trace_read waits for the recorded events, then writes up to `max`
 * entries (kernel name, launches, summed milliseconds) and the entry count
 * to *n_out; it clears the record.  Host functions. */
typedef struct {
    char name[48];
    int64_t launches;
    double total_ms;
} gcsgd_trace_entry;
int gcsgd_trace_enable(int32_t on);
int gcsgd_trace_read(gcsgd_trace_entry* entries, int32_t max, int32_t* n_out);
/* Restricts tracing to the launches of one kernel name (as reported by
 * gcsgd_trace_read), so that the events of the others do not sit between
 * kernels of a timed region; NULL or "" traces every kernel again.  The name
 * is copied.  Returns GCSGD_ERR_INVALID_ARG for a name of 48 bytes or more.
 * Host. */
int gcsgd_trace_only(const char* name);

#ifdef __cplusplus
}
#endif

#endif /* GCSGD_H */

// api.cu -- the C ABI of libgcsgd: argument checks, error text, launch
// counting and per-kernel event tracing.  All compute lives in dgc.cu,
// adacomp.cu, spavg.cu and dcd.cu.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "dgc.cuh"

namespace gcsgd {

size_t adacomp_workspace_bytes(const int64_t* off, const int32_t* lt, int S, int K, int64_t cap);
int adacomp_launch(const int64_t* off, int S, const int32_t* lt, int K, const float* dW, float* R, gcsgd_pair* out,
                   int64_t cap, int64_t* counts, float* scales, int64_t* totals, void* ws, size_t ws_bytes,
                   cudaStream_t stream, int defer, int pending);
int adacomp_settle_launch(const int64_t* off, int S, const int32_t* lt, int K, float* R, const gcsgd_pair* out,
                          int64_t cap, const int64_t* counts, const int64_t* totals, void* ws, size_t ws_bytes,
                          cudaStream_t stream);
int spavg_launch(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int K, int64_t n, float* out,
                 cudaStream_t stream, bool update, float lr);
size_t spavg_ws_bytes(int K, int64_t n);
int spavg_ws_launch(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int K, int64_t n, float* out,
                    void* ws, cudaStream_t stream, bool update, float lr);
int spavg_ws_status(const void* ws, int K, int64_t n, cudaStream_t stream, int32_t* status);
int dcd_launch(int n, int64_t d, const float* w, float* xhat, const float* grad, float gamma, double p, uint64_t seed,
               uint32_t t, cudaStream_t stream);
int dcd_rows_launch(int rows, int64_t d, int64_t first_node, const float* w, float* xhat, const float* grad,
                    float gamma, double p, uint64_t seed, uint32_t t, gcsgd_pair* c_first, gcsgd_pair* c_last,
                    int64_t cap, int64_t* counts, cudaStream_t stream);
int dcd_copy_add_launch(float* x, int64_t d, const gcsgd_pair* pairs, const int64_t* count, int64_t cap,
                        bool zero_pass, cudaStream_t stream);
int ecd_launch(int n, int64_t d, const float* w, const float* x, float* x_prev, float* xt, const float* grad,
               float gamma, double p, uint64_t seed, uint32_t t, cudaStream_t stream);
int wire_dgc_encode(const gcsgd_pair* lists, int64_t cap, const int64_t* totals, int K, uint8_t* streams,
                    int64_t stream_cap, int64_t* nbytes, cudaStream_t stream);
int wire_dgc_decode(const uint8_t* streams, int64_t stream_cap, const int64_t* nbytes, int K, gcsgd_pair* lists,
                    int64_t cap, int64_t* totals, cudaStream_t stream);
int wire_ada_encode(const int64_t* off, int S, const gcsgd_pair* lists, int64_t cap, const int64_t* counts,
                    const float* scales, int K, uint8_t* streams, int64_t stream_cap, int64_t* nbytes,
                    cudaStream_t stream);
int wire_ada_decode(const int64_t* off, int S, const uint8_t* streams, int64_t stream_cap, const int64_t* nbytes,
                    int K, gcsgd_pair* lists, int64_t cap, int64_t* totals, cudaStream_t stream);

// ------------------------------------------------------------------ errors

static thread_local char g_err[512] = "";

int set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int check_launch(const char* name) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(GCSGD_ERR_CUDA, "%s: launch failed: %s", name, cudaGetErrorString(e));
    return GCSGD_OK;
}

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

// ------------------------------------------------------- launches, tracing

static std::atomic<int64_t> g_launches{0};
static std::atomic<bool> g_trace{false};
static std::mutex g_trace_mu;
static std::string g_trace_name;  // only this kernel is traced when non-empty (guarded by g_trace_mu)
struct PendingEvent {
    std::string name;
    cudaEvent_t a, b;
};
static std::vector<PendingEvent> g_pending;
static std::vector<cudaEvent_t> g_free_events;

static cudaEvent_t take_event() {
    if (!g_free_events.empty()) {
        cudaEvent_t e = g_free_events.back();
        g_free_events.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// A trace event is recorded as an external event node when the stream is
// being captured into a CUDA graph (so each replay records it again and the
// replays can be timed from outside the graph), as a plain record otherwise;
// the external flag is refused on a stream that is not capturing.
static void record_trace_event(cudaEvent_t e, cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else
        cudaEventRecord(e, s);
}

// Any error left over from an earlier runtime call is cleared before the
// launch, so check_launch reports this launch's own.
LaunchScope::LaunchScope(const char* n, cudaStream_t s) : name(n), stream(s), slot(-1) {
    (void)cudaGetLastError();
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_trace.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!g_trace_name.empty() && g_trace_name != n) return;
    cudaEvent_t a = take_event(), b = take_event();
    if (!a || !b) {  // untraced launch; keep whichever event was made
        if (a) g_free_events.push_back(a);
        if (b) g_free_events.push_back(b);
        return;
    }
    record_trace_event(a, s);
    g_pending.push_back({std::string(n), a, b});
    slot = (int)g_pending.size() - 1;
}

LaunchScope::~LaunchScope() {
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (slot < (int)g_pending.size()) record_trace_event(g_pending[slot].b, stream);
}

// ------------------------------------------------------------ validation

static int check_layout(const char* fn, const int64_t* off, int32_t S) {
    if (!off) return set_error(GCSGD_ERR_INVALID_ARG, "%s: seg_offsets is NULL", fn);
    if (S < 1 || S > GCSGD_MAX_SEGMENTS)
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: n_seg = %d outside [1, %d]", fn, S, GCSGD_MAX_SEGMENTS);
    if (off[0] != 0) return set_error(GCSGD_ERR_INVALID_ARG, "%s: seg_offsets[0] must be 0", fn);
    for (int s = 0; s < S; ++s)
        if (off[s + 1] < off[s])
            return set_error(GCSGD_ERR_INVALID_ARG, "%s: seg_offsets decreases at segment %d", fn, s);
    if (off[S] >= (int64_t)1 << 32)
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: N = %lld does not fit uint32 indices", fn, (long long)off[S]);
    return GCSGD_OK;
}

static int check_ws(const char* fn, const void* ws, size_t bytes, size_t need) {
    if (bytes < need)
        return set_error(GCSGD_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, bytes, need);
    if (need > 0 && (!ws || ((uintptr_t)ws & 255)))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: workspace must be non-NULL and 256-byte aligned", fn);
    return GCSGD_OK;
}

static size_t dgc_ws_bytes(const int64_t* off, int32_t S, int32_t K, double density, double sample_frac) {
    dgc::HostPlan hp;
    dgc::host_plan(off, S, density, sample_frac, &hp);
    return dgc_workspace_layout(S, K, hp, sample_frac > 0.0, nullptr, nullptr);
}

}  // namespace gcsgd

using namespace gcsgd;

extern "C" {

const char* gcsgd_last_error(void) { return g_err; }

int32_t gcsgd_version(void) { return 100; }

int64_t gcsgd_launch_count(void) { return g_launches.load(); }

void gcsgd_launch_count_reset(void) { g_launches.store(0); }

int gcsgd_trace_enable(int32_t on) {
    g_trace.store(on != 0);
    return GCSGD_OK;
}

int gcsgd_trace_only(const char* name) {
    if (name && strlen(name) >= sizeof(((gcsgd_trace_entry*)nullptr)->name))
        return set_error(GCSGD_ERR_INVALID_ARG, "gcsgd_trace_only: name longer than 47 bytes");
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace_name = name ? name : "";
    return GCSGD_OK;
}

int gcsgd_trace_read(gcsgd_trace_entry* entries, int32_t max, int32_t* n_out) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    std::map<std::string, std::pair<int64_t, double>> agg;
    std::vector<std::string> order;
    int rc = GCSGD_OK;
    for (auto& p : g_pending) {
        float ms = 0.0f;
        if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) {
            rc = set_error(GCSGD_ERR_CUDA, "gcsgd_trace_read: event timing failed");
            (void)cudaGetLastError();  // not left pending for the next launch check
        }
        if (!agg.count(p.name)) order.push_back(p.name);
        agg[p.name].first += 1;
        agg[p.name].second += ms;
        g_free_events.push_back(p.a);
        g_free_events.push_back(p.b);
    }
    g_pending.clear();
    int32_t n = 0;
    for (auto& name : order) {
        if (entries && n < max) {
            memset(&entries[n], 0, sizeof(gcsgd_trace_entry));
            strncpy(entries[n].name, name.c_str(), sizeof(entries[n].name) - 1);
            entries[n].launches = agg[name].first;
            entries[n].total_ms = agg[name].second;
        }
        ++n;
    }
    if (n_out) *n_out = n;
    return rc;
}

int64_t gcsgd_dgc_k(double density, int64_t n) {
    if (n <= 0) return 0;
    return (int64_t)dgc_k_of(density, (uint64_t)n);
}

int gcsgd_dgc_workspace_size(const int64_t* seg_offsets, int32_t n_seg, int32_t K, double density, size_t* bytes) {
    int rc;
    if ((rc = check_layout("gcsgd_dgc_workspace_size", seg_offsets, n_seg))) return rc;
    if (K < 1 || !bytes) return set_error(GCSGD_ERR_INVALID_ARG, "gcsgd_dgc_workspace_size: K < 1 or bytes NULL");
    if (!(density > 0.0 && density <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "gcsgd_dgc_workspace_size: density %g outside (0, 1]", density);
    *bytes = dgc_ws_bytes(seg_offsets, n_seg, K, density, 0.0);
    return GCSGD_OK;
}

int gcsgd_dgc_sampled_workspace_size(const int64_t* seg_offsets, int32_t n_seg, int32_t K, double density,
                                     double sample_frac, size_t* bytes) {
    const char* fn = "gcsgd_dgc_sampled_workspace_size";
    int rc;
    if ((rc = check_layout(fn, seg_offsets, n_seg))) return rc;
    if (K < 1 || !bytes) return set_error(GCSGD_ERR_INVALID_ARG, "%s: K < 1 or bytes NULL", fn);
    if (!(density > 0.0 && density <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: density %g outside (0, 1]", fn, density);
    if (!(sample_frac > 0.0 && sample_frac <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: sample_frac %g outside (0, 1]", fn, sample_frac);
    *bytes = dgc_ws_bytes(seg_offsets, n_seg, K, density, sample_frac);
    return GCSGD_OK;
}

static int dgc_common(const char* fn, const int64_t* seg_offsets, int32_t n_seg, int32_t K, const float* grad,
                      float* u, float* v, double density, double sample_frac, float momentum, bool nesterov,
                      float clip_thr, int32_t clip_nodes, gcsgd_pair* out, int64_t cap, int64_t* counts,
                      int64_t* totals, void* workspace, size_t workspace_bytes, void* stream) {
    int rc;
    if ((rc = check_layout(fn, seg_offsets, n_seg))) return rc;
    if (K < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: K = %d < 1", fn, K);
    if (!(density > 0.0 && density <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: density %g outside (0, 1]", fn, density);
    if (!isfinite(momentum) || !isfinite(clip_thr))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: momentum and clip_thr must be finite", fn);
    if (clip_nodes < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: clip_nodes = %d < 1", fn, clip_nodes);
    if (cap < 0) return set_error(GCSGD_ERR_INVALID_ARG, "%s: cap < 0", fn);
    if (seg_offsets[n_seg] > 0 && (!grad || !u || !v))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: grad, u and v must be non-NULL", fn);
    if (!counts) return set_error(GCSGD_ERR_INVALID_ARG, "%s: counts is NULL", fn);
    if (cap > 0 && !out) return set_error(GCSGD_ERR_INVALID_ARG, "%s: out is NULL", fn);
    if ((rc = check_ws(fn, workspace, workspace_bytes, dgc_ws_bytes(seg_offsets, n_seg, K, density, sample_frac))))
        return rc;
    return dgc_launch(seg_offsets, n_seg, K, grad, u, v, density, sample_frac, momentum, nesterov, clip_thr,
                      clip_nodes, out, cap, counts, totals, workspace, workspace_bytes, (cudaStream_t)stream);
}

int dgc_compress(const int64_t* seg_offsets, int32_t n_seg, int32_t K, const float* grad, float* u, float* v,
                 double density, float momentum, float clip_thr, int32_t clip_nodes, gcsgd_pair* out, int64_t cap,
                 int64_t* counts, int64_t* totals, void* workspace, size_t workspace_bytes, void* stream) {
    return dgc_common("dgc_compress", seg_offsets, n_seg, K, grad, u, v, density, 0.0, momentum, false, clip_thr,
                      clip_nodes, out, cap, counts, totals, workspace, workspace_bytes, stream);
}

int dgc_compress_nesterov(const int64_t* seg_offsets, int32_t n_seg, int32_t K, const float* grad, float* u,
                          float* v, double density, float momentum, float clip_thr, int32_t clip_nodes,
                          gcsgd_pair* out, int64_t cap, int64_t* counts, int64_t* totals, void* workspace,
                          size_t workspace_bytes, void* stream) {
    return dgc_common("dgc_compress_nesterov", seg_offsets, n_seg, K, grad, u, v, density, 0.0, momentum, true,
                      clip_thr, clip_nodes, out, cap, counts, totals, workspace, workspace_bytes, stream);
}

int dgc_compress_sampled(const int64_t* seg_offsets, int32_t n_seg, int32_t K, const float* grad, float* u, float* v,
                         double density, double sample_frac, float momentum, float clip_thr, int32_t clip_nodes,
                         gcsgd_pair* out, int64_t cap, int64_t* counts, int64_t* totals, void* workspace,
                         size_t workspace_bytes, void* stream) {
    if (!(sample_frac > 0.0 && sample_frac <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "dgc_compress_sampled: sample_frac %g outside (0, 1]", sample_frac);
    return dgc_common("dgc_compress_sampled", seg_offsets, n_seg, K, grad, u, v, density, sample_frac, momentum,
                      false, clip_thr, clip_nodes, out, cap, counts, totals, workspace, workspace_bytes, stream);
}

int gcsgd_dgc_stats(const int64_t* seg_offsets, int32_t n_seg, int32_t K, double density, const void* workspace,
                    void* stream, gcsgd_dgc_stats_t* out) {
    int rc;
    if ((rc = check_layout("gcsgd_dgc_stats", seg_offsets, n_seg))) return rc;
    if (K < 1 || !workspace || !out || !(density > 0.0 && density <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "gcsgd_dgc_stats: bad argument");
    return dgc_collect_stats(seg_offsets, n_seg, K, density, workspace, (cudaStream_t)stream, out);
}

int gcsgd_adacomp_workspace_size(const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt, int32_t K,
                                 int64_t cap, size_t* bytes) {
    const char* fn = "gcsgd_adacomp_workspace_size";
    int rc;
    if ((rc = check_layout(fn, seg_offsets, n_seg))) return rc;
    if (!lt || K < 1 || cap < 0 || !bytes) return set_error(GCSGD_ERR_INVALID_ARG, "%s: bad argument", fn);
    for (int s = 0; s < n_seg; ++s)
        if (lt[s] < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: lt[%d] = %d < 1", fn, s, lt[s]);
    *bytes = adacomp_workspace_bytes(seg_offsets, lt, n_seg, K, cap);
    return GCSGD_OK;
}

static int adacomp_check(const char* fn, const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt, int32_t K,
                         const float* dW, float* residue, gcsgd_pair* out, int64_t cap, int64_t* counts,
                         float* scales, int64_t* totals, void* workspace, size_t workspace_bytes) {
    int rc;
    if ((rc = check_layout(fn, seg_offsets, n_seg))) return rc;
    if (!lt) return set_error(GCSGD_ERR_INVALID_ARG, "%s: lt is NULL", fn);
    for (int s = 0; s < n_seg; ++s)
        if (lt[s] < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: lt[%d] = %d < 1", fn, s, lt[s]);
    if (K < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: K = %d < 1", fn, K);
    if (cap < 0 || cap >= (int64_t)1 << 32) return set_error(GCSGD_ERR_INVALID_ARG, "%s: cap outside [0, 2^32)", fn);
    if (seg_offsets[n_seg] > 0 && (!dW || !residue))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: dW and residue must be non-NULL", fn);
    if (!counts || !scales || !totals)
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: counts, scales and totals must be non-NULL", fn);
    if (cap > 0 && !out) return set_error(GCSGD_ERR_INVALID_ARG, "%s: out is NULL", fn);
    return check_ws(fn, workspace, workspace_bytes, adacomp_workspace_bytes(seg_offsets, lt, n_seg, K, cap));
}

int adacomp_compress(const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt, int32_t K, const float* dW,
                     float* residue, gcsgd_pair* out, int64_t cap, int64_t* counts, float* scales, int64_t* totals,
                     void* workspace, size_t workspace_bytes, void* stream) {
    int rc = adacomp_check("adacomp_compress", seg_offsets, n_seg, lt, K, dW, residue, out, cap, counts, scales,
                           totals, workspace, workspace_bytes);
    if (rc) return rc;
    return adacomp_launch(seg_offsets, n_seg, lt, K, dW, residue, out, cap, counts, scales, totals, workspace,
                          workspace_bytes, (cudaStream_t)stream, 0, 0);
}

int adacomp_compress_deferred(const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt, int32_t K,
                              const float* dW, float* residue, gcsgd_pair* out, int64_t cap, int64_t* counts,
                              float* scales, int64_t* totals, int32_t pending, void* workspace,
                              size_t workspace_bytes, void* stream) {
    const char* fn = "adacomp_compress_deferred";
    int rc = adacomp_check(fn, seg_offsets, n_seg, lt, K, dW, residue, out, cap, counts, scales, totals, workspace,
                           workspace_bytes);
    if (rc) return rc;
    if (pending != 0 && pending != 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: pending = %d, not 0 or 1", fn, pending);
    return adacomp_launch(seg_offsets, n_seg, lt, K, dW, residue, out, cap, counts, scales, totals, workspace,
                          workspace_bytes, (cudaStream_t)stream, 1, pending);
}

int adacomp_settle(const int64_t* seg_offsets, int32_t n_seg, const int32_t* lt, int32_t K, float* residue,
                   const gcsgd_pair* out, int64_t cap, const int64_t* counts, const int64_t* totals, void* workspace,
                   size_t workspace_bytes, void* stream) {
    const char* fn = "adacomp_settle";
    int rc;
    if ((rc = check_layout(fn, seg_offsets, n_seg))) return rc;
    if (!lt) return set_error(GCSGD_ERR_INVALID_ARG, "%s: lt is NULL", fn);
    for (int s = 0; s < n_seg; ++s)
        if (lt[s] < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: lt[%d] = %d < 1", fn, s, lt[s]);
    if (K < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: K = %d < 1", fn, K);
    if (cap < 0 || cap >= (int64_t)1 << 32) return set_error(GCSGD_ERR_INVALID_ARG, "%s: cap outside [0, 2^32)", fn);
    if (seg_offsets[n_seg] > 0 && !residue) return set_error(GCSGD_ERR_INVALID_ARG, "%s: residue is NULL", fn);
    if (!counts || !totals) return set_error(GCSGD_ERR_INVALID_ARG, "%s: counts and totals must be non-NULL", fn);
    if (cap > 0 && !out) return set_error(GCSGD_ERR_INVALID_ARG, "%s: out is NULL", fn);
    if ((rc = check_ws(fn, workspace, workspace_bytes, adacomp_workspace_bytes(seg_offsets, lt, n_seg, K, cap))))
        return rc;
    return adacomp_settle_launch(seg_offsets, n_seg, lt, K, residue, out, cap, counts, totals, workspace,
                                 workspace_bytes, (cudaStream_t)stream);
}

static int check_average(const char* fn, const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K,
                         int64_t n, const float* out) {
    if (K < 1 || K > 512) return set_error(GCSGD_ERR_INVALID_ARG, "%s: K = %d outside [1, 512]", fn, K);
    if (n < 0 || n > ((int64_t)1 << 32)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: n outside [0, 2^32]", fn);
    if (cap < 0) return set_error(GCSGD_ERR_INVALID_ARG, "%s: cap < 0", fn);
    if (!counts || (n > 0 && !out) || (cap > 0 && !lists))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    return GCSGD_OK;
}

int sparse_average(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K, int64_t n, float* out,
                   void* stream) {
    int rc = check_average("sparse_average", lists, cap, counts, K, n, out);
    if (rc) return rc;
    return spavg_launch(lists, cap, counts, K, n, out, (cudaStream_t)stream, false, 0.0f);
}

int gcsgd_sparse_average_workspace_size(int32_t K, int64_t n, size_t* bytes) {
    if (K < 1 || K > 512) return set_error(GCSGD_ERR_INVALID_ARG, "gcsgd_sparse_average_workspace_size: K = %d outside [1, 512]", K);
    if (n < 0 || n > ((int64_t)1 << 32))
        return set_error(GCSGD_ERR_INVALID_ARG, "gcsgd_sparse_average_workspace_size: n outside [0, 2^32]");
    if (!bytes) return set_error(GCSGD_ERR_INVALID_ARG, "gcsgd_sparse_average_workspace_size: bytes is NULL");
    *bytes = spavg_ws_bytes(K, n);
    return GCSGD_OK;
}

int sparse_average_ws(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K, int64_t n, float* out,
                      void* workspace, size_t workspace_bytes, void* stream) {
    const char* fn = "sparse_average_ws";
    int rc = check_average(fn, lists, cap, counts, K, n, out);
    if (rc) return rc;
    if (n == 0) return GCSGD_OK;
    if (!workspace) return set_error(GCSGD_ERR_INVALID_ARG, "%s: workspace is NULL", fn);
    if (((uintptr_t)workspace & 255) != 0) return set_error(GCSGD_ERR_INVALID_ARG, "%s: workspace not 256-byte aligned", fn);
    if (workspace_bytes < spavg_ws_bytes(K, n))
        return set_error(GCSGD_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                         spavg_ws_bytes(K, n));
    return spavg_ws_launch(lists, cap, counts, K, n, out, workspace, (cudaStream_t)stream, false, 0.0f);
}

int sparse_average_update_ws(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K, int64_t n,
                             float lr, float* w, void* workspace, size_t workspace_bytes, void* stream) {
    const char* fn = "sparse_average_update_ws";
    int rc = check_average(fn, lists, cap, counts, K, n, w);
    if (rc) return rc;
    if (!isfinite(lr)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: lr is not finite", fn);
    if (n == 0) return GCSGD_OK;
    if (!workspace) return set_error(GCSGD_ERR_INVALID_ARG, "%s: workspace is NULL", fn);
    if (((uintptr_t)workspace & 255) != 0) return set_error(GCSGD_ERR_INVALID_ARG, "%s: workspace not 256-byte aligned", fn);
    if (workspace_bytes < spavg_ws_bytes(K, n))
        return set_error(GCSGD_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                         spavg_ws_bytes(K, n));
    return spavg_ws_launch(lists, cap, counts, K, n, w, workspace, (cudaStream_t)stream, true, lr);
}

int gcsgd_sparse_average_status(const void* workspace, int32_t K, int64_t n, void* stream, int32_t* status) {
    const char* fn = "gcsgd_sparse_average_status";
    if (K < 1 || K > 512) return set_error(GCSGD_ERR_INVALID_ARG, "%s: K = %d outside [1, 512]", fn, K);
    if (n < 1 || n > ((int64_t)1 << 32)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: n outside [1, 2^32]", fn);
    if (!workspace || !status) return set_error(GCSGD_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    return spavg_ws_status(workspace, K, n, (cudaStream_t)stream, status);
}

int sparse_average_update(const gcsgd_pair* lists, int64_t cap, const int64_t* counts, int32_t K, int64_t n,
                          float lr, float* w, void* stream) {
    int rc = check_average("sparse_average_update", lists, cap, counts, K, n, w);
    if (rc) return rc;
    if (!isfinite(lr)) return set_error(GCSGD_ERR_INVALID_ARG, "sparse_average_update: lr is not finite");
    return spavg_launch(lists, cap, counts, K, n, w, (cudaStream_t)stream, true, lr);
}

int dcd_step(int32_t n_nodes, int64_t d, const float* w_ring, float* xhat, const float* grad, float gamma,
             double keep_p, uint64_t seed, uint32_t t, void* stream) {
    const char* fn = "dcd_step";
    if (n_nodes < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: n_nodes < 1", fn);
    if (d < 0 || d >= ((int64_t)1 << 36)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: d outside [0, 2^36)", fn);
    if (!w_ring) return set_error(GCSGD_ERR_INVALID_ARG, "%s: w_ring is NULL", fn);
    if (d > 0 && (!xhat || !grad)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: xhat and grad must be non-NULL", fn);
    if (!(keep_p > 0.0 && keep_p <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: keep_p %g outside (0, 1]", fn, keep_p);
    if (!isfinite(gamma) || !isfinite(w_ring[0]) || !isfinite(w_ring[1]) || !isfinite(w_ring[2]))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: gamma and weights must be finite", fn);
    return dcd_launch(n_nodes, d, w_ring, xhat, grad, gamma, keep_p, seed, t, (cudaStream_t)stream);
}

int dcd_step_rows(int32_t rows, int64_t d, int64_t first_node, const float* w_ring, float* xhat, const float* grad,
                  float gamma, double keep_p, uint64_t seed, uint32_t t, gcsgd_pair* c_first, gcsgd_pair* c_last,
                  int64_t cap, int64_t* counts, void* stream) {
    const char* fn = "dcd_step_rows";
    if (rows < 3) return set_error(GCSGD_ERR_INVALID_ARG, "%s: rows = %d < 3 (two copies and an own node)", fn, rows);
    if (d < 0 || d > ((int64_t)1 << 32)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: d outside [0, 2^32]", fn);
    if (first_node < 0 || first_node + rows - 2 > ((int64_t)1 << 32))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: node indices outside [0, 2^32)", fn);
    if (!w_ring) return set_error(GCSGD_ERR_INVALID_ARG, "%s: w_ring is NULL", fn);
    if (!counts) return set_error(GCSGD_ERR_INVALID_ARG, "%s: counts is NULL", fn);
    if (d > 0 && (!xhat || !grad)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: xhat and grad must be non-NULL", fn);
    if (cap < 0 || (cap > 0 && (!c_first || !c_last)))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: cap < 0 or NULL lists", fn);
    if (!(keep_p > 0.0 && keep_p <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: keep_p %g outside (0, 1]", fn, keep_p);
    if (!isfinite(gamma) || !isfinite(w_ring[0]) || !isfinite(w_ring[1]) || !isfinite(w_ring[2]))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: gamma and weights must be finite", fn);
    return dcd_rows_launch(rows, d, first_node, w_ring, xhat, grad, gamma, keep_p, seed, t, c_first, c_last, cap,
                           counts, (cudaStream_t)stream);
}

int dcd_copy_add(float* x_row, int64_t d, const gcsgd_pair* pairs, const int64_t* count, int64_t cap,
                 int32_t zero_pass, void* stream) {
    const char* fn = "dcd_copy_add";
    if (d < 0 || d > ((int64_t)1 << 32)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: d outside [0, 2^32]", fn);
    if (cap < 0) return set_error(GCSGD_ERR_INVALID_ARG, "%s: cap < 0", fn);
    if (d > 0 && !x_row) return set_error(GCSGD_ERR_INVALID_ARG, "%s: x_row is NULL", fn);
    if (cap > 0 && (!pairs || !count)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: NULL list", fn);
    return dcd_copy_add_launch(x_row, d, pairs, count, cap, zero_pass != 0, (cudaStream_t)stream);
}

int ecd_step(int32_t n_nodes, int64_t d, const float* w_ring, const float* x, float* x_prev, float* xtilde,
             const float* grad, float gamma, double keep_p, uint64_t seed, uint32_t t, void* stream) {
    const char* fn = "ecd_step";
    if (n_nodes < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: n_nodes < 1", fn);
    if (d < 0 || d >= ((int64_t)1 << 36)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: d outside [0, 2^36)", fn);
    if (t < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: t = 0 (iterations count from 1)", fn);
    if (!w_ring) return set_error(GCSGD_ERR_INVALID_ARG, "%s: w_ring is NULL", fn);
    if (d > 0 && (!x || !x_prev || !xtilde || !grad))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: x, x_prev, xtilde and grad must be non-NULL", fn);
    if (!(keep_p > 0.0 && keep_p <= 1.0))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: keep_p %g outside (0, 1]", fn, keep_p);
    if (!isfinite(gamma)) return set_error(GCSGD_ERR_INVALID_ARG, "%s: gamma is not finite", fn);
    return ecd_launch(n_nodes, d, w_ring, x, x_prev, xtilde, grad, gamma, keep_p, seed, t, (cudaStream_t)stream);
}

static int check_streams(const char* fn, int32_t K, const void* streams, int64_t stream_cap, const void* a,
                         const void* b) {
    if (K < 1) return set_error(GCSGD_ERR_INVALID_ARG, "%s: K = %d < 1", fn, K);
    if (stream_cap < 0 || (stream_cap & 15))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: stream_cap must be a non-negative multiple of 16", fn);
    if (!streams || ((uintptr_t)streams & 15))
        return set_error(GCSGD_ERR_INVALID_ARG, "%s: streams must be non-NULL and 16-byte aligned", fn);
    if (!a || !b) return set_error(GCSGD_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    return GCSGD_OK;
}

int dgc_encode(const gcsgd_pair* lists, int64_t cap, const int64_t* totals, int32_t K, uint8_t* streams,
               int64_t stream_cap, int64_t* nbytes, void* stream) {
    int rc = check_streams("dgc_encode", K, streams, stream_cap, totals, nbytes);
    if (rc) return rc;
    if (cap < 0 || (cap > 0 && !lists)) return set_error(GCSGD_ERR_INVALID_ARG, "dgc_encode: bad lists or cap");
    return wire_dgc_encode(lists, cap, totals, K, streams, stream_cap, nbytes, (cudaStream_t)stream);
}

int dgc_decode(const uint8_t* streams, int64_t stream_cap, const int64_t* nbytes, int32_t K, gcsgd_pair* lists,
               int64_t cap, int64_t* totals, void* stream) {
    int rc = check_streams("dgc_decode", K, streams, stream_cap, nbytes, totals);
    if (rc) return rc;
    if (cap < 0 || (cap > 0 && !lists)) return set_error(GCSGD_ERR_INVALID_ARG, "dgc_decode: bad lists or cap");
    return wire_dgc_decode(streams, stream_cap, nbytes, K, lists, cap, totals, (cudaStream_t)stream);
}

int adacomp_encode(const int64_t* seg_offsets, int32_t n_seg, const gcsgd_pair* lists, int64_t cap,
                   const int64_t* counts, const float* scales, int32_t K, uint8_t* streams, int64_t stream_cap,
                   int64_t* nbytes, void* stream) {
    int rc;
    if ((rc = check_layout("adacomp_encode", seg_offsets, n_seg))) return rc;
    if ((rc = check_streams("adacomp_encode", K, streams, stream_cap, counts, nbytes))) return rc;
    if (!scales || cap < 0 || (cap > 0 && !lists))
        return set_error(GCSGD_ERR_INVALID_ARG, "adacomp_encode: bad lists, cap or scales");
    return wire_ada_encode(seg_offsets, n_seg, lists, cap, counts, scales, K, streams, stream_cap, nbytes,
                           (cudaStream_t)stream);
}

int adacomp_decode(const int64_t* seg_offsets, int32_t n_seg, const uint8_t* streams, int64_t stream_cap,
                   const int64_t* nbytes, int32_t K, gcsgd_pair* lists, int64_t cap, int64_t* totals, void* stream) {
    int rc;
    if ((rc = check_layout("adacomp_decode", seg_offsets, n_seg))) return rc;
    if ((rc = check_streams("adacomp_decode", K, streams, stream_cap, nbytes, totals))) return rc;
    if (cap < 0 || (cap > 0 && !lists)) return set_error(GCSGD_ERR_INVALID_ARG, "adacomp_decode: bad lists or cap");
    return wire_ada_decode(seg_offsets, n_seg, streams, stream_cap, nbytes, K, lists, cap, totals,
                           (cudaStream_t)stream);
}

}  // extern "C"

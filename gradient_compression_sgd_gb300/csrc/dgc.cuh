// dgc.cuh -- plan and workspace structures of the DGC kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gcsgd.h"

namespace gcsgd {
namespace dgc {

enum : uint32_t { kKindEmpty = 0, kKindRaw = 1, kKindPool = 2 };

// Per-segment plan, computed on the device by dgc_plan (48 bytes).
struct SegPlan {
    uint32_t off;       // first element of the segment within a learner
    uint32_t n;         // elements
    uint32_t k;         // entries sent
    uint32_t kind;      // kKindEmpty / kKindRaw (select from v') / kKindPool (candidates)
    uint32_t cap;       // candidate pool capacity
    uint32_t m;         // sample size (whole 64-value blocks)
    uint32_t a;         // rank of the hint (or of tau, sampled) within the sample
    uint32_t pool_off;  // first pool slot within a learner's pool
    uint32_t tile_off;  // first tile within a learner's tiles
    uint32_t ntiles;    // tiles of 4096 elements
    uint32_t out_off;   // first message slot within a learner's list
    uint32_t sampled;   // 1: sampled threshold (the hint is the selection threshold)
};

// Segment offsets passed by value to dgc_plan (no host-to-device copy).
template <int MAXS>
struct SegOffsets {
    uint32_t off[MAXS + 1];
};

// Segments with a candidate pool, from the host plan (passed by value; the
// sampling CTAs recompute each segment's sample size and rank).
template <int MAXS>
struct PoolList {
    uint32_t n_pool;
    uint16_t seg[MAXS];
    uint32_t koff[MAXS];  // sampled threshold, samples above kSampleMax: first key in the learner's spill region
    uint16_t order[MAXS];  // all segments by size, largest first (dgc_select's order)
};

struct HostPlan {
    uint64_t tiles_per_learner;
    uint64_t pool_per_learner;
    uint64_t out_per_learner;
    uint64_t pool_segments;
    uint64_t skeys_per_learner;  // sampled threshold: spilled sample keys per learner
};

struct DgcWorkspace {
    SegPlan* plan;
    float* clip_c;
    double* clip_part;
    uint16_t* order;  // segments by size, largest first
    uint32_t* hint;
    uint32_t* pool_cnt;
    uint2* tile_tab;
    uint2* pool;
    gcsgd_pair* msg;  // sampled threshold: per-tensor regions before packing
    uint32_t* skeys;  // sampled threshold: sample keys of pool segments above kSampleMax
};

int host_plan(const int64_t* off, int S, double density, double sample_frac, HostPlan* hp);

}  // namespace dgc

size_t dgc_workspace_layout(int S, int K, const dgc::HostPlan& hp, bool sampled, void* base, dgc::DgcWorkspace* w);

int dgc_collect_stats(const int64_t* off, int S, int K, double density, const void* ws, cudaStream_t stream,
                      gcsgd_dgc_stats_t* st);

int dgc_launch(const int64_t* off, int S, int K, const float* grad, float* u, float* v, double density,
               double sample_frac, float momentum, bool nesterov, float clip_thr, int clip_nodes, gcsgd_pair* out,
               int64_t cap, int64_t* counts, int64_t* totals, void* ws, size_t ws_bytes, cudaStream_t stream);

}  // namespace gcsgd

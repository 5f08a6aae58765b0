// plmla_internal.cuh -- definitions shared by the CUDA translation units of
// libplmla (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace plmla {

constexpr int kLatent = 512;      // compressed latent width (c_kv)
constexpr int kRope = 64;         // rope key width
constexpr int kRow = kLatent + kRope;
constexpr int kPageTokens = 1536; // token rows per MLA page
constexpr int kMaxLayers = 1024;  // layers of one mla_decode_layers step
constexpr int kTile = 128;        // KV tokens per decode tile; chunks are multiples of it
constexpr int kMaxReqs = 1024;
// query tokens per request: draft tokens of a verify step (4) up to a chunk of
// new tokens of an extend (prefill) step, causal among themselves
constexpr int kMaxNq = 256;
constexpr int kMaxPlanSplits = 32768; // chunks the device planner can schedule
constexpr int kChunksPerMember = 104; // default chunk budget per persistent CTA
// Planner cost of starting a segment, in 128-token tiles: a request's first
// chunk carries it (query load, first-tile softmax, the previous segment's
// partial-state epilogue).
constexpr int kSegmentCostTiles = 2;

constexpr int kMaxSms = 256;            // persistent CTAs per row group the schedule covers

struct PlanBuffers {
    int32_t *status;            // [1] device status word, reset to 0 by the plan kernel
    int32_t *indptr;            // [R + 1] per-request chunk counts, prefix-summed
    int64_t *chunk;             // [1] chunk length in tokens
    // persistent schedule (all null when only the split plan is wanted)
    int32_t *seg_count;         // [1] number of segments S
    int4 *segments;             // [S] (request, t0, t1, member)
    int32_t *seg_req_indptr;    // [R + 1] segments of request r: [r], [r + 1]
    int32_t *seg_member_indptr; // [members + 1] segments of member k: [k], [k + 1]
    int32_t *done;              // [n_done] finished-segment counters, zeroed by the plan kernel
    int32_t n_done;
    // FP8 decode: extra CTAs of the plan grid quantise the queries (null: none)
    const __nv_bfloat16 *q_nope; // [q_rows, 512]
    const __nv_bfloat16 *q_rope; // [q_rows, 64]
    uint8_t *q8;                 // [2, q_rows, 576] E4M3 hi and lo parts of q * 2^-e
    int32_t *qexp;               // [q_rows] e
    int32_t q_rows;
};

struct DecodeArgs {
    const __nv_bfloat16 *q_nope;   // [R*n_q, H, 512]
    const __nv_bfloat16 *q_rope;   // [R*n_q, H, 64]
    const void *slab;              // bf16 elements, or E4M3 bytes when fp8
    int64_t page_stride;           // elements
    int64_t num_pages;
    const int32_t *page_table;
    int64_t table_ld;
    const int32_t *seq_lens;
    int32_t num_reqs, n_q, num_heads;
    int32_t rows_per_req;          // n_q * H
    int32_t group_rows;            // rows owned by one CTA: 16, 32 or 64
    int32_t num_groups;            // rows_per_req / group_rows (teams)
    int32_t members;               // CTAs per team
    int32_t cluster;               // teams of one member per thread-block cluster (1, 2, 4)
    float scale_log2;              // softmax scale * log2(e)
    const int4 *segments;
    const int32_t *seg_member_indptr;
    const int32_t *seg_count;
    float *o_part;                 // [groups * S, group_rows, 512]
    float *lse_part;               // [groups * S, group_rows], natural log
    int32_t *status;               // device status word (0 = ok, else the failed wait)
    int32_t *done;                 // [groups * R] segments of (team, request) written
    // FP8 pages: slab holds E4M3 bytes (value = kv_scale * byte), the queries are
    // read as E4M3 codes q8 with per-row exponents qexp (written by the plan grid)
    int32_t fp8;
    float kv_scale;
    const uint8_t *q8;             // [2, R*n_q*H, 576]: hi plane, then lo plane
    const int32_t *qexp;           // [R*n_q*H]
};

// E4M3's largest finite value and the plan grid's query-quantising CTAs.
constexpr float kE4m3Max = 448.f;
constexpr int kQuantRowsPerCta = 64;

// Largest of 64, 32, 16 that divides `rows`, or 0.
inline int group_rows_for(int rows)
{
    if (rows % 64 == 0) return 64;
    if (rows % 32 == 0) return 32;
    if (rows % 16 == 0) return 16;
    return 0;
}

size_t plan_smem_bytes();
// uniform != 0: every request with history gets budget / (such requests) splits
// (the uniform baseline of the split rule), else the per-request rule.
cudaError_t launch_plan(const int32_t *seq_lens, int num_reqs, int budget, int members,
                        int uniform, PlanBuffers plan, cudaStream_t stream);
cudaError_t launch_decode_tc(const DecodeArgs &args, cudaStream_t stream);
// Teams of 64 query rows that share each KV item through a thread-block
// cluster (the KV tiles multicast by TMA): 4 or 2 (at most max_teams, and a
// divisor of the team count), or 1 for the E4M3 decode and narrower teams.
// kClusterTeams is the default of max_teams: pairs (measured on the 128-team
// extend, where clusters of 4 were slower than pairs).  The library uses
// clusters only for teams of few members (plmla_abi.cu).
constexpr int kClusterTeams = 2;
int decode_cluster_teams(int group_rows, int groups, bool fp8, int max_teams);
// Clusters of `cluster` (2 or 4) decode CTAs the current device holds at once
// (0 if it cannot say).
int decode_max_clusters(int cluster);
// The FP8 decode's query quantiser as a kernel of its own (rows of 576 values;
// q8 holds the hi plane, then the lo plane).
cudaError_t launch_quantize(const __nv_bfloat16 *q_nope, const __nv_bfloat16 *q_rope, int rows,
                            uint8_t *q8, int32_t *qexp, cudaStream_t stream);
// KV append (plmla_append.cu): status codes it writes for a bad row.
constexpr int32_t kStatusAppendPosition = 32;   // seq_lens[r] < n_new
constexpr int32_t kStatusAppendPage = 33;       // page ID outside [0, num_pages)
cudaError_t launch_append(const void *latent, const void *rope, void *slab, int64_t num_pages,
                          int64_t page_stride, const int32_t *table, int64_t table_ld,
                          const int32_t *seq_lens, int num_reqs, int n_new, int32_t *status,
                          cudaStream_t stream);
// The same into E4M3 pages: each value stored as the E4M3 code of x / kv_scale.
cudaError_t launch_append_fp8(const void *latent, const void *rope, void *slab,
                              int64_t num_pages, int64_t page_stride, float kv_scale,
                              const int32_t *table, int64_t table_ld, const int32_t *seq_lens,
                              int num_reqs, int n_new, int32_t *status, cudaStream_t stream);

// Shared by the query quantiser (plan grid) and the FP8 append: one E4M3 byte
// pair from two floats, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Merge of chunk partials + sigmoid gate.  Row rw of request r (rw = j*H + h)
// lives in group g = rw / group_rows at row rw % group_rows of the partials
// of segments [g*stride + indptr[r], g*stride + indptr[r + 1]), where stride is
// *seg_stride (or 0 when seg_stride is null).
// With `done` (and `status`) set, the combine is launched while the decode is
// still running and waits, per request, until done[team * R + r] counts `epoch`
// times the request's segments (the counters run on across the layers of one
// step: epoch = layer + 1); without it, it waits for the previous grid to finish.
cudaError_t launch_combine(const float *o_part, const float *lse_part, const int32_t *indptr,
                           const int32_t *seg_stride, int group_rows,
                           const __nv_bfloat16 *gate, int num_reqs, int n_q, int num_heads,
                           __nv_bfloat16 *out, float *lse, const int32_t *done,
                           int32_t *status, int epoch, cudaStream_t stream);

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace plmla

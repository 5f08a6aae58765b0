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
constexpr int kTile = 128;        // KV tokens per decode tile; chunks are multiples of it
constexpr int kMaxReqs = 1024;
constexpr int kMaxNq = 16;

// One unit of decode work: KV tokens [t0, t1) of request `req`, whose partial
// softmax state is stored at split id `split` (the request's splits are
// consecutive ids starting at split_indptr[req]).
struct __align__(16) WorkItem {
    int32_t req;
    int32_t split;
    int32_t t0;
    int32_t t1;
};

struct PlanBuffers {
    int32_t *status;   // [1] device status word, reset to 0 by the plan kernel
    int32_t *indptr;   // [R + 1]
    int64_t *chunk;    // [1]
    int32_t *count;    // [1] number of work items
    WorkItem *items;   // [max_items], longest request first
};

struct DecodeArgs {
    const __nv_bfloat16 *q_nope;   // [R*n_q, H, 512]
    const __nv_bfloat16 *q_rope;   // [R*n_q, H, 64]
    const __nv_bfloat16 *slab;
    int64_t page_stride;           // elements
    int64_t num_pages;
    const int32_t *page_table;
    int64_t table_ld;
    const int32_t *seq_lens;
    int32_t num_reqs, n_q, num_heads;
    int32_t rows_per_req;          // n_q * H
    int32_t group_rows;            // rows owned by one CTA: 16, 32 or 64
    int32_t num_groups;            // rows_per_req / group_rows
    float scale_log2;              // softmax scale * log2(e)
    const WorkItem *items;
    const int32_t *item_count;
    float *o_part;                 // [splits, rows_per_req, 512]
    float *lse_part;               // [splits, rows_per_req], natural log
    int32_t *status;               // device status word (0 = ok, else the failed wait)
};

// Largest of 64, 32, 16 that divides `rows`, or 0.
inline int group_rows_for(int rows)
{
    if (rows % 64 == 0) return 64;
    if (rows % 32 == 0) return 32;
    if (rows % 16 == 0) return 16;
    return 0;
}

cudaError_t launch_plan(const int32_t *seq_lens, int num_reqs, int budget, PlanBuffers plan,
                        cudaStream_t stream);
cudaError_t launch_decode_tc(const DecodeArgs &args, int max_items, cudaStream_t stream);
cudaError_t launch_combine(const float *o_part, const float *lse_part, const int32_t *indptr,
                           const __nv_bfloat16 *gate, int num_reqs, int n_q, int num_heads,
                           __nv_bfloat16 *out, float *lse, cudaStream_t stream);

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace plmla

// plmla_abi.cu -- host implementation of the C ABI declared in include/plmla.h.
//
// Validates arguments, lays out the caller's workspace, and enqueues the plan,
// split-decode and combine kernels on the caller's stream.  Nothing here
// allocates device memory, synchronises, or reads device data back.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>

#include "plmla.h"
#include "plmla_internal.cuh"

using namespace plmla;

namespace plmla {
// plmla_check.cu: the opt-in page-table check after a decode step.
cudaError_t launch_check_pages(const int32_t *seq_lens, int num_reqs, const int32_t *page_table,
                               int64_t table_ld, int64_t num_pages, int32_t *status,
                               cudaStream_t stream);
// plmla_combine.cu: merge of G ranks' gated partial outputs and LSEs.
cudaError_t launch_merge_partials(const __nv_bfloat16 *parts, const float *lse_parts, int world,
                                  int64_t rows, __nv_bfloat16 *out, float *lse,
                                  cudaStream_t stream);
// plmla_dcp.cu: one rank's page-table rows and history lengths.
cudaError_t launch_dcp_shard(const int32_t *table, int64_t ld, const int32_t *lens, int num_reqs,
                             int world, int rank, int32_t *table_out, int64_t out_ld,
                             int32_t *lens_out, cudaStream_t stream);
}  // namespace plmla

namespace {

constexpr size_t kAlign = 256;

// Page-table checks after each decode step: off unless PLMLA_CHECK_PAGES (or the
// general debug switch PLMLA_DEBUG) is set to something other than "0" in the
// environment, or mla_set_page_checks(1).
bool env_on(const char *name)
{
    const char *v = getenv(name);
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
}
int initial_page_checks() { return env_on("PLMLA_CHECK_PAGES") || env_on("PLMLA_DEBUG"); }
std::atomic<int> g_page_checks{initial_page_checks()};   // set and read from any host thread

// Split rule of the planner: 0 = per-request (default), 1 = uniform split counts;
// PLMLA_SPLIT_MODE=uniform in the environment selects 1 when the library loads.
int initial_split_mode()
{
    const char *v = getenv("PLMLA_SPLIT_MODE");
    return (v != nullptr && v[0] == 'u') ? 1 : 0;
}
std::atomic<int> g_split_mode{initial_split_mode()};

// Widest cluster of 64-row teams that share KV loads (1 = none, 2 or 4).
std::atomic<int> g_team_clusters{kClusterTeams};

// Teams share loads in clusters only when each has at most this many members:
// then every CTA streams long stretches of history alone (measured: the
// 128-team extend, one member per team, 2.6% faster in pairs; the 4-draft
// decode, 38 members per team, 1.6% slower).
constexpr int32_t kClusterMaxMembers = 8;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int current_sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return -1;
    if (dev < 64 && cached[dev] > 0)
        return cached[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    if (dev < 64)
        cached[dev] = sms;
    return sms;
}

bool shape_ok(int32_t num_reqs, int32_t n_q, int32_t num_heads)
{
    return num_reqs >= 1 && num_reqs <= kMaxReqs && n_q >= 1 && n_q <= kMaxNq &&
           num_heads >= 16 && num_heads <= 128 && num_heads % 16 == 0;
}

struct WorkspaceLayout {
    size_t status, indptr, chunk, seg_count, segments, seg_req, seg_member, done, o_part,
        lse_part, q8, qexp, total;
    int32_t max_segments;
};

struct Shape {
    int32_t rows_per_req, group_rows, groups, members, budget;
};

// Split budget and team layout for a decode shape (see mla_split_budget).
bool shape_for(int32_t num_reqs, int32_t n_q, int32_t num_heads, int32_t cta_budget,
               int32_t min_splits, Shape *out)
{
    if (!shape_ok(num_reqs, n_q, num_heads) || cta_budget < 0 || min_splits < 1)
        return false;
    Shape sh;
    sh.rows_per_req = n_q * num_heads;
    sh.group_rows = group_rows_for(sh.rows_per_req);
    if (sh.group_rows == 0)
        return false;
    sh.groups = sh.rows_per_req / sh.group_rows;
    const int64_t slots = cta_budget > 0 ? cta_budget : current_sm_count();
    if (slots <= 0)
        return false;
    sh.members = (int32_t)(slots / sh.groups > 0 ? slots / sh.groups : 1);
    if (sh.members > kMaxSms)   // the schedule keeps per-member tables of kMaxSms entries
        return false;
    int64_t budget = (int64_t)kChunksPerMember * sh.members;
    const int64_t wanted = (int64_t)num_reqs * min_splits;
    if (wanted > budget)
        budget = wanted;
    if (budget > kMaxPlanSplits)
        budget = kMaxPlanSplits;
    if (wanted > budget)
        return false;
    sh.budget = (int32_t)budget;
    *out = sh;
    return true;
}

// Workspace of one decode step; the FP8 decode adds the quantised queries.
WorkspaceLayout layout_for(int32_t num_reqs, const Shape &sh, bool fp8)
{
    WorkspaceLayout w;
    // a segment starts only where the request or the CTA changes along the
    // request-ordered chunks, so there are at most R + members - 1 of them
    const int32_t max_chunks = sh.budget > num_reqs ? sh.budget : num_reqs;
    const int32_t max_runs = num_reqs + sh.members;
    w.max_segments = max_chunks < max_runs ? max_chunks : max_runs;
    size_t off = 0;
    w.status = off;
    off = align_up(off + sizeof(int32_t));
    w.indptr = off;
    off = align_up(off + sizeof(int32_t) * (size_t)(num_reqs + 1));
    w.chunk = off;
    off = align_up(off + sizeof(int64_t));
    w.seg_count = off;
    off = align_up(off + sizeof(int32_t));
    w.segments = off;
    off = align_up(off + sizeof(int4) * (size_t)w.max_segments);
    w.seg_req = off;
    off = align_up(off + sizeof(int32_t) * (size_t)(num_reqs + 1));
    w.seg_member = off;
    off = align_up(off + sizeof(int32_t) * (size_t)(sh.members + 1));
    w.done = off;
    off = align_up(off + sizeof(int32_t) * (size_t)sh.groups * num_reqs);
    const size_t part_rows = (size_t)sh.groups * w.max_segments * sh.group_rows;
    w.o_part = off;
    off = align_up(off + sizeof(float) * part_rows * kLatent);
    w.lse_part = off;
    off = align_up(off + sizeof(float) * part_rows);
    const size_t q_rows = (size_t)num_reqs * sh.rows_per_req;
    w.q8 = off;
    off = fp8 ? align_up(off + 2 * (size_t)kRow * q_rows) : off;   // hi and lo planes
    w.qexp = off;
    off = fp8 ? align_up(off + sizeof(int32_t) * q_rows) : off;
    w.total = off;
    return w;
}

}  // namespace

extern "C" const char *mla_strerror(plmla_status status)
{
    switch (status) {
    case PLMLA_OK: return "PLMLA_OK";
    case PLMLA_INVALID_ARGUMENT: return "PLMLA_INVALID_ARGUMENT";
    case PLMLA_UNSUPPORTED: return "PLMLA_UNSUPPORTED";
    case PLMLA_WORKSPACE_TOO_SMALL: return "PLMLA_WORKSPACE_TOO_SMALL";
    case PLMLA_CUDA_ERROR: return "PLMLA_CUDA_ERROR";
    }
    return "PLMLA_UNKNOWN_STATUS";
}

extern "C" int32_t mla_split_budget(int32_t num_reqs, int32_t n_q, int32_t num_heads,
                                    int32_t cta_budget, int32_t min_splits_per_req)
{
    Shape sh;
    if (!shape_for(num_reqs, n_q, num_heads, cta_budget, min_splits_per_req, &sh))
        return -1;
    return sh.budget;
}

extern "C" size_t mla_workspace_size(int32_t num_reqs, int32_t n_q, int32_t num_heads,
                                     int32_t cta_budget, int32_t min_splits_per_req)
{
    Shape sh;
    if (!shape_for(num_reqs, n_q, num_heads, cta_budget, min_splits_per_req, &sh))
        return 0;
    return layout_for(num_reqs, sh, false).total;
}

extern "C" size_t mla_workspace_size_fp8(int32_t num_reqs, int32_t n_q, int32_t num_heads,
                                         int32_t cta_budget, int32_t min_splits_per_req)
{
    Shape sh;
    if (!shape_for(num_reqs, n_q, num_heads, cta_budget, min_splits_per_req, &sh))
        return 0;
    return layout_for(num_reqs, sh, true).total;
}

extern "C" plmla_status mla_plan_splits(const int32_t *seq_lens, int32_t num_reqs,
                                        int32_t split_budget, int32_t *split_indptr,
                                        int64_t *split_chunk, void *stream)
{
    if (seq_lens == nullptr || split_indptr == nullptr || split_chunk == nullptr ||
        num_reqs < 1 || num_reqs > kMaxReqs || split_budget < 1 || !aligned(seq_lens, 4) ||
        !aligned(split_indptr, 4) || !aligned(split_chunk, 8))
        return PLMLA_INVALID_ARGUMENT;
    if (split_budget > kMaxPlanSplits)
        return PLMLA_UNSUPPORTED;
    // Same kernel as inside mla_decode, without the persistent schedule.
    PlanBuffers plan = {};
    plan.indptr = split_indptr;
    plan.chunk = split_chunk;
    cudaError_t err = launch_plan(seq_lens, num_reqs, split_budget, 1,
                                  g_split_mode.load(std::memory_order_relaxed), plan,
                                  static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PLMLA_OK : PLMLA_CUDA_ERROR;
}

extern "C" void mla_set_page_checks(int32_t on)
{
    g_page_checks.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
}

extern "C" int32_t mla_get_page_checks(void)
{
    return g_page_checks.load(std::memory_order_relaxed);
}

extern "C" plmla_status mla_set_split_mode(int32_t mode)
{
    if (mode != 0 && mode != 1)
        return PLMLA_INVALID_ARGUMENT;
    g_split_mode.store(mode, std::memory_order_relaxed);
    return PLMLA_OK;
}

extern "C" int32_t mla_get_split_mode(void)
{
    return g_split_mode.load(std::memory_order_relaxed);
}

extern "C" plmla_status mla_set_team_clusters(int32_t max_teams)
{
    if (max_teams != 1 && max_teams != 2 && max_teams != 4)
        return PLMLA_INVALID_ARGUMENT;
    g_team_clusters.store(max_teams, std::memory_order_relaxed);
    return PLMLA_OK;
}

extern "C" int32_t mla_get_team_clusters(void)
{
    return g_team_clusters.load(std::memory_order_relaxed);
}

extern "C" plmla_status mla_merge_partials(const void *out_parts, const float *lse_parts,
                                           int32_t world, int64_t rows, void *out, float *lse,
                                           void *stream)
{
    if (out_parts == nullptr || lse_parts == nullptr || out == nullptr || world < 1 ||
        world > 4096 || rows < 0 || rows > (int64_t)kMaxReqs * kMaxNq * 128)
        return PLMLA_INVALID_ARGUMENT;
    if (!aligned(out_parts, 16) || !aligned(lse_parts, 4) || !aligned(out, 16) ||
        (lse != nullptr && !aligned(lse, 4)))
        return PLMLA_INVALID_ARGUMENT;
    cudaError_t err = launch_merge_partials(static_cast<const __nv_bfloat16 *>(out_parts),
                                            lse_parts, world, rows,
                                            static_cast<__nv_bfloat16 *>(out), lse,
                                            static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PLMLA_OK : PLMLA_CUDA_ERROR;
}

extern "C" plmla_status mla_dcp_shard(const int32_t *page_table, int64_t page_table_ld,
                                      const int32_t *seq_lens, int32_t num_reqs, int32_t world,
                                      int32_t rank, int32_t *table_out, int64_t table_out_ld,
                                      int32_t *lens_out, void *stream)
{
    if (page_table == nullptr || seq_lens == nullptr || table_out == nullptr ||
        lens_out == nullptr || num_reqs < 1 || num_reqs > kMaxReqs || world < 1 ||
        world > 4096 || rank < 0 || rank >= world || page_table_ld < 1 ||
        table_out_ld < (page_table_ld + world - 1) / world || !aligned(page_table, 4) ||
        !aligned(seq_lens, 4) || !aligned(table_out, 4) || !aligned(lens_out, 4))
        return PLMLA_INVALID_ARGUMENT;
    const cudaError_t err = launch_dcp_shard(page_table, page_table_ld, seq_lens, num_reqs, world,
                                             rank, table_out, table_out_ld, lens_out,
                                             static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PLMLA_OK : PLMLA_CUDA_ERROR;
}

extern "C" plmla_status mla_split_combine(const float *o_part, const float *lse_part,
                                          const int32_t *split_indptr, const void *gate,
                                          int32_t num_reqs, int32_t n_q_per_req,
                                          int32_t num_heads, void *out, float *lse,
                                          void *stream)
{
    if (o_part == nullptr || lse_part == nullptr || split_indptr == nullptr ||
        gate == nullptr || out == nullptr)
        return PLMLA_INVALID_ARGUMENT;
    if (!shape_ok(num_reqs, n_q_per_req, num_heads))
        return PLMLA_INVALID_ARGUMENT;
    if (!aligned(o_part, 16) || !aligned(lse_part, 4) || !aligned(gate, 8) ||
        !aligned(out, 8) || (lse != nullptr && !aligned(lse, 4)))
        return PLMLA_INVALID_ARGUMENT;
    cudaError_t err = launch_combine(o_part, lse_part, split_indptr, nullptr,
                                     n_q_per_req * num_heads,
                                     static_cast<const __nv_bfloat16 *>(gate), num_reqs,
                                     n_q_per_req, num_heads, static_cast<__nv_bfloat16 *>(out),
                                     lse, nullptr, nullptr, 1, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PLMLA_OK : PLMLA_CUDA_ERROR;
}

namespace {
cudaError_t record(void *event, cudaStream_t stream)
{
    return event != nullptr ? cudaEventRecord(static_cast<cudaEvent_t>(event), stream)
                            : cudaSuccess;
}
}  // namespace

namespace {

// Cache format of one decode call: bf16 pages, or E4M3 pages with their scale.
struct KvFormat {
    bool fp8;
    float kv_scale;
};

// One decode step of `layers` attention layers that share the page table and
// the history lengths (one paged layout for every layer's pool): one split plan
// for the step, then per layer the split decode and the gated combine.  The
// finished-segment counters are zeroed by the plan and count on across the
// layers, so layer l's combine waits for (l + 1) times each request's segments;
// layer l's decode starts only after layer l - 1's combine (programmatic
// launch), so the partial states can be reused.  Layer-indexed arrays are host
// arrays of device pointers; kv_scale (E4M3 pages) is a host array too.
plmla_status decode_layers_impl(int32_t layers, const void *const *q_nope_absorbed,
                                const void *const *q_rope, const void *const *gate,
                                const void *const *slab_base, const float *kv_scale,
                                int64_t num_pages, int64_t page_stride_elems,
                                const int32_t *page_table, int64_t page_table_ld,
                                const int32_t *seq_lens, int32_t num_reqs, int32_t n_q_per_req,
                                int32_t num_heads, float scale, void *const *out,
                                float *const *lse, void *workspace, size_t workspace_bytes,
                                int32_t cta_budget, int32_t min_splits_per_req, void *stream,
                                const plmla_stage_events *events, bool fp8)
{
    if (layers < 1 || layers > kMaxLayers || q_nope_absorbed == nullptr || q_rope == nullptr ||
        gate == nullptr || slab_base == nullptr || out == nullptr ||
        (fp8 && kv_scale == nullptr) || (events != nullptr && layers != 1))
        return PLMLA_INVALID_ARGUMENT;
    if (page_table == nullptr || seq_lens == nullptr || workspace == nullptr)
        return PLMLA_INVALID_ARGUMENT;
    if (!shape_ok(num_reqs, n_q_per_req, num_heads) || min_splits_per_req < 1 || cta_budget < 0)
        return PLMLA_INVALID_ARGUMENT;
    // page strides are multiples of 16 bytes (a TMA requirement): 8 bf16 or 16 E4M3 elements
    if (num_pages < 1 || num_pages > INT32_MAX || page_table_ld < 1 ||
        page_stride_elems < (int64_t)kPageTokens * kRow ||
        page_stride_elems % (fp8 ? 16 : 8) != 0)
        return PLMLA_INVALID_ARGUMENT;
    if (!(isfinite(scale)))
        return PLMLA_INVALID_ARGUMENT;
    if (!aligned(workspace, kAlign) || !aligned(page_table, 4) || !aligned(seq_lens, 4))
        return PLMLA_INVALID_ARGUMENT;
    for (int32_t l = 0; l < layers; ++l) {
        if (q_nope_absorbed[l] == nullptr || q_rope[l] == nullptr || gate[l] == nullptr ||
            slab_base[l] == nullptr || out[l] == nullptr)
            return PLMLA_INVALID_ARGUMENT;
        if (fp8 && !(isfinite(kv_scale[l]) && kv_scale[l] > 0.f))
            return PLMLA_INVALID_ARGUMENT;
        if (!aligned(q_nope_absorbed[l], 16) || !aligned(q_rope[l], 16) ||
            !aligned(gate[l], 16) || !aligned(slab_base[l], 16) || !aligned(out[l], 16) ||
            (lse != nullptr && lse[l] != nullptr && !aligned(lse[l], 4)))
            return PLMLA_INVALID_ARGUMENT;
    }

    Shape sh;
    if (!shape_for(num_reqs, n_q_per_req, num_heads, cta_budget, min_splits_per_req, &sh))
        return (cta_budget == 0 && current_sm_count() <= 0) ? PLMLA_CUDA_ERROR
                                                            : PLMLA_UNSUPPORTED;
    const WorkspaceLayout w = layout_for(num_reqs, sh, fp8);
    if (workspace_bytes < w.total)
        return PLMLA_WORKSPACE_TOO_SMALL;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    PlanBuffers plan = {};
    plan.status = reinterpret_cast<int32_t *>(ws + w.status);
    plan.indptr = reinterpret_cast<int32_t *>(ws + w.indptr);
    plan.chunk = reinterpret_cast<int64_t *>(ws + w.chunk);
    plan.seg_count = reinterpret_cast<int32_t *>(ws + w.seg_count);
    plan.segments = reinterpret_cast<int4 *>(ws + w.segments);
    plan.seg_req_indptr = reinterpret_cast<int32_t *>(ws + w.seg_req);
    plan.seg_member_indptr = reinterpret_cast<int32_t *>(ws + w.seg_member);
    plan.done = reinterpret_cast<int32_t *>(ws + w.done);
    plan.n_done = sh.groups * num_reqs;
    // E4M3 pages: the plan grid also quantises the first layer's queries
    plan.q_nope = static_cast<const __nv_bfloat16 *>(q_nope_absorbed[0]);
    plan.q_rope = static_cast<const __nv_bfloat16 *>(q_rope[0]);
    plan.q8 = fp8 ? reinterpret_cast<uint8_t *>(ws + w.q8) : nullptr;
    plan.qexp = fp8 ? reinterpret_cast<int32_t *>(ws + w.qexp) : nullptr;
    plan.q_rows = num_reqs * sh.rows_per_req;
    float *o_part = reinterpret_cast<float *>(ws + w.o_part);
    float *lse_part = reinterpret_cast<float *>(ws + w.lse_part);

    const plmla_stage_events none = {nullptr, nullptr, nullptr, nullptr};
    const plmla_stage_events &ev = events != nullptr ? *events : none;
    if (record(ev.plan_begin, s) != cudaSuccess)
        return PLMLA_CUDA_ERROR;
    cudaError_t err = launch_plan(seq_lens, num_reqs, sh.budget, sh.members,
                                  g_split_mode.load(std::memory_order_relaxed), plan, s);
    if (err != cudaSuccess)
        return PLMLA_CUDA_ERROR;

    DecodeArgs a = {};
    a.page_stride = page_stride_elems;
    a.num_pages = num_pages;
    a.page_table = page_table;
    a.table_ld = page_table_ld;
    a.seq_lens = seq_lens;
    a.num_reqs = num_reqs;
    a.n_q = n_q_per_req;
    a.num_heads = num_heads;
    a.rows_per_req = sh.rows_per_req;
    a.group_rows = sh.group_rows;
    a.num_groups = sh.groups;
    a.members = sh.members;
    // teams of a member in one cluster share its KV items (multicast), when the
    // device holds every cluster of the grid at once; the arithmetic, and so
    // every output bit, is the same either way
    a.cluster = sh.members <= kClusterMaxMembers
                    ? decode_cluster_teams(sh.group_rows, sh.groups, fp8,
                                           g_team_clusters.load(std::memory_order_relaxed))
                    : 1;
    while (a.cluster > 1 &&
           (int64_t)sh.members * (sh.groups / a.cluster) > decode_max_clusters(a.cluster))
        a.cluster /= 2;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.segments = plan.segments;
    a.seg_member_indptr = plan.seg_member_indptr;
    a.seg_count = plan.seg_count;
    a.o_part = o_part;
    a.lse_part = lse_part;
    a.status = plan.status;
    a.done = plan.done;
    a.fp8 = fp8 ? 1 : 0;
    a.q8 = plan.q8;
    a.qexp = plan.qexp;
    for (int32_t l = 0; l < layers; ++l) {
        if (fp8 && l > 0 &&
            launch_quantize(static_cast<const __nv_bfloat16 *>(q_nope_absorbed[l]),
                            static_cast<const __nv_bfloat16 *>(q_rope[l]), plan.q_rows, plan.q8,
                            plan.qexp, s) != cudaSuccess)
            return PLMLA_CUDA_ERROR;
        if (record(ev.decode_begin, s) != cudaSuccess)
            return PLMLA_CUDA_ERROR;
        a.q_nope = static_cast<const __nv_bfloat16 *>(q_nope_absorbed[l]);
        a.q_rope = static_cast<const __nv_bfloat16 *>(q_rope[l]);
        a.slab = slab_base[l];
        a.kv_scale = fp8 ? kv_scale[l] : 1.f;
        err = launch_decode_tc(a, s);
        if (err != cudaSuccess || record(ev.combine_begin, s) != cudaSuccess)
            return PLMLA_CUDA_ERROR;
        err = launch_combine(o_part, lse_part, plan.seg_req_indptr, plan.seg_count,
                             sh.group_rows, static_cast<const __nv_bfloat16 *>(gate[l]), num_reqs,
                             n_q_per_req, num_heads, static_cast<__nv_bfloat16 *>(out[l]),
                             lse != nullptr ? lse[l] : nullptr, plan.done, plan.status, l + 1,
                             s);
        if (err != cudaSuccess || record(ev.combine_end, s) != cudaSuccess)
            return PLMLA_CUDA_ERROR;
    }
    if (g_page_checks.load(std::memory_order_relaxed) != 0 &&
        launch_check_pages(seq_lens, num_reqs, page_table, page_table_ld,
                                            num_pages, plan.status, s) != cudaSuccess)
        return PLMLA_CUDA_ERROR;
    return PLMLA_OK;
}

// One layer (mla_decode, mla_decode_fp8 and their _ex forms).
plmla_status decode_impl(const void *q_nope_absorbed, const void *q_rope, const void *gate,
                         const void *slab_base, int64_t num_pages, int64_t page_stride_elems,
                         const int32_t *page_table, int64_t page_table_ld,
                         const int32_t *seq_lens, int32_t num_reqs, int32_t n_q_per_req,
                         int32_t num_heads, float scale, void *out, float *lse, void *workspace,
                         size_t workspace_bytes, int32_t cta_budget, int32_t min_splits_per_req,
                         void *stream, const plmla_stage_events *events, const KvFormat &fmt)
{
    void *out_l[1] = {out};
    float *lse_l[1] = {lse};
    const float kv_l[1] = {fmt.kv_scale};
    return decode_layers_impl(1, &q_nope_absorbed, &q_rope, &gate, &slab_base,
                              fmt.fp8 ? kv_l : nullptr, num_pages, page_stride_elems, page_table,
                              page_table_ld, seq_lens, num_reqs, n_q_per_req, num_heads, scale,
                              out_l, lse_l, workspace, workspace_bytes, cta_budget,
                              min_splits_per_req, stream, events, fmt.fp8);
}

}  // namespace

extern "C" plmla_status mla_decode_layers(int32_t num_layers, const void *const *q_nope_absorbed,
                                          const void *const *q_rope, const void *const *gate,
                                          const void *const *slab_base, int64_t num_pages,
                                          int64_t page_stride_elems, const int32_t *page_table,
                                          int64_t page_table_ld, const int32_t *seq_lens,
                                          int32_t num_reqs, int32_t n_q_per_req,
                                          int32_t num_heads, float scale, void *const *out,
                                          float *const *lse, void *workspace,
                                          size_t workspace_bytes, int32_t cta_budget,
                                          int32_t min_splits_per_req, void *stream)
{
    return decode_layers_impl(num_layers, q_nope_absorbed, q_rope, gate, slab_base, nullptr,
                              num_pages, page_stride_elems, page_table, page_table_ld, seq_lens,
                              num_reqs, n_q_per_req, num_heads, scale, out, lse, workspace,
                              workspace_bytes, cta_budget, min_splits_per_req, stream, nullptr,
                              false);
}

extern "C" plmla_status mla_decode_layers_fp8(
    int32_t num_layers, const void *const *q_nope_absorbed, const void *const *q_rope,
    const void *const *gate, const void *const *slab_base, const float *kv_scale,
    int64_t num_pages, int64_t page_stride_elems, const int32_t *page_table,
    int64_t page_table_ld, const int32_t *seq_lens, int32_t num_reqs, int32_t n_q_per_req,
    int32_t num_heads, float scale, void *const *out, float *const *lse, void *workspace,
    size_t workspace_bytes, int32_t cta_budget, int32_t min_splits_per_req, void *stream)
{
    if (kv_scale == nullptr)
        return PLMLA_INVALID_ARGUMENT;
    return decode_layers_impl(num_layers, q_nope_absorbed, q_rope, gate, slab_base, kv_scale,
                              num_pages, page_stride_elems, page_table, page_table_ld, seq_lens,
                              num_reqs, n_q_per_req, num_heads, scale, out, lse, workspace,
                              workspace_bytes, cta_budget, min_splits_per_req, stream, nullptr,
                              true);
}

extern "C" plmla_status mla_decode_ex(const void *q_nope_absorbed, const void *q_rope,
                                      const void *gate, const void *slab_base,
                                      int64_t num_pages, int64_t page_stride_elems,
                                      const int32_t *page_table, int64_t page_table_ld,
                                      const int32_t *seq_lens, int32_t num_reqs,
                                      int32_t n_q_per_req, int32_t num_heads, float scale,
                                      void *out, float *lse, void *workspace,
                                      size_t workspace_bytes, int32_t cta_budget,
                                      int32_t min_splits_per_req, void *stream,
                                      const plmla_stage_events *events)
{
    return decode_impl(q_nope_absorbed, q_rope, gate, slab_base, num_pages, page_stride_elems,
                       page_table, page_table_ld, seq_lens, num_reqs, n_q_per_req, num_heads,
                       scale, out, lse, workspace, workspace_bytes, cta_budget,
                       min_splits_per_req, stream, events, KvFormat{false, 1.f});
}

extern "C" plmla_status mla_decode_fp8_ex(const void *q_nope_absorbed, const void *q_rope,
                                          const void *gate, const void *slab_base,
                                          int64_t num_pages, int64_t page_stride_elems,
                                          float kv_scale, const int32_t *page_table,
                                          int64_t page_table_ld, const int32_t *seq_lens,
                                          int32_t num_reqs, int32_t n_q_per_req,
                                          int32_t num_heads, float scale, void *out, float *lse,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t cta_budget, int32_t min_splits_per_req,
                                          void *stream, const plmla_stage_events *events)
{
    return decode_impl(q_nope_absorbed, q_rope, gate, slab_base, num_pages, page_stride_elems,
                       page_table, page_table_ld, seq_lens, num_reqs, n_q_per_req, num_heads,
                       scale, out, lse, workspace, workspace_bytes, cta_budget,
                       min_splits_per_req, stream, events, KvFormat{true, kv_scale});
}

extern "C" plmla_status mla_decode_fp8(const void *q_nope_absorbed, const void *q_rope,
                                       const void *gate, const void *slab_base,
                                       int64_t num_pages, int64_t page_stride_elems,
                                       float kv_scale, const int32_t *page_table,
                                       int64_t page_table_ld, const int32_t *seq_lens,
                                       int32_t num_reqs, int32_t n_q_per_req, int32_t num_heads,
                                       float scale, void *out, float *lse, void *workspace,
                                       size_t workspace_bytes, int32_t cta_budget,
                                       int32_t min_splits_per_req, void *stream)
{
    return mla_decode_fp8_ex(q_nope_absorbed, q_rope, gate, slab_base, num_pages,
                             page_stride_elems, kv_scale, page_table, page_table_ld, seq_lens,
                             num_reqs, n_q_per_req, num_heads, scale, out, lse, workspace,
                             workspace_bytes, cta_budget, min_splits_per_req, stream, nullptr);
}

extern "C" plmla_status mla_decode(const void *q_nope_absorbed, const void *q_rope,
                                   const void *gate, const void *slab_base, int64_t num_pages,
                                   int64_t page_stride_elems, const int32_t *page_table,
                                   int64_t page_table_ld, const int32_t *seq_lens,
                                   int32_t num_reqs, int32_t n_q_per_req, int32_t num_heads,
                                   float scale, void *out, float *lse, void *workspace,
                                   size_t workspace_bytes, int32_t cta_budget,
                                   int32_t min_splits_per_req, void *stream)
{
    return mla_decode_ex(q_nope_absorbed, q_rope, gate, slab_base, num_pages, page_stride_elems,
                         page_table, page_table_ld, seq_lens, num_reqs, n_q_per_req, num_heads,
                         scale, out, lse, workspace, workspace_bytes, cta_budget,
                         min_splits_per_req, stream, nullptr);
}

extern "C" plmla_status mla_kv_append(const void *latent_new, const void *rope_new,
                                      void *slab_base, int64_t num_pages,
                                      int64_t page_stride_elems, const int32_t *page_table,
                                      int64_t page_table_ld, const int32_t *seq_lens,
                                      int32_t num_reqs, int32_t n_new, int32_t *status,
                                      void *stream)
{
    if (num_reqs < 1 || n_new < 0)
        return PLMLA_INVALID_ARGUMENT;
    if (n_new == 0)
        return PLMLA_OK;
    if (latent_new == nullptr || rope_new == nullptr || slab_base == nullptr ||
        page_table == nullptr || seq_lens == nullptr)
        return PLMLA_INVALID_ARGUMENT;
    if (!aligned(latent_new, 16) || !aligned(rope_new, 16) || !aligned(slab_base, 16) ||
        !aligned(page_table, 4) || !aligned(seq_lens, 4) ||
        (status != nullptr && !aligned(status, 4)))
        return PLMLA_INVALID_ARGUMENT;
    if (num_pages < 1 || page_table_ld < 1 || page_stride_elems < (int64_t)kPageTokens * kRow ||
        page_stride_elems % 8 != 0)
        return PLMLA_INVALID_ARGUMENT;
    const cudaError_t err = launch_append(latent_new, rope_new, slab_base, num_pages,
                                          page_stride_elems, page_table, page_table_ld, seq_lens,
                                          num_reqs, n_new, status,
                                          static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PLMLA_OK : PLMLA_CUDA_ERROR;
}

extern "C" plmla_status mla_kv_append_fp8(const void *latent_new, const void *rope_new,
                                          void *slab_base, int64_t num_pages,
                                          int64_t page_stride_elems, float kv_scale,
                                          const int32_t *page_table, int64_t page_table_ld,
                                          const int32_t *seq_lens, int32_t num_reqs,
                                          int32_t n_new, int32_t *status, void *stream)
{
    if (num_reqs < 1 || n_new < 0)
        return PLMLA_INVALID_ARGUMENT;
    if (n_new == 0)
        return PLMLA_OK;
    if (latent_new == nullptr || rope_new == nullptr || slab_base == nullptr ||
        page_table == nullptr || seq_lens == nullptr)
        return PLMLA_INVALID_ARGUMENT;
    if (!aligned(latent_new, 16) || !aligned(rope_new, 16) || !aligned(slab_base, 16) ||
        !aligned(page_table, 4) || !aligned(seq_lens, 4) ||
        (status != nullptr && !aligned(status, 4)))
        return PLMLA_INVALID_ARGUMENT;
    if (num_pages < 1 || page_table_ld < 1 || page_stride_elems < (int64_t)kPageTokens * kRow ||
        page_stride_elems % 16 != 0 || !(isfinite(kv_scale) && kv_scale > 0.f))
        return PLMLA_INVALID_ARGUMENT;
    const cudaError_t err = launch_append_fp8(latent_new, rope_new, slab_base, num_pages,
                                              page_stride_elems, kv_scale, page_table,
                                              page_table_ld, seq_lens, num_reqs, n_new, status,
                                              static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PLMLA_OK : PLMLA_CUDA_ERROR;
}

extern "C" plmla_status mla_quantize_queries_fp8(const void *q_nope_absorbed, const void *q_rope,
                                                 int64_t rows, void *q8, int32_t *qexp,
                                                 void *stream)
{
    if (rows < 0 || rows > (int64_t)1 << 30)
        return PLMLA_INVALID_ARGUMENT;
    if (rows == 0)
        return PLMLA_OK;
    if (q_nope_absorbed == nullptr || q_rope == nullptr || q8 == nullptr || qexp == nullptr ||
        !aligned(q_nope_absorbed, 16) || !aligned(q_rope, 16) || !aligned(q8, 16) ||
        !aligned(qexp, 4))
        return PLMLA_INVALID_ARGUMENT;
    const cudaError_t err = launch_quantize(static_cast<const __nv_bfloat16 *>(q_nope_absorbed),
                                            static_cast<const __nv_bfloat16 *>(q_rope), (int)rows,
                                            static_cast<uint8_t *>(q8), qexp,
                                            static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PLMLA_OK : PLMLA_CUDA_ERROR;
}

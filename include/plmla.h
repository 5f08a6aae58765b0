/*
 * plmla.h -- C ABI of libplmla: gated Multi-head Latent Attention (MLA) decode
 * over a flat, paged KV pool, for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operation (web pages, cited by title and section):
 *   [K3]  TokenSpeed, Day-0 Kimi K3 post (lightseek.org/blog/tokenspeed-kimi-k3.html):
 *         architecture list (Gated MLA: full softmax attention over stored
 *         compressed latent KV, with a gate on its output); section "A Generic,
 *         Unified Flat KV Layout for Cache Management" (one page pool, 1,536-token
 *         MLA pages, one global page ID per page across slabs); section "Gluon
 *         kernels on AMD GPUs", Gated MLA decode paragraph (split the history
 *         along the context, merge partial softmax states in a second kernel).
 *   [AX]  "331 output tokens/s per GPU on AgentX: Serving Kimi K3 on GB300 with
 *         TokenSpeed": section "Balance MLA work with per-request KV splitting"
 *         (Figure 4: chunk length from total history and parallelism budget,
 *         more splits for longer requests, CUDA-graph compatible); section
 *         "Kernel fusion and overlap complete the decode path" (sigmoid output
 *         gating); section "Use TP4 selectively ..." (four drafted tokens are
 *         verified per request).
 *   [IX]  "AgentX - InferenceXv3: Does CUDA Moat Hold up in Agentic Inferencing?":
 *         the ROCm AITER section (64-bit MLA offsets for pools above 2 GB); the
 *         TensorRT-LLM section (honour block-index strides); the SGLang section
 *         (context length as a runtime scalar, no per-step device-to-host sync).
 *
 * Fixed shape of the latent cache: every token row holds 576 bf16 values, the
 * 512-wide compressed latent c_kv followed by the 64-wide rope key; a page holds
 * 1,536 consecutive token rows.
 *
 * Conventions shared by every entry point:
 *   - bf16 means IEEE bfloat16 (2 bytes); pointers to bf16 data are void*.
 *   - Every pointer is a DEVICE pointer of the current CUDA device, owned by
 *     the caller.  The library never allocates, frees or synchronises on these
 *     calls; all work is enqueued on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and no call reads device data back to the host, so the
 *     calls can be captured in a CUDA graph.
 *   - Errors are returned as plmla_status; nothing is thrown across the ABI.
 *     PLMLA_CUDA_ERROR means a launch failed: cudaGetLastError() has the cause.
 *     Arguments are checked on the host before anything is enqueued.
 */
#ifndef PLMLA_H
#define PLMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum plmla_status {
    PLMLA_OK = 0,
    PLMLA_INVALID_ARGUMENT = 1,     /* null or misaligned pointer, bad size or count */
    PLMLA_UNSUPPORTED = 2,          /* valid request outside what the kernels cover */
    PLMLA_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < mla_workspace_size(...) */
    PLMLA_CUDA_ERROR = 4,           /* a CUDA runtime/driver call failed */
} plmla_status;

enum {
    PLMLA_LATENT_DIM = 512,  /* c_kv width */
    PLMLA_ROPE_DIM = 64,     /* rope key width */
    PLMLA_ROW_DIM = 576,     /* elements per token row in a page */
    PLMLA_PAGE_TOKENS = 1536 /* token rows per MLA page [K3, flat KV layout] */
};

/* Human-readable name of a status code (static storage, never NULL). */
const char *mla_strerror(plmla_status status);

/*
 * mla_split_budget -- the chunk budget mla_decode plans with: how many KV chunks
 * the per-request split rule of [AX, Figure 4] may create for this shape, taken
 * from the machine as [IX] asks (a hard-coded budget starved a large GPU).  Pure
 * host arithmetic.
 *
 *   group_rows = the largest of 64, 32, 16 dividing n_q * num_heads (query rows
 *                one CTA owns); row_groups = n_q * num_heads / group_rows
 *   slots      = cta_budget, or the current device's SM count when 0
 *   members    = max(1, floor(slots / row_groups))   (persistent CTAs per group)
 *   budget     = max(104 * members, num_reqs * min_splits_per_req), at most 32768
 *
 * mla_decode runs row_groups x members persistent CTAs; each takes a contiguous
 * run of the chunks holding an equal share of their cost (128-token tiles plus a
 * charge for starting a request).  The schedule depends only on seq_lens and
 * this shape, so repeated calls on the same inputs give the same bits, in any
 * process.  Returns the budget, or -1 for invalid arguments, members above 256,
 * num_reqs * min_splits_per_req above 32768, or no CUDA device when
 * cta_budget == 0.
 */
int32_t mla_split_budget(int32_t num_reqs, int32_t n_q, int32_t num_heads, int32_t cta_budget,
                         int32_t min_splits_per_req);

/*
 * mla_workspace_size -- bytes of device workspace mla_decode needs for this
 * shape: the plan and schedule arrays, and fp32 partial outputs and partial
 * log-sum-exps for at most row_groups x (num_reqs + members) segments.  0 on
 * invalid arguments.  Pure host arithmetic.
 */
size_t mla_workspace_size(int32_t num_reqs, int32_t n_q, int32_t num_heads, int32_t cta_budget,
                          int32_t min_splits_per_req);

/*
 * mla_set_page_checks -- process-wide switch (not part of the method) for a
 * check of the page table after every mla_decode / mla_decode_fp8 step: one
 * extra kernel reads each request's table entries 0 .. ceil(L / 1536) - 1 and
 * sets the step's status word to 40 if any lies outside [0, num_pages), or to 41
 * if a history needs more than page_table_ld columns.  Off by
 * default; the environment variable PLMLA_CHECK_PAGES or PLMLA_DEBUG (any value
 * but "0") turns it on when the library loads.  mla_get_page_checks returns the setting.
 */
void mla_set_page_checks(int32_t on);
int32_t mla_get_page_checks(void);

/*
 * mla_set_split_mode -- process-wide choice of the split rule that mla_decode,
 * mla_decode_fp8 and mla_plan_splits plan with (not part of the method's
 * default; it exists to reproduce the comparison of [AX, Figure 5]):
 *   0  per-request split counts [AX, Figure 4] (the default, see mla_plan_splits)
 *   1  uniform split counts, the baseline that figure compares against: every
 *      request with history gets su = split_budget / (requests with history)
 *      chunks (at least 1), so request r's chunk is ceil(L_r / su) rounded up to
 *      a multiple of 128 and splits_r = ceil(L_r / that chunk)
 * The environment variable PLMLA_SPLIT_MODE=uniform selects 1 when the library
 * loads.  The decode's outputs agree under both rules within rounding (the
 * partial states merge to the same softmax); under 1, mla_plan_splits writes
 * split_chunk = 0 (the chunk differs per request).  Returns
 * PLMLA_INVALID_ARGUMENT for another mode.  mla_get_split_mode returns it.
 */
plmla_status mla_set_split_mode(int32_t mode);
int32_t mla_get_split_mode(void);

/*
 * mla_set_team_clusters -- process-wide widest thread-block cluster of query-row
 * teams (1, 2 or 4; default 2) for the bf16 decode.  When a step has two or more
 * teams of 64 rows (n_q * num_heads a multiple of 128) and each team has at most
 * 8 persistent CTAs (members; e.g. a chunked extend of 128 tokens at 64 heads),
 * the CTAs that hold the same member's work for 2 or 4 teams run as one cluster
 * and every KV tile is read from memory once and multicast by TMA into all of
 * them, instead of once per team.  The width used is the largest of 4, 2 within
 * max_teams that divides the team count and whose clusters the device holds at
 * once (all of the grid's CTAs must be resident together), else 1.  Only the loads change: the outputs
 * are bit-identical for every setting.  PLMLA_INVALID_ARGUMENT for another value.
 * mla_get_team_clusters returns the setting.
 */
plmla_status mla_set_team_clusters(int32_t max_teams);
int32_t mla_get_team_clusters(void);

/*
 * mla_plan_splits -- per-request KV split plan [AX, Figure 4], on the device.
 *
 *   chunk     = ceil(sum_r L_r / split_budget) rounded up to a multiple of 128,
 *               then grown by 128 while sum_r ceil(L_r / chunk) > split_budget,
 *               never past the longest history (then every request has 1 chunk)
 *   splits_r  = ceil(L_r / chunk)  (0 when L_r = 0)
 *   split s of request r covers tokens [s*chunk, min((s+1)*chunk, L_r)).
 *
 * seq_lens      [num_reqs] int32, device, L_r >= 0;  num_reqs 1 .. 1024.
 * split_budget  1 .. 32768 (PLMLA_UNSUPPORTED above).
 * split_indptr  [num_reqs + 1] int32, device, written: exclusive prefix sum of
 *               splits_r in request order (split ids of request r are
 *               split_indptr[r] .. split_indptr[r+1]-1).
 * split_chunk   [1] int64, device, written: chunk.
 * Runs as one kernel; never reads device data on the host.
 */
plmla_status mla_plan_splits(const int32_t *seq_lens, int32_t num_reqs, int32_t split_budget,
                             int32_t *split_indptr, int64_t *split_chunk, void *stream);

/*
 * mla_decode -- one gated-MLA decode step for a batch of requests [K3, AX].
 *
 * For request r, draft token j < n_q_per_req and head h, with
 * L' = seq_lens[r] - (n_q_per_req - 1 - j) (drafts see each other causally) and
 * token row x_t = slab_base[page_table[r*page_table_ld + t/1536]*page_stride_elems
 *                           + (t % 1536)*576 + 0..575]:
 *
 *   s_t = scale * (q_nope_absorbed[r,j,h,:] . x_t[0:512] + q_rope[r,j,h,:] . x_t[512:576])
 *   o   = sum_{t < L'} softmax(s)_t * x_t[0:512]
 *   lse = ln sum_{t < L'} exp(s_t)                      (natural log, before the gate)
 *   out = bf16_rn( sigmoid(gate[r,j,h,:]) * o )        (elementwise gate)
 *
 * Rows with L' <= 0 give out = 0 and lse = -inf.  Token rows at t >= L' and
 * pages the table does not reach are never used, whatever they hold (NaN safe).
 *
 * q_nope_absorbed  bf16 [num_reqs*n_q_per_req, num_heads, 512], contiguous
 * q_rope           bf16 [num_reqs*n_q_per_req, num_heads, 64], contiguous
 * gate             bf16 [num_reqs*n_q_per_req, num_heads, 512] gate logits
 * slab_base        bf16 pool of num_pages pages, 16-byte aligned
 * num_pages        pages in the pool (1 .. 2^31-1); offsets are computed in 64 bits
 * page_stride_elems elements from one page to the next, >= 1536*576, multiple of 8
 * page_table       int32, row r at page_table + r*page_table_ld (row stride honoured)
 * page_table_ld    >= ceil(max_r L_r / 1536)
 * seq_lens         int32 [num_reqs], device (history incl. the n_q drafts)
 * num_reqs         1 .. 1024;  n_q_per_req 1 .. 256 (draft tokens of a verify step,
 *                  or a chunk of new tokens: a chunked extend / prefill over the
 *                  pages, whose KV rows were appended before the call);
 *                  num_heads multiple of 16, <= 128
 * scale            softmax scale (1/sqrt(192) for a 128+64 head)
 * out              bf16 [num_reqs*n_q_per_req, num_heads, 512], written
 * lse              fp32 [num_reqs*n_q_per_req, num_heads], written (may be NULL)
 * workspace        device scratch of workspace_bytes >= mla_workspace_size(...),
 *                  256-byte aligned; contents on entry are irrelevant.  After the
 *                  step, its first 4 bytes hold the device status word (int32):
 *                  0 = ok; 40 = a used page ID out of range, 41 = a history
 *                  longer than the table row (both with page checks on); another nonzero value = a pipeline wait inside the decode kernel
 *                  gave up after its time bound and the outputs are invalid
 *                  (the kernel never traps or spins forever)
 * cta_budget       concurrent CTA slots for the split budget (0 = SM count)
 * min_splits_per_req  >= 1; raises the budget so that equal-length requests get
 *                  at least this many chunks each
 * stream           cudaStream_t
 *
 * Enqueues: plan kernel (split plan + persistent schedule) -> split-decode
 * kernel (one persistent CTA per SM and row group; with two or more 64-row
 * groups, in 2-CTA clusters that share each KV tile's load, see
 * mla_set_team_clusters) -> combine/gate kernel.
 * Page IDs are not checked on the hot path: an ID outside [0, num_pages) is a
 * tensor-map coordinate out of range, which the TMA unit reads as zeros (no
 * fault), so the affected rows come out wrong.  With page checks on (see
 * mla_set_page_checks) a small kernel after the step checks every table entry
 * a history uses and writes status 40 into the status word if one is out of
 * range.
 */
plmla_status mla_decode(const void *q_nope_absorbed, const void *q_rope, const void *gate,
                        const void *slab_base, int64_t num_pages, int64_t page_stride_elems,
                        const int32_t *page_table, int64_t page_table_ld,
                        const int32_t *seq_lens, int32_t num_reqs, int32_t n_q_per_req,
                        int32_t num_heads, float scale, void *out, float *lse, void *workspace,
                        size_t workspace_bytes, int32_t cta_budget, int32_t min_splits_per_req,
                        void *stream);

/*
 * mla_decode_layers -- the decode step of num_layers MLA layers at once [K3,
 * section "A Generic, Unified Flat KV Layout for Cache Management": the pool's
 * slabs each hold one MLA page per global page ID, so every layer reads the
 * same page table with its own slab base].  Each layer l computes exactly what
 * mla_decode computes with q_nope_absorbed[l], q_rope[l], gate[l], slab_base[l],
 * out[l] and lse[l] (bit for bit: same plan, same kernels); the split plan and
 * persistent schedule, which depend only on seq_lens and the shape, are made
 * once for the step instead of once per layer.
 *
 * num_layers       1 .. 1024
 * q_nope_absorbed, q_rope, gate, slab_base, out
 *                  HOST arrays of num_layers device pointers, each as in
 *                  mla_decode (the slabs share num_pages and page_stride_elems)
 * lse              NULL (no LSE for any layer), or a host array of num_layers
 *                  device pointers, each NULL or as in mla_decode
 * other arguments  as in mla_decode; the workspace is mla_workspace_size(...)
 *                  bytes, the same as for one layer, and its status word covers
 *                  the whole step (a failed layer makes the later ones stop)
 *
 * Enqueues: plan kernel -> for each layer: split-decode kernel -> combine/gate
 * kernel (each layer's decode starts once the previous layer's combine is
 * done).  The host arrays are read during the call only.
 */
plmla_status mla_decode_layers(int32_t num_layers, const void *const *q_nope_absorbed,
                               const void *const *q_rope, const void *const *gate,
                               const void *const *slab_base, int64_t num_pages,
                               int64_t page_stride_elems, const int32_t *page_table,
                               int64_t page_table_ld, const int32_t *seq_lens, int32_t num_reqs,
                               int32_t n_q_per_req, int32_t num_heads, float scale,
                               void *const *out, float *const *lse, void *workspace,
                               size_t workspace_bytes, int32_t cta_budget,
                               int32_t min_splits_per_req, void *stream);

/* Size of the scratch array compiled into the library for mla_decode_static_scratch. */
#define PLMLA_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * mla_decode_static_scratch -- mla_decode for callers that cannot allocate
 * device memory.  The source pages have no counterpart to this entry point: it
 * exists for the library's callers, not for the method.
 *
 * Who needs it: a serving engine that reserved nearly all device memory for its
 * KV page pool up front and allows no later cudaMalloc; a plugin running inside
 * a framework that owns the device allocator; a latency-critical loop that
 * cannot afford the device synchronisation cudaMalloc/cudaFree may cause.
 *
 * Arguments, results and errors are those of mla_decode without `workspace`
 * and `workspace_bytes`.  The workspace is a PLMLA_STATIC_SCRATCH_BYTES (32 MiB)
 * array compiled into the library; every GPU that loads the library holds it
 * until the process exits.  A shape whose mla_workspace_size(...) exceeds that
 * size is rejected with PLMLA_WORKSPACE_TOO_SMALL before anything is enqueued.
 * The call allocates nothing (no cudaMalloc/cudaFree, no allocating library
 * routine).
 *
 * The first call on each device, made with that device current, looks up the
 * array's device address once (cudaGetSymbolAddress) and caches it; make that
 * first call before any stream capture.  The cached address is only valid for
 * the CUDA context that was current then: do not keep using the library after
 * cudaDeviceReset or after the primary context was destroyed and re-created.
 * All calls on a device share the one array, which keeps the previous call's
 * contents (nothing in it needs to start at zero: each call's plan kernel
 * rewrites every entry the later kernels read).  Calls whose executions overlap
 * on the GPU -- on different streams, or from several host threads -- race on
 * the array and corrupt each other's results: serialise them, e.g. on one
 * stream.  The step's device status word (see mla_decode's `workspace`) lives
 * in the array; mla_static_scratch_status reads it.
 */
plmla_status mla_decode_static_scratch(const void *q_nope_absorbed, const void *q_rope,
                                       const void *gate, const void *slab_base,
                                       int64_t num_pages, int64_t page_stride_elems,
                                       const int32_t *page_table, int64_t page_table_ld,
                                       const int32_t *seq_lens, int32_t num_reqs,
                                       int32_t n_q_per_req, int32_t num_heads, float scale,
                                       void *out, float *lse, int32_t cta_budget,
                                       int32_t min_splits_per_req, void *stream);

/*
 * mla_static_scratch_status -- enqueue, on `stream`, a copy of the device status
 * word of the last mla_decode_static_scratch step on the current device into
 * `status_out` (4 bytes; device memory or pinned host memory, or pageable host
 * memory, for which the copy completes before the call returns).  Values as for
 * mla_decode's workspace status word: 0 = ok, 40 / 41 = page check failures,
 * another nonzero value = a bounded pipeline wait gave up and the outputs are
 * invalid.  Allocates nothing.  Like the decode entry point, the first call on a
 * device looks up the array's address; call it after the step on the same
 * stream.  Returns PLMLA_INVALID_ARGUMENT for a null or misaligned
 * status_out, PLMLA_CUDA_ERROR if the copy cannot be enqueued.
 */
plmla_status mla_static_scratch_status(int32_t *status_out, void *stream);

/*
 * Optional stage events for mla_decode_ex: each non-NULL member is a cudaEvent_t
 * that is recorded on `stream` at that point of the step (before the plan
 * kernel, before the split-decode kernel, before the combine kernel, after the
 * combine kernel).  Used to time each kernel inside a measured step; recording
 * adds no device work.
 */
typedef struct plmla_stage_events {
    void *plan_begin;
    void *decode_begin;
    void *combine_begin;
    void *combine_end;
} plmla_stage_events;

/*
 * mla_decode_ex -- mla_decode with optional stage events (NULL = none).  Same
 * arguments, results and errors as mla_decode.
 */
plmla_status mla_decode_ex(const void *q_nope_absorbed, const void *q_rope, const void *gate,
                           const void *slab_base, int64_t num_pages, int64_t page_stride_elems,
                           const int32_t *page_table, int64_t page_table_ld,
                           const int32_t *seq_lens, int32_t num_reqs, int32_t n_q_per_req,
                           int32_t num_heads, float scale, void *out, float *lse,
                           void *workspace, size_t workspace_bytes, int32_t cta_budget,
                           int32_t min_splits_per_req, void *stream,
                           const plmla_stage_events *events);

/*
 * mla_workspace_size_fp8 -- workspace bytes of mla_decode_fp8 for a shape: that
 * of mla_decode plus the two-part FP8 queries (num_reqs*n_q*num_heads rows of
 * 2 x 576 bytes and one int32 exponent each).  0 for an unsupported shape.
 */
size_t mla_workspace_size_fp8(int32_t num_reqs, int32_t n_q, int32_t num_heads,
                              int32_t cta_budget, int32_t min_splits_per_req);

/*
 * mla_decode_fp8 -- mla_decode over FP8 pages, the deployment's cache format
 * ("FP8 target/drafter KV cache": TokenSpeed AgentX post, memory-budget
 * paragraph; float8_e4m3fn, as named in the AMD notes of the AgentX -
 * InferenceXv3 report).
 *
 * Every slab element is one OCP E4M3 byte (bias 7, 3 mantissa bits, no
 * infinity, S.1111.111 = NaN) and stands for kv_scale * its value; a token row
 * is 576 bytes (512 latent, then 64 rope).  The operation is mla_decode's with
 * x_t = kv_scale * decoded bytes and the bf16 query as given:
 *
 *   s_t = scale * (q_nope_absorbed . x_t[0:512] + q_rope . x_t[512:576])
 *   o   = sum_{t < L'} softmax(s)_t * x_t[0:512]
 *   lse = ln sum_{t < L'} exp(s_t);   out = bf16_rn(sigmoid(gate) * o)
 *
 * How it is computed: the FP8 tensor-core MMA multiplies E4M3 by E4M3, so each
 * query row q = [q_nope | q_rope] is scaled to v = q * 2^-e (e the smallest
 * integer >= -126 with max|q| * 2^-e <= 448; 0 for an all-zero row) and enters
 * as two E4M3 parts, hi = E4M3(v) and lo = E4M3(v - hi), each multiplied with
 * the cache in its own MMA into one fp32 accumulator.  hi + lo equals v
 * exactly where |v| >= 2^-2 and is within 2^-10 below it, so the scores are
 * those of the bf16 query up to that.  The probabilities enter the value MMA
 * as E4M3 (relative rounding <= 2^-4 in E4M3's normal range, <= 2^-10 absolute
 * below it, with the row's largest probability scaled to >= 16); their sum for
 * the normaliser and lse stays fp32.
 *
 * Arguments as mla_decode, except:
 * slab_base          E4M3 bytes, 16-byte aligned
 * page_stride_elems  bytes from one page to the next, >= 1536*576, multiple of 16
 * kv_scale           finite, > 0
 * workspace_bytes    >= mla_workspace_size_fp8(...)
 * Enqueues: plan kernel (its grid also quantises the queries) -> split-decode
 * kernel -> combine/gate kernel.  Returns PLMLA_INVALID_ARGUMENT also for a
 * non-finite or non-positive kv_scale.
 */
plmla_status mla_decode_fp8(const void *q_nope_absorbed, const void *q_rope, const void *gate,
                            const void *slab_base, int64_t num_pages, int64_t page_stride_elems,
                            float kv_scale, const int32_t *page_table, int64_t page_table_ld,
                            const int32_t *seq_lens, int32_t num_reqs, int32_t n_q_per_req,
                            int32_t num_heads, float scale, void *out, float *lse,
                            void *workspace, size_t workspace_bytes, int32_t cta_budget,
                            int32_t min_splits_per_req, void *stream);

/*
 * mla_decode_layers_fp8 -- mla_decode_layers over E4M3 pages: layer l computes
 * what mla_decode_fp8 computes with kv_scale[l] (a HOST array of num_layers
 * scales) and the layer's pointers; the workspace is mla_workspace_size_fp8(...)
 * bytes.  The first layer's queries are quantised by the plan grid, each later
 * layer's by a quantiser kernel before its decode.
 */
plmla_status mla_decode_layers_fp8(int32_t num_layers, const void *const *q_nope_absorbed,
                                   const void *const *q_rope, const void *const *gate,
                                   const void *const *slab_base, const float *kv_scale,
                                   int64_t num_pages, int64_t page_stride_elems,
                                   const int32_t *page_table, int64_t page_table_ld,
                                   const int32_t *seq_lens, int32_t num_reqs,
                                   int32_t n_q_per_req, int32_t num_heads, float scale,
                                   void *const *out, float *const *lse, void *workspace,
                                   size_t workspace_bytes, int32_t cta_budget,
                                   int32_t min_splits_per_req, void *stream);

/*
 * mla_quantize_queries_fp8 -- the query step of mla_decode_fp8 on its own: rows
 * of [q_nope | q_rope] (512 + 64 bf16 values, row i at q_nope + 512 i and
 * q_rope + 64 i) become two E4M3 parts of v = q * 2^-e (round to nearest even):
 * q8[576 i .. 576 i + 575] = hi = E4M3(v) and q8[576 (rows + i) ..] = lo =
 * E4M3(v - hi), and qexp[i] = e, the smallest integer >= -126 with
 * max|q| * 2^-e <= 448 (0 for an all-zero row).  q8 holds 2 * rows * 576 bytes
 * (the hi plane, then the lo plane).  q_nope, q_rope and q8 16-byte aligned;
 * rows 0 .. 2^30.  Asynchronous on `stream`.
 */
plmla_status mla_quantize_queries_fp8(const void *q_nope_absorbed, const void *q_rope,
                                      int64_t rows, void *q8, int32_t *qexp, void *stream);

/* mla_decode_fp8 with optional stage events (as mla_decode_ex). */
plmla_status mla_decode_fp8_ex(const void *q_nope_absorbed, const void *q_rope, const void *gate,
                               const void *slab_base, int64_t num_pages,
                               int64_t page_stride_elems, float kv_scale,
                               const int32_t *page_table, int64_t page_table_ld,
                               const int32_t *seq_lens, int32_t num_reqs, int32_t n_q_per_req,
                               int32_t num_heads, float scale, void *out, float *lse,
                               void *workspace, size_t workspace_bytes, int32_t cta_budget,
                               int32_t min_splits_per_req, void *stream,
                               const plmla_stage_events *events);

/*
 * mla_split_combine -- merge the partial softmax states of each request's KV
 * chunks and apply the sigmoid output gate [K3, Gated MLA decode paragraph;
 * AX, gating bullet].  Split order is fixed, so results are deterministic.
 *
 *   lse = ln sum_i exp(lse_part_i);  o = sum_i exp(lse_part_i - lse) * o_part_i
 *   out = bf16_rn(sigmoid(gate) * o)
 *
 * o_part       fp32 [num_splits, n_q_per_req*num_heads, 512]: split i's output,
 *              normalised over its own chunk (row index j*num_heads + h)
 * lse_part     fp32 [num_splits, n_q_per_req*num_heads], natural log; -inf for
 *              an empty chunk
 * split_indptr int32 [num_reqs + 1], device; request r owns splits
 *              split_indptr[r] .. split_indptr[r+1]-1 (none: out = 0, lse = -inf)
 * gate, out    bf16 [num_reqs*n_q_per_req, num_heads, 512]
 * lse          fp32 [num_reqs*n_q_per_req, num_heads] (may be NULL)
 */
plmla_status mla_split_combine(const float *o_part, const float *lse_part,
                               const int32_t *split_indptr, const void *gate, int32_t num_reqs,
                               int32_t n_q_per_req, int32_t num_heads, void *out, float *lse,
                               void *stream);

/*
 * mla_merge_partials -- the exchange step of decode context parallelism [AX,
 * "AgentX benchmark results": ranks combine partial attention results]: each
 * of `world` ranks decoded (with mla_decode) a disjoint part of every request's
 * history -- its own pages -- and the gathered results are merged.  The gate is
 * elementwise and the same for every part, so gated parts merge directly:
 *
 *   lse = ln sum_k exp(lse_parts[k]);  out = bf16_rn(sum_k exp(lse_parts[k] - lse) * out_parts[k])
 *
 * out_parts  bf16 [world, rows, 512], 16-byte aligned: rank k's gated output
 *            (rows = num_reqs * n_q * num_heads, the order of mla_decode's out)
 * lse_parts  fp32 [world, rows], natural log; -inf where rank k's part is empty
 * world      1 .. 4096;  rows >= 0
 * out        bf16 [rows, 512], written;  lse fp32 [rows], written (may be NULL);
 *            a row that no rank saw gives 0 and -inf
 * Ranks are merged in a fixed order, so the result does not depend on timing.
 * The bf16 rounding of each part adds at most 2^-9 relative error per part.
 */
plmla_status mla_merge_partials(const void *out_parts, const float *lse_parts, int32_t world,
                                int64_t rows, void *out, float *lse, void *stream);

/*
 * mla_dcp_shard -- one rank's part of every request's history for decode
 * context parallelism over `world` ranks [AX, "AgentX benchmark results": the
 * ranks decode parts of the context and combine partial attention results].
 * Page column c of request r (its tokens [1536 c, 1536 (c + 1)) of the
 * history) belongs to rank (c + r) mod world: every rank holds the same number
 * of a request's pages up to one, and the rotation by r spreads the leftover
 * pages over the ranks.  For rank `rank` this writes, per request, the page IDs
 * of its columns in column order into table_out row r, and into lens_out[r]
 * the tokens they hold (1536 per page; the request's last page, if this rank
 * holds it, only its L - 1536 (n - 1) tokens).  mla_decode on (table_out,
 * lens_out) with single-token queries then gives the rank's gated part (the
 * order of the tokens does not change the softmax), and mla_merge_partials of
 * the ranks' parts gives mla_decode over the whole history.
 *
 * page_table    int32, row r at page_table + r * page_table_ld (as mla_decode);
 *               columns 0 .. ceil(L_r / 1536) - 1 are read, at most
 *               page_table_ld of them (a longer history keeps the row's pages)
 * seq_lens      int32 [num_reqs], num_reqs 1 .. 1024
 * world         1 .. 4096; rank in [0, world)
 * table_out     int32 [num_reqs, table_out_ld], table_out_ld >=
 *               ceil(page_table_ld / world); entries past a row's page count are
 *               not written
 * lens_out      int32 [num_reqs], written
 * Device pointers; asynchronous on `stream`; reads nothing back.  Returns
 * PLMLA_INVALID_ARGUMENT for null or misaligned pointers and bad sizes.
 */
plmla_status mla_dcp_shard(const int32_t *page_table, int64_t page_table_ld,
                           const int32_t *seq_lens, int32_t num_reqs, int32_t world, int32_t rank,
                           int32_t *table_out, int64_t table_out_ld, int32_t *lens_out,
                           void *stream);

/*
 * mla_kv_append -- write each request's new latent and rope rows into the flat
 * page pool, the step before attention: under MLA a new token's rows are
 * appended after the request's history and no earlier row changes (vLLM blog
 * "Kimi K3 Inference Backend Evolution", section "State Overwrite: How KDA
 * Breaks Traditional KV Cache"); pages as in mla_decode (TokenSpeed Kimi K3
 * post, "A Generic, Unified Flat KV Layout for Cache Management").
 *
 * latent_new   [num_reqs * n_new, 512] bf16, row r * n_new + j = request r's
 *              new token j, contiguous rows, 16-byte aligned
 * rope_new     [num_reqs * n_new, 64] bf16, same rows, 16-byte aligned
 * slab_base, num_pages, page_stride_elems, page_table, page_table_ld
 *              the pool and table exactly as for mla_decode
 * seq_lens     [num_reqs] int32 histories AFTER the append (mla_decode's
 *              convention): new token j of request r goes to position
 *              seq_lens[r] - n_new + j, i.e. page page_table[r, p / 1536],
 *              row p % 1536, as 512 latent then 64 rope values
 * n_new        new tokens per request (0: nothing to do)
 * status       optional device int32: set to 32 if some seq_lens[r] < n_new and
 *              to 33 if a position's page column p / 1536 is >= page_table_ld or
 *              its page ID lies outside [0, num_pages); such rows are skipped,
 *              no table entry past a row's page_table_ld columns is read and
 *              nothing is written outside the pool
 *
 * Ownership: caller owns every buffer.  Asynchronous on `stream`.  Returns
 * PLMLA_INVALID_ARGUMENT for null or misaligned pointers and bad sizes,
 * PLMLA_CUDA_ERROR if the launch fails.
 */
plmla_status mla_kv_append(const void *latent_new, const void *rope_new, void *slab_base,
                           int64_t num_pages, int64_t page_stride_elems, const int32_t *page_table,
                           int64_t page_table_ld, const int32_t *seq_lens, int32_t num_reqs,
                           int32_t n_new, int32_t *status, void *stream);

/*
 * mla_kv_append_fp8 -- mla_kv_append into E4M3 pages (see mla_decode_fp8): each
 * new bf16 value x is stored as the E4M3 code of x / kv_scale (one correctly
 * rounded fp32 division, then round to nearest even, saturating at +-448; NaN
 * stays NaN).  Positions, pages, the status word and errors as mla_kv_append;
 * page_stride_elems counts bytes (>= 1536*576, multiple of 16) and kv_scale
 * must be finite and > 0.
 */
plmla_status mla_kv_append_fp8(const void *latent_new, const void *rope_new, void *slab_base,
                               int64_t num_pages, int64_t page_stride_elems, float kv_scale,
                               const int32_t *page_table, int64_t page_table_ld,
                               const int32_t *seq_lens, int32_t num_reqs, int32_t n_new,
                               int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PLMLA_H */

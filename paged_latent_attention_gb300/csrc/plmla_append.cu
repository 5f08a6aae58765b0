// plmla_append.cu -- KV append: each request's new latent and rope rows into the
// flat page pool.
//
// vLLM blog "Kimi K3 Inference Backend Evolution", section "State Overwrite: How
// KDA Breaks Traditional KV Cache": under MLA a new token's key/value rows are
// appended after the request's history and no earlier row changes.  The pool is
// the flat layout of the TokenSpeed Kimi K3 post ("A Generic, Unified Flat KV
// Layout for Cache Management"): one global page ID per 1,536-token page, token
// row t of page p at p * page_stride + t * 576 (512 latent, then 64 rope).
//
// seq_lens counts the history after the append (the decode's convention for
// draft tokens), so new token j of request r lands at position
// seq_lens[r] - n_new + j.  One warp per new row: the 1,152-byte row is
// contiguous in its page, so 72 16-byte stores cover it, reading the latent row
// (1,024 bytes) and the rope row (128 bytes) with 16-byte loads.  A position
// below zero, a position past the table's row (p / 1536 >= table_ld) or a page ID
// outside the pool skips the row and sets the status word (when given); nothing
// is read past the table's row and nothing is written outside the pool.
// append_fp8_kernel writes the same rows into E4M3 pages (the FP8 cache, 576
// bytes per token row), each value quantised with the cache's scale.
#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kAppendThreads = 256;   // 8 rows per CTA
constexpr int kLatentChunks = kLatent * 2 / 16;   // 64
constexpr int kRopeChunks = kRope * 2 / 16;       // 8

__global__ void __launch_bounds__(kAppendThreads)
append_kernel(const uint4 *__restrict__ latent, const uint4 *__restrict__ rope,
              __nv_bfloat16 *__restrict__ slab, int64_t num_pages, int64_t page_stride,
              const int32_t *__restrict__ table, int64_t table_ld,
              const int32_t *__restrict__ seq_lens, int num_reqs, int n_new, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5);
    if (row >= (int64_t)num_reqs * n_new)
        return;
    const int r = (int)(row / n_new), j = (int)(row % n_new);
    const int p = seq_lens[r] - n_new + j;
    if (p < 0) {
        if (lane == 0 && status != nullptr)
            atomicExch(status, kStatusAppendPosition);
        return;
    }
    if (p / kPageTokens >= table_ld) {     // past the table's row: no page to name
        if (lane == 0 && status != nullptr)
            atomicExch(status, kStatusAppendPage);
        return;
    }
    const int page = table[(int64_t)r * table_ld + p / kPageTokens];
    if (page < 0 || (int64_t)page >= num_pages) {
        if (lane == 0 && status != nullptr)
            atomicExch(status, kStatusAppendPage);
        return;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(slab + (int64_t)page * page_stride +
                                           (int64_t)(p % kPageTokens) * kRow);
    const uint4 *sl = latent + row * kLatentChunks;
    const uint4 *sr = rope + row * kRopeChunks;
    const uint4 a = __ldg(sl + lane), b = __ldg(sl + lane + 32);
    uint4 c = make_uint4(0u, 0u, 0u, 0u);
    if (lane < kRopeChunks)
        c = __ldg(sr + lane);
    dst[lane] = a;
    dst[lane + 32] = b;
    if (lane < kRopeChunks)
        dst[kLatentChunks + lane] = c;
}

// The same rows into E4M3 pages (576 bytes per token row): value x is stored as
// the E4M3 code of x / kv_scale (one correctly rounded fp32 division, then
// round to nearest even, saturating at +-448).  Lane l converts latent values
// [16 l, 16 l + 16) into 16 bytes and, for l < 8, rope values [8 l, 8 l + 8).
__global__ void __launch_bounds__(kAppendThreads)
append_fp8_kernel(const uint4 *__restrict__ latent, const uint4 *__restrict__ rope,
                  uint8_t *__restrict__ slab, int64_t num_pages, int64_t page_stride,
                  float kv_scale, const int32_t *__restrict__ table, int64_t table_ld,
                  const int32_t *__restrict__ seq_lens, int num_reqs, int n_new,
                  int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5);
    if (row >= (int64_t)num_reqs * n_new)
        return;
    const int r = (int)(row / n_new), j = (int)(row % n_new);
    const int p = seq_lens[r] - n_new + j;
    if (p < 0) {
        if (lane == 0 && status != nullptr)
            atomicExch(status, kStatusAppendPosition);
        return;
    }
    if (p / kPageTokens >= table_ld) {
        if (lane == 0 && status != nullptr)
            atomicExch(status, kStatusAppendPage);
        return;
    }
    const int page = table[(int64_t)r * table_ld + p / kPageTokens];
    if (page < 0 || (int64_t)page >= num_pages) {
        if (lane == 0 && status != nullptr)
            atomicExch(status, kStatusAppendPage);
        return;
    }
    uint8_t *dst = slab + (int64_t)page * page_stride + (int64_t)(p % kPageTokens) * kRow;
    const uint4 *sl = latent + row * kLatentChunks;
    const uint4 *sr = rope + row * kRopeChunks;
    const uint4 a = __ldg(sl + 2 * lane), b = __ldg(sl + 2 * lane + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = __fdiv_rn(__uint_as_float(w[2 * i] << 16), kv_scale);
        const float x1 = __fdiv_rn(__uint_as_float(w[2 * i] & 0xFFFF0000u), kv_scale);
        const float x2 = __fdiv_rn(__uint_as_float(w[2 * i + 1] << 16), kv_scale);
        const float x3 = __fdiv_rn(__uint_as_float(w[2 * i + 1] & 0xFFFF0000u), kv_scale);
        q[i] = (uint32_t)e4m3x2(x0, x1) | ((uint32_t)e4m3x2(x2, x3) << 16);
    }
    *reinterpret_cast<uint4 *>(dst + 16 * lane) = make_uint4(q[0], q[1], q[2], q[3]);
    if (lane < kRopeChunks) {
        const uint4 c = __ldg(sr + lane);
        const uint32_t u[4] = {c.x, c.y, c.z, c.w};
        uint32_t rq[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float x0 = __fdiv_rn(__uint_as_float(u[2 * i] << 16), kv_scale);
            const float x1 = __fdiv_rn(__uint_as_float(u[2 * i] & 0xFFFF0000u), kv_scale);
            const float x2 = __fdiv_rn(__uint_as_float(u[2 * i + 1] << 16), kv_scale);
            const float x3 = __fdiv_rn(__uint_as_float(u[2 * i + 1] & 0xFFFF0000u), kv_scale);
            rq[i] = (uint32_t)e4m3x2(x0, x1) | ((uint32_t)e4m3x2(x2, x3) << 16);
        }
        *reinterpret_cast<uint2 *>(dst + kLatent + 8 * lane) = make_uint2(rq[0], rq[1]);
    }
}

}  // namespace

cudaError_t launch_append_fp8(const void *latent, const void *rope, void *slab,
                              int64_t num_pages, int64_t page_stride, float kv_scale,
                              const int32_t *table, int64_t table_ld, const int32_t *seq_lens,
                              int num_reqs, int n_new, int32_t *status, cudaStream_t stream)
{
    const int64_t rows = (int64_t)num_reqs * n_new;
    if (rows == 0)
        return cudaSuccess;
    const int64_t blocks = (rows + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
    append_fp8_kernel<<<(unsigned)blocks, kAppendThreads, 0, stream>>>(
        static_cast<const uint4 *>(latent), static_cast<const uint4 *>(rope),
        static_cast<uint8_t *>(slab), num_pages, page_stride, kv_scale, table, table_ld,
        seq_lens, num_reqs, n_new, status);
    return cudaGetLastError();
}

cudaError_t launch_append(const void *latent, const void *rope, void *slab, int64_t num_pages,
                          int64_t page_stride, const int32_t *table, int64_t table_ld,
                          const int32_t *seq_lens, int num_reqs, int n_new, int32_t *status,
                          cudaStream_t stream)
{
    const int64_t rows = (int64_t)num_reqs * n_new;
    if (rows == 0)
        return cudaSuccess;
    const int64_t blocks = (rows + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
    append_kernel<<<(unsigned)blocks, kAppendThreads, 0, stream>>>(
        static_cast<const uint4 *>(latent), static_cast<const uint4 *>(rope),
        static_cast<__nv_bfloat16 *>(slab), num_pages, page_stride, table, table_ld, seq_lens,
        num_reqs, n_new, status);
    return cudaGetLastError();
}

}  // namespace plmla

// plmla_combine.cu -- partial-softmax (LSE) merge of KV chunks + sigmoid gate.
//
// TokenSpeed Kimi K3 post, section "Gluon kernels on AMD GPUs" (Gated MLA decode:
// chunk states are merged in a second kernel) and the AgentX post's decode
// context parallelism paragraph (ranks combine partial attention results).  The
// gate is the sigmoid output gate of Gated MLA (AgentX post, "Kernel fusion and
// overlap complete the decode path").
//
// SPLIT warps per output row (draft token, head), each with 512 / SPLIT of its
// latent columns; a lane owns 4 / SPLIT float4 groups (lane + 32k of the warp's
// part), so every split's row is read with fully coalesced 512-byte
// transactions.  Splits are visited in a fixed order, and every warp of a row
// computes the same weights, so the result does not depend on scheduling or on
// SPLIT.  Few rows (a handful of long requests) take SPLIT = 4 so that enough
// warps merge in parallel once the decode's last segments are published.
#include <math.h>

#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kThreads = 256;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr int32_t kStatusCombineWait = 16;

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int ld_acquire(const int32_t *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Lane 0 waits (bounded) until `need` segments of the row's request have been
// published by the decode kernel; false if the wait gave up or the decode
// reported an error.
__device__ bool wait_segments(const int32_t *counter, int need, int32_t *status)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
        const unsigned long long t0 = global_ns();
        while (ld_acquire(counter) < need) {
            if (*reinterpret_cast<volatile int32_t *>(status) != 0) {
                ok = false;
                break;
            }
            if (global_ns() - t0 > kWaitLimitNs) {
                atomicExch(status, kStatusCombineWait);
                ok = false;
                break;
            }
            __nanosleep(256);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    // every lane takes its own acquire of the (final) count before reading
    if (ok)
        (void)ld_acquire(counter);
    return ok;
}

template <int SPLIT>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
               const int32_t *__restrict__ indptr, const int32_t *__restrict__ seg_stride,
               int group_rows, const __nv_bfloat16 *__restrict__ gate, int num_reqs, int n_q,
               int num_heads, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
               const int32_t *__restrict__ done, int32_t *status, int epoch)
{
    // The next kernel on the stream may launch now (the decode step's planner
    // waits on entry for this grid to complete).
    asm volatile("griddepcontrol.launch_dependents;");
    // Without counters: launched as a programmatic dependent of the decode
    // kernel (or on its own), wait for the previous grid's partial states.
    if (done == nullptr)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int KG = 4 / SPLIT;                // float4 groups per lane
    const int lane = threadIdx.x & 31;
    const int64_t wid = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int64_t row = wid / SPLIT;
    const int part = (int)(wid % SPLIT);
    const int f0 = part * 32 * KG + lane;        // this lane's first float4 of the row
    const int64_t rows = (int64_t)num_reqs * n_q * num_heads;
    if (row >= rows)
        return;
    const int rows_per_req = n_q * num_heads;
    const int r = (int)(row / rows_per_req);
    const int rw = (int)(row % rows_per_req);   // j * H + h within the request
    const int g = rw / group_rows;               // row group (team) of this row
    const int gi = rw % group_rows;              // row inside the group's partials
    const int base = seg_stride != nullptr ? g * __ldcg(seg_stride) : 0;
    const int s0 = base + __ldcg(indptr + r), s1 = base + __ldcg(indptr + r + 1);
    // the gate logits are an input of the step: read them before waiting
    const uint2 *gp = reinterpret_cast<const uint2 *>(gate + row * kLatent);
    uint2 graw[KG];
#pragma unroll
    for (int k = 0; k < KG; ++k)
        graw[k] = gp[f0 + 32 * k];
    // With counters: this request's partial states are complete once all its
    // segments of this team are published for this layer (other requests may
    // still run; the counters hold the earlier layers' segments too).
    if (done != nullptr && !wait_segments(done + g * num_reqs + r, (s1 - s0) * epoch, status))
        return;

    // The segments' log-sum-exps are read by the lanes in parallel, 32 at a
    // time (one round trip instead of one per segment); the maximum and the
    // weights follow with warp shuffles, and the weighted rows are read with
    // several segments' loads in flight.  The order of every sum is fixed.
    float m = -INFINITY;
    for (int b = s0; b < s1; b += 32) {
        const int s = b + lane;
        if (s < s1)
            m = fmaxf(m, __ldcg(lse_part + (int64_t)s * group_rows + gi));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float4 acc[KG];
#pragma unroll
    for (int k = 0; k < KG; ++k)
        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (m != -INFINITY) {
        for (int b = s0; b < s1; b += 32) {
            const int s = b + lane;
            const float l = s < s1 ? __ldcg(lse_part + (int64_t)s * group_rows + gi) : -INFINITY;
            const float wl = l == -INFINITY ? 0.f : expf(l - m);   // this lane's segment weight
            wsum += wl;
            const int n = min(32, s1 - b);
            const float4 *src0 = reinterpret_cast<const float4 *>(
                o_part + ((int64_t)b * group_rows + gi) * kLatent);
            const int64_t seg_step = (int64_t)group_rows * kLatent / 4;   // float4 per segment
#pragma unroll 4
            for (int k = 0; k < n; ++k) {
                const float w = __shfl_sync(0xffffffffu, wl, k);
                if (w == 0.f)
                    continue;                    // warp-uniform: an empty segment
                const float4 *src = src0 + k * seg_step;
#pragma unroll
                for (int j = 0; j < KG; ++j) {
                    const float4 v = __ldcg(src + f0 + 32 * j);
                    acc[j].x = fmaf(w, v.x, acc[j].x);
                    acc[j].y = fmaf(w, v.y, acc[j].y);
                    acc[j].z = fmaf(w, v.z, acc[j].z);
                    acc[j].w = fmaf(w, v.w, acc[j].w);
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2 *dst = reinterpret_cast<uint2 *>(out + row * kLatent);
#pragma unroll
    for (int k = 0; k < KG; ++k) {
        const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&graw[k].x));
        const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&graw[k].y));
        const float o0 = acc[k].x * inv / (1.f + expf(-g01.x));
        const float o1 = acc[k].y * inv / (1.f + expf(-g01.y));
        const float o2 = acc[k].z * inv / (1.f + expf(-g23.x));
        const float o3 = acc[k].w * inv / (1.f + expf(-g23.y));
        const __nv_bfloat162 p01 = __floats2bfloat162_rn(o0, o1);
        const __nv_bfloat162 p23 = __floats2bfloat162_rn(o2, o3);
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t *>(&p01);
        packed.y = *reinterpret_cast<const uint32_t *>(&p23);
        dst[f0 + 32 * k] = packed;
    }
    if (lse != nullptr && lane == 0 && part == 0)
        lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

// Decode context parallelism: G ranks each decoded a disjoint part of every
// request's history (its pages), giving a gated bf16 output and the LSE of
// its part; merge them.  The gate is elementwise and the same for every part,
// so the merged gated row is the LSE-weighted sum of the gated parts:
//   lse = ln sum_k e^{lse_k},   out = sum_k e^{lse_k - lse} out_k
// (AgentX post, "AgentX benchmark results": decode context parallelism, ranks
// combine partial attention results; the merge rule is the split merge above).
// One warp per row, ranks in a fixed order; a row no rank saw gives 0, -inf.
__global__ void __launch_bounds__(kThreads)
merge_partials_kernel(const __nv_bfloat16 *__restrict__ parts, const float *__restrict__ lse_parts,
                      int world, int64_t rows, __nv_bfloat16 *__restrict__ out,
                      float *__restrict__ lse)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows)
        return;
    float m = -INFINITY;
    for (int k0 = 0; k0 < world; k0 += 32) {
        const int k = k0 + lane;
        if (k < world)
            m = fmaxf(m, __ldg(lse_parts + (int64_t)k * rows + row));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        acc[i] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
        for (int k = 0; k < world; ++k) {
            const float l = __ldg(lse_parts + (int64_t)k * rows + row);
            if (l == -INFINITY)
                continue;
            const float w = expf(l - m);
            wsum += w;
            // lane owns columns [8 lane, 8 lane + 8) and [256 + 8 lane, 256 + 8 lane + 8)
            const uint4 *src = reinterpret_cast<const uint4 *>(parts + ((int64_t)k * rows + row) * kLatent);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint4 v = __ldg(src + lane + 32 * h);
                const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wd[e]));
                    acc[8 * h + 2 * e] = fmaf(w, f.x, acc[8 * h + 2 * e]);
                    acc[8 * h + 2 * e + 1] = fmaf(w, f.y, acc[8 * h + 2 * e + 1]);
                }
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint4 *dst = reinterpret_cast<uint4 *>(out + row * kLatent);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t wd[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p =
                __floats2bfloat162_rn(acc[8 * h + 2 * e] * inv, acc[8 * h + 2 * e + 1] * inv);
            wd[e] = *reinterpret_cast<const uint32_t *>(&p);
        }
        dst[lane + 32 * h] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
    if (lse != nullptr && lane == 0)
        lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge_partials(const __nv_bfloat16 *parts, const float *lse_parts, int world,
                                  int64_t rows, __nv_bfloat16 *out, float *lse,
                                  cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    const int64_t blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
    merge_partials_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(parts, lse_parts, world, rows,
                                                                   out, lse);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *o_part, const float *lse_part, const int32_t *indptr,
                           const int32_t *seg_stride, int group_rows,
                           const __nv_bfloat16 *gate, int num_reqs, int n_q, int num_heads,
                           __nv_bfloat16 *out, float *lse, const int32_t *done,
                           int32_t *status, int epoch, cudaStream_t stream)
{
    const int64_t rows = (int64_t)num_reqs * n_q * num_heads;
    // warps per row: enough warps for about one CTA of 8 per SM
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    const int64_t target = (int64_t)sms * (kThreads / 32);
    const int split = rows >= target ? 1 : (2 * rows >= target ? 2 : 4);
    const int64_t blocks = (rows * split + kThreads / 32 - 1) / (kThreads / 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((done == nullptr) != (status == nullptr) || epoch < 1)
        return cudaErrorInvalidValue;
    auto kernel = split == 1 ? combine_kernel<1> : (split == 2 ? combine_kernel<2> : combine_kernel<4>);
    return cudaLaunchKernelEx(&cfg, kernel, o_part, lse_part, indptr, seg_stride, group_rows, gate,
                              num_reqs, n_q, num_heads, out, lse, done, status, epoch);
}

}  // namespace plmla

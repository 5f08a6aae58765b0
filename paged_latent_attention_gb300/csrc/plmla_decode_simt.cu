// plmla_decode_simt.cu -- split-KV gated-MLA decode on CUDA cores (fp32 FMA).
//
// One CTA per (work item, row group): the CTA owns `NG` query rows (draft token
// j, head h) of one request and one KV chunk [t0, t1).  It streams the chunk in
// 32-token tiles through shared memory, computes the 576-long scores, keeps an
// fp32 online softmax per row (running max m and sum l, base-2 exponent with
// log2(e) folded into the scale), and accumulates O += P V with one thread per
// latent column.  The chunk's partial state (O / l, m + ln l) goes to the
// workspace for the combine kernel.
//
// Rows past a request's history (and past each draft's causal limit) are never
// read into the dot products: the tile load writes zeros there, so stale or NaN
// page contents cannot reach the output.
#include <math.h>

#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kThreads = 512;          // one thread per latent column
constexpr int kTT = 32;                // tokens per tile
constexpr int kKStride = kRow + 2;     // bf16 elements per staged KV row (odd word stride)
constexpr float kLn2 = 0.69314718055994530942f;

template <int NG>
struct SimtSmem {
    static constexpr size_t q_bytes = size_t(NG) * kRow * 2;
    static constexpr size_t k_bytes = size_t(kTT) * kKStride * 2;
    static constexpr size_t s_bytes = size_t(NG) * kTT * 4;
    static constexpr size_t total = q_bytes + k_bytes + s_bytes + 4 * NG * 4;
};

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int NG>
__global__ void __launch_bounds__(kThreads, 1) decode_simt_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __nv_bfloat16 *Qs = reinterpret_cast<__nv_bfloat16 *>(smem);
    __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(smem + SimtSmem<NG>::q_bytes);
    float *S = reinterpret_cast<float *>(smem + SimtSmem<NG>::q_bytes + SimtSmem<NG>::k_bytes);
    float *m_s = S + NG * kTT;
    float *l_s = m_s + NG;
    float *alpha_s = l_s + NG;
    int *lrow_s = reinterpret_cast<int *>(alpha_s + NG);

    if ((int)blockIdx.x >= *a.item_count)
        return;
    const WorkItem it = a.items[blockIdx.x];
    const int row0 = blockIdx.y * NG;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int L = a.seq_lens[it.req];

    const int64_t qrow0 = (int64_t)it.req * a.rows_per_req + row0;
    for (int i = tid; i < NG * (kRow / 8); i += kThreads) {
        const int row = i / (kRow / 8), c8 = i % (kRow / 8);
        uint4 v;
        if (c8 < kLatent / 8)
            v = reinterpret_cast<const uint4 *>(a.q_nope + (qrow0 + row) * kLatent)[c8];
        else
            v = reinterpret_cast<const uint4 *>(a.q_rope + (qrow0 + row) * kRope)[c8 - kLatent / 8];
        reinterpret_cast<uint4 *>(Qs + row * kRow)[c8] = v;
    }
    if (tid < NG) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
        const int j = (row0 + tid) / a.num_heads;
        lrow_s[tid] = L - (a.n_q - 1 - j);
    }
    float acc[NG];
#pragma unroll
    for (int r = 0; r < NG; ++r)
        acc[r] = 0.f;
    __syncthreads();

    const int32_t *table_row = a.page_table + (int64_t)it.req * a.table_ld;
    for (int t0 = it.t0; t0 < it.t1; t0 += kTT) {
        // stage the tile (zeros past the chunk end)
        for (int i = tid; i < kTT * (kRow / 8); i += kThreads) {
            const int tt = i / (kRow / 8), c8 = i % (kRow / 8);
            const int t = t0 + tt;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (t < it.t1) {
                const int64_t page = table_row[t / kPageTokens];
                const __nv_bfloat16 *rowp =
                    a.slab + page * a.page_stride + (int64_t)(t % kPageTokens) * kRow;
                v = reinterpret_cast<const uint4 *>(rowp)[c8];
            }
            uint32_t *dst = reinterpret_cast<uint32_t *>(Ks + tt * kKStride + c8 * 8);
            dst[0] = v.x;
            dst[1] = v.y;
            dst[2] = v.z;
            dst[3] = v.w;
        }
        __syncthreads();
        // scores: one warp per (row, 32 tokens); the query row is a broadcast read
        for (int p = tid; p < NG * kTT; p += kThreads) {
            const int row = p / kTT, tt = p % kTT;
            const int t = t0 + tt;
            float s = -INFINITY;
            if (t < it.t1 && t < lrow_s[row]) {
                const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(Qs + row * kRow);
                const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(Ks + tt * kKStride);
                float dot = 0.f;
#pragma unroll 8
                for (int d = 0; d < kRow / 2; ++d) {
                    const float2 qf = __bfloat1622float2(q2[d]);
                    const float2 kf = __bfloat1622float2(k2[d]);
                    dot = fmaf(qf.x, kf.x, dot);
                    dot = fmaf(qf.y, kf.y, dot);
                }
                s = dot * a.scale_log2;
            }
            S[row * kTT + tt] = s;
        }
        __syncthreads();
        // online softmax, one warp per row, lane = token
        for (int row = warp; row < NG; row += kThreads / 32) {
            const float s = S[row * kTT + lane];
            const float m_old = m_s[row];
            const float m_new = fmaxf(m_old, warp_max(s));
            float alpha = 1.f, p = 0.f;
            if (m_new != -INFINITY) {
                alpha = fast_exp2(m_old - m_new);
                p = fast_exp2(s - m_new);
            }
            const float psum = warp_sum(p);
            S[row * kTT + lane] = p;
            if (lane == 0) {
                m_s[row] = m_new;
                l_s[row] = l_s[row] * alpha + psum;
                alpha_s[row] = alpha;
            }
        }
        __syncthreads();
        // O = O * alpha + P V, thread = latent column
#pragma unroll
        for (int r = 0; r < NG; ++r)
            acc[r] *= alpha_s[r];
        for (int tt = 0; tt < kTT; ++tt) {
            const float v = __bfloat162float(Ks[tt * kKStride + tid]);
#pragma unroll
            for (int r = 0; r < NG; ++r)
                acc[r] = fmaf(S[r * kTT + tt], v, acc[r]);
        }
        __syncthreads();
    }

    const int64_t obase = ((int64_t)it.split * a.rows_per_req + row0) * kLatent;
#pragma unroll
    for (int r = 0; r < NG; ++r) {
        const float l = l_s[r];
        a.o_part[obase + (int64_t)r * kLatent + tid] = l > 0.f ? acc[r] / l : 0.f;
    }
    if (tid < NG) {
        const float l = l_s[tid];
        a.lse_part[(int64_t)it.split * a.rows_per_req + row0 + tid] =
            l > 0.f ? (m_s[tid] + log2f(l)) * kLn2 : -INFINITY;
    }
}

template <int NG>
cudaError_t launch_ng(const DecodeArgs &a, int max_items, cudaStream_t stream)
{
    const size_t smem = SimtSmem<NG>::total;
    cudaError_t err = cudaFuncSetAttribute(decode_simt_kernel<NG>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    dim3 grid(max_items, a.num_groups);
    decode_simt_kernel<NG><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs &args, int max_items, cudaStream_t stream)
{
    switch (args.group_rows) {
    case 64: return launch_ng<64>(args, max_items, stream);
    case 32: return launch_ng<32>(args, max_items, stream);
    case 16: return launch_ng<16>(args, max_items, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace plmla

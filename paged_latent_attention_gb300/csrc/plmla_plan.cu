// plmla_plan.cu -- device-side per-request KV split planner.
//
// TokenSpeed AgentX post, section "Balance MLA work with per-request KV
// splitting" (Figure 4): a target chunk length follows from the batch's total
// history and the parallelism budget, and each request gets as many chunks as
// its own history needs.  The plan is computed on the device from seq_lens, so a
// decode step never waits for the host and a captured CUDA graph stays valid
// as histories grow (AgentX - InferenceXv3 report, SGLang section: runtime
// lengths, no per-step device-to-host length sync).
//
// chunk = ceil(sum L / budget) rounded up to kTile; if the chunks do not fit the
// budget, chunk grows (smallest multiple of kTile that fits, found by binary
// search because the chunk count only falls as the chunk grows), but never
// beyond the longest history rounded up to kTile.  Work items are emitted
// longest request first, so the block scheduler starts the longest chunks first.
#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPerThread = kMaxReqs / kPlanThreads;  // elements per thread in scans

__device__ __forceinline__ long long ceil_div_ll(long long a, long long b)
{
    return (a + b - 1) / b;
}

template <typename T>
__device__ T block_sum(T v, T *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    T total = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w)
        total += red[w];
    return total;
}

__device__ int block_max_int(int v, int *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    int m = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w)
        m = max(m, red[w]);
    return m;
}

// Exclusive prefix sum of vals[0..n) in place (n <= kMaxReqs); returns the total.
__device__ int block_exclusive_scan(int *vals, int n, int *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int base = threadIdx.x * kPerThread;
    int local[kPerThread];
    int run = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        int v = (base + i < n) ? vals[base + i] : 0;
        local[i] = run;
        run += v;
    }
    // inclusive warp scan of the per-thread totals
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int up = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += up;
    }
    __syncthreads();
    if (lane == 31)
        red[warp] = incl;
    __syncthreads();
    int warp_off = 0, total = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
        if (w < warp)
            warp_off += red[w];
        total += red[w];
    }
    const int thread_off = warp_off + incl - run;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i)
        if (base + i < n)
            vals[base + i] = thread_off + local[i];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(const int32_t *__restrict__ seq_lens, int num_reqs, int budget, PlanBuffers plan)
{
    __shared__ int lens[kMaxReqs];
    __shared__ int splits[kMaxReqs];   // split count, then split id base (request order)
    __shared__ int ranked[kMaxReqs];   // split count in rank order, then item base
    __shared__ int rank_of[kMaxReqs];
    __shared__ long long red64[kPlanThreads / 32];
    __shared__ int red32[kPlanThreads / 32];

    const int tid = threadIdx.x;
    long long local_sum = 0;
    int local_max = 0;
    for (int r = tid; r < num_reqs; r += kPlanThreads) {
        int L = max(0, seq_lens[r]);
        lens[r] = L;
        local_sum += L;
        local_max = max(local_max, L);
    }
    __syncthreads();
    const long long total = block_sum<long long>(local_sum, red64);
    const int longest_len = block_max_int(local_max, red32);

    long long chunk = kTile;
    if (total > 0) {
        const long long c0 = ceil_div_ll(ceil_div_ll(total, budget), kTile) * kTile;
        const long long longest = ceil_div_ll(longest_len, kTile) * kTile;
        chunk = c0;
        if (c0 < longest) {
            // smallest k in [0, K] with count(c0 + k*kTile) <= budget, else K
            long long lo = 0, hi = (longest - c0) / kTile;
            while (lo < hi) {
                const long long mid = (lo + hi) / 2;
                const long long c = c0 + mid * kTile;
                long long cnt = 0;
                for (int r = tid; r < num_reqs; r += kPlanThreads)
                    cnt += ceil_div_ll(lens[r], c);
                cnt = block_sum<long long>(cnt, red64);
                if (cnt <= budget)
                    hi = mid;
                else
                    lo = mid + 1;
            }
            chunk = c0 + lo * kTile;
        }
    }

    for (int r = tid; r < num_reqs; r += kPlanThreads) {
        const int L = lens[r];
        splits[r] = (int)ceil_div_ll(L, chunk);
        // rank: longer histories first, ties by request index
        int rank = 0;
        for (int q = 0; q < num_reqs; ++q) {
            const int Lq = lens[q];
            rank += (Lq > L) || (Lq == L && q < r);
        }
        rank_of[r] = rank;
    }
    __syncthreads();
    for (int r = tid; r < num_reqs; r += kPlanThreads)
        ranked[rank_of[r]] = splits[r];
    __syncthreads();
    const int n_items = block_exclusive_scan(ranked, num_reqs, red32);
    const int n_splits = block_exclusive_scan(splits, num_reqs, red32);

    for (int r = tid; r < num_reqs; r += kPlanThreads) {
        plan.indptr[r] = splits[r];
        const int L = lens[r];
        const int n = (int)ceil_div_ll(L, chunk);
        const int item0 = ranked[rank_of[r]];
        for (int s = 0; s < n && plan.items != nullptr; ++s) {
            WorkItem it;
            it.req = r;
            it.split = splits[r] + s;
            it.t0 = (int)(s * chunk);
            it.t1 = (int)min((long long)L, (s + 1) * chunk);
            plan.items[item0 + s] = it;
        }
    }
    if (tid == 0) {
        if (plan.status != nullptr)
            *plan.status = 0;
        plan.indptr[num_reqs] = n_splits;
        *plan.chunk = chunk;
        if (plan.count != nullptr)
            *plan.count = n_items;
    }
}

}  // namespace

cudaError_t launch_plan(const int32_t *seq_lens, int num_reqs, int budget, PlanBuffers plan,
                        cudaStream_t stream)
{
    plan_kernel<<<1, kPlanThreads, 0, stream>>>(seq_lens, num_reqs, budget, plan);
    return cudaGetLastError();
}

}  // namespace plmla

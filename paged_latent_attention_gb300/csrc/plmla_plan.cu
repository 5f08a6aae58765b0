// plmla_plan.cu -- device-side KV split planner and the persistent-CTA schedule.
//
// Split plan (TokenSpeed AgentX post, section "Balance MLA work with per-request
// KV splitting", Figure 4): a target chunk length follows from the batch's total
// history and a parallelism budget, and each request gets as many chunks as its
// own history needs.  chunk = ceil(sum L / budget) rounded up to kTile; if the
// chunks do not fit the budget, chunk grows (the smallest multiple of kTile
// that fits, found by a 32-way parallel search because the chunk count only falls as the
// chunk grows), never beyond the longest history rounded up to kTile.
//
// Schedule (the GB300 side): the decode kernel runs one persistent CTA per SM.
// The chunks, in request order, are dealt out as contiguous runs so that every
// CTA ("member") gets its share of the cost up to half a chunk, cost counted in
// 128-token tiles plus a fixed charge for each request's first chunk (starting
// a segment): chunk i goes to the member whose share holds the chunk's cost
// midpoint (cost before i + cost of i / 2).  Shares are equal until the decode
// has measured each SM's speed (SmCalib), then proportional to it.  Consecutive chunks of one request that land on one member form
// a segment, which the CTA processes without writing an intermediate partial
// state.  Every row group of the queries repeats the same schedule on its own
// team of members, so teams read the same KV tiles at about the same time.
//
// Everything is computed on the device from seq_lens, so a decode step never
// waits for the host and a captured CUDA graph stays valid as histories grow
// (AgentX - InferenceXv3 report, SGLang section: runtime lengths, no per-step
// device-to-host length sync).
#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kSegmentCostTiles = 2;
constexpr int kScanPerThread = kMaxPlanSplits / kPlanThreads;

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

// Exclusive prefix sum of vals[0..n) in place (n <= kMaxPlanSplits); returns the total.
__device__ int block_exclusive_scan(int *vals, int n, int *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int base = threadIdx.x * kScanPerThread;
    int local[kScanPerThread];
    int run = 0;
#pragma unroll
    for (int i = 0; i < kScanPerThread; ++i) {
        const int v = (base + i < n) ? vals[base + i] : 0;
        local[i] = run;
        run += v;
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, incl, o);
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
    for (int i = 0; i < kScanPerThread; ++i)
        if (base + i < n)
            vals[base + i] = thread_off + local[i];
    __syncthreads();
    return total;
}

struct PlanSmem {
    int lens[kMaxReqs];
    int split_base[kMaxReqs];
    int sp_req[kMaxPlanSplits];
    int sp_t0[kMaxPlanSplits];
    int sp_t1[kMaxPlanSplits];
    int sp_tiles[kMaxPlanSplits];   // tiles of each chunk, then their exclusive prefix
    int sp_member[kMaxPlanSplits];
    int sp_seg[kMaxPlanSplits];     // segment-start flag, then the segment id
    long long red64[kPlanThreads / 32];
    int red32[kPlanThreads / 32];
    int cand_k[kPlanThreads / 32];
    int cand_fits[kPlanThreads / 32];
    float wprefix[kMaxSms + 1];     // inclusive prefix of member weights (speed-scaled shares)
    float wrun[kMaxSms];
    int weighted;                   // 1 when wprefix holds measured weights
};

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(const int32_t *__restrict__ seq_lens, int num_reqs, int budget, int members,
            PlanBuffers plan)
{
    extern __shared__ __align__(16) unsigned char plan_smem_raw[];
    PlanSmem &sm = *reinterpret_cast<PlanSmem *>(plan_smem_raw);
    const int tid = threadIdx.x;
    // the decode kernel may start its prologue now; it waits for this grid's
    // completion before reading the plan
    asm volatile("griddepcontrol.launch_dependents;");

    // finished-segment counters and CTA claims of this call's decode start from zero
    if (plan.done != nullptr)
        for (int i = tid; i < plan.n_done; i += kPlanThreads)
            plan.done[i] = 0;
    if (plan.claim != nullptr)
        for (int i = tid; i < plan.n_claim; i += kPlanThreads)
            plan.claim[i] = 0;

    // ---- split plan (per request)
    long long local_sum = 0;
    int local_max = 0;
    for (int r = tid; r < num_reqs; r += kPlanThreads) {
        const int L = max(0, seq_lens[r]);
        sm.lens[r] = L;
        local_sum += L;
        local_max = max(local_max, L);
    }
    __syncthreads();
    const long long total = block_sum<long long>(local_sum, sm.red64);
    const int longest_len = block_max_int(local_max, sm.red32);

    long long chunk = kTile;
    if (total > 0) {
        const long long c0 = ceil_div_ll(ceil_div_ll(total, budget), kTile) * kTile;
        const long long longest = ceil_div_ll(longest_len, kTile) * kTile;
        chunk = c0;
        if (c0 < longest) {
            // smallest k in [0, K] with count(c0 + k*kTile) <= budget, else K;
            // count only falls as the chunk grows, so each round splits [lo, hi]
            // into 32 parts, one candidate per warp.  32-bit arithmetic only:
            // histories and chunks are below 2^31, and a count is only compared
            // with the budget, so it saturates at budget + 1.
            int lo = 0, hi = (int)((longest - c0) / kTile);
            const unsigned c0u = (unsigned)c0;
            const int lane = tid & 31, warp = tid >> 5;
            while (lo < hi) {
                const int span = hi - lo;
                const int k = lo + (int)(((long long)span * (warp + 1)) / 33);   // in [lo, hi)
                const unsigned c = c0u + (unsigned)k * kTile;
                int cnt = 0;
                for (int r = lane; r < num_reqs; r += 32) {
                    const unsigned L = (unsigned)sm.lens[r];
                    cnt = min(cnt + (int)((L + c - 1u) / c), budget + 1);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    cnt = min(cnt + __shfl_xor_sync(0xffffffffu, cnt, o), budget + 1);
                __syncthreads();
                if (lane == 0) {
                    sm.cand_k[warp] = k;
                    sm.cand_fits[warp] = cnt <= budget;
                }
                __syncthreads();
                // candidates ascend with the warp index: the first fitting one
                // bounds hi, the one before it (failing) bounds lo
                const unsigned fits = __ballot_sync(0xffffffffu, sm.cand_fits[lane] != 0);
                const int first = fits ? __ffs(fits) - 1 : kPlanThreads / 32;
                if (first < kPlanThreads / 32)
                    hi = sm.cand_k[first];
                if (first > 0)
                    lo = max(lo, sm.cand_k[first - 1] + 1);
            }
            chunk = c0 + (long long)lo * kTile;
        }
    }
    for (int r = tid; r < num_reqs; r += kPlanThreads)
        sm.split_base[r] = (int)ceil_div_ll(sm.lens[r], chunk);
    __syncthreads();
    const int n_splits = block_exclusive_scan(sm.split_base, num_reqs, sm.red32);
    for (int r = tid; r < num_reqs; r += kPlanThreads)
        plan.indptr[r] = sm.split_base[r];
    if (tid == 0) {
        if (plan.status != nullptr)
            *plan.status = 0;
        plan.indptr[num_reqs] = n_splits;
        *plan.chunk = chunk;
    }
    if (plan.segments == nullptr)
        return;
    if (n_splits > kMaxPlanSplits) {   // excluded by the host-side budget limit
        if (tid == 0 && plan.status != nullptr)
            *plan.status = 8;
        return;
    }

    // ---- member shares: CTA c of the decode grid runs on the SM with id c when
    // it can (it claims that index), so once every such SM's speed is measured,
    // member m of every team gets a share of the cost proportional to the mean
    // speed of SMs team*members + m; until then the shares are equal
    {
        const SmCalib *cal = plan.calib;
        const int n_cta = plan.n_claim;
        const int teams = n_cta / max(members, 1);
        const bool usable = cal != nullptr && teams >= 1 && n_cta <= kMaxSms;
        float rate = 0.f;
        bool measured = true;
        if (usable && tid < n_cta) {
            const float c = cal->cost[tid], t = cal->time_ns[tid];
            measured = c >= kCalibCost && t > 0.f;
            rate = measured ? c / t : 0.f;
            sm.wprefix[tid + 1] = rate;              // per-CTA rate, reduced below
        }
        const int ready = __syncthreads_and(usable && measured);
        if (ready) {
            // member rate (mean over teams), then an inclusive prefix in warp 0:
            // lane l owns members [8l, 8l + 8)
            if (tid < members) {
                float r = 0.f;
                for (int g = 0; g < teams; ++g)
                    r += sm.wprefix[g * members + tid + 1];
                sm.wrun[tid] = r / teams;
            }
            __syncthreads();
            if (tid < 32) {
                constexpr int per = kMaxSms / 32;
                float loc[per];
                float run = 0.f;
#pragma unroll
                for (int i = 0; i < per; ++i) {
                    const int m = tid * per + i;
                    run += m < members ? sm.wrun[m] : 0.f;
                    loc[i] = run;
                }
                float incl = run;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float up = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o)
                        incl += up;
                }
                const float off = incl - run;
#pragma unroll
                for (int i = 0; i < per; ++i) {
                    const int m = tid * per + i;
                    if (m < members)
                        sm.wprefix[m + 1] = off + loc[i];
                }
                if (tid == 0)
                    sm.wprefix[0] = 0.f;
            }
        }
        if (tid == 0)
            sm.weighted = ready ? 1 : 0;
        __syncthreads();
    }

    // ---- schedule: chunks in request order, dealt to members by cost
    for (int i = tid; i < n_splits; i += kPlanThreads) {
        // request of chunk i: the last r with split_base[r] <= i
        int lo = 0, hi = num_reqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm.split_base[mid] <= i)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int r = lo;
        const int s = i - sm.split_base[r];
        const int L = sm.lens[r];
        const int t0 = (int)(s * chunk);
        const int t1 = (int)min((long long)L, (s + 1) * chunk);
        sm.sp_req[i] = r;
        sm.sp_t0[i] = t0;
        sm.sp_t1[i] = t1;
        // cost in tiles; a request's first chunk also carries the cost of
        // starting a segment (query load, first-tile softmax, epilogue)
        sm.sp_tiles[i] = (t1 - t0 + kTile - 1) / kTile + (s == 0 ? kSegmentCostTiles : 0);
        sm.sp_member[i] = sm.sp_tiles[i];   // keep the cost for the midpoint
    }
    __syncthreads();
    const int total_tiles = block_exclusive_scan(sm.sp_tiles, n_splits, sm.red32);
    for (int i = tid; i < n_splits; i += kPlanThreads) {
        // midpoint of chunk i as a fraction of the total cost
        const long long mid2 = 2LL * sm.sp_tiles[i] + sm.sp_member[i];  // 2*prefix + cost
        const float frac = (float)mid2 / (2.f * (float)max(total_tiles, 1));
        int m;
        if (sm.weighted) {
            // the member whose share [wprefix[m], wprefix[m + 1]) holds the midpoint
            const float target = frac * sm.wprefix[members];
            int lo = 0, hi = members - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (sm.wprefix[mid] <= target)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            m = lo;
        } else {
            m = (int)(frac * (float)members);
        }
        sm.sp_member[i] = min(members - 1, max(0, m));
    }
    __syncthreads();
    for (int i = tid; i < n_splits; i += kPlanThreads)
        sm.sp_seg[i] = (i == 0) || sm.sp_req[i] != sm.sp_req[i - 1] ||
                       sm.sp_member[i] != sm.sp_member[i - 1];
    __syncthreads();
    const int n_segs = block_exclusive_scan(sm.sp_seg, n_splits, sm.red32);
    for (int i = tid; i < n_splits; i += kPlanThreads) {
        // sp_seg now holds the number of segment starts before chunk i, so a
        // chunk that continues a segment belongs to segment sp_seg[i] - 1
        const bool starts = (i == 0) || sm.sp_req[i] != sm.sp_req[i - 1] ||
                            sm.sp_member[i] != sm.sp_member[i - 1];
        const int seg = sm.sp_seg[i] - (starts ? 0 : 1);
        const bool ends = (i == n_splits - 1) || sm.sp_req[i + 1] != sm.sp_req[i] ||
                          sm.sp_member[i + 1] != sm.sp_member[i];
        if (starts) {
            plan.segments[seg].x = sm.sp_req[i];
            plan.segments[seg].y = sm.sp_t0[i];
            plan.segments[seg].w = sm.sp_member[i];
            // members (previous chunk's member, this member] start at this segment
            const int prev = (i == 0) ? -1 : sm.sp_member[i - 1];
            for (int k = prev + 1; k <= sm.sp_member[i]; ++k)
                plan.seg_member_indptr[k] = seg;
        }
        if (ends)
            plan.segments[seg].z = sm.sp_t1[i];
    }
    // first segment of each request: the segment id of its first chunk (for a
    // request without chunks, the id of the next request's first chunk)
    for (int r = tid; r < num_reqs; r += kPlanThreads) {
        const int i = sm.split_base[r];
        plan.seg_req_indptr[r] = i < n_splits ? sm.sp_seg[i] : n_segs;
    }
    if (tid == 0) {
        plan.seg_req_indptr[num_reqs] = n_segs;
        const int last = n_splits > 0 ? sm.sp_member[n_splits - 1] : -1;
        for (int k = last + 1; k <= members; ++k)
            plan.seg_member_indptr[k] = n_segs;
        *plan.seg_count = n_segs;
    }
}

}  // namespace

size_t plan_smem_bytes() { return sizeof(PlanSmem); }

cudaError_t launch_plan(const int32_t *seq_lens, int num_reqs, int budget, int members,
                        PlanBuffers plan, cudaStream_t stream)
{
    const int smem = (int)sizeof(PlanSmem);
    cudaError_t err =
        cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess)
        return err;
    plan_kernel<<<1, kPlanThreads, smem, stream>>>(seq_lens, num_reqs, budget, members, plan);
    return cudaGetLastError();
}

}  // namespace plmla

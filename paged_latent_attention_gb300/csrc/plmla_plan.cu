// plmla_plan.cu -- device-side KV split planner and the persistent-CTA schedule.
//
// Split plan (TokenSpeed AgentX post, section "Balance MLA work with per-request
// KV splitting", Figure 4): a target chunk length follows from the batch's total
// history and a parallelism budget, and each request gets as many chunks as its
// own history needs.  chunk = ceil(sum L / budget) rounded up to kTile; if the
// chunks do not fit the budget, chunk grows (the smallest multiple of kTile
// that fits, found by a parallel search because the chunk count only falls as
// the chunk grows), never beyond the longest history rounded up to kTile.
// Uniform mode (the baseline of that section's Figure 5 comparison): every
// request with history gets the same split count su = budget / (requests with
// history), so request r's chunk is ceil(L_r / su) rounded up to kTile.
//
// Schedule (the GB300 side): the decode kernel runs one persistent CTA per SM.
// The chunks, in request order, are dealt out as contiguous runs so that every
// CTA ("member") gets its share of the cost up to half a chunk, cost counted in
// 128-token tiles plus a fixed charge for each request's first chunk (starting
// a segment): a chunk goes to the member whose equal share holds the chunk's
// cost midpoint (cost before it + half its cost).  The schedule depends only on
// the histories and the grid shape, never on timing, so a step's outputs are
// the same bits on every call and in every process.  The chunks
// of one request all have the same length (the last may be shorter), so the
// cost before any chunk has a closed form from a per-request prefix, and each
// member's chunk range comes from a binary search over requests, without a
// per-chunk table.  Consecutive chunks of one request that land on one member
// form a segment, which the CTA processes without writing an intermediate
// partial state.  Every row group of the queries repeats the same schedule on
// its own team of members, so teams read the same KV tiles at about the same
// time.
//
// Everything is computed on the device from seq_lens, so a decode step never
// waits for the host and a captured CUDA graph stays valid as histories grow
// (AgentX - InferenceXv3 report, SGLang section: runtime lengths, no per-step
// device-to-host length sync).
#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kReqPerThread = kMaxReqs / kPlanThreads;   // thread t owns requests [4t, 4t + 4)

struct PlanSmem {
    int lens[kMaxReqs];
    int sb[kMaxReqs + 1];        // exclusive prefix of chunks per request (split base)
    int cost0[kMaxReqs + 1];     // exclusive prefix of request cost (tiles + start charge)
    int lastm[kMaxReqs];         // running max of each request's last-chunk doubled midpoint
    int nonempty[kMaxReqs + 1];  // exclusive prefix of requests with at least one chunk
    int ctile[kMaxReqs];         // chunk length of each request, in tiles
    int first[kMaxSms + 1];      // first chunk of each member (members + 1 entries)
    int nseg[kMaxSms + 1];       // exclusive prefix of segments per member
    long long red64[kPlanWarps];
    int red32[kPlanWarps];
    int cand_k[kPlanWarps];
    int cand_fits[kPlanWarps];
};

// Block-wide sum / max of one value per thread; every thread gets the result.
__device__ long long block_sum64(long long v, long long *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    long long t = 0;
#pragma unroll
    for (int w = 0; w < kPlanWarps; ++w)
        t += red[w];
    __syncthreads();
    return t;
}

__device__ int block_max32(int v, int *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    int m = 0;
#pragma unroll
    for (int w = 0; w < kPlanWarps; ++w)
        m = max(m, red[w]);
    __syncthreads();
    return m;
}

// Exclusive block scan (sum) of one value per thread, in thread order; the
// block total goes to *total.
__device__ int block_scan_excl(int v, int *red, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += up;
    }
    if (lane == 31)
        red[warp] = incl;
    __syncthreads();
    int off = 0, t = 0;
#pragma unroll
    for (int w = 0; w < kPlanWarps; ++w) {
        off += w < warp ? red[w] : 0;
        t += red[w];
    }
    __syncthreads();
    *total = t;
    return off + incl - v;
}

// Exclusive block scan (max, identity -1) of one value per thread.
__device__ int block_scan_max_excl(int v, int *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl = max(incl, up);
    }
    int excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0)
        excl = -1;
    if (lane == 31)
        red[warp] = incl;
    __syncthreads();
    int off = -1;
#pragma unroll
    for (int w = 0; w < kPlanWarps; ++w)
        off = w < warp ? max(off, red[w]) : off;
    __syncthreads();
    return max(off, excl);
}

// Number of chunks of length c (a multiple of kTile, below 2^31) the requests
// need, counted by one warp and saturated at cap + 1.
__device__ int warp_chunk_count(const int *lens, int num_reqs, unsigned c, int cap)
{
    const int lane = threadIdx.x & 31;
    int cnt = 0;
    for (int r = lane; r < num_reqs; r += 32)
        cnt = min(cnt + (int)(((unsigned)lens[r] + c - 1u) / c), cap + 1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        cnt = min(cnt + __shfl_xor_sync(0xffffffffu, cnt, o), cap + 1);
    return cnt;
}

// Doubled cost midpoint of chunk s of a request whose cost prefix is `cost0`
// and which has `tiles` tiles: the first chunk carries the segment charge.
__device__ __forceinline__ int chunk_mid2(int cost0, int tiles, int chunk_tiles, int s)
{
    const int t = min(chunk_tiles, tiles - s * chunk_tiles);
    return s == 0 ? 2 * cost0 + t + kSegmentCostTiles
                  : 2 * cost0 + 2 * kSegmentCostTiles + 2 * s * chunk_tiles + t;
}

// Two E4M3 values (low byte first) widened exactly to floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    float lo, hi;
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
    return make_float2(lo, hi);
}

// The remainder v - decode(hi) of one scaled value: exact in fp32 (v and
// decode(hi) are within a factor of two, or decode(hi) is zero).  A nonzero q
// whose scaled value underflowed fp32 has the exact remainder v itself, a tiny
// number of q's sign, whose E4M3 code is q's signed zero.
__device__ __forceinline__ float remainder_of(float q, float v, float hi)
{
    return (v == 0.f && q != 0.f) ? copysignf(0.f, q) : v - hi;
}

// E4M3 codes of four values times p2 as one word (hi part), and the E4M3 codes
// of their remainders (lo part); both round to nearest even.
__device__ __forceinline__ void split4(const float *q, float p2, uint32_t &hi, uint32_t &lo)
{
    const float a = q[0] * p2, b = q[1] * p2, c = q[2] * p2, d = q[3] * p2;
    const uint16_t h0 = e4m3x2(a, b), h1 = e4m3x2(c, d);
    const float2 f0 = e4m3x2_to_float2(h0), f1 = e4m3x2_to_float2(h1);
    hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
    lo = (uint32_t)e4m3x2(remainder_of(q[0], a, f0.x), remainder_of(q[1], b, f0.y)) |
         ((uint32_t)e4m3x2(remainder_of(q[2], c, f1.x), remainder_of(q[3], d, f1.y)) << 16);
}

// FP8 queries for the FP8 decode (its tensor-core kind multiplies E4M3 by E4M3):
// row i of [q_nope | q_rope] (576 values) is scaled to v = q * 2^-e, with e the
// smallest exponent for which max |q| * 2^-e <= 448 (E4M3's largest finite
// value), at least -126, and 0 for an all-zero row; the scaling by a power of
// two is exact.  v enters as two E4M3 parts: hi = E4M3(v) (plane 0 of q8) and
// lo = E4M3(v - hi) (plane 1, rows q_rows further on).  v has bf16's 8
// significant bits, hi keeps 4 and the remainder's at most 4 others fit lo
// exactly while |v| >= 2^-2 (below it lo is subnormal, off by at most 2^-10),
// so the decode's scores use the bf16 query itself, up to that last bit.  One
// warp per row: lane l takes latent values [16 l, 16 l + 16) and, for l < 8,
// rope values [8 l, 8 l + 8).
__device__ void quantize_queries(const PlanBuffers &plan, int cta)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row_end = min(plan.q_rows, (cta + 1) * kQuantRowsPerCta);
    for (int row = cta * kQuantRowsPerCta + warp; row < row_end; row += kPlanWarps) {
        const uint4 *qn = reinterpret_cast<const uint4 *>(plan.q_nope + (int64_t)row * kLatent);
        const uint4 *qr = reinterpret_cast<const uint4 *>(plan.q_rope + (int64_t)row * kRope);
        uint32_t w[12];
        const uint4 a = qn[2 * lane], b = qn[2 * lane + 1];
        const uint4 c = lane < 8 ? qr[lane] : make_uint4(0u, 0u, 0u, 0u);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        w[8] = c.x; w[9] = c.y; w[10] = c.z; w[11] = c.w;
        float v[24];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 12; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const uint32_t bits = __float_as_uint(amax);
        const int biased = (int)((bits >> 23) & 0xFFu);
        int e = 0;
        if (amax > 0.f) {
            if (biased == 0) {
                e = -126;                               // subnormal maximum
            } else {
                // amax = (1 + f) 2^k: 2^(k-8) keeps it <= 448 = 1.75 * 2^8 iff f <= 0.75
                const int k = biased - 127;
                e = max((bits & 0x7FFFFFu) <= 0x600000u ? k - 8 : k - 7, -126);
            }
        }
        const float p2 = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e, exact
        uint32_t hi[4], lo[4], rope_hi[2], rope_lo[2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            split4(v + 4 * i, p2, hi[i], lo[i]);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            split4(v + 16 + 4 * i, p2, rope_hi[i], rope_lo[i]);
        uint8_t *dst = plan.q8 + (int64_t)row * kRow;
        uint8_t *dst_lo = plan.q8 + ((int64_t)plan.q_rows + row) * kRow;
        *reinterpret_cast<uint4 *>(dst + 16 * lane) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(dst_lo + 16 * lane) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (lane < 8) {
            *reinterpret_cast<uint2 *>(dst + kLatent + 8 * lane) = make_uint2(rope_hi[0], rope_hi[1]);
            *reinterpret_cast<uint2 *>(dst_lo + kLatent + 8 * lane) =
                make_uint2(rope_lo[0], rope_lo[1]);
        }
        if (lane == 0)
            plan.qexp[row] = e;
    }
}

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(const int32_t *__restrict__ seq_lens, int num_reqs, int budget, int members,
            int uniform, PlanBuffers plan)
{
    extern __shared__ __align__(16) unsigned char plan_smem_raw[];
    PlanSmem &sm = *reinterpret_cast<PlanSmem *>(plan_smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Launched as a programmatic dependent of whatever ran before it on the
    // stream: wait for that grid (it may have written seq_lens or the queries,
    // or still read this workspace) before touching memory.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the decode kernel may start its prologue now; it waits for this grid's
    // completion before reading the plan (and the FP8 queries)
    asm volatile("griddepcontrol.launch_dependents;");
    if (blockIdx.x > 0) {
        quantize_queries(plan, blockIdx.x - 1);
        return;
    }

    // ---- histories
    const int r0 = tid * kReqPerThread;
    int L[kReqPerThread];
    long long local_sum = 0;
    int local_max = 0, local_live = 0;
#pragma unroll
    for (int k = 0; k < kReqPerThread; ++k) {
        const int r = r0 + k;
        L[k] = r < num_reqs ? max(0, seq_lens[r]) : 0;
        if (r < num_reqs)
            sm.lens[r] = L[k];
        local_sum += L[k];
        local_max = max(local_max, L[k]);
        local_live += L[k] > 0 ? 1 : 0;
    }
    // finished-segment counters of this call's decode start from zero
    if (plan.done != nullptr)
        for (int i = tid; i < plan.n_done; i += kPlanThreads)
            plan.done[i] = 0;
    const long long total = block_sum64(local_sum, sm.red64);   // also publishes sm.lens
    const int longest_len = block_max32(local_max, sm.red32);
    const int live = (int)block_sum64(local_live, sm.red64);
    // uniform mode: split count of every request with history
    const long long su = max(1, budget / max(1, live));

    // ---- chunk length (per-request mode)
    long long chunk = kTile;
    if (total > 0 && !uniform) {
        const long long c0 = (((total + budget - 1) / budget + kTile - 1) / kTile) * kTile;
        const long long longest = ((longest_len + kTile - 1) / (long long)kTile) * kTile;
        chunk = c0;
        // c0 usually fits the budget already; otherwise the smallest k in
        // [1, K] with count(c0 + k*kTile) <= budget (K if none): the count only
        // falls as the chunk grows, so each round splits [lo, hi] into
        // kPlanWarps + 1 parts, one candidate per warp.  Histories and chunks
        // are below 2^31, and a count is only compared with the budget, so it
        // saturates at budget + 1.
        if (c0 < longest && warp_chunk_count(sm.lens, num_reqs, (unsigned)c0, budget) > budget) {
            int lo = 1, hi = (int)((longest - c0) / kTile);
            const unsigned c0u = (unsigned)c0;
            while (lo < hi) {
                const int span = hi - lo;
                const int k = lo + (int)(((long long)span * (warp + 1)) / (kPlanWarps + 1));
                const int cnt = warp_chunk_count(sm.lens, num_reqs, c0u + (unsigned)k * kTile,
                                                 budget);
                if (lane == 0) {
                    sm.cand_k[warp] = k;
                    sm.cand_fits[warp] = cnt <= budget;
                }
                __syncthreads();
                // candidates ascend with the warp index: the first fitting one
                // bounds hi, the one before it (failing) bounds lo
                int first = kPlanWarps;
                for (int w = kPlanWarps - 1; w >= 0; --w)
                    if (sm.cand_fits[w])
                        first = w;
                if (first < kPlanWarps)
                    hi = sm.cand_k[first];
                if (first > 0)
                    lo = max(lo, sm.cand_k[first - 1] + 1);
                __syncthreads();
            }
            chunk = c0 + (long long)lo * kTile;
        }
    }

    // ---- per request: chunk length, chunks, tiles, cost (tiles plus the start
    // charge); prefixes
    int ns[kReqPerThread], nt[kReqPerThread], ct[kReqPerThread];
    int my_chunks = 0, my_cost = 0, my_nonempty = 0;
#pragma unroll
    for (int k = 0; k < kReqPerThread; ++k) {
        long long c = chunk;
        if (uniform) {
            const long long per = (L[k] + su - 1) / su;
            c = max(1LL, (per + kTile - 1) / kTile) * kTile;
        }
        ct[k] = (int)(c / kTile);
        if (r0 + k < num_reqs)
            sm.ctile[r0 + k] = ct[k];
        ns[k] = (int)((L[k] + c - 1) / c);
        nt[k] = (L[k] + kTile - 1) / kTile;
        my_chunks += ns[k];
        my_cost += nt[k] + (ns[k] > 0 ? kSegmentCostTiles : 0);
        my_nonempty += ns[k] > 0 ? 1 : 0;
    }
    int n_splits, total_cost, n_nonempty;
    int sb_run = block_scan_excl(my_chunks, sm.red32, &n_splits);
    int cost_run = block_scan_excl(my_cost, sm.red32, &total_cost);
    int ne_run = block_scan_excl(my_nonempty, sm.red32, &n_nonempty);
    int lm[kReqPerThread];
    int my_lm = -1;
    {
        int c = cost_run;
#pragma unroll
        for (int k = 0; k < kReqPerThread; ++k) {
            lm[k] = ns[k] > 0 ? chunk_mid2(c, nt[k], ct[k], ns[k] - 1) : -1;
            my_lm = max(my_lm, lm[k]);
            c += nt[k] + (ns[k] > 0 ? kSegmentCostTiles : 0);
        }
    }
    int lm_run = block_scan_max_excl(my_lm, sm.red32);
#pragma unroll
    for (int k = 0; k < kReqPerThread; ++k) {
        const int r = r0 + k;
        lm_run = max(lm_run, lm[k]);
        if (r < num_reqs) {
            sm.sb[r] = sb_run;
            sm.cost0[r] = cost_run;
            sm.nonempty[r] = ne_run;
            sm.lastm[r] = lm_run;
        }
        sb_run += ns[k];
        cost_run += nt[k] + (ns[k] > 0 ? kSegmentCostTiles : 0);
        ne_run += ns[k] > 0 ? 1 : 0;
    }
    if (tid == 0) {
        sm.sb[num_reqs] = n_splits;
        sm.cost0[num_reqs] = total_cost;
        sm.nonempty[num_reqs] = n_nonempty;
    }
    __syncthreads();

    // ---- the split plan itself
    for (int r = tid; r <= num_reqs; r += kPlanThreads)
        plan.indptr[r] = sm.sb[r];
    if (tid == 0) {
        if (plan.status != nullptr)
            *plan.status = 0;
        *plan.chunk = uniform ? 0 : chunk;
    }
    if (plan.segments == nullptr)
        return;
    if (members > kMaxSms || n_splits > kMaxPlanSplits) {   // excluded on the host
        if (tid == 0 && plan.status != nullptr)
            *plan.status = 8;
        return;
    }

    // ---- first chunk of every member: the first chunk whose doubled cost
    // midpoint reaches the member's doubled share boundary
    for (int m = tid; m <= members; m += kPlanThreads) {
        int firstc = n_splits;
        if (m == 0) {
            firstc = 0;
        } else if (m < members) {
            // a doubled midpoint v reaches member m's boundary when
            // v >= 2 * total_cost * m / members: an integer threshold that rises
            // with m, so each chunk has exactly one member
            const long long thr = (2LL * total_cost * m + members - 1) / members;
            auto reaches = [&](int v) -> bool { return (long long)v >= thr; };
            // the first request whose last chunk reaches it (lastm is a running
            // maximum, so this request has chunks)
            int lo = 0, hi = num_reqs;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (reaches(sm.lastm[mid]))
                    hi = mid;
                else
                    lo = mid + 1;
            }
            if (lo < num_reqs) {
                const int r = lo;
                const int tiles = (sm.lens[r] + kTile - 1) / kTile;
                const int nsr = sm.sb[r + 1] - sm.sb[r];
                const int c = sm.cost0[r];
                int s = 0;
                const int chunk_tiles = sm.ctile[r];
                if (!reaches(chunk_mid2(c, tiles, chunk_tiles, 0))) {
                    int a = 1, b = nsr - 1;   // the last chunk reaches
                    while (a < b) {
                        const int mid = (a + b) >> 1;
                        if (reaches(chunk_mid2(c, tiles, chunk_tiles, mid)))
                            b = mid;
                        else
                            a = mid + 1;
                    }
                    s = a;
                }
                firstc = sm.sb[r] + s;
            }
        }
        sm.first[m] = firstc;
    }
    __syncthreads();

    // request of chunk i: the last r with sb[r] <= i (a request with chunks)
    auto req_of = [&](int chunk_i) -> int {
        int lo = 0, hi = num_reqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm.sb[mid] <= chunk_i)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    };

    // ---- segments per member: one per request with chunks in the member's range
    int my_nseg = 0, my_rfirst = 0;
    if (tid < members) {
        const int c0i = sm.first[tid], c1i = sm.first[tid + 1];
        if (c1i > c0i) {
            my_rfirst = req_of(c0i);
            const int rlast = req_of(c1i - 1);
            my_nseg = sm.nonempty[rlast + 1] - sm.nonempty[my_rfirst];
        }
    }
    int n_segs;
    const int seg0 = block_scan_excl(tid < members ? my_nseg : 0, sm.red32, &n_segs);
    if (tid < members) {
        sm.nseg[tid] = seg0;
        plan.seg_member_indptr[tid] = seg0;
    }
    if (tid == 0) {
        sm.nseg[members] = n_segs;
        plan.seg_member_indptr[members] = n_segs;
        *plan.seg_count = n_segs;
        plan.seg_req_indptr[num_reqs] = n_segs;
    }
    if (tid < members && my_nseg > 0) {
        const int c0i = sm.first[tid], c1i = sm.first[tid + 1];
        int id = seg0;
        for (int r = my_rfirst; id < seg0 + my_nseg; ++r) {
            if (sm.sb[r + 1] == sm.sb[r])
                continue;                            // a request without chunks
            const int a = max(c0i, sm.sb[r]) - sm.sb[r];
            const int b = min(c1i, sm.sb[r + 1]) - sm.sb[r];
            int4 seg;
            seg.x = r;
            const long long cr = (long long)sm.ctile[r] * kTile;
            seg.y = (int)(a * cr);
            seg.z = (int)min((long long)sm.lens[r], b * cr);
            seg.w = tid;
            plan.segments[id] = seg;
            ++id;
        }
    }
    __syncthreads();

    // ---- first segment of each request (for a request without chunks, that of
    // the next request with chunks, or the total)
    for (int r = tid; r < num_reqs; r += kPlanThreads) {
        int rr = r;
        if (sm.sb[r + 1] == sm.sb[r]) {
            const int want = sm.nonempty[r];          // that request's rank among them
            if (want >= n_nonempty) {
                plan.seg_req_indptr[r] = n_segs;
                continue;
            }
            int lo = r + 1, hi = num_reqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (sm.nonempty[mid + 1] > want)
                    hi = mid;
                else
                    lo = mid + 1;
            }
            rr = lo;
        }
        // the member holding the request's first chunk (the last member whose
        // range starts at or before it), and the request's place among that
        // member's requests
        const int c = sm.sb[rr];
        int lo = 0, hi = members - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm.first[mid] <= c)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int rf = req_of(sm.first[lo]);
        plan.seg_req_indptr[r] = sm.nseg[lo] + (sm.nonempty[rr] - sm.nonempty[rf]);
    }
}

// The query quantiser on its own (the FP8 decode runs it inside the plan grid).
__global__ void __launch_bounds__(kPlanThreads)
quantize_kernel(PlanBuffers plan)
{
    quantize_queries(plan, blockIdx.x);
}

}  // namespace

cudaError_t launch_quantize(const __nv_bfloat16 *q_nope, const __nv_bfloat16 *q_rope, int rows,
                            uint8_t *q8, int32_t *qexp, cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    PlanBuffers plan = {};
    plan.q_nope = q_nope;
    plan.q_rope = q_rope;
    plan.q8 = q8;
    plan.qexp = qexp;
    plan.q_rows = rows;
    quantize_kernel<<<(rows + kQuantRowsPerCta - 1) / kQuantRowsPerCta, kPlanThreads, 0, stream>>>(
        plan);
    return cudaGetLastError();
}

size_t plan_smem_bytes() { return sizeof(PlanSmem); }

cudaError_t launch_plan(const int32_t *seq_lens, int num_reqs, int budget, int members,
                        int uniform, PlanBuffers plan, cudaStream_t stream)
{
    const int smem = (int)sizeof(PlanSmem);
    cudaError_t err =
        cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess)
        return err;
    const int qctas =
        plan.q8 != nullptr ? (plan.q_rows + kQuantRowsPerCta - 1) / kQuantRowsPerCta : 0;
    // programmatic stream serialization: the launch overlaps the tail of the
    // previous kernel, whose completion the kernel waits for on entry
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(1 + qctas));
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan_kernel, seq_lens, num_reqs, budget, members, uniform,
                              plan);
}

}  // namespace plmla

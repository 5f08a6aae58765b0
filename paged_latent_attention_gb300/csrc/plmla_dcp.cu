// plmla_dcp.cu -- decode context parallelism: one rank's part of every
// request's history (TokenSpeed AgentX post, "AgentX benchmark results": ranks
// decode parts of the context and combine the partial attention results).
//
// Page column c of request r belongs to rank (c + r) mod world: each request's
// pages are dealt round-robin, so every rank holds the same number of its pages
// up to one, and the starting rank rotates with the request so that the
// requests' leftover pages spread over the ranks.  A rank's pages, in column
// order, form its own page-table row; softmax attention does not depend on the
// order of the tokens, so the rank decodes them as one history whose length is
// its pages' tokens (the request's last page, wherever it lands, is the only
// partial one).
#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kDcpThreads = 128;

__global__ void __launch_bounds__(kDcpThreads)
dcp_shard_kernel(const int32_t *__restrict__ table, int64_t ld, const int32_t *__restrict__ lens,
                 int num_reqs, int world, int rank, int32_t *__restrict__ table_out,
                 int64_t out_ld, int32_t *__restrict__ lens_out)
{
    const int r = blockIdx.x;
    if (r >= num_reqs)
        return;
    const int L = max(0, lens[r]);
    // pages of the history; a history longer than its table row keeps the
    // row's pages only (the decode has the same precondition)
    const int64_t n_full = ((int64_t)L + kPageTokens - 1) / kPageTokens;
    const int n = (int)(n_full < ld ? n_full : ld);
    const int c0 = ((rank - r) % world + world) % world;   // this rank's first column
    const int cnt = n > c0 ? (n - c0 + world - 1) / world : 0;
    for (int i = threadIdx.x; i < cnt; i += kDcpThreads)
        table_out[(int64_t)r * out_ld + i] = table[(int64_t)r * ld + c0 + (int64_t)i * world];
    if (threadIdx.x == 0) {
        // tokens in the row's pages, and in this rank's pages: all full but the
        // last column's, which holds the rest of the history
        const int64_t held = n == n_full ? (int64_t)L : (int64_t)n * kPageTokens;
        int64_t tokens = (int64_t)cnt * kPageTokens;
        if (cnt > 0 && (n - 1 - c0) % world == 0)
            tokens -= (int64_t)n * kPageTokens - held;
        lens_out[r] = (int32_t)tokens;
    }
}

}  // namespace

cudaError_t launch_dcp_shard(const int32_t *table, int64_t ld, const int32_t *lens, int num_reqs,
                             int world, int rank, int32_t *table_out, int64_t out_ld,
                             int32_t *lens_out, cudaStream_t stream)
{
    dcp_shard_kernel<<<num_reqs, kDcpThreads, 0, stream>>>(table, ld, lens, num_reqs, world, rank,
                                                           table_out, out_ld, lens_out);
    return cudaGetLastError();
}

}  // namespace plmla

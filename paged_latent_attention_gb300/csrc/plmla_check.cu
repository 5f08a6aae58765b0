// plmla_check.cu -- opt-in check of the page table a decode step reads.
//
// The decode reads page IDs from the table and hands them to the TMA unit as
// coordinates of the slab's [page][token][576] tensor map: an ID outside
// [0, num_pages) is never dereferenced, the unit fills such a tile with zeros,
// and the step's result is silently wrong.  With checks on, a kernel launched
// after the step looks at every table entry a request's history uses
// (columns 0 .. ceil(L / 1536) - 1) and, if one is out of range, writes a status
// code into the step's status word (it never traps); a history longer than the
// table's row stride allows is reported too.  So a caller can tell a bad
// table from a good one (the pages' flat-layout section: one global page ID per
// page, honoured through the table's row stride).
#include "plmla_internal.cuh"

namespace plmla {
namespace {

constexpr int kCheckThreads = 256;
constexpr int32_t kStatusBadPage = 40;      // a used page-table entry outside [0, num_pages)
constexpr int32_t kStatusTableTooShort = 41; // a history needs more columns than the row holds

__global__ void __launch_bounds__(kCheckThreads)
check_pages_kernel(const int32_t *__restrict__ seq_lens, int num_reqs,
                   const int32_t *__restrict__ page_table, int64_t table_ld, int64_t num_pages,
                   int32_t *status)
{
    // one block per request, threads over its page columns
    const int r = blockIdx.x;
    if (r >= num_reqs)
        return;
    const int L = max(0, seq_lens[r]);
    const int64_t need = (L + kPageTokens - 1) / kPageTokens;
    if (need > table_ld && threadIdx.x == 0)
        atomicExch(status, kStatusTableTooShort);
    const int cols = (int)min(need, table_ld);   // never read past the row
    const int32_t *row = page_table + (int64_t)r * table_ld;
    for (int c = threadIdx.x; c < cols; c += kCheckThreads) {
        const int32_t p = row[c];
        if (p < 0 || (int64_t)p >= num_pages)
            atomicExch(status, kStatusBadPage);
    }
}

}  // namespace

cudaError_t launch_check_pages(const int32_t *seq_lens, int num_reqs, const int32_t *page_table,
                               int64_t table_ld, int64_t num_pages, int32_t *status,
                               cudaStream_t stream)
{
    check_pages_kernel<<<num_reqs, kCheckThreads, 0, stream>>>(seq_lens, num_reqs, page_table,
                                                               table_ld, num_pages, status);
    return cudaGetLastError();
}

}  // namespace plmla

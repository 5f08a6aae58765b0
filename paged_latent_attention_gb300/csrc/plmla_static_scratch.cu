// plmla_static_scratch.cu -- mla_decode for callers that cannot allocate.
//
// Some callers have no way to hand the library a device workspace: a serving
// engine that reserved nearly all device memory for its KV page pool up front
// and forbids later cudaMalloc calls, a plugin living inside a framework that
// owns the device allocator, or a latency-critical loop that cannot afford the
// implicit device synchronisation cudaMalloc/cudaFree may cause.  For them this
// entry point runs the same plan -> split-decode -> combine kernels as
// mla_decode, with the workspace carved from a fixed array compiled into the
// library instead of from caller memory.
//
// The array is a file-scope static __device__ object, so every GPU that loads
// the library holds it until the process exits.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in object),
// so the first call on each device looks the real address up with
// cudaGetSymbolAddress while that device is current, checks the result, and
// caches it; later calls reuse the cached pointer.  The cache is keyed by device
// ordinal only, so it does not survive a device reset (documented in the header).
// The step's status word is the array's first 4 bytes (mla_decode's workspace
// layout); mla_static_scratch_status copies it out without allocating.
#include <stdint.h>

#include <mutex>

#include <cuda_runtime.h>

#include "plmla.h"

namespace {

constexpr size_t kScratchBytes = PLMLA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_lookup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device (looked up once).
plmla_status scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return PLMLA_CUDA_ERROR;
    if (dev >= kMaxDevices)
        return PLMLA_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_lookup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr)
            return PLMLA_CUDA_ERROR;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return PLMLA_OK;
}

}  // namespace

extern "C" plmla_status mla_decode_static_scratch(
    const void *q_nope_absorbed, const void *q_rope, const void *gate, const void *slab_base,
    int64_t num_pages, int64_t page_stride_elems, const int32_t *page_table,
    int64_t page_table_ld, const int32_t *seq_lens, int32_t num_reqs, int32_t n_q_per_req,
    int32_t num_heads, float scale, void *out, float *lse, int32_t cta_budget,
    int32_t min_splits_per_req, void *stream)
{
    void *scratch = nullptr;
    plmla_status st = scratch_for_current_device(&scratch);
    if (st != PLMLA_OK)
        return st;
    const size_t need = mla_workspace_size(num_reqs, n_q_per_req, num_heads, cta_budget,
                                           min_splits_per_req);
    if (need == 0)
        return PLMLA_INVALID_ARGUMENT;
    if (need > kScratchBytes)
        return PLMLA_WORKSPACE_TOO_SMALL;
    // Nothing in the scratch has to start at zero: each call's plan kernel
    // writes every plan entry, split state and counter the later kernels read.
    return mla_decode(q_nope_absorbed, q_rope, gate, slab_base, num_pages, page_stride_elems,
                      page_table, page_table_ld, seq_lens, num_reqs, n_q_per_req, num_heads,
                      scale, out, lse, scratch, kScratchBytes, cta_budget, min_splits_per_req,
                      stream);
}

extern "C" plmla_status mla_static_scratch_status(int32_t *status_out, void *stream)
{
    if (status_out == nullptr || (reinterpret_cast<uintptr_t>(status_out) % 4) != 0)
        return PLMLA_INVALID_ARGUMENT;
    void *scratch = nullptr;
    const plmla_status st = scratch_for_current_device(&scratch);
    if (st != PLMLA_OK)
        return st;
    // the status word sits at offset 0 of mla_decode's workspace
    const cudaError_t err = cudaMemcpyAsync(status_out, scratch, sizeof(int32_t),
                                            cudaMemcpyDefault,
                                            static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PLMLA_OK : PLMLA_CUDA_ERROR;
}

// mla_noalloc.cu -- dense decode for callers that cannot allocate device memory.
//
// mla_decode needs a caller-provided workspace (the error word plus the fp32
// per-split partials that the split-K reduce merges).  Some callers cannot get
// one: code that runs where cudaMalloc is unavailable or forbidden (inside a
// region that must not allocate, such as a latency-critical serving loop with a
// fixed memory budget, or a host framework that hands over only its input and
// output buffers).  This entry point serves them: the scratch lives in a
// file-scope __device__ array that the library owns, so the call allocates
// nothing.  The pages have no counterpart of this entry point.
#include <mutex>

#include "mla_internal.h"

namespace {

// The static scratch: every GPU that loads the library holds these bytes until
// the process exits.
__device__ __align__(256) unsigned char g_mla_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices];  // device address of the array, per device

// Once per device, with that device current: look up the array's device
// address.  In host code the array's name is only a host-side stand-in, so the
// kernels must be given this address instead.
int scratch_for_current_device(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mla_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MLA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_noalloc(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                                  const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                                  const int32_t* kv_indices, const int32_t* kv_indptr,
                                  int32_t batch, int32_t q_len, int32_t num_heads, float scale,
                                  float kv_scale, void* o_lat, float* lse, void* stream)
{
    if (!plan) return MLA_ERR_INVALID_ARG;
    // The scratch need comes from the plan's shape and split count, not from
    // its workspace_bytes field, which a caller could have edited; mla_decode
    // rejects a plan whose field disagrees with that need.
    if (mla::needed_workspace(plan) > (int64_t)MLA_NOALLOC_SCRATCH_BYTES)
        return MLA_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc != MLA_OK) return rc;
    // The array keeps the previous call's contents.  Nothing in it has to start
    // at zero: the split kernel writes every partial and LSE before the reduce
    // reads them, and the error word at its head is only ever ORed into (this
    // entry point never reads it back, so stale bits there are harmless).
    return mla_decode(plan, q_lat, q_pe, pool, pool_rows, seq_lens, kv_indices, kv_indptr,
                      batch, q_len, num_heads, scale, kv_scale, o_lat, lse, scratch,
                      (int64_t)MLA_NOALLOC_SCRATCH_BYTES, stream);
}

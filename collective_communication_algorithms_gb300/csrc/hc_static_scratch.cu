// hc_static_scratch.cu -- hc_reduce_scatter_static_scratch: the step-mode
// ReduceScatter for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and are not
// allowed to allocate device memory themselves: a plugin inside a host
// framework that owns every device allocation through its own pool, or a
// latency-critical path that cannot afford cudaMalloc's implicit
// synchronisation or its failure under memory pressure.  The ordinary
// step-mode ReduceScatter needs a caller-provided scratch buffer whenever a
// rank's output is not inside its input; this entry point instead uses a
// fixed array that the library itself places in every GPU's memory when the
// library is loaded (HC_STATIC_SCRATCH_BYTES per GPU, held until the process
// exits), and allocates nothing.
#include <cuda_runtime.h>

#include <atomic>

#include "hc_internal.h"

// The scratch itself.  Host code must never use this name as a device
// address (on the host it is only a stand-in object); its device address is
// fetched with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char hc_static_scratch[HC_STATIC_SCRATCH_BYTES];

namespace {

// Device address of hc_static_scratch, per device, looked up on the first
// call made with that device current.
std::atomic<void*> g_static_scratch_addr[hc::kMaxRanks];  // null-initialised (static storage)

hc_status_t static_scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HC_ERR_CUDA;
    if (dev < 0 || dev >= hc::kMaxRanks) return HC_ERR_CUDA;
    void* a = g_static_scratch_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        // two threads may both look it up; they store the same address
        if (cudaGetSymbolAddress(&a, hc_static_scratch) != cudaSuccess || !a) return HC_ERR_CUDA;
        g_static_scratch_addr[dev].store(a, std::memory_order_release);
    }
    *out = a;
    return HC_OK;
}

}  // namespace

extern "C" hc_status_t hc_reduce_scatter_static_scratch(
    const void* const* send, void* const* recv, int P, size_t count, hc_dtype_t dtype,
    hc_op_t op, hc_algo_t algo, int ranks_per_server, size_t max_loop_bytes, hc_stream_t stream) {
    // Reject work that does not fit before touching the device.  For invalid
    // arguments hc_scratch_bytes returns 0 and hc_reduce_scatter reports them.
    const size_t need = hc_scratch_bytes(algo, P, count, dtype);
    if (need > (size_t)HC_STATIC_SCRATCH_BYTES) return HC_ERR_SCRATCH;
    void* scratch = nullptr;
    const hc_status_t st = static_scratch_address(&scratch);
    if (st != HC_OK) return st;
    hc_opts_t o;
    o.struct_size = sizeof(hc_opts_t);
    o.mode = HC_MODE_STEP;
    o.ranks_per_server = ranks_per_server;
    o.max_loop_bytes = max_loop_bytes;
    o.scratch = scratch;
    o.scratch_bytes = HC_STATIC_SCRATCH_BYTES;
    o.host_buffers = 0;
    return hc_reduce_scatter(send, recv, P, count, dtype, op, algo, &o, stream);
}

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
// fixed array of HC_STATIC_SCRATCH_BYTES that the library itself places in
// the memory of every GPU it runs on, held until the process exits, and
// allocates nothing.
//
// When the array is committed depends on the CUDA runtime's module loading.
// Under lazy loading (CUDA_MODULE_LOADING=LAZY, the default of current
// runtimes) the module holding it is loaded by the first address lookup on a
// device, i.e. inside the first call that needs the scratch, and that call
// fails with HC_ERR_CUDA if the device cannot give it 32 MiB at that moment;
// with CUDA_MODULE_LOADING=EAGER it is committed when the runtime first
// initialises each device.
#include <cuda_runtime.h>

#include <atomic>

#include "hc_internal.h"

// The scratch itself.  Host code must never use this name as a device
// address (on the host it is only a stand-in object); its device address is
// fetched with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char hc_static_scratch[HC_STATIC_SCRATCH_BYTES];

namespace {

// Device address of hc_static_scratch, per device ordinal, looked up on the
// first call that needs it with that device current.  The address is never
// looked up again, so the library must not be used across a
// cudaDeviceReset() of that device (which unloads the module and may place
// the array elsewhere when it is loaded again).
std::atomic<void*> g_static_scratch_addr[hc::kMaxDevices];  // null-initialised (static storage)

hc_status_t static_scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HC_ERR_CUDA;
    if (dev < 0 || dev >= hc::kMaxDevices) return HC_ERR_CUDA;
    void* a = g_static_scratch_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        // two threads may both look it up; they store the same address
        if (cudaGetSymbolAddress(&a, hc_static_scratch) != cudaSuccess || !a) {
            cudaGetLastError();  // leave no pending error behind for the caller
            return HC_ERR_CUDA;
        }
        g_static_scratch_addr[dev].store(a, std::memory_order_release);
    }
    *out = a;
    return HC_OK;
}

}  // namespace

extern "C" hc_status_t hc_reduce_scatter_static_scratch(
    const void* const* send, void* const* recv, int P, size_t count, hc_dtype_t dtype,
    hc_op_t op, hc_algo_t algo, int ranks_per_server, size_t max_loop_bytes, hc_stream_t stream) {
    hc_opts_t o;
    o.struct_size = sizeof(hc_opts_t);
    o.mode = HC_MODE_STEP;
    o.ranks_per_server = ranks_per_server;
    o.max_loop_bytes = max_loop_bytes;
    o.scratch = nullptr;
    o.scratch_bytes = 0;
    o.host_buffers = 0;
    // Validate every argument before the device is touched.  Without a
    // scratch, prepare() answers HC_ERR_SCRATCH only when some rank is out of
    // place (and every other argument is valid); when every rank is in place
    // the call needs no scratch at all.
    hc::Prepared c;
    hc_status_t st = hc::prepare(HC_COLL_REDUCE_SCATTER, send, recv, P, count, dtype, op, algo, &o,
                                 -1, &c);
    if (st == HC_OK) return hc::execute(c, (cudaStream_t)stream);
    if (st != HC_ERR_SCRATCH) return st;
    if (hc_scratch_bytes(algo, P, count, dtype) > (size_t)HC_STATIC_SCRATCH_BYTES) return HC_ERR_SCRATCH;
    void* scratch = nullptr;
    st = static_scratch_address(&scratch);
    if (st != HC_OK) return st;
    o.scratch = scratch;
    o.scratch_bytes = HC_STATIC_SCRATCH_BYTES;
    st = hc::prepare(HC_COLL_REDUCE_SCATTER, send, recv, P, count, dtype, op, algo, &o, -1, &c);
    if (st != HC_OK) return st;
    return hc::execute(c, (cudaStream_t)stream);
}

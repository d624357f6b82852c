// hc_fused_pipe.cu -- fused kernels (register path and TMA-staged) of one schedule (Pipeline intra-server chains, then the inter-server chain):
// AllReduce and ReduceScatter, 1 vector per thread.  One translation unit per schedule keeps each compile short.
#include "hc_device.cuh"

namespace hc {

void* pick_fused_pipe(int coll, hc_dtype_t dt, hc_op_t op, int V) {
    if (V != 1) return nullptr;
    return coll == 0 ? pick_fused_dt<HC_ALGO_PIPELINE, 0, 1>(dt, op) : pick_fused_dt<HC_ALGO_PIPELINE, 1, 1>(dt, op);
}

void* pick_fused_pipe_tma(int coll, hc_dtype_t dt, hc_op_t op) { return pick_tma<HC_ALGO_PIPELINE>(coll, dt, op); }

}  // namespace hc

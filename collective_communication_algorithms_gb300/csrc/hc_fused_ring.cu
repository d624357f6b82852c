// hc_fused_ring.cu -- fused kernels (register path and TMA-staged) of one schedule (Ring chain ((X_{k+1} (+) X_{k+2}) (+) ...) (+) X_k):
// AllReduce and ReduceScatter, 1 vector per thread.  One translation unit per schedule keeps each compile short.
#include "hc_device.cuh"

namespace hc {

void* pick_fused_ring(int coll, hc_dtype_t dt, hc_op_t op, int V) {
    if (V != 1) return nullptr;
    return coll == 0 ? pick_fused_dt<HC_ALGO_RING, 0, 1>(dt, op) : pick_fused_dt<HC_ALGO_RING, 1, 1>(dt, op);
}

void* pick_fused_ring_tma(int coll, hc_dtype_t dt, hc_op_t op) { return pick_tma<HC_ALGO_RING>(coll, dt, op); }

}  // namespace hc

// hc_fused_hier.cu -- fused kernels (register path and TMA-staged) of one schedule (plain hierarchical: RHD tree over servers of intra-server chains):
// AllReduce only, 1 vector per thread.  One translation unit per schedule keeps each compile short.
#include "hc_device.cuh"

namespace hc {

void* pick_fused_hier(int coll, hc_dtype_t dt, hc_op_t op, int V) {
    if (V != 1 || coll != 0) return nullptr;
    return pick_fused_dt<HC_ALGO_HIER, 0, 1>(dt, op);
}

void* pick_fused_hier_tma(int coll, hc_dtype_t dt, hc_op_t op) {
    if (coll != 0) return nullptr;  // AllReduce only
    switch (dt) {
    case HC_INT32: return pick_tma_op<HC_ALGO_HIER, 0, HC_INT32>(op);
    case HC_FLOAT32: return pick_tma_op<HC_ALGO_HIER, 0, HC_FLOAT32>(op);
    default: return pick_tma_op<HC_ALGO_HIER, 0, HC_BFLOAT16>(op);
    }
}

}  // namespace hc

// hc_fused_rhd.cu -- fused kernels (register path and TMA-staged) of one schedule (RHD fold + balanced pairwise tree):
// AllReduce and ReduceScatter with 1 vector per thread, and the bf16
// sum / prod AllReduce with 2 vectors per thread (the only shape that
// measured faster with 2); separate kernels for 16 or more ranks.  One translation unit per schedule keeps each compile short.
#include "hc_device.cuh"

namespace hc {

void* pick_fused_rhd(int coll, hc_dtype_t dt, hc_op_t op, int V, bool large) {
    if (large) {
        if (V != 1) return nullptr;
        return coll == 0 ? pick_fused_dt<kAlgoRhdLarge, 0, 1>(dt, op) : pick_fused_dt<kAlgoRhdLarge, 1, 1>(dt, op);
    }
    if (V == 2) {
        if (coll != 0 || dt != HC_BFLOAT16) return nullptr;
        if (op == HC_SUM) return (void*)fused_reduce<HC_ALGO_RHD, 0, HC_BFLOAT16, HC_SUM, 2>;
        if (op == HC_PROD) return (void*)fused_reduce<HC_ALGO_RHD, 0, HC_BFLOAT16, HC_PROD, 2>;
        return nullptr;
    }
    return coll == 0 ? pick_fused_dt<HC_ALGO_RHD, 0, 1>(dt, op) : pick_fused_dt<HC_ALGO_RHD, 1, 1>(dt, op);
}

void* pick_fused_rhd_tma(int coll, hc_dtype_t dt, hc_op_t op, bool large) {
    return large ? pick_tma<kAlgoRhdLarge>(coll, dt, op) : pick_tma<HC_ALGO_RHD>(coll, dt, op);
}

}  // namespace hc

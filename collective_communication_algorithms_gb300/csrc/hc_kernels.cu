// hc_kernels.cu -- sm_103a kernels of libhc.
//
//  step_kernel  (step-faithful mode): one launch per schedule step; every item
//               reads its operands' 16-byte vectors from the peers' buffers,
//               reduces them in the item's order and writes every output.  It
//               is the "recv_ptr[i] = reduce_op(recv_ptr[i], local_ptr[i])"
//               loop of the ring pseudo-code ("Ring AllReduce带宽最优的环形流水线"),
//               the halving reduce / doubling memcpy of the RHD pseudo-code,
//               and the Pipeline article's LocalCopy, with the HCOMM transfer
//               replaced by a load from the peer's buffer.
//  fused_*      (fused mode): one launch per collective; each thread takes a
//               16-byte vector of a segment, loads it from every rank, reduces
//               in registers in exactly the association order the schedule
//               implies (Ring chain, RHD fold + pairwise tree, Pipeline
//               intra-server chain then inter-server chain) and stores it to
//               every output.  Minimum traffic: AllReduce reads and writes
//               P n b bytes.
//
// Arithmetic (must match the reduction semantics in hc.h bit for bit):
//  int32 wrap; fp32 IEEE RNE via __fadd_rn / __fmul_rn (no contraction, no
//  flush to zero); bf16 widened to fp32, op, then cvt.rn.bf16x2.f32;
//  max/min by IEEE totalOrder keys on the bit patterns.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "hc_internal.h"

namespace hc {
namespace {

// ---------------------------------------------------------------------------
// element-wise operators on 32-bit words (one fp32/int32, or two bf16)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key32(uint32_t u) {
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint32_t key16(uint32_t h) {  // h in the low 16 bits
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <hc_dtype_t DT, hc_op_t OP>
struct WordOp;

template <hc_op_t OP>
struct WordOp<HC_INT32, OP> {
    __device__ __forceinline__ static uint32_t f(uint32_t a, uint32_t b) {
        if (OP == HC_SUM) return a + b;
        if (OP == HC_PROD) return a * b;
        if (OP == HC_MAX) return ((int32_t)a < (int32_t)b) ? b : a;
        return ((int32_t)b < (int32_t)a) ? b : a;
    }
};

template <hc_op_t OP>
struct WordOp<HC_FLOAT32, OP> {
    __device__ __forceinline__ static uint32_t f(uint32_t a, uint32_t b) {
        if (OP == HC_SUM) return __float_as_uint(__fadd_rn(__uint_as_float(a), __uint_as_float(b)));
        if (OP == HC_PROD) return __float_as_uint(__fmul_rn(__uint_as_float(a), __uint_as_float(b)));
        if (OP == HC_MAX) return key32(a) < key32(b) ? b : a;
        return key32(b) < key32(a) ? b : a;
    }
};

template <hc_op_t OP>
struct WordOp<HC_BFLOAT16, OP> {
    __device__ __forceinline__ static uint32_t f(uint32_t a, uint32_t b) {
        if (OP == HC_SUM)
            return pack_bf16x2(__fadd_rn(bf_lo(a), bf_lo(b)), __fadd_rn(bf_hi(a), bf_hi(b)));
        if (OP == HC_PROD)
            return pack_bf16x2(__fmul_rn(bf_lo(a), bf_lo(b)), __fmul_rn(bf_hi(a), bf_hi(b)));
        uint32_t alo = a & 0xFFFFu, blo = b & 0xFFFFu, ahi = a >> 16, bhi = b >> 16;
        uint32_t lo, hi;
        if (OP == HC_MAX) {
            lo = key16(alo) < key16(blo) ? blo : alo;
            hi = key16(ahi) < key16(bhi) ? bhi : ahi;
        } else {
            lo = key16(blo) < key16(alo) ? blo : alo;
            hi = key16(bhi) < key16(ahi) ? bhi : ahi;
        }
        return lo | (hi << 16);
    }
};

template <hc_dtype_t DT, hc_op_t OP>
__device__ __forceinline__ uint4 vop(const uint4& a, const uint4& b) {
    using W = WordOp<DT, OP>;
    return make_uint4(W::f(a.x, b.x), W::f(a.y, b.y), W::f(a.z, b.z), W::f(a.w, b.w));
}
template <hc_dtype_t DT, hc_op_t OP>
__device__ __forceinline__ uint32_t vop(uint32_t a, uint32_t b) {
    return WordOp<DT, OP>::f(a, b);
}

// ---------------------------------------------------------------------------
// memory access: 16-byte vectors, or one element (ragged end of a vector)
// ---------------------------------------------------------------------------
template <int ES>
__device__ __forceinline__ uint32_t ld_elem(uintptr_t p) {
    if (ES == 2) return *(const uint16_t*)p;
    return *(const uint32_t*)p;
}
template <int ES>
__device__ __forceinline__ void st_elem(uintptr_t p, uint32_t v) {
    if (ES == 2) *(uint16_t*)p = (uint16_t)v;
    else *(uint32_t*)p = v;
}
__device__ __forceinline__ uint4 ld_vec(uintptr_t p) { return *(const uint4*)p; }
__device__ __forceinline__ void st_vec(uintptr_t p, const uint4& v) { *(uint4*)p = v; }
// streaming variants for data touched once by the fused kernels
__device__ __forceinline__ uint4 ld_stream(uintptr_t p) { return __ldcs((const uint4*)p); }
__device__ __forceinline__ void st_stream(uintptr_t p, const uint4& v) { __stcs((uint4*)p, v); }

template <hc_dtype_t DT>
struct DT_ {
    static constexpr int ES = DT == HC_BFLOAT16 ? 2 : 4;
    static constexpr int A = 16 / ES;
};

// ---------------------------------------------------------------------------
// step kernel
// ---------------------------------------------------------------------------
constexpr int kStepThreads = 256;

template <hc_dtype_t DT, hc_op_t OP, int MAXI>
__global__ void __launch_bounds__(kStepThreads)
step_kernel(const __grid_constant__ StepParams<MAXI> p) {
    constexpr int ES = DT_<DT>::ES;
    constexpr int A = DT_<DT>::A;
    const int b = blockIdx.x;
    int it = 0;
    while (it + 1 < p.nitems && p.items[it + 1].cta_begin <= b) it++;
    const DevItem& I = p.items[it];
    const int cend = (it + 1 < p.nitems) ? p.items[it + 1].cta_begin : p.total_ctas;
    const int64_t nthreads = (int64_t)(cend - I.cta_begin) * blockDim.x;
    const int64_t t0 = (int64_t)(b - I.cta_begin) * blockDim.x + threadIdx.x;
    const int nseg = I.seg_width * I.seg_reps;

    for (int si = 0; si < nseg; si++) {
        const int seg = I.seg_first + (si / I.seg_width) * I.seg_stride + (si % I.seg_width);
        const int64_t sbeg = (int64_t)seg * p.L;
        int64_t send_ = sbeg + p.L;
        if (send_ > p.n) send_ = p.n;
        int64_t hi = sbeg + p.hi;
        if (hi > send_) hi = send_;
        const int64_t lo = sbeg + p.lo;
        for (int64_t e = lo + t0 * A; e < hi; e += nthreads * A) {
            const uintptr_t off = (uintptr_t)e * ES;
            int r = I.in_rot;
            if (e + A <= hi) {
                uint4 v = ld_vec(p.base[I.in_loc][I.in_base + r] + off);
                for (int j = 1; j < I.in_cnt; j++) {
                    if (++r == I.in_mod) r = 0;
                    v = vop<DT, OP>(v, ld_vec(p.base[I.in_loc][I.in_base + r] + off));
                }
                if (I.acc_rank >= 0) v = vop<DT, OP>(ld_vec(p.base[I.acc_loc][I.acc_rank] + off), v);
                int o = I.out_rot;
                for (int j = 0; j < I.out_cnt; j++) {
                    st_vec(p.base[I.out_loc][I.out_base + o] + off, v);
                    if (++o == I.out_mod) o = 0;
                }
            } else {
                // ragged end of the rank vector: element by element
                for (int64_t x = e; x < hi; x++) {
                    const uintptr_t xo = (uintptr_t)x * ES;
                    int rr = I.in_rot;
                    uint32_t v = ld_elem<ES>(p.base[I.in_loc][I.in_base + rr] + xo);
                    for (int j = 1; j < I.in_cnt; j++) {
                        if (++rr == I.in_mod) rr = 0;
                        v = vop<DT, OP>(v, ld_elem<ES>(p.base[I.in_loc][I.in_base + rr] + xo));
                    }
                    if (I.acc_rank >= 0)
                        v = vop<DT, OP>(ld_elem<ES>(p.base[I.acc_loc][I.acc_rank] + xo), v);
                    int o = I.out_rot;
                    for (int j = 0; j < I.out_cnt; j++) {
                        st_elem<ES>(p.base[I.out_loc][I.out_base + o] + xo, v);
                        if (++o == I.out_mod) o = 0;
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// fused kernels
// ---------------------------------------------------------------------------
struct FusedParams {
    uintptr_t src[kMaxRanks];  // global-indexed input view of each rank
    uintptr_t dst[kMaxRanks];  // global-indexed output view of each rank
    int64_t L;
    int64_t n;
    int P;
    int p_intra;
    int pp;                    // RHD: power-of-two core size
    int rfold;                 // RHD: number of folded pairs
    unsigned long long skip_mask;  // AllGather: ranks whose own segment is already in place
};

constexpr int kFusedThreads = 256;
constexpr int kBatch = 8;

// Reduce a chain x_0 (+) x_1 (+) ... (+) x_{cnt-1}, x_i = load(rank(i)), with
// loads issued kBatch at a time for memory-level parallelism.
template <hc_dtype_t DT, hc_op_t OP, class V, class Load>
__device__ __forceinline__ V chain_reduce(int cnt, int base, int rot, int mod, Load load) {
    int r = rot;
    V acc = load(base + r);
    int i = 1;
    for (; i + kBatch <= cnt; i += kBatch) {
        V x[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; j++) {
            if (++r == mod) r = 0;
            x[j] = load(base + r);
        }
#pragma unroll
        for (int j = 0; j < kBatch; j++) acc = vop<DT, OP>(acc, x[j]);
    }
    for (; i < cnt; i++) {
        if (++r == mod) r = 0;
        acc = vop<DT, OP>(acc, load(base + r));
    }
    return acc;
}

// Balanced pairwise tree over leaves [w0, w0 + N), N a power of two.
template <hc_dtype_t DT, hc_op_t OP, int N, class V, class Leaf>
__device__ __forceinline__ V tree_fixed(int w0, Leaf leaf) {
    if constexpr (N == 1) {
        return leaf(w0);
    } else {
        V a = tree_fixed<DT, OP, N / 2, V>(w0, leaf);
        V b = tree_fixed<DT, OP, N / 2, V>(w0 + N / 2, leaf);
        return vop<DT, OP>(a, b);
    }
}

// RHD tree: leaves u_w = X_{2w+1} (+) X_{2w} for w < rfold (the fold step:
// rank 2w+1's data arrives at rank 2w), else X_{w + rfold}; balanced
// pairwise tree over the pp leaves, partner bit 0 first.
template <hc_dtype_t DT, hc_op_t OP, class V, class Load>
__device__ __forceinline__ V rhd_reduce(int pp, int rfold, Load load) {
    auto leaf = [&](int w) -> V {
        if (w < rfold) return vop<DT, OP>(load(2 * w + 1), load(2 * w));
        return load(w + rfold);
    };
    switch (pp) {
    case 1: return tree_fixed<DT, OP, 1, V>(0, leaf);
    case 2: return tree_fixed<DT, OP, 2, V>(0, leaf);
    case 4: return tree_fixed<DT, OP, 4, V>(0, leaf);
    default: break;
    }
    // pp >= 8: subtrees of 8 leaves combined pairwise as soon as both halves
    // exist (same tree, fewer live registers)
    V t0 = tree_fixed<DT, OP, 8, V>(0, leaf);
    if (pp == 8) return t0;
    t0 = vop<DT, OP>(t0, tree_fixed<DT, OP, 8, V>(8, leaf));
    if (pp == 16) return t0;
    V t1 = tree_fixed<DT, OP, 8, V>(16, leaf);
    t1 = vop<DT, OP>(t1, tree_fixed<DT, OP, 8, V>(24, leaf));
    t0 = vop<DT, OP>(t0, t1);
    if (pp == 32) return t0;
    V t2 = tree_fixed<DT, OP, 8, V>(32, leaf);
    t2 = vop<DT, OP>(t2, tree_fixed<DT, OP, 8, V>(40, leaf));
    V t3 = tree_fixed<DT, OP, 8, V>(48, leaf);
    t3 = vop<DT, OP>(t3, tree_fixed<DT, OP, 8, V>(56, leaf));
    return vop<DT, OP>(t0, vop<DT, OP>(t2, t3));
}

// The association order of segment k for each algorithm.
template <hc_algo_t ALGO, hc_dtype_t DT, hc_op_t OP, class V, class Load>
__device__ __forceinline__ V segment_reduce(const FusedParams& p, int k, Load load) {
    if constexpr (ALGO == HC_ALGO_RING) {
        // chain X_{k+1} (+) X_{k+2} (+) ... (+) X_k
        return chain_reduce<DT, OP, V>(p.P, 0, (k + 1) % p.P, p.P, load);
    } else if constexpr (ALGO == HC_ALGO_RHD) {
        return rhd_reduce<DT, OP, V>(p.pp, p.rfold, load);
    } else {
        // intra-server chains rotated from l, then the inter-server chain from s+1
        const int pin = p.p_intra, pout = p.P / p.p_intra;
        const int s = k / pin, l = k % pin;
        int t = s + 1 == pout ? 0 : s + 1;
        V acc = chain_reduce<DT, OP, V>(pin, t * pin, l, pin, load);
        for (int i = 1; i < pout; i++) {
            if (++t == pout) t = 0;
            acc = vop<DT, OP>(acc, chain_reduce<DT, OP, V>(pin, t * pin, l, pin, load));
        }
        return acc;
    }
}

// AllReduce (COLL = 0) and ReduceScatter (COLL = 1).  grid.y = segment.
template <hc_algo_t ALGO, int COLL, hc_dtype_t DT, hc_op_t OP>
__global__ void __launch_bounds__(kFusedThreads)
fused_reduce(const __grid_constant__ FusedParams p) {
    constexpr int ES = DT_<DT>::ES;
    constexpr int A = DT_<DT>::A;
    const int k = blockIdx.y;
    const int64_t sbeg = (int64_t)k * p.L;
    if (sbeg >= p.n) return;
    const int64_t send_ = (sbeg + p.L < p.n) ? sbeg + p.L : p.n;
    const int64_t nfull = (send_ - sbeg) / A;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nfull; v += stride) {
        const uintptr_t off = (uintptr_t)(sbeg + v * A) * ES;
        auto load = [&](int r) -> uint4 { return ld_stream(p.src[r] + off); };
        uint4 acc = segment_reduce<ALGO, DT, OP, uint4>(p, k, load);
        if (COLL == 0) {
            for (int r = 0; r < p.P; r++) st_stream(p.dst[r] + off, acc);
        } else {
            st_stream(p.dst[k] + off, acc);
        }
    }
    // ragged end: fewer than A elements after the last full vector
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int64_t x = sbeg + nfull * A; x < send_; x++) {
            const uintptr_t xo = (uintptr_t)x * ES;
            auto load = [&](int r) -> uint32_t { return ld_elem<ES>(p.src[r] + xo); };
            uint32_t acc = segment_reduce<ALGO, DT, OP, uint32_t>(p, k, load);
            if (COLL == 0) {
                for (int r = 0; r < p.P; r++) st_elem<ES>(p.dst[r] + xo, acc);
            } else {
                st_elem<ES>(p.dst[k] + xo, acc);
            }
        }
    }
}

// AllGather: segment k read once from its owner, written to every rank
// (the owner's own copy only when it is not already in place).
template <int ES>
__global__ void __launch_bounds__(kFusedThreads)
fused_allgather(const __grid_constant__ FusedParams p) {
    constexpr int A = 16 / ES;
    const int k = blockIdx.y;
    const int64_t sbeg = (int64_t)k * p.L;
    if (sbeg >= p.n) return;
    const int64_t send_ = (sbeg + p.L < p.n) ? sbeg + p.L : p.n;
    const int64_t nfull = (send_ - sbeg) / A;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const bool skip_own = (p.skip_mask >> k) & 1ull;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nfull; v += stride) {
        const uintptr_t off = (uintptr_t)(sbeg + v * A) * ES;
        const uint4 x = ld_stream(p.src[k] + off);
        for (int r = 0; r < p.P; r++)
            if (r != k || !skip_own) st_stream(p.dst[r] + off, x);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int64_t x = sbeg + nfull * A; x < send_; x++) {
            const uintptr_t xo = (uintptr_t)x * ES;
            const uint32_t val = ld_elem<ES>(p.src[k] + xo);
            for (int r = 0; r < p.P; r++)
                if (r != k || !skip_own) st_elem<ES>(p.dst[r] + xo, val);
        }
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <hc_algo_t ALGO, int COLL, hc_dtype_t DT>
void* pick_reduce_op(hc_op_t op) {
    switch (op) {
    case HC_SUM: return (void*)fused_reduce<ALGO, COLL, DT, HC_SUM>;
    case HC_PROD: return (void*)fused_reduce<ALGO, COLL, DT, HC_PROD>;
    case HC_MAX: return (void*)fused_reduce<ALGO, COLL, DT, HC_MAX>;
    default: return (void*)fused_reduce<ALGO, COLL, DT, HC_MIN>;
    }
}
template <hc_algo_t ALGO, int COLL>
void* pick_reduce_dt(hc_dtype_t dt, hc_op_t op) {
    switch (dt) {
    case HC_INT32: return pick_reduce_op<ALGO, COLL, HC_INT32>(op);
    case HC_FLOAT32: return pick_reduce_op<ALGO, COLL, HC_FLOAT32>(op);
    default: return pick_reduce_op<ALGO, COLL, HC_BFLOAT16>(op);
    }
}
template <int COLL>
void* pick_reduce(hc_algo_t algo, hc_dtype_t dt, hc_op_t op) {
    switch (algo) {
    case HC_ALGO_RING: return pick_reduce_dt<HC_ALGO_RING, COLL>(dt, op);
    case HC_ALGO_RHD: return pick_reduce_dt<HC_ALGO_RHD, COLL>(dt, op);
    default: return pick_reduce_dt<HC_ALGO_PIPELINE, COLL>(dt, op);
    }
}

template <int MAXI, hc_dtype_t DT>
void* pick_step_op(hc_op_t op) {
    switch (op) {
    case HC_SUM: return (void*)step_kernel<DT, HC_SUM, MAXI>;
    case HC_PROD: return (void*)step_kernel<DT, HC_PROD, MAXI>;
    case HC_MAX: return (void*)step_kernel<DT, HC_MAX, MAXI>;
    default: return (void*)step_kernel<DT, HC_MIN, MAXI>;
    }
}
template <int MAXI>
void* pick_step(hc_dtype_t dt, hc_op_t op) {
    switch (dt) {
    case HC_INT32: return pick_step_op<MAXI, HC_INT32>(op);
    case HC_FLOAT32: return pick_step_op<MAXI, HC_FLOAT32>(op);
    default: return pick_step_op<MAXI, HC_BFLOAT16>(op);
    }
}

constexpr int kSmallItems = 48;   // parameter block under 4 KB
constexpr int kLargeItems = 256;  // large kernel parameter block

template <int MAXI>
cudaError_t launch_step_items(const Plan& plan, const PlanLaunch& L, size_t first, size_t count,
                              hc_dtype_t dt, hc_op_t op,
                              const uintptr_t (&base)[LOC_COUNT][kMaxRanks],
                              cudaStream_t stream, int max_ctas) {
    static thread_local StepParams<MAXI> p;  // large: keep it off the stack
    std::memcpy(p.base, base, sizeof(p.base));
    p.L = plan.lay.L;
    p.n = plan.lay.n;
    p.lo = L.lo;
    p.hi = L.hi;
    p.vecs = (L.hi - L.lo + plan.lay.A - 1) / plan.lay.A;
    PlanLaunch part;
    part.lo = L.lo;
    part.hi = L.hi;
    part.items.assign(L.items.begin() + first, L.items.begin() + first + count);
    const int grid = assign_ctas(part, plan.lay, kStepThreads, max_ctas);
    p.nitems = (int)count;
    p.total_ctas = grid;
    std::memcpy(p.items, part.items.data(), count * sizeof(DevItem));
    void* fn = pick_step<MAXI>(dt, op);
    void* args[] = {&p};
    return cudaLaunchKernel(fn, dim3(grid), dim3(kStepThreads), args, 0, stream);
}

}  // namespace

cudaError_t launch_step(const Plan& plan, int P, hc_dtype_t dt, hc_op_t op,
                        const uintptr_t (&base)[LOC_COUNT][kMaxRanks], cudaStream_t stream,
                        int sm_count) {
    (void)P;
    const int max_ctas = sm_count * (2048 / kStepThreads);
    for (const PlanLaunch& L : plan.launches) {
        size_t ni = L.items.size();
        cudaError_t e = cudaSuccess;
        if (ni <= (size_t)kSmallItems) {
            e = launch_step_items<kSmallItems>(plan, L, 0, ni, dt, op, base, stream, max_ctas);
        } else {
            // items of one step are independent, so a step may be split
            for (size_t f = 0; f < ni && e == cudaSuccess; f += kLargeItems)
                e = launch_step_items<kLargeItems>(plan, L, f, std::min(ni - f, (size_t)kLargeItems),
                                                   dt, op, base, stream, max_ctas);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream, int sm_count) {
    FusedParams p;
    std::memset(&p, 0, sizeof p);
    const int es = elem_bytes(a.dtype);
    const Layout& lay = a.lay;
    for (int r = 0; r < a.P; r++) {
        if (a.coll == HC_COLL_ALLGATHER) {
            // owner's segment view: send[k] holds segment k from its start
            const uintptr_t seg_off = (uintptr_t)lay.seg_lo(r) * es;
            const uintptr_t s = a.send ? (uintptr_t)a.send[r] : (uintptr_t)a.recv[r] + seg_off;
            p.src[r] = s - seg_off;
            p.dst[r] = (uintptr_t)a.recv[r];
            if (a.ag_in_place[r]) p.skip_mask |= 1ull << r;
        } else {
            p.src[r] = (uintptr_t)a.send[r];
            if (a.coll == HC_COLL_REDUCE_SCATTER)
                p.dst[r] = (uintptr_t)a.recv[r] - (uintptr_t)lay.seg_lo(r) * es;
            else
                p.dst[r] = (uintptr_t)a.recv[r];
        }
    }
    p.L = lay.L;
    p.n = lay.n;
    p.P = a.P;
    p.p_intra = a.p_intra;
    int pp = 1;
    while (pp * 2 <= a.P) pp *= 2;
    p.pp = pp;
    p.rfold = a.P - pp;
    int S = lay.S;
    if (a.algo == HC_ALGO_RHD && a.coll == HC_COLL_ALLREDUCE) {
        // the RHD tree is the same for every element: spread over P segments of
        // the p'-segment layout (the grid only needs the element range)
        S = lay.S;
    }
    const int64_t vecs_per_seg = (lay.L + lay.A - 1) / lay.A;
    const int64_t want = std::max<int64_t>(1, (vecs_per_seg + kFusedThreads - 1) / kFusedThreads);
    const int64_t cap = std::max<int64_t>(1, (int64_t)sm_count * (2048 / kFusedThreads) / S);
    const int gx = (int)std::min(want, cap);
    void* fn;
    if (a.coll == HC_COLL_ALLGATHER) {
        fn = es == 2 ? (void*)fused_allgather<2> : (void*)fused_allgather<4>;
    } else if (a.coll == HC_COLL_ALLREDUCE) {
        fn = pick_reduce<0>(a.algo, a.dtype, a.op);
    } else {
        fn = pick_reduce<1>(a.algo, a.dtype, a.op);
    }
    void* args[] = {&p};
    return cudaLaunchKernel(fn, dim3(gx, S), dim3(kFusedThreads), args, 0, stream);
}

}  // namespace hc

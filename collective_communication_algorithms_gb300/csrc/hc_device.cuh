// hc_device.cuh -- device-side building blocks shared by the kernel
// translation units of libhc: the element-wise operators (int32 wrap, fp32
// RNE without contraction or flush to zero, bf16 widened to fp32 and rounded
// back with cvt.rn.bf16x2.f32, max/min by IEEE totalOrder keys), 16-byte
// memory access, bulk copies with bounded mbarrier waits, and the fused
// kernel templates (register path and TMA-staged) with the association order
// of every schedule.  Internal; not installed.
#pragma once

#include <cuda_runtime.h>

#include "hc_internal.h"

namespace hc {

struct FusedParams {
    uintptr_t src[kMaxRanks];  // global-indexed input view of each rank
    uintptr_t dst[kMaxRanks];  // global-indexed output view of each rank
    int64_t L;
    int64_t n;
    int P;
    int p_intra;
    int pp;                    // RHD: power-of-two core size
    int rfold;                 // RHD: number of folded pairs
    int hold;                  // TMA kernels: 1 = the wait-expiry test mode (see hc_test_expire_waits)
    int owner;                 // Broadcast: the root owns the single segment (-1: segment k's owner is k)
    unsigned long long skip_mask;  // AllGather / Broadcast: ranks whose data is already in place
    unsigned long long wait_ns;    // TMA kernels: limit of the first wait on the copies' mbarrier
    int prefetch;              // AllGather / Broadcast: 1 = the first S blocks each prefetch one owner's segment into L2
    int* err;                  // device address of the library's error flag (HC_ERR_TIMEOUT on a wait that gave up)
};

// Register-path fused kernels, one translation unit per algorithm.
// coll: 0 AllReduce, 1 ReduceScatter; V: vectors per thread (1, or 2 where
// provided).  Returns nullptr for a combination that is not provided.
void* pick_fused_ring(int coll, hc_dtype_t dt, hc_op_t op, int V);
// large: P >= 16 (power-of-two core of 16 or more ranks)
void* pick_fused_rhd(int coll, hc_dtype_t dt, hc_op_t op, int V, bool large);
void* pick_fused_pipe(int coll, hc_dtype_t dt, hc_op_t op, int V);
void* pick_fused_hier(int coll, hc_dtype_t dt, hc_op_t op, int V);
// TMA-staged fused kernels (fused_reduce_tma) of the same schedules.
void* pick_fused_ring_tma(int coll, hc_dtype_t dt, hc_op_t op);
void* pick_fused_rhd_tma(int coll, hc_dtype_t dt, hc_op_t op, bool large);
void* pick_fused_pipe_tma(int coll, hc_dtype_t dt, hc_op_t op);
void* pick_fused_hier_tma(int coll, hc_dtype_t dt, hc_op_t op);

namespace {

// Kernel-table tag of the RHD kernels for 16 or more ranks (pp >= 16).
constexpr hc_algo_t kAlgoRhdLarge = (hc_algo_t)100;


// ---------------------------------------------------------------------------
// element-wise operators on 32-bit words (one fp32/int32, or two bf16)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key32(uint32_t u) {
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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

// Both halves of a bf16x2 word mapped at once to their totalOrder keys
// (per half: a negative value complemented, any other with its top bit set,
// as key32 does for fp32), so that unsigned 16-bit order is totalOrder, and
// back.
__device__ __forceinline__ uint32_t keys16x2(uint32_t w) {
    const uint32_t neg = ((w >> 15) & 0x00010001u) * 0xFFFFu;  // 0xFFFF in each negative half
    return w ^ (neg | 0x80008000u);
}
__device__ __forceinline__ uint32_t unkeys16x2(uint32_t k) {
    const uint32_t neg = ((~k >> 15) & 0x00010001u) * 0x7FFFu;  // halves whose key has the top bit clear
    return k ^ (neg | 0x80008000u);
}

template <hc_op_t OP>
struct WordOp<HC_BFLOAT16, OP> {
    __device__ __forceinline__ static uint32_t f(uint32_t a, uint32_t b) {
        if (OP == HC_SUM)
            return pack_bf16x2(__fadd_rn(bf_lo(a), bf_lo(b)), __fadd_rn(bf_hi(a), bf_hi(b)));
        if (OP == HC_PROD)
            return pack_bf16x2(__fmul_rn(bf_lo(a), bf_lo(b)), __fmul_rn(bf_hi(a), bf_hi(b)));
        // max / min by totalOrder, both halves in one SIMD instruction on
        // their keys; the key map is a bijection, so equal keys are equal
        // values and the result is the same word whichever operand wins
        const uint32_t ka = keys16x2(a), kb = keys16x2(b);
        uint32_t k;
        if (OP == HC_MAX) asm("max.u16x2 %0, %1, %2;" : "=r"(k) : "r"(ka), "r"(kb));
        else asm("min.u16x2 %0, %1, %2;" : "=r"(k) : "r"(ka), "r"(kb));
        return unkeys16x2(k);
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
// the same with an L2 eviction-priority policy (createpolicy)
__device__ __forceinline__ uint4 ld_vec_hint(uintptr_t p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}
__device__ __forceinline__ void st_vec_hint(uintptr_t p, const uint4& v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}
// streaming variants for data touched once by the fused kernels
__device__ __forceinline__ uint4 ld_stream(uintptr_t p) { return __ldcs((const uint4*)p); }
__device__ __forceinline__ void st_stream(uintptr_t p, const uint4& v) { __stcs((uint4*)p, v); }

// ---------------------------------------------------------------------------
// bulk copies (cp.async.bulk) and mbarriers with bounded waits
// ---------------------------------------------------------------------------
// Limit of every wait on an mbarrier: a copy that has not landed after this
// long is reported (HC_ERR_TIMEOUT) instead of being waited for forever.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
// Limit of the first wait in the wait-expiry test mode (hc_test_expire_waits).
constexpr unsigned long long kTestWaitLimitNs = 1000000ull;

__device__ __forceinline__ unsigned smem_addr(const void* p) {
    return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* m, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(m)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* m, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(m)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* m, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(m)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Poll an mbarrier phase for at most limit_ns.
__device__ bool mbar_wait_bounded(uint64_t* m, unsigned parity, unsigned long long limit_ns) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(m, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* m) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(m)) : "memory");
}
// After a first wait on the copies' mbarrier `full` has expired: record
// HC_ERR_TIMEOUT, release the arrival the test mode held back (hold = 1, on
// the thread that issued the copies), and wait again, bounded by
// kWaitLimitNs, until the bulk copies into this block's shared memory have
// landed, so the block never exits with a copy into its shared memory in
// flight.  A second expiry (a copy stuck for seconds) ends the wait anyway.
__device__ __noinline__ void mbar_expired(uint64_t* full, int* err, int hold, bool issuer) {
    atomicExch(err, (int)HC_ERR_TIMEOUT);
    if (hold && issuer) mbar_arrive(full);
    mbar_wait_bounded(full, 0, kWaitLimitNs);
}
__device__ __forceinline__ void bulk_g2s(void* smem_dst, uintptr_t gsrc, unsigned bytes, uint64_t* m) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(m))
        : "memory");
}
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, uintptr_t gsrc, unsigned bytes, uint64_t* m,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(m)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void bulk_s2g(uintptr_t gdst, const void* smem_src, unsigned bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
}
// The same store with an L2 eviction-priority policy (createpolicy).
__device__ __forceinline__ void bulk_s2g_hint(uintptr_t gdst, const void* smem_src, unsigned bytes,
                                              uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
                 "r"(smem_addr(smem_src)), "r"(bytes), "l"(policy)
                 : "memory");
}
// Policies: lines accessed through them are the first (the last) evicted
// from L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Asynchronous prefetch of [gsrc, gsrc + bytes) into L2 with a cache policy
// (16-byte aligned address, size a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2_hint(uintptr_t gsrc, unsigned bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(gsrc), "r"(bytes),
                 "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// wait until every committed bulk store has read its shared-memory source
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}


template <hc_dtype_t DT>
struct DT_ {
    static constexpr int ES = DT == HC_BFLOAT16 ? 2 : 4;
    static constexpr int A = 16 / ES;
};

// ---------------------------------------------------------------------------
// fused kernels
// ---------------------------------------------------------------------------


constexpr int kFusedThreads = 256;
constexpr int kBatch = 8;

// V 16-byte vectors handled together by one thread (more loads in flight)
template <int V>
struct VecN {
    uint4 v[V];
};
template <hc_dtype_t DT, hc_op_t OP, int V>
__device__ __forceinline__ VecN<V> vop(const VecN<V>& a, const VecN<V>& b) {
    VecN<V> r;
#pragma unroll
    for (int j = 0; j < V; j++) r.v[j] = vop<DT, OP>(a.v[j], b.v[j]);
    return r;
}

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

// Balanced pairwise tree over `count` leaves (a power of two) evaluated with
// a runtime loop: leaf w is merged with the pending left subtrees of the
// levels where w has a 1 bit (left operand = left subtree, exactly as the
// recursive tree_fixed), so the leaf code is instantiated once.
template <hc_dtype_t DT, hc_op_t OP, class V, class Leaf>
__device__ __forceinline__ V balanced_loop(int count, Leaf leaf) {
    V st[7];
    for (int w = 0; w < count; w++) {
        V x = leaf(w);
#pragma unroll
        for (int h = 0; h < 7; h++) {
            if ((w >> h) & 1) {
                x = vop<DT, OP>(st[h], x);
            } else {
                st[h] = x;
                break;
            }
        }
    }
    V res = st[0];
#pragma unroll
    for (int h = 1; h < 7; h++)
        if ((1 << h) == count) res = st[h];
    return res;
}

// RHD tree: leaves u_w = X_{2w+1} (+) X_{2w} for w < rfold (the fold step:
// rank 2w+1's data arrives at rank 2w), else X_{w + rfold}; balanced
// pairwise tree over the pp leaves, partner bit 0 first.
// LARGE = false: pp <= 8 (P < 16), trees unrolled at compile time, so that
// all loads are in flight together and the kernel keeps few registers;
// LARGE = true: pp = 16 unrolled, 32 and 64 by a runtime loop over
// compile-time subtrees of 8 leaves (separate kernels, so the small case does
// not pay the registers of the large ones).
template <hc_dtype_t DT, hc_op_t OP, bool LARGE, class V, class Load>
__device__ __forceinline__ V rhd_reduce(int pp, int rfold, Load load) {
    auto leaf = [&](int w) -> V {
        if (w < rfold) return vop<DT, OP>(load(2 * w + 1), load(2 * w));
        return load(w + rfold);
    };
    if constexpr (!LARGE) {
        switch (pp) {
        case 1: return tree_fixed<DT, OP, 1, V>(0, leaf);
        case 2: return tree_fixed<DT, OP, 2, V>(0, leaf);
        case 4: return tree_fixed<DT, OP, 4, V>(0, leaf);
        default: return tree_fixed<DT, OP, 8, V>(0, leaf);
        }
    } else {
        if (pp == 16) return tree_fixed<DT, OP, 16, V>(0, leaf);
        return balanced_loop<DT, OP, V>(pp / 8, [&](int g) -> V { return tree_fixed<DT, OP, 8, V>(8 * g, leaf); });
    }
}

// The same RHD tree with a leaf that is itself a long computation (the
// hierarchical AllReduce's intra-server chains): one runtime loop over the
// pp leaves, so the group code is instantiated twice rather than pp times.
template <hc_dtype_t DT, hc_op_t OP, class V, class Group>
__device__ __forceinline__ V rhd_reduce_loop(int pp, int rfold, Group group) {
    return balanced_loop<DT, OP, V>(pp, [&](int w) -> V {
        return w < rfold ? vop<DT, OP>(group(2 * w + 1), group(2 * w)) : group(w + rfold);
    });
}

// The association order of segment k for each algorithm.
template <hc_algo_t ALGO, hc_dtype_t DT, hc_op_t OP, class V, class Load>
__device__ __forceinline__ V segment_reduce(const FusedParams& p, int k, Load load) {
    if constexpr (ALGO == HC_ALGO_RING) {
        // chain X_{k+1} (+) X_{k+2} (+) ... (+) X_k
        return chain_reduce<DT, OP, V>(p.P, 0, (k + 1) % p.P, p.P, load);
    } else if constexpr (ALGO == HC_ALGO_RHD) {
        return rhd_reduce<DT, OP, false, V>(p.pp, p.rfold, load);
    } else if constexpr (ALGO == kAlgoRhdLarge) {
        return rhd_reduce<DT, OP, true, V>(p.pp, p.rfold, load);
    } else if constexpr (ALGO == HC_ALGO_HIER) {
        // RHD tree over servers (pp / rfold are the server-level core size and
        // folded pairs) whose leaves are the intra-server chains rotated from
        // the intra segment l = k / pp
        const int pin = p.p_intra, l = k / p.pp;
        auto server = [&](int s) -> V { return chain_reduce<DT, OP, V>(pin, s * pin, l, pin, load); };
        return rhd_reduce_loop<DT, OP, V>(p.pp, p.rfold, server);
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

// Ragged end of segment k: the fewer than A elements after its last full
// vector, element by element (one thread).
template <hc_algo_t ALGO, int COLL, hc_dtype_t DT, hc_op_t OP>
__device__ void ragged_tail(const FusedParams& p, int k, int64_t from, int64_t to) {
    constexpr int ES = DT_<DT>::ES;
    for (int64_t x = from; x < to; x++) {
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

// AllReduce (COLL = 0) and ReduceScatter (COLL = 1), register path: every
// thread loads V vectors of a segment from every rank straight into
// registers.  grid.y = segment.
template <hc_algo_t ALGO, int COLL, hc_dtype_t DT, hc_op_t OP, int V>
__global__ void __launch_bounds__(kFusedThreads)
fused_reduce(const __grid_constant__ FusedParams p) {
    constexpr int ES = DT_<DT>::ES;
    constexpr int A = DT_<DT>::A;
    const int k = blockIdx.y;
    const int64_t sbeg = (int64_t)k * p.L;
    if (sbeg >= p.n) return;
    const int64_t send_ = (sbeg + p.L < p.n) ? sbeg + p.L : p.n;
    const int64_t nfull = (send_ - sbeg) / A;
    const int64_t chunk = (int64_t)V * blockDim.x;
    // programmatic dependent launch: wait for the previous grid on the
    // stream (and its writes) before touching a buffer, then let the next
    // grid be scheduled
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t base = (int64_t)blockIdx.x * chunk; base < nfull; base += (int64_t)gridDim.x * chunk) {
        auto load = [&](int r) -> VecN<V> {
            VecN<V> x;
#pragma unroll
            for (int j = 0; j < V; j++) {
                const int64_t v = base + threadIdx.x + (int64_t)j * blockDim.x;
                x.v[j] = v < nfull ? ld_stream(p.src[r] + (uintptr_t)(sbeg + v * A) * ES)
                                   : make_uint4(0u, 0u, 0u, 0u);
            }
            return x;
        };
        const VecN<V> acc = segment_reduce<ALGO, DT, OP, VecN<V>>(p, k, load);
#pragma unroll
        for (int j = 0; j < V; j++) {
            const int64_t v = base + threadIdx.x + (int64_t)j * blockDim.x;
            if (v >= nfull) continue;
            const uintptr_t off = (uintptr_t)(sbeg + v * A) * ES;
            if (COLL == 0) {
                for (int r = 0; r < p.P; r++) st_stream(p.dst[r] + off, acc.v[j]);
            } else {
                st_stream(p.dst[k] + off, acc.v[j]);
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) ragged_tail<ALGO, COLL, DT, OP>(p, k, sbeg + nfull * A, send_);
}


// AllReduce (COLL = 0) and ReduceScatter (COLL = 1), TMA-staged: block
// (t, k) moves tile t of segment k (kTmaTile bytes, 16 per thread) of every
// rank into shared memory with one bulk copy per rank, all completing on one
// mbarrier; then each thread reduces its 16-byte vector from shared memory
// in the schedule's order and stores it to every output (AllReduce) or to the
// owner's (ReduceScatter).  Shared memory: P tiles, so P <= kTmaMaxRanks.
// The mbarrier wait is bounded (p.wait_ns): on expiry the thread records
// HC_ERR_TIMEOUT in *p.err, waits (bounded) for the block's copies in flight
// and returns without storing (the call's outputs are then undefined).  In
// the wait-expiry test mode (p.hold = 1) the mbarrier expects one arrival
// more than the block makes before that first wait, so the first wait
// expires although every copy lands; the copies' issuer makes the held
// arrival once its own wait has expired.
constexpr int kTmaThreads = 128;
constexpr int kTmaTile = kTmaThreads * 16;  // bytes per rank per block
constexpr int kTmaMaxRanks = 32;            // 64 KB of tiles per block

template <hc_algo_t ALGO, int COLL, hc_dtype_t DT, hc_op_t OP>
__global__ void __launch_bounds__(kTmaThreads)
fused_reduce_tma(const __grid_constant__ FusedParams p) {
    constexpr int ES = DT_<DT>::ES;
    constexpr int A = DT_<DT>::A;
    extern __shared__ __align__(128) unsigned char smem[];
    const int k = blockIdx.y;
    const int64_t sbeg = (int64_t)k * p.L;
    if (sbeg >= p.n) return;  // empty trailing segment
    const int64_t send_ = (sbeg + p.L < p.n) ? sbeg + p.L : p.n;
    const int64_t nfull = (send_ - sbeg) / A;
    const int64_t nbytes = nfull * 16;
    const int64_t t0 = (int64_t)blockIdx.x * kTmaTile;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // programmatic dependent launch
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (t0 < nbytes) {
        const int64_t left = nbytes - t0;
        const unsigned tb = (unsigned)(left < kTmaTile ? left : kTmaTile);
        const uintptr_t off = (uintptr_t)sbeg * ES + (uintptr_t)t0;
        uint64_t* full = (uint64_t*)(smem + (size_t)p.P * kTmaTile);
        if (threadIdx.x == 0) {
            mbar_init(full, 1 + p.hold);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            mbar_arrive_expect_tx(full, tb * (unsigned)p.P);
            for (int r = 0; r < p.P; r++) bulk_g2s(smem + (size_t)r * kTmaTile, p.src[r] + off, tb, full);
        }
        __syncthreads();  // the mbarrier is initialised before anyone polls it
        if (!mbar_wait_bounded(full, 0, p.wait_ns)) {
            mbar_expired(full, p.err, p.hold, threadIdx.x == 0);
            return;
        }
        const unsigned vo = threadIdx.x * 16u;
        if (vo < tb) {
            auto load = [&](int r) -> uint4 { return *(const uint4*)(smem + (size_t)r * kTmaTile + vo); };
            const uint4 acc = segment_reduce<ALGO, DT, OP, uint4>(p, k, load);
            if (COLL == 0) {
                for (int r = 0; r < p.P; r++) st_stream(p.dst[r] + off + vo, acc);
            } else {
                st_stream(p.dst[k] + off + vo, acc);
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) ragged_tail<ALGO, COLL, DT, OP>(p, k, sbeg + nfull * A, send_);
}

// Kernel table of the TMA-staged kernels of one algorithm.
template <hc_algo_t ALGO, int COLL, hc_dtype_t DT>
void* pick_tma_op(hc_op_t op) {
    switch (op) {
    case HC_SUM: return (void*)fused_reduce_tma<ALGO, COLL, DT, HC_SUM>;
    case HC_PROD: return (void*)fused_reduce_tma<ALGO, COLL, DT, HC_PROD>;
    case HC_MAX: return (void*)fused_reduce_tma<ALGO, COLL, DT, HC_MAX>;
    default: return (void*)fused_reduce_tma<ALGO, COLL, DT, HC_MIN>;
    }
}
template <hc_algo_t ALGO>
void* pick_tma(int coll, hc_dtype_t dt, hc_op_t op) {
    switch (dt) {
    case HC_INT32: return coll == 0 ? pick_tma_op<ALGO, 0, HC_INT32>(op) : pick_tma_op<ALGO, 1, HC_INT32>(op);
    case HC_FLOAT32: return coll == 0 ? pick_tma_op<ALGO, 0, HC_FLOAT32>(op) : pick_tma_op<ALGO, 1, HC_FLOAT32>(op);
    default: return coll == 0 ? pick_tma_op<ALGO, 0, HC_BFLOAT16>(op) : pick_tma_op<ALGO, 1, HC_BFLOAT16>(op);
    }
}

// Kernel table of one algorithm: the register-path kernels for every dtype,
// op, collective and (where instantiated) vectors per thread.
template <hc_algo_t ALGO, int COLL, hc_dtype_t DT, int V>
void* pick_fused_op(hc_op_t op) {
    switch (op) {
    case HC_SUM: return (void*)fused_reduce<ALGO, COLL, DT, HC_SUM, V>;
    case HC_PROD: return (void*)fused_reduce<ALGO, COLL, DT, HC_PROD, V>;
    case HC_MAX: return (void*)fused_reduce<ALGO, COLL, DT, HC_MAX, V>;
    default: return (void*)fused_reduce<ALGO, COLL, DT, HC_MIN, V>;
    }
}
template <hc_algo_t ALGO, int COLL, int V>
void* pick_fused_dt(hc_dtype_t dt, hc_op_t op) {
    switch (dt) {
    case HC_INT32: return pick_fused_op<ALGO, COLL, HC_INT32, V>(op);
    case HC_FLOAT32: return pick_fused_op<ALGO, COLL, HC_FLOAT32, V>(op);
    default: return pick_fused_op<ALGO, COLL, HC_BFLOAT16, V>(op);
    }
}

}  // namespace
}  // namespace hc

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
//               16-byte vector of a segment, reads it from every rank, reduces
//               in registers in exactly the association order the schedule
//               implies (Ring chain, RHD fold + pairwise tree, Pipeline
//               intra-server chain then inter-server chain) and stores it to
//               every output.  Up to 32 ranks the inputs are staged in shared
//               memory by bulk copies (fused_reduce_tma, hc_device.cuh); the
//               AllGather / Broadcast bulk-stores 32 KB tiles from shared
//               memory.  Minimum traffic: AllReduce reads and writes P n b
//               bytes.
//
// Arithmetic (must match the reduction semantics in hc.h bit for bit):
//  int32 wrap; fp32 IEEE RNE via __fadd_rn / __fmul_rn (no contraction, no
//  flush to zero); bf16 widened to fp32, op, then cvt.rn.bf16x2.f32;
//  max/min by IEEE totalOrder keys on the bit patterns.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "hc_device.cuh"

namespace hc {

// Wait-expiry test mode (hc_test_expire_waits): read at each launch of a
// TMA-staged kernel.
std::atomic<int> g_test_expire_waits{0};

namespace {

// ---------------------------------------------------------------------------
// step kernel
// ---------------------------------------------------------------------------
constexpr int kStepThreads = 256;
constexpr int kStepBatch = 8;  // input loads in flight per vector
// Vectors per thread per loop pass for single-input items (a copy, or
// acc (+) one input: every Ring and RHD step, the inter-server steps): all
// their loads are issued before any is reduced.  On GB300 two measured
// 0.96 of the copy bandwidth for the Ring AllReduce fp32 step mode against
// 0.83 with one, and the hierarchical steps 0.91 against 0.87.
constexpr int kStepUnroll = 2;

// Calls f(rank, kept) for every output of an item: its output set, then its
// second output set (a merged copy of the same block).  `kept`: a later step
// of the call reads that set's block (DevItem::keep).
template <class F>
__device__ __forceinline__ void each_output(const DevItem& I, F f) {
    int o = I.out_rot;
    for (int j = 0; j < I.out_cnt; j++) {
        f(I.out_base + o, (I.keep & 1) != 0);
        if (++o == I.out_mod) o = 0;
    }
    o = I.out2_rot;
    for (int j = 0; j < I.out2_cnt; j++) {
        f(I.out2_base + o, (I.keep & 2) != 0);
        if (++o == I.out2_mod) o = 0;
    }
}

// BATCH: input loads issued before reducing (1 for launches whose items
// have at most two inputs, where 8 blocks per SM give the loads in flight;
// kStepBatch for wider items, e.g. the Pipeline's intra-server mesh reduce)
template <hc_dtype_t DT, hc_op_t OP, int MAXI, int BATCH>
__global__ void __launch_bounds__(kStepThreads, BATCH == 1 ? 8 : 4)
step_kernel(const __grid_constant__ StepParams<MAXI> p) {
    constexpr int ES = DT_<DT>::ES;
    constexpr int A = DT_<DT>::A;
    const int b = blockIdx.x;
    int it = 0;
    while (it + 1 < p.nitems && p.items[it + 1].cta_begin <= b) it++;
    const DevItem& I = p.items[it];
    const int cend = (it + 1 < p.nitems) ? p.items[it + 1].cta_begin : p.total_ctas;
    const int ncta = cend - I.cta_begin;
    const int bl = b - I.cta_begin;
    const int nseg = I.seg_width * I.seg_reps;
    // An item that spans several segments gives each segment its own blocks
    // (ncta / nseg of them; the host assigns at least one per segment), and
    // each segment's blocks stride over its slice.  (All of an item's threads
    // striding over one segment after another left those past a segment's
    // vector count idle and made the others visit every segment in turn: RHD
    // steps, whose items span up to P / 2 segments, paid that latency per
    // segment.)  With fewer blocks than segments a block takes every
    // ncta-th segment.
    int si_begin = 0, si_step = 1, cps = ncta, cb = bl;  // cb: block within its segment's
    if (nseg > 1) {
        if (ncta >= nseg) {
            cps = ncta / nseg;
            si_begin = bl / cps;
            si_step = nseg;
            if (si_begin >= nseg) return;  // the remainder of the division
            cb = bl - si_begin * cps;
        } else {
            cps = 1;
            si_begin = bl;
            si_step = ncta;
            cb = 0;
        }
    }
    const int64_t nthreads = (int64_t)cps * blockDim.x;
    const int64_t t0 = (int64_t)cb * blockDim.x + threadIdx.x;
    // Operands no other item of this launch reads are loaded with an L2
    // evict-first policy, so that what stays in L2 is what the next steps
    // read again (this step's outputs).  On GB300 this took the Ring
    // AllReduce fp32 step mode from 0.94 to 1.15 of the copy bandwidth on its
    // own bytes (the accumulators then come from L2), the Ring
    // ReduceScatter / AllGather steps from 0.84 / 0.85 to 0.99.  Outputs no
    // later step reads (the results of the last steps) are stored with the
    // same policy: Ring AllGather step mode 1.11 -> 1.15, bf16 AllReduce
    // steps 0.916 -> 0.926.
    const uint64_t first_out = l2_evict_first_policy();
    auto ld_vec = [&](uintptr_t a) -> uint4 { return I.once ? ld_vec_hint(a, first_out) : hc::ld_vec(a); };
    // Programmatic dependent launch: this grid may be scheduled while the
    // previous step's grid drains.  Wait for that grid to complete (and its
    // writes to be visible) before touching any buffer, then let the next
    // step's grid be scheduled.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    for (int si = si_begin; si < nseg; si += si_step) {
        const int seg = I.seg_first + (si / I.seg_width) * I.seg_stride + (si % I.seg_width);
        const int64_t sbeg = (int64_t)seg * p.L;
        int64_t send_ = sbeg + p.L;
        if (send_ > p.n) send_ = p.n;
        int64_t hi = sbeg + p.hi;
        if (hi > send_) hi = send_;
        const int64_t lo = sbeg + p.lo;
        for (int64_t e = lo + t0 * A; e < hi; e += nthreads * A) {
            if (BATCH == 1 && I.in_cnt == 1 && e + (kStepUnroll - 1) * nthreads * A + A <= hi) {
                // kStepUnroll full vectors, nthreads * A elements apart
                uintptr_t o[kStepUnroll];
                uint4 x[kStepUnroll];
                const uintptr_t ib = p.base[I.in_loc][I.in_base + I.in_rot];
#pragma unroll
                for (int u = 0; u < kStepUnroll; u++) {
                    o[u] = (uintptr_t)(e + u * nthreads * A) * ES;
                    x[u] = ld_vec(ib + o[u]);
                }
                if (I.acc_rank >= 0) {
                    const uintptr_t ab = p.base[I.acc_loc][I.acc_rank];
                    uint4 a[kStepUnroll];
#pragma unroll
                    for (int u = 0; u < kStepUnroll; u++) a[u] = ld_vec(ab + o[u]);
#pragma unroll
                    for (int u = 0; u < kStepUnroll; u++) x[u] = vop<DT, OP>(a[u], x[u]);
                }
                each_output(I, [&](int r, bool kept) {
                    const uintptr_t ob = p.base[I.out_loc][r];
                    if (kept) {
#pragma unroll
                        for (int u = 0; u < kStepUnroll; u++) st_vec(ob + o[u], x[u]);
                    } else {
#pragma unroll
                        for (int u = 0; u < kStepUnroll; u++) st_vec_hint(ob + o[u], x[u], first_out);
                    }
                });
                e += (kStepUnroll - 1) * nthreads * A;  // the loop step adds the last stride
                continue;
            }
            const uintptr_t off = (uintptr_t)e * ES;
            if (e + A <= hi) {
                // issue the accumulator's and up to BATCH inputs' loads
                // before reducing them in the item's order
                uint4 acc = make_uint4(0, 0, 0, 0);
                if (I.acc_rank >= 0) acc = ld_vec(p.base[I.acc_loc][I.acc_rank] + off);
                uint4 v = acc;
                int r = I.in_rot;
                for (int c = 0; c < I.in_cnt; c += BATCH) {
                    const int m = I.in_cnt - c < BATCH ? I.in_cnt - c : BATCH;
                    uint4 x[BATCH];
#pragma unroll
                    for (int q = 0; q < BATCH; q++) {
                        if (q < m) {
                            x[q] = ld_vec(p.base[I.in_loc][I.in_base + r] + off);
                            if (++r == I.in_mod) r = 0;
                        }
                    }
#pragma unroll
                    for (int q = 0; q < BATCH; q++)
                        if (q < m) v = (c == 0 && q == 0) ? x[0] : vop<DT, OP>(v, x[q]);
                }
                if (I.acc_rank >= 0) v = vop<DT, OP>(acc, v);
                each_output(I, [&](int r, bool kept) {
                    if (kept) st_vec(p.base[I.out_loc][r] + off, v);
                    else st_vec_hint(p.base[I.out_loc][r] + off, v, first_out);
                });
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
                    each_output(I, [&](int r, bool) { st_elem<ES>(p.base[I.out_loc][r] + xo, v); });
                }
            }
        }
    }
}

// Step kernel, TMA-staged: for launches whose items combine three or more
// operands (the intra-server mesh reduce of the Pipeline and of the
// hierarchical AllReduce: up to p_intra inputs plus the partial that arrived
// on the inter-server ring), launches of pure broadcasts, and large launches
// of narrow items (below).  Block (item, segment, tile) bulk-copies tile
// `tile` (TILE bytes) of the launch's slice of that segment from every
// operand -- the item's inputs in their order, then its accumulator -- into
// consecutive TILE-byte slots of shared memory, all completing on one
// mbarrier.  The threads then combine its 16-byte vectors exactly as
// step_kernel does (in[0] (+) in[1] (+) ..., then acc (+) that) and store
// them to every output.  The mbarrier waits are bounded like
// fused_reduce_tma's.  On GB300 the register path (BATCH = 8, 4 blocks per
// SM) ran the wide launches at 0.79 of the copy bandwidth.
constexpr int kStepTmaMaxOperands = kTmaMaxRanks;  // shared memory <= 64 KB per block
// Narrow launches (items of at most two operands: the Ring and RHD steps,
// the inter-server steps) take this kernel too once a launch moves at least
// kNarrowTmaMinBytes, with 8 KB tiles: on GB300 the Ring AllReduce fp32 step
// mode went from 1.17 to 1.30 of the copy bandwidth on its own bytes, the
// Ring AllGather steps from 1.15 to 1.31, the bf16 Ring / RHD AllReduce
// steps (128 MiB per rank) from 0.93 to 1.04 / 1.06.  With 2 KB tiles they
// ran at 0.5 - 0.6; launches of small items (Ring with 32 ranks below 4 Mi
// elements) measured 4 - 12 % slower than on the register kernel.
constexpr int kNarrowTmaTile = 8192;
constexpr int64_t kNarrowTmaMinBytes = 8 << 20;

// TILE: bytes per operand per block (kTmaTile, or kNarrowTmaTile)
template <hc_dtype_t DT, hc_op_t OP, int MAXI, int TILE>
__global__ void __launch_bounds__(kTmaThreads)
step_kernel_tma(const __grid_constant__ StepParams<MAXI> p) {
    constexpr int ES = DT_<DT>::ES;
    constexpr int A = DT_<DT>::A;
    extern __shared__ __align__(128) unsigned char smem[];
    const int b = blockIdx.x;
    int it = 0;
    while (it + 1 < p.nitems && p.items[it + 1].cta_begin <= b) it++;
    const DevItem& I = p.items[it];
    const int64_t local = b - I.cta_begin;
    const int si = (int)(local / p.tiles);
    const int64_t tile = local - (int64_t)si * p.tiles;
    const int seg = I.seg_first + (si / I.seg_width) * I.seg_stride + (si % I.seg_width);
    const int64_t sbeg = (int64_t)seg * p.L;
    const int64_t send_ = sbeg + p.L < p.n ? sbeg + p.L : p.n;
    const int64_t hi = sbeg + p.hi < send_ ? sbeg + p.hi : send_;
    const int64_t lo = sbeg + p.lo;
    const int64_t nfull = lo < hi ? (hi - lo) / A : 0;
    const int64_t t0 = tile * TILE;
    const int acc_slot = I.acc_rank >= 0 ? I.in_cnt : -1;
    const int nops = I.in_cnt + (acc_slot >= 0 ? 1 : 0);
    const bool staged = t0 < nfull * 16;
    const int64_t left = nfull * 16 - t0;
    const unsigned tb = (unsigned)(left < TILE ? left : TILE);
    const uintptr_t off = (uintptr_t)lo * ES + (uintptr_t)t0;
    uint64_t* full = (uint64_t*)(smem + (size_t)nops * TILE);
    // Inputs that no launch of this call writes may be requested before the
    // programmatic wait, overlapping the previous launch's tail; everything
    // else (the accumulator, every store) comes after it.
    const bool early = staged && p.early && I.early;
    // L2 policies as in step_kernel: operands read by this item only leave
    // L2 first; outputs a later step reads leave it last (on GB300 the
    // Pipeline 4 x 8 step mode went from 0.82 to 0.86 of the copy bandwidth
    // on its own bytes, the hierarchical from 0.92 to 0.94), outputs nobody
    // reads again leave it first (Pipeline 4 x 8 AllReduce / AllGather step
    // mode 0.92 / 0.88 -> 0.95 / 0.93, hierarchical 1.03 -> 1.05)
    const uint64_t first_out = l2_evict_first_policy();
    auto load = [&](int slot, uintptr_t src) {
        if (I.once) bulk_g2s_hint(smem + (size_t)slot * TILE, src, tb, full, first_out);
        else bulk_g2s(smem + (size_t)slot * TILE, src, tb, full);
    };
    auto issue_inputs = [&]() {
        int r = I.in_rot;
        for (int j = 0; j < I.in_cnt; j++) {
            load(j, p.base[I.in_loc][I.in_base + r] + off);
            if (++r == I.in_mod) r = 0;
        }
    };
    if (staged && threadIdx.x == 0) {
        mbar_init(full, 1 + p.hold);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(full, tb * (unsigned)nops);
        if (early) issue_inputs();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // programmatic dependent launch
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (lo >= hi) return;  // the slice misses this (short) segment
    if (staged) {
        if (threadIdx.x == 0) {
            if (!early) issue_inputs();
            if (acc_slot >= 0) load(acc_slot, p.base[I.acc_loc][I.acc_rank] + off);
        }
        __syncthreads();  // the mbarrier is initialised before anyone polls it
        if (!mbar_wait_bounded(full, 0, p.wait_ns)) {
            mbar_expired(full, p.err, p.hold, threadIdx.x == 0);
            return;
        }
        if (I.in_cnt == 1 && acc_slot < 0) {
            // a copy: the tile goes from shared memory to every output by
            // bulk stores; the block leaves once they have read it
            if (threadIdx.x == 0) {
                const uint64_t last_out = l2_evict_last_policy();
                each_output(I, [&](int r, bool kept) {
                    bulk_s2g_hint(p.base[I.out_loc][r] + off, smem, tb, kept ? last_out : first_out);
                });
                bulk_commit();
                bulk_wait_read_all();
            }
        } else {
            for (unsigned vo = threadIdx.x * 16u; vo < tb; vo += kTmaThreads * 16u) {
                uint4 v = *(const uint4*)(smem + vo);
                for (int j = 1; j < I.in_cnt; j++)
                    v = vop<DT, OP>(v, *(const uint4*)(smem + (size_t)j * TILE + vo));
                if (acc_slot >= 0) v = vop<DT, OP>(*(const uint4*)(smem + (size_t)acc_slot * TILE + vo), v);
                const uint64_t last_out = l2_evict_last_policy();
                each_output(I, [&](int r, bool kept) {
                    st_vec_hint(p.base[I.out_loc][r] + off + vo, v, kept ? last_out : first_out);
                });
            }
        }
    }
    if (tile == 0 && threadIdx.x == 0) {
        // ragged end of the rank vector (< 16 bytes): element by element
        for (int64_t x = lo + nfull * A; x < hi; x++) {
            const uintptr_t xo = (uintptr_t)x * ES;
            int rr = I.in_rot;
            uint32_t v = ld_elem<ES>(p.base[I.in_loc][I.in_base + rr] + xo);
            for (int j = 1; j < I.in_cnt; j++) {
                if (++rr == I.in_mod) rr = 0;
                v = vop<DT, OP>(v, ld_elem<ES>(p.base[I.in_loc][I.in_base + rr] + xo));
            }
            if (acc_slot >= 0) v = vop<DT, OP>(ld_elem<ES>(p.base[I.acc_loc][I.acc_rank] + xo), v);
            each_output(I, [&](int r, bool) { st_elem<ES>(p.base[I.out_loc][r] + xo, v); });
        }
    }
}

constexpr int kAgPrefetchChunk = 32768;  // bytes per L2 prefetch request

// AllGather, register path: segment k read once from its owner, written to
// every rank (the owner's own copy only when it is not already in place).
// Broadcast is the same kernel with one segment owned by the root.
template <int ES>
__global__ void __launch_bounds__(kFusedThreads)
fused_allgather(const __grid_constant__ FusedParams p) {
    constexpr int A = 16 / ES;
    const int seg = blockIdx.y;
    const int k = p.owner >= 0 ? p.owner : seg;
    const int64_t sbeg = (int64_t)seg * p.L;
    if (sbeg >= p.n) return;
    const int64_t send_ = (sbeg + p.L < p.n) ? sbeg + p.L : p.n;
    const int64_t nfull = (send_ - sbeg) / A;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const bool skip_own = (p.skip_mask >> k) & 1ull;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // programmatic dependent launch
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (p.prefetch && threadIdx.x == 0) {
        // the first gridDim.y blocks in launch order each request one owner's
        // segment into L2 (evict-last, so that the stream of stores does not
        // push it out before the later blocks read it)
        const int64_t lin = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
        if (lin < gridDim.y) {
            const int s2 = (int)lin;
            const int k2 = p.owner >= 0 ? p.owner : s2;
            const int64_t b2 = (int64_t)s2 * p.L;
            const int64_t e2 = b2 + p.L < p.n ? b2 + p.L : p.n;
            const int64_t nb = e2 > b2 ? ((e2 - b2) * ES) / 16 * 16 : 0;
            const uint64_t keep = l2_evict_last_policy();
            for (int64_t t = 0; t < nb; t += kAgPrefetchChunk) {
                const unsigned by = (unsigned)(nb - t < kAgPrefetchChunk ? nb - t : kAgPrefetchChunk);
                bulk_prefetch_l2_hint(p.src[k2] + (uintptr_t)b2 * ES + (uintptr_t)t, by, keep);
            }
        }
    }
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

// Library error flag of the kernels' bounded waits (HC_ERR_TIMEOUT), read and
// cleared by hc_device_status.
__device__ int hc_device_error;

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
// Register-path kernel of (algo, collective, dtype, op, vectors per thread).
void* pick_reduce(hc_algo_t algo, int coll, hc_dtype_t dt, hc_op_t op, int V, int P) {
    switch (algo) {
    case HC_ALGO_RING: return pick_fused_ring(coll, dt, op, V);
    case HC_ALGO_RHD: return pick_fused_rhd(coll, dt, op, V, P >= 16);
    case HC_ALGO_HIER: return pick_fused_hier(coll, dt, op, V);
    default: return pick_fused_pipe(coll, dt, op, V);
    }
}

// TMA-staged fused reduce of (algo, collective, dtype, op).
void* pick_reduce_tma(hc_algo_t algo, int coll, hc_dtype_t dt, hc_op_t op, int P) {
    switch (algo) {
    case HC_ALGO_RING: return pick_fused_ring_tma(coll, dt, op);
    case HC_ALGO_RHD: return pick_fused_rhd_tma(coll, dt, op, P >= 16);
    case HC_ALGO_HIER: return pick_fused_hier_tma(coll, dt, op);
    default: return pick_fused_pipe_tma(coll, dt, op);
    }
}

// Device address of hc_device_error on the current device (looked up once
// per device).
int* device_error_flag() {
    static std::atomic<int*> addr[kMaxDevices];  // null-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* a = addr[dev].load(std::memory_order_acquire);
    if (!a) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, hc_device_error) != cudaSuccess) return nullptr;
        a = (int*)p;
        addr[dev].store(a, std::memory_order_release);
    }
    return a;
}

// Launch with programmatic stream serialization: the kernel waits for the
// previous grid on the stream itself (griddepcontrol.wait), so its launch
// and block scheduling overlap that grid's tail.
cudaError_t launch_pdl(void* fn, dim3 grid, dim3 block, void** args, size_t smem,
                       cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Raise a kernel's dynamic shared memory limit to at least `bytes` (the
// attribute is per kernel and device, so remember the largest value set for
// each pair).
std::mutex g_kernel_attr_mu;  // guards the per-kernel caches below

bool allow_smem(void* fn, int bytes) {
    static void* fns[512];
    static int devs[512];
    static int set[512];
    static int nfns = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_kernel_attr_mu);  // the attribute is per device
    int i = 0;
    while (i < nfns && (fns[i] != fn || devs[i] != dev)) i++;
    if (i < nfns && set[i] >= bytes) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    if (i == nfns && nfns < 512) {
        fns[nfns] = fn;
        devs[nfns++] = dev;
    }
    if (i < nfns) set[i] = bytes;
    return true;
}

template <int MAXI, int BATCH, hc_dtype_t DT>
void* pick_step_op(hc_op_t op) {
    switch (op) {
    case HC_SUM: return (void*)step_kernel<DT, HC_SUM, MAXI, BATCH>;
    case HC_PROD: return (void*)step_kernel<DT, HC_PROD, MAXI, BATCH>;
    case HC_MAX: return (void*)step_kernel<DT, HC_MAX, MAXI, BATCH>;
    default: return (void*)step_kernel<DT, HC_MIN, MAXI, BATCH>;
    }
}
template <int MAXI, int TILE, hc_dtype_t DT>
void* pick_step_tma_op(hc_op_t op) {
    switch (op) {
    case HC_SUM: return (void*)step_kernel_tma<DT, HC_SUM, MAXI, TILE>;
    case HC_PROD: return (void*)step_kernel_tma<DT, HC_PROD, MAXI, TILE>;
    case HC_MAX: return (void*)step_kernel_tma<DT, HC_MAX, MAXI, TILE>;
    default: return (void*)step_kernel_tma<DT, HC_MIN, MAXI, TILE>;
    }
}
template <int MAXI, int TILE>
void* pick_step_tma(hc_dtype_t dt, hc_op_t op) {
    switch (dt) {
    case HC_INT32: return pick_step_tma_op<MAXI, TILE, HC_INT32>(op);
    case HC_FLOAT32: return pick_step_tma_op<MAXI, TILE, HC_FLOAT32>(op);
    default: return pick_step_tma_op<MAXI, TILE, HC_BFLOAT16>(op);
    }
}

template <int MAXI, int BATCH>
void* pick_step(hc_dtype_t dt, hc_op_t op) {
    switch (dt) {
    case HC_INT32: return pick_step_op<MAXI, BATCH, HC_INT32>(op);
    case HC_FLOAT32: return pick_step_op<MAXI, BATCH, HC_FLOAT32>(op);
    default: return pick_step_op<MAXI, BATCH, HC_BFLOAT16>(op);
    }
}

// Blocks of a step kernel resident per SM (cached per kernel).
int resident_blocks(void* fn) {
    static void* fns[256];
    static int val[256];
    static int nfns = 0;
    std::lock_guard<std::mutex> lock(g_kernel_attr_mu);
    for (int i = 0; i < nfns; i++)
        if (fns[i] == fn) return val[i];
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fn, kStepThreads, 0) != cudaSuccess || v < 1)
        v = 1;
    if (nfns < 256) {
        fns[nfns] = fn;
        val[nfns++] = v;
    }
    return v;
}

constexpr int kSmallItems = 48;   // parameter block under 4 KB
constexpr int kLargeItems = 256;  // large kernel parameter block

// early: not the call's first kernel launch (StepParams::early)
template <int MAXI>
cudaError_t launch_step_items(const Plan& plan, const PlanLaunch& L, size_t first, size_t count,
                              hc_dtype_t dt, hc_op_t op,
                              const uintptr_t (&base)[LOC_COUNT][kMaxRanks],
                              cudaStream_t stream, int sm_count, bool host_buffers, bool early) {
    static thread_local StepParams<MAXI> p;  // large: keep it off the stack
    std::memcpy(p.base, base, sizeof(p.base));
    p.L = plan.lay.L;
    p.n = plan.lay.n;
    p.lo = L.lo;
    p.hi = L.hi;
    p.vecs = (L.hi - L.lo + plan.lay.A - 1) / plan.lay.A;
    p.tiles = 0;
    p.early = early ? 1 : 0;
    p.hold = g_test_expire_waits.load() ? 1 : 0;
    p.wait_ns = p.hold ? kTestWaitLimitNs : kWaitLimitNs;
    p.err = nullptr;
    PlanLaunch part;
    part.lo = L.lo;
    part.hi = L.hi;
    part.items.assign(L.items.begin() + first, L.items.begin() + first + count);
    int widest = 1, operands = 1;
    for (const DevItem& it : part.items) {
        widest = std::max(widest, (int)it.in_cnt);
        operands = std::max(operands, it.in_cnt + (it.acc_rank >= 0 ? 1 : 0));
    }
    p.nitems = (int)count;
    // Launches of pure broadcasts (every item copies one input to three or
    // more outputs: the mesh AllGather of the hierarchical AllReduce, the
    // Pipeline AllGather steps whose forward and intra-server sends of a
    // block are one item) also take the TMA-staged kernel, whose bulk stores
    // write a tile from shared memory to every output.  These launches keep
    // most of their traffic in L2 and were bound by per-thread stores: on
    // GB300 the hierarchical 4 x 8 step mode went from 0.96 to 1.03 of the
    // copy bandwidth on its own bytes, the Pipeline 4 x 8 AllReduce step mode
    // from 0.410 to 0.397 ms per call and its AllGather from 0.223 to 0.208.
    // Launches that mix broadcasts with 1 -> 1 copies keep the register
    // kernel (the Pipeline AllGather steps before their sends were merged
    // measured 0.89 -> 0.77 on bulk copies).
    bool broadcasts = true;
    int64_t launch_bytes = 0;  // every item's operands and outputs over the slice
    for (const DevItem& it : part.items) {
        broadcasts = broadcasts && it.in_cnt == 1 && it.acc_rank < 0 && item_outputs(it) >= 3;
        launch_bytes += (int64_t)it.seg_width * it.seg_reps * p.vecs * 16 *
                        (it.in_cnt + (it.acc_rank >= 0 ? 1 : 0) + item_outputs(it));
    }
    const bool wide = widest >= 3 || broadcasts;
    const bool narrow = !wide && launch_bytes >= kNarrowTmaMinBytes;
    if ((wide || narrow) && operands <= kStepTmaMaxOperands && !host_buffers) {
        // TMA-staged: one block per tile of every segment of every item
        const int tile = wide ? kTmaTile : kNarrowTmaTile;
        void* fn = wide ? pick_step_tma<MAXI, kTmaTile>(dt, op) : pick_step_tma<MAXI, kNarrowTmaTile>(dt, op);
        p.err = device_error_flag();
        if (!p.err) return cudaErrorInvalidValue;
        const int smem = operands * tile + 16;
        if (!allow_smem(fn, smem)) return cudaErrorInvalidValue;
        p.tiles = std::max<int64_t>(1, (p.vecs * 16 + tile - 1) / tile);
        int64_t begin = 0;
        for (DevItem& it : part.items) {
            it.cta_begin = (int32_t)begin;
            begin += (int64_t)it.seg_width * it.seg_reps * p.tiles;
        }
        if (begin > INT32_MAX) return cudaErrorInvalidValue;
        p.total_ctas = (int)begin;
        std::memcpy(p.items, part.items.data(), count * sizeof(DevItem));
        void* args[] = {&p};
        return launch_pdl(fn, dim3((unsigned)begin), dim3(kTmaThreads), args, smem, stream);
    }
    void* fn = widest >= 3 ? pick_step<MAXI, kStepBatch>(dt, op) : pick_step<MAXI, 1>(dt, op);
    // one wave of resident blocks
    const int grid = assign_ctas(part, plan.lay, kStepThreads, sm_count * resident_blocks(fn));
    p.total_ctas = grid;
    std::memcpy(p.items, part.items.data(), count * sizeof(DevItem));
    void* args[] = {&p};
    return launch_pdl(fn, dim3(grid), dim3(kStepThreads), args, 0, stream);
}

}  // namespace

cudaError_t launch_step(const Plan& plan, int P, hc_dtype_t dt, hc_op_t op,
                        const uintptr_t (&base)[LOC_COUNT][kMaxRanks], cudaStream_t stream,
                        int sm_count, bool host_buffers) {
    (void)P;
    uint64_t index = 0;
    int kernels = 0;  // kernel launches of this call so far
    for (const PlanLaunch& L : plan.launches) {
        const TraceRange range("hc step launch", 0, index++);
        size_t ni = L.items.size();
        cudaError_t e = cudaSuccess;
        if (ni <= (size_t)kSmallItems) {
            e = launch_step_items<kSmallItems>(plan, L, 0, ni, dt, op, base, stream, sm_count,
                                               host_buffers, kernels++ > 0);
        } else {
            // items of one step are independent, so a step may be split
            for (size_t f = 0; f < ni && e == cudaSuccess; f += kLargeItems)
                e = launch_step_items<kLargeItems>(plan, L, f, std::min(ni - f, (size_t)kLargeItems),
                                                   dt, op, base, stream, sm_count, host_buffers,
                                                   kernels++ > 0);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

void set_test_expire_waits(bool on) { g_test_expire_waits.store(on ? 1 : 0); }

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream, int sm_count) {
    FusedParams p;
    std::memset(&p, 0, sizeof p);
    const int es = elem_bytes(a.dtype);
    const Layout& lay = a.lay;
    p.owner = -1;
    p.hold = g_test_expire_waits.load() ? 1 : 0;
    p.wait_ns = p.hold ? kTestWaitLimitNs : kWaitLimitNs;
    for (int r = 0; r < a.P; r++) {
        if (a.coll == HC_COLL_BROADCAST) {
            // the root's input is the whole vector (segment 0 starts at 0)
            p.src[r] = (uintptr_t)(a.send && a.send[r] ? a.send[r] : a.recv[r]);
            p.dst[r] = (uintptr_t)a.recv[r];
            if (a.ag_in_place[r]) p.skip_mask |= 1ull << r;
            p.owner = a.root;
        } else if (a.coll == HC_COLL_ALLGATHER) {
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
    // RHD core: over ranks, or over servers for the hierarchical AllReduce
    const int groups = a.algo == HC_ALGO_HIER ? a.P / a.p_intra : a.P;
    int pp = 1;
    while (pp * 2 <= groups) pp *= 2;
    p.pp = pp;
    p.rfold = groups - pp;
    const int S = lay.S;
    const int64_t seg_bytes = lay.L * es;
    void* args[] = {&p};

    // Device buffers: one block per chunk of the segment (a 32 KB tile, or
    // V x 256 vectors), so blocks are scheduled in index order and the stores
    // sweep every output from its start.  On GB300 this measured 3 - 9 %
    // faster than a persistent grid of a few blocks per SM striding over the
    // segment, for every collective; plain stores from one-shot blocks
    // reached 7.47 TB/s where grid-stride stores of the same bytes reached
    // 6.3 TB/s.  Buffers in page-locked host memory keep a persistent grid
    // (the host link, not HBM, bounds them).
    if (a.coll == HC_COLL_ALLGATHER || a.coll == HC_COLL_BROADCAST) {
        // The plain load / store path at every rank count.  A TMA-staged
        // variant (one 32 KB tile per block, bulk-loaded once and
        // bulk-stored to every rank) measured on GB300 (fp32, out of place,
        // one call) between 5.0 and 7.2 TB/s on (P + 1) n b depending on the
        // grid's shape: 20 - 30 % slower than this path at 4 Mi elements per
        // rank for 16, 32 and 64 ranks (P = 32: 106 against 82 us), 3 - 6 %
        // faster at 8 Mi, with no layout, tile size or store order that
        // removed the dips; this path stays at 6.6 - 6.95 TB/s over 8 to 64
        // ranks and 1 to 32 Mi elements.  The same store pattern without the
        // loads takes 73.8 us at P = 8, 64 MiB per rank, against 89 - 93 us
        // with them: reads and writes share the DRAM bus.
        // From 16 ranks, with segments of at most 1 MiB and a source of at
        // least 8 MiB, the first blocks also prefetch the whole source into
        // L2 (evict-last).  On GB300 (fp32, out of place, same call): P = 16,
        // 2 / 4 Mi elements per rank 22.3 -> 21.0 / 42.6 -> 38.7 us; P = 32,
        // 4 / 8 Mi 83.1 -> 76.2 / 161.6 -> 155.7 us (bf16 8 Mi: 83.1 ->
        // 76.2); P = 64, 2 / 4 / 8 Mi 84.2 -> 80.5 / 160.8 -> 151.3 / 314 ->
        // 303 us.  With fewer ranks the segments are long and one thread per
        // segment cannot issue the requests in time (P = 8, 64 MiB per rank:
        // 90 -> 131 us); a separate prefetch launch cost 2 us per call and
        // slowed that case too (93 us); sources under 8 MiB gained nothing
        // (P = 32, 1 Mi: 22.1 -> 23.0 us).
        p.prefetch = (a.P >= 16 && seg_bytes <= (1 << 20) && lay.n * es >= (8 << 20) && !a.host_buffers) ? 1 : 0;
        void* fn = es == 2 ? (void*)fused_allgather<2> : (void*)fused_allgather<4>;
        const int64_t vecs = (lay.L + lay.A - 1) / lay.A;
        const int64_t want = std::max<int64_t>(1, (vecs + kFusedThreads - 1) / kFusedThreads);
        const int64_t gx = a.host_buffers ? std::min(want, std::max<int64_t>(1, (int64_t)sm_count * 4 / S)) : want;
        return launch_pdl(fn, dim3((unsigned)gx, S), dim3(kFusedThreads), args, 0, stream);
    }

    const int COLL = a.coll == HC_COLL_ALLREDUCE ? 0 : 1;
    // TMA-staged path: device buffers and P <= kTmaMaxRanks (P tiles of
    // shared memory per block), one block per kTmaTile bytes of a segment.
    // Against the register path on GB300 (fraction of the measured copy
    // bandwidth, same call): Pipeline fp32 4x8 1.007 vs 0.953, hierarchical
    // 0.994 vs 0.930, Ring ReduceScatter fp32 1.010 vs 0.964, Ring bf16 max
    // 0.967 vs 0.935, RHD bf16 max 0.990 vs 0.975; Ring fp32 and bf16 and
    // RHD bf16 sum AllReduce within 0.2 %.
    if (!a.host_buffers && a.P <= kTmaMaxRanks) {
        void* fn = pick_reduce_tma(a.algo, COLL, a.dtype, a.op, a.P);
        if (fn) {
            p.err = device_error_flag();
            if (!p.err) return cudaErrorInvalidValue;
            const int smem = a.P * kTmaTile + 16;
            if (!allow_smem(fn, smem)) return cudaErrorInvalidValue;
            const int64_t tiles = std::max<int64_t>(1, (seg_bytes + kTmaTile - 1) / kTmaTile);
            return launch_pdl(fn, dim3((unsigned)tiles, S), dim3(kTmaThreads), args, smem, stream);
        }
    }
    // Register path, one block per chunk of V x 256 vectors.  V from
    // measurements on GB300 (fraction of the measured copy bandwidth, one
    // call, one-shot grids): bf16 sum / prod RHD AllReduce V2 (1.016, against
    // 0.930 with V1); every other shape V1 (Ring fp32 AllReduce 0.97 - 1.00
    // against 0.96 with V2).
    int V = 1;
    if (COLL == 0 && a.P <= 16 && es == 2 && a.algo == HC_ALGO_RHD &&
        (a.op == HC_SUM || a.op == HC_PROD))
        V = 2;
    // Page-locked host buffers: the host link (about 210 GB/s each way, 330
    // GB/s both ways at once on GB300 with Grace), not HBM, bounds the kernel;
    // 1 to 16 blocks per SM measured within 4 % of each other, 1 the fastest.
    if (a.host_buffers) V = 1;
    void* fn = pick_reduce(a.algo, COLL, a.dtype, a.op, V, a.P);
    if (!fn && V != 1) {  // shape not instantiated: one vector per thread
        V = 1;
        fn = pick_reduce(a.algo, COLL, a.dtype, a.op, V, a.P);
    }
    if (!fn) return cudaErrorInvalidValue;
    const int64_t vecs = (lay.L + lay.A - 1) / lay.A;
    const int64_t want = std::max<int64_t>(1, (vecs + (int64_t)V * kFusedThreads - 1) / ((int64_t)V * kFusedThreads));
    const int64_t gx = a.host_buffers ? std::min(want, std::max<int64_t>(1, (int64_t)sm_count / S)) : want;
    return launch_pdl(fn, dim3((unsigned)gx, S), dim3(kFusedThreads), args, 0, stream);
}

cudaError_t read_device_error(bool clear, int* status) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, hc_device_error, sizeof(int));
    if (e != cudaSuccess) return e;
    *status = v;
    if (clear && v) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(hc_device_error, &zero, sizeof(int));
    }
    return e;
}

}  // namespace hc

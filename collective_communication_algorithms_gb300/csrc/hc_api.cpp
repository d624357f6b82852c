// hc_api.cpp -- the C ABI of libhc (see include/hc.h): argument validation,
// in-place detection, step-plan cache and dispatch to the kernels.
#include <algorithm>
#include <atomic>
#include <cstddef>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>
#include <vector>

#include <cuda_runtime.h>

#include "hc_internal.h"

using namespace hc;

namespace {

bool valid_dtype(hc_dtype_t d) { return d == HC_INT32 || d == HC_FLOAT32 || d == HC_BFLOAT16; }
bool valid_op(hc_op_t o) { return o == HC_SUM || o == HC_PROD || o == HC_MAX || o == HC_MIN; }
bool valid_algo(hc_algo_t a) {
    return a == HC_ALGO_RING || a == HC_ALGO_RHD || a == HC_ALGO_PIPELINE || a == HC_ALGO_HIER;
}
bool valid_coll(hc_coll_t c) {
    return c == HC_COLL_ALLREDUCE || c == HC_COLL_REDUCE_SCATTER || c == HC_COLL_ALLGATHER ||
           c == HC_COLL_BROADCAST;
}

struct Opts {
    hc_mode_t mode = HC_MODE_FUSED;
    int p_intra = 1;
    int64_t loop_bytes = 0;
    void* scratch = nullptr;
    size_t scratch_bytes = 0;
    bool host_buffers = false;
};

hc_status_t read_opts(const hc_opts_t* o, hc_algo_t algo, int P, Opts* out) {
    *out = Opts();
    if (!o) return HC_OK;
    // callers built before host_buffers existed pass the shorter size
    if (o->struct_size < offsetof(hc_opts_t, host_buffers)) return HC_ERR_INVALID_ARG;
    if (o->struct_size >= sizeof(hc_opts_t)) {
        if (o->host_buffers != 0 && o->host_buffers != 1) return HC_ERR_INVALID_ARG;
        out->host_buffers = o->host_buffers == 1;
    }
    if (o->mode != HC_MODE_FUSED && o->mode != HC_MODE_STEP) return HC_ERR_INVALID_ARG;
    out->mode = o->mode;
    if (algo == HC_ALGO_PIPELINE || algo == HC_ALGO_HIER) {
        if (o->ranks_per_server < 1 || P % o->ranks_per_server) return HC_ERR_INVALID_ARG;
        out->p_intra = o->ranks_per_server;
    }
    if (o->max_loop_bytes > (size_t)INT64_MAX) return HC_ERR_INVALID_ARG;
    out->loop_bytes = (int64_t)o->max_loop_bytes;
    out->scratch = o->scratch;
    out->scratch_bytes = o->scratch_bytes;
    return HC_OK;
}

// true when some two intervals overlap (empty intervals ignored); sorts v
bool any_overlap(std::vector<Interval>& v) {
    v.erase(std::remove_if(v.begin(), v.end(), [](const Interval& x) { return x.hi <= x.lo; }),
            v.end());
    std::sort(v.begin(), v.end(), [](const Interval& a, const Interval& b) { return a.lo < b.lo; });
    uintptr_t end = 0;
    for (size_t i = 0; i < v.size(); i++) {
        if (i > 0 && v[i].lo < end) return true;
        end = std::max(end, v[i].hi);
    }
    return false;
}

// The CUDA error behind the last HC_ERR_CUDA returned on this thread.
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

hc_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return HC_OK;
    g_last_cuda_error = e;
    return HC_ERR_CUDA;
}

// A buffer the kernels may dereference at its own address: device or managed
// memory, or page-locked host memory mapped at the same address (unified
// addressing).  Pageable memory, or host memory mapped elsewhere, is refused.
hc_status_t check_device_accessible(const void* p) {
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // leave no pending error behind for the caller
        return cuda_status(e);
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return HC_OK;
    if (at.type == cudaMemoryTypeHost && at.devicePointer == p) return HC_OK;
    return HC_ERR_INVALID_ARG;
}

int sm_count_of_current_device() {
    static std::atomic<int> cache[kMaxDevices];  // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c) return c;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

// ---------------------------------------------------------------- plan cache
using PlanKey = std::tuple<int, int, int, int, int, int64_t, int, int64_t, unsigned long long,
                           unsigned long long>;
std::map<PlanKey, std::shared_ptr<const Plan>>& plan_cache() {
    static std::map<PlanKey, std::shared_ptr<const Plan>> m;
    return m;
}
// Guards plan_cache(): host threads may call the collectives concurrently.
std::mutex g_plan_cache_mu;

std::shared_ptr<const Plan> get_plan(hc_algo_t algo, hc_coll_t coll, int P, int p_intra, int root,
                                     int64_t n, hc_dtype_t dt, int64_t loop_bytes,
                                     const Aliasing& al) {
    unsigned long long m1 = 0, m2 = 0;
    for (int r = 0; r < P; r++) {
        if (al.orig_is_work[r]) m1 |= 1ull << r;
        if (al.final_is_work[r]) m2 |= 1ull << r;
    }
    PlanKey key{(int)algo, (int)coll, P, p_intra, root, n, (int)dt, loop_bytes, m1, m2};
    std::lock_guard<std::mutex> lock(g_plan_cache_mu);
    auto& cache = plan_cache();
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    if (cache.size() >= 256) cache.clear();  // plans still held by callers stay alive
    auto plan = std::make_shared<Plan>();
    if (!build_plan(algo, coll, P, p_intra, root, n, dt, loop_bytes, al, plan.get())) return nullptr;
    cache.emplace(key, plan);
    log_plan(algo, coll, P, p_intra, n, dt, loop_bytes, *plan);
    return plan;
}

size_t scratch_stride(size_t n, hc_dtype_t dt) {
    size_t b = n * (size_t)elem_bytes(dt);
    return (b + 255) / 256 * 256;
}

}  // namespace

namespace hc {

// Validate one collective call and record everything its launch needs.
hc_status_t prepare(hc_coll_t coll, const void* const* send, void* const* recv, int P, size_t count,
                    hc_dtype_t dtype, hc_op_t op, hc_algo_t algo, const hc_opts_t* opts, int root,
                    Prepared* out) {
    *out = Prepared();
    if (!valid_dtype(dtype) || !valid_op(op) || !valid_algo(algo)) return HC_ERR_INVALID_ARG;
    if (P < 1 || P > kMaxRanks) return HC_ERR_INVALID_ARG;
    const bool bcast = coll == HC_COLL_BROADCAST;
    if (bcast && (root < 0 || root >= P)) return HC_ERR_INVALID_ARG;
    if (bcast && algo != HC_ALGO_RHD) return HC_ERR_UNSUPPORTED;
    if (algo == HC_ALGO_HIER && coll != HC_COLL_ALLREDUCE) return HC_ERR_UNSUPPORTED;
    Opts o;
    hc_status_t st = read_opts(opts, algo, P, &o);
    if (st != HC_OK) return st;
    Prepared& c = *out;
    c.coll = coll;
    c.algo = algo;
    c.dtype = dtype;
    c.op = op;
    c.P = P;
    c.count = count;
    c.mode = o.mode;
    c.p_intra = o.p_intra;
    c.root = bcast ? root : -1;
    c.loop_bytes = o.loop_bytes;
    c.empty = count == 0;
    if (c.empty) return HC_OK;
    if (count > (size_t)INT64_MAX / 16) return HC_ERR_INVALID_ARG;
    if (!recv) return HC_ERR_INVALID_ARG;
    if (!send && coll != HC_COLL_ALLGATHER && !bcast) return HC_ERR_INVALID_ARG;

    const int64_t n = (int64_t)count;
    const int es = elem_bytes(dtype);
    c.lay = make_layout(algo, coll, P, n, dtype, o.p_intra);
    const Layout& own = c.lay;  // the per-rank segment of RS / AG is the rank's own

    // a buffer of zero elements (the ReduceScatter output or AllGather input
    // of an empty trailing segment) is never touched: it may be NULL or
    // unaligned; every other buffer must be non-null and 16-byte aligned
    for (int r = 0; r < P; r++) {
        const bool seg_empty = bcast ? false : own.seg_hi(r) == own.seg_lo(r);
        const bool recv_used = !(coll == HC_COLL_REDUCE_SCATTER && seg_empty);
        const bool send_used = bcast ? (send && r == root && send[r])
                                     : send && !(coll == HC_COLL_ALLGATHER && seg_empty);
        if ((recv_used && !recv[r]) || (send_used && !send[r])) return HC_ERR_INVALID_ARG;
        if ((recv_used && ((uintptr_t)recv[r] & 15)) || (send_used && ((uintptr_t)send[r] & 15)))
            return HC_ERR_ALIGN;
        if (o.host_buffers) {
            if (recv_used && (st = check_device_accessible(recv[r])) != HC_OK) return st;
            if (send_used && (st = check_device_accessible(send[r])) != HC_OK) return st;
        }
    }
    c.host_buffers = o.host_buffers;

    std::memset(&c.al, 0, sizeof c.al);
    std::vector<Interval> iv;
    iv.reserve(2 * (size_t)P + 1);  // one allocation each, not one per growth
    c.reads.reserve((size_t)P);
    c.writes.reserve((size_t)P + 1);
    const uintptr_t full = (uintptr_t)n * es;
    for (int r = 0; r < P; r++) {
        const uintptr_t d = (uintptr_t)recv[r];
        c.recv[r] = d;
        if (coll == HC_COLL_ALLREDUCE) {
            const uintptr_t s = (uintptr_t)send[r];
            c.send[r] = s;
            c.al.orig_is_work[r] = (s == d);
            c.al.final_is_work[r] = true;
            iv.push_back({d, d + full});
            c.writes.push_back({d, d + full});
            if (s != d) {
                iv.push_back({s, s + full});
                c.reads.push_back({s, s + full});
            }
        } else if (coll == HC_COLL_REDUCE_SCATTER) {
            const uintptr_t s = (uintptr_t)send[r];
            c.send[r] = s;
            const uintptr_t off = (uintptr_t)own.seg_lo(r) * es;
            const uintptr_t len = (uintptr_t)(own.seg_hi(r) - own.seg_lo(r)) * es;
            c.rs_in_place[r] = (d == s + off);
            iv.push_back({s, s + full});
            c.reads.push_back({s, s + full});
            if (!c.rs_in_place[r]) {
                iv.push_back({d, d + len});
                c.writes.push_back({d, d + len});
            } else {
                c.writes.push_back({s, s + full});  // the input is working memory
            }
        } else if (bcast) {
            // only the root has an input; it is in place when it is recv[root]
            const uintptr_t s = (r == root && send && send[r]) ? (uintptr_t)send[r] : d;
            c.send[r] = s;
            c.ag_in_place[r] = (s == d);
            c.al.orig_is_work[r] = c.ag_in_place[r];
            c.al.final_is_work[r] = true;
            if (r == root && s != d) {
                iv.push_back({s, s + full});
                c.reads.push_back({s, s + full});
            }
            if (r != root || s != d) {
                iv.push_back({d, d + full});
                c.writes.push_back({d, d + full});
            } else {
                iv.push_back({d, d + full});
                c.reads.push_back({d, d + full});
            }
        } else {
            const uintptr_t off = (uintptr_t)own.seg_lo(r) * es;
            const uintptr_t len = (uintptr_t)(own.seg_hi(r) - own.seg_lo(r)) * es;
            const uintptr_t s = send ? (uintptr_t)send[r] : d + off;
            c.send[r] = s;
            c.ag_in_place[r] = (s == d + off);
            c.al.orig_is_work[r] = c.ag_in_place[r];
            c.al.final_is_work[r] = true;
            iv.push_back({d, d + full});
            c.writes.push_back({d, d + full});
            if (!c.ag_in_place[r]) {
                iv.push_back({s, s + len});
                c.reads.push_back({s, s + len});
            }
        }
    }
    c.has_send = send != nullptr;

    // step-mode ReduceScatter: working memory is the input (in place) or scratch
    bool need_scratch = false;
    if (coll == HC_COLL_REDUCE_SCATTER && o.mode == HC_MODE_STEP) {
        for (int r = 0; r < P; r++) {
            c.al.orig_is_work[r] = c.rs_in_place[r];
            c.al.final_is_work[r] = c.rs_in_place[r];
            if (!c.rs_in_place[r]) need_scratch = true;
        }
    }
    if (need_scratch) {
        const size_t need = (size_t)P * scratch_stride(count, dtype);
        if (!o.scratch || o.scratch_bytes < need) return HC_ERR_SCRATCH;
        if ((uintptr_t)o.scratch & 15) return HC_ERR_ALIGN;
        iv.push_back({(uintptr_t)o.scratch, (uintptr_t)o.scratch + need});
        c.writes.push_back({(uintptr_t)o.scratch, (uintptr_t)o.scratch + need});
        c.scratch = (uintptr_t)o.scratch;
    }
    if (any_overlap(iv)) return HC_ERR_INVALID_ARG;
    if (o.mode == HC_MODE_STEP) {
        c.plan = get_plan(algo, coll, P, o.p_intra, bcast ? root : 0, n, dtype, o.loop_bytes, c.al);
        if (!c.plan) return HC_ERR_INVALID_ARG;
    }
    return HC_OK;
}

// Launch a prepared call on a stream.
hc_status_t execute(const Prepared& c, cudaStream_t stream) {
    if (c.empty) return HC_OK;
    const TraceRange range(c.coll, trace_category(c.algo, c.mode), (uint64_t)c.count);
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return cuda_status(cudaErrorNoDevice);
    const int es = elem_bytes(c.dtype);
    const Layout& own = c.lay;
    if (c.mode == HC_MODE_FUSED) {
        log_fused(c);
        const void* sp[kMaxRanks];
        void* rp[kMaxRanks];
        for (int r = 0; r < c.P; r++) {
            sp[r] = (const void*)c.send[r];
            rp[r] = (void*)c.recv[r];
        }
        FusedArgs a;
        a.algo = c.algo;
        a.coll = c.coll;
        a.dtype = c.dtype;
        a.op = c.op;
        a.P = c.P;
        a.p_intra = c.p_intra;
        a.n = (int64_t)c.count;
        a.lay = c.lay;
        a.send = sp;
        a.recv = rp;
        std::memcpy(a.ag_in_place, c.ag_in_place, sizeof a.ag_in_place);
        std::memcpy(a.rs_in_place, c.rs_in_place, sizeof a.rs_in_place);
        a.root = c.root;
        a.host_buffers = c.host_buffers;
        return cuda_status(launch_fused(a, stream, sms));
    }
    uintptr_t base[LOC_COUNT][kMaxRanks];
    std::memset(base, 0, sizeof base);
    for (int r = 0; r < c.P; r++) {
        const uintptr_t d = c.recv[r], s = c.send[r];
        if (c.coll == HC_COLL_ALLREDUCE) {
            base[LOC_ORIG][r] = s;
            base[LOC_WORK][r] = d;
            base[LOC_FINAL][r] = d;
        } else if (c.coll == HC_COLL_REDUCE_SCATTER) {
            base[LOC_ORIG][r] = s;
            base[LOC_WORK][r] = c.rs_in_place[r] ? s : c.scratch + (uintptr_t)r * scratch_stride(c.count, c.dtype);
            base[LOC_FINAL][r] = d - (uintptr_t)own.seg_lo(r) * es;
        } else if (c.coll == HC_COLL_BROADCAST) {
            base[LOC_ORIG][r] = s;
            base[LOC_WORK][r] = d;
            base[LOC_FINAL][r] = d;
        } else {
            const uintptr_t off = (uintptr_t)own.seg_lo(r) * es;
            base[LOC_ORIG][r] = s - off;
            base[LOC_WORK][r] = d;
            base[LOC_FINAL][r] = d;
        }
    }
    return cuda_status(launch_step(*c.plan, c.P, c.dtype, c.op, base, stream, sms, c.host_buffers));
}

bool conflicts(const Prepared& a, const Prepared& b) {
    auto hit = [](const std::vector<Interval>& x, const std::vector<Interval>& y) {
        for (const Interval& i : x)
            for (const Interval& j : y)
                if (i.lo < j.hi && j.lo < i.hi && i.lo < i.hi && j.lo < j.hi) return true;
        return false;
    };
    return hit(a.writes, b.writes) || hit(a.writes, b.reads) || hit(a.reads, b.writes);
}

}  // namespace hc

namespace {

hc_status_t run(hc_coll_t coll, const void* const* send, void* const* recv, int P, size_t count,
                hc_dtype_t dtype, hc_op_t op, hc_algo_t algo, const hc_opts_t* opts,
                cudaStream_t stream) {
    Prepared c;
    const hc_status_t st = prepare(coll, send, recv, P, count, dtype, op, algo, opts, -1, &c);
    if (st != HC_OK) return st;
    return execute(c, stream);
}

}  // namespace

extern "C" {

hc_status_t hc_allreduce(const void* const* send, void* const* recv, int P, size_t count,
                         hc_dtype_t dtype, hc_op_t op, hc_algo_t algo, const hc_opts_t* opts,
                         hc_stream_t stream) {
    return run(HC_COLL_ALLREDUCE, send, recv, P, count, dtype, op, algo, opts,
               (cudaStream_t)stream);
}

hc_status_t hc_reduce_scatter(const void* const* send, void* const* recv, int P, size_t count,
                              hc_dtype_t dtype, hc_op_t op, hc_algo_t algo,
                              const hc_opts_t* opts, hc_stream_t stream) {
    return run(HC_COLL_REDUCE_SCATTER, send, recv, P, count, dtype, op, algo, opts,
               (cudaStream_t)stream);
}

hc_status_t hc_broadcast(const void* send, void* const* recv, int P, size_t count,
                         hc_dtype_t dtype, int root, hc_algo_t algo, const hc_opts_t* opts,
                         hc_stream_t stream) {
    if (P < 1 || P > kMaxRanks) return HC_ERR_INVALID_ARG;
    const void* sendv[kMaxRanks] = {nullptr};
    if (root >= 0 && root < P) sendv[root] = send;
    Prepared c;
    const hc_status_t st = prepare(HC_COLL_BROADCAST, sendv, recv, P, count, dtype, HC_SUM, algo,
                                   opts, root, &c);
    if (st != HC_OK) return st;
    return execute(c, (cudaStream_t)stream);
}

hc_status_t hc_allgather(const void* const* send, void* const* recv, int P, size_t count,
                         hc_dtype_t dtype, hc_algo_t algo, const hc_opts_t* opts,
                         hc_stream_t stream) {
    return run(HC_COLL_ALLGATHER, send, recv, P, count, dtype, HC_SUM, algo, opts,
               (cudaStream_t)stream);
}

int hc_num_segments(hc_algo_t algo, hc_coll_t coll, int P) {
    if (!valid_algo(algo) || !valid_coll(coll) || P < 1 || P > kMaxRanks) return 0;
    if (algo == HC_ALGO_HIER) return 0;  // depends on ranks_per_server
    return num_segments(algo, coll, P);
}

hc_status_t hc_segment_range(hc_algo_t algo, hc_coll_t coll, int P, size_t count,
                             hc_dtype_t dtype, int k, size_t* off, size_t* len) {
    if (!valid_algo(algo) || !valid_coll(coll) || !valid_dtype(dtype)) return HC_ERR_INVALID_ARG;
    if (P < 1 || P > kMaxRanks || !off || !len) return HC_ERR_INVALID_ARG;
    if (count > (size_t)INT64_MAX / 16) return HC_ERR_INVALID_ARG;
    if (algo == HC_ALGO_HIER) return HC_ERR_UNSUPPORTED;
    Layout lay = make_layout(algo, coll, P, (int64_t)count, dtype);
    if (k < 0 || k >= lay.S) return HC_ERR_INVALID_ARG;
    *off = (size_t)lay.seg_lo(k);
    *len = (size_t)(lay.seg_hi(k) - lay.seg_lo(k));
    return HC_OK;
}

size_t hc_scratch_bytes(hc_algo_t algo, int P, size_t count, hc_dtype_t dtype) {
    if (!valid_algo(algo) || !valid_dtype(dtype) || P < 1 || P > kMaxRanks) return 0;
    return (size_t)P * scratch_stride(count, dtype);
}

hc_status_t hc_schedule_stats(hc_algo_t algo, hc_coll_t coll, int P, int ranks_per_server,
                              size_t count, hc_dtype_t dtype, size_t max_loop_bytes,
                              hc_stats_t* stats, unsigned long long* bytes_sent) {
    if (!valid_algo(algo) || !valid_coll(coll) || !valid_dtype(dtype)) return HC_ERR_INVALID_ARG;
    if (P < 1 || P > kMaxRanks || count > (size_t)INT64_MAX / 16) return HC_ERR_INVALID_ARG;
    if (stats && stats->struct_size < sizeof(hc_stats_t)) return HC_ERR_INVALID_ARG;
    int p_intra = (algo == HC_ALGO_PIPELINE || algo == HC_ALGO_HIER) ? ranks_per_server : 1;
    if (p_intra < 1 || P % p_intra) return HC_ERR_INVALID_ARG;
    const int64_t n = (int64_t)count;
    int spl = 0;
    if (!schedule_traffic(algo, coll, P, p_intra, 0, n, dtype, (int64_t)max_loop_bytes, &spl,
                          bytes_sent))
        return HC_ERR_INVALID_ARG;
    if (!stats) return HC_OK;
    Aliasing al;
    for (int r = 0; r < P; r++) { al.orig_is_work[r] = true; al.final_is_work[r] = true; }
    Plan plan;
    if (!build_plan(algo, coll, P, p_intra, 0, n, dtype, (int64_t)max_loop_bytes, al, &plan))
        return HC_ERR_INVALID_ARG;
    const int es = elem_bytes(dtype);
    stats->steps_per_loop = spl;
    stats->loops = plan.sl.loops;
    stats->chunk = (size_t)plan.sl.chunk;
    stats->tail = (size_t)plan.sl.tail;
    stats->launches_step = (int)plan.launches.size();
    stats->launches_fused = n > 0 ? 1 : 0;
    unsigned long long sb = 0;
    for (const PlanLaunch& L : plan.launches)
        for (const DevItem& it : L.items)
            for (int i = 0; i < it.seg_width * it.seg_reps; i++) {
                int k = it.seg_first + (i / it.seg_width) * it.seg_stride + i % it.seg_width;
                int64_t lo = std::min(plan.lay.seg_lo(k) + L.lo, plan.lay.seg_hi(k));
                int64_t hi = std::min(plan.lay.seg_lo(k) + L.hi, plan.lay.seg_hi(k));
                unsigned long long len = (unsigned long long)(hi - lo) * es;
                sb += len * (unsigned long long)(it.in_cnt + (it.acc_rank >= 0) + item_outputs(it));
            }
    stats->step_bytes = sb;
    const unsigned long long nb = (unsigned long long)n * es;
    if (coll == HC_COLL_ALLREDUCE) stats->fused_bytes = 2ull * P * nb;
    else stats->fused_bytes = (unsigned long long)(P + 1) * nb;  // RS, AG and Broadcast out of place
    return HC_OK;
}

hc_status_t hc_step_plan(hc_algo_t algo, hc_coll_t coll, int P, int ranks_per_server,
                         size_t count, hc_dtype_t dtype, size_t max_loop_bytes, int in_place,
                         int root, hc_plan_record_t* records, size_t cap, size_t* n_out,
                         int* launches) {
    if (!valid_algo(algo) || !valid_coll(coll) || !valid_dtype(dtype) || !n_out)
        return HC_ERR_INVALID_ARG;
    if (P < 1 || P > kMaxRanks || count > (size_t)INT64_MAX / 16) return HC_ERR_INVALID_ARG;
    int p_intra = (algo == HC_ALGO_PIPELINE || algo == HC_ALGO_HIER) ? ranks_per_server : 1;
    if (p_intra < 1 || P % p_intra) return HC_ERR_INVALID_ARG;
    Aliasing al;
    for (int r = 0; r < P; r++) {
        al.orig_is_work[r] = in_place != 0;
        al.final_is_work[r] = in_place != 0;
        if (coll == HC_COLL_ALLREDUCE) al.final_is_work[r] = true;
        if (coll == HC_COLL_ALLGATHER || coll == HC_COLL_BROADCAST) al.final_is_work[r] = true;
    }
    if (coll == HC_COLL_BROADCAST && (root < 0 || root >= P)) return HC_ERR_INVALID_ARG;
    Plan plan;
    if (!build_plan(algo, coll, P, p_intra, coll == HC_COLL_BROADCAST ? root : 0, (int64_t)count,
                    dtype, (int64_t)max_loop_bytes, al, &plan))
        return HC_ERR_INVALID_ARG;
    size_t m = 0;
    for (size_t li = 0; li < plan.launches.size(); li++) {
        const PlanLaunch& L = plan.launches[li];
        for (const DevItem& it : L.items)
            for (int i = 0; i < it.seg_width * it.seg_reps; i++) {
                int k = it.seg_first + (i / it.seg_width) * it.seg_stride + i % it.seg_width;
                if (records && m < cap) {
                    hc_plan_record_t& R = records[m];
                    std::memset(&R, 0, sizeof R);
                    R.launch = (int32_t)li;
                    R.seg = k;
                    R.lo = std::min(plan.lay.seg_lo(k) + L.lo, plan.lay.seg_hi(k));
                    R.hi = std::min(plan.lay.seg_lo(k) + L.hi, plan.lay.seg_hi(k));
                    R.acc_rank = it.acc_rank;
                    R.acc_loc = it.acc_loc;
                    R.in_loc = it.in_loc;
                    R.in_cnt = it.in_cnt;
                    R.out_loc = it.out_loc;
                    R.out_cnt = item_outputs(it);
                    for (int j = 0; j < it.in_cnt; j++)
                        R.in_ranks[j] = it.in_base + (it.in_rot + j) % it.in_mod;
                    for (int j = 0; j < it.out_cnt; j++)
                        R.out_ranks[j] = it.out_base + (it.out_rot + j) % it.out_mod;
                    for (int j = 0; j < it.out2_cnt; j++)
                        R.out_ranks[it.out_cnt + j] = it.out2_base + (it.out2_rot + j) % it.out2_mod;
                }
                m++;
            }
    }
    *n_out = m;
    if (launches) *launches = (int)plan.launches.size();
    return HC_OK;
}

hc_status_t hc_select_algo(hc_coll_t coll, int P, int ranks_per_server, size_t count,
                           hc_dtype_t dtype, hc_mode_t mode, hc_algo_t* out_algo,
                           double* predicted_us) {
    // Constants measured on GB300 (a C caller; bench.py --sweep select, the
    // benchmark's configurations and a C timing loop around the entry points),
    // the device terms fitted to the measured table by least squares on the
    // log of the time:
    //  host: 0.55 us of the library's own work per call, 1.4 us per launch;
    //  step mode: the device time per dependent launch of each schedule (Ring
    //    1.8 us, RHD 2.0, Pipeline 1.9, hierarchical 2.6 -- fewer but heavier
    //    launches) plus 0.02 us per rank (the launch's items), and the
    //    fraction of the copy bandwidth each schedule's steps reach on their
    //    own bytes (above 1 where a step's outputs come back from L2 as the
    //    next step's operands);
    //  fused mode: a fixed device cost per call plus a per-rank cost of the
    //    schedule's reduction in one block (the Ring chain, the RHD tree --
    //    compile-time below 16 ranks, looped above --, the Pipeline and
    //    hierarchical two-level trees, the AllGather's plain copies), then the
    //    bytes at the path's fraction of the bandwidth (AllReduce /
    //    ReduceScatter TMA-staged up to 32 ranks, register path above; the
    //    AllGather, prefetching its source into L2 from 16 ranks);
    //  both modes: a call whose ranks' vectors fit in L2 (P n b <= 96 MiB)
    //    moves its bytes 1.44 times faster when its buffers are L2-resident, as
    //    for calls repeated on the same buffers.
    const double kHostCallUs = 0.55, kHostLaunchUs = 1.4;
    const double kFusedBaseUs = 1.3, kBandwidth = 6800e9;
    const double kLaunchPerRankUs = 0.02, kL2HotBytes = 96.0 * (1 << 20), kL2HotFactor = 1.44;
    if (!out_algo || !valid_coll(coll) || !valid_dtype(dtype)) return HC_ERR_INVALID_ARG;
    if (mode != HC_MODE_FUSED && mode != HC_MODE_STEP) return HC_ERR_INVALID_ARG;
    if (P < 1 || P > kMaxRanks) return HC_ERR_INVALID_ARG;
    std::vector<hc_algo_t> cands = {HC_ALGO_RING, HC_ALGO_RHD};
    if (coll == HC_COLL_BROADCAST) cands = {HC_ALGO_RHD};
    const bool servers = ranks_per_server > 1 && P % ranks_per_server == 0;
    if (servers && coll != HC_COLL_BROADCAST) cands.push_back(HC_ALGO_PIPELINE);
    if (servers && coll == HC_COLL_ALLREDUCE) cands.push_back(HC_ALGO_HIER);
    const bool copy = coll == HC_COLL_ALLGATHER || coll == HC_COLL_BROADCAST;
    double best = 0, best_dev = 0;
    bool have = false;
    for (hc_algo_t a : cands) {
        hc_stats_t st;
        std::memset(&st, 0, sizeof st);
        st.struct_size = sizeof st;
        const int rps = (a == HC_ALGO_PIPELINE || a == HC_ALGO_HIER) ? ranks_per_server : 1;
        if (hc_schedule_stats(a, coll, P, rps, count, dtype, 0, &st, nullptr) != HC_OK) continue;
        double host, dev;
        const double bw = kBandwidth *
                          ((double)P * (double)count * elem_bytes(dtype) <= kL2HotBytes ? kL2HotFactor : 1.0);
        if (mode == HC_MODE_STEP) {
            const double launch_us = (a == HC_ALGO_RING       ? 1.8
                                      : a == HC_ALGO_RHD      ? 2.0
                                      : a == HC_ALGO_PIPELINE ? 1.9
                                                              : 2.6) +
                                     kLaunchPerRankUs * P;
            const double f = a == HC_ALGO_RING       ? 1.48
                             : a == HC_ALGO_RHD      ? 1.24
                             : a == HC_ALGO_PIPELINE ? 1.17
                                                     : 1.12;
            host = kHostCallUs + st.launches_step * kHostLaunchUs;
            dev = st.launches_step * launch_us + (double)st.step_bytes / (f * bw) * 1e6;
        } else {
            double per_rank, f;
            if (copy) {
                per_rank = 0.042;
                f = P < 16 ? 1.05 : 1.09;
            } else {
                per_rank = a == HC_ALGO_RING       ? 0.064
                           : a == HC_ALGO_RHD      ? (P < 16 ? 0.057 : 0.076)
                           : a == HC_ALGO_PIPELINE ? 0.076
                                                   : 0.098;
                f = P <= 32 ? 1.03 : 0.99;
            }
            host = kHostCallUs + st.launches_fused * kHostLaunchUs;
            dev = st.launches_fused ? kFusedBaseUs + per_rank * P +
                                          (double)st.fused_bytes / (f * bw) * 1e6
                                    : 0.0;
        }
        // launches are queued asynchronously: the host cost and the device
        // time overlap and the larger decides; between equal costs the lower
        // device time, then the earlier candidate
        const double t = host > dev ? host : dev;
        if (!have || t < best || (t == best && dev < best_dev)) {
            best = t;
            best_dev = dev;
            *out_algo = a;
            have = true;
        }
    }
    if (!have) return HC_ERR_INVALID_ARG;
    if (predicted_us) *predicted_us = best;
    return HC_OK;
}

hc_status_t hc_device_status(int clear) {
    int v = 0;
    const hc_status_t st = cuda_status(read_device_error(clear != 0, &v));
    if (st != HC_OK) return st;
    return v ? (hc_status_t)v : HC_OK;
}

hc_status_t hc_test_expire_waits(int enable) {
    if (enable != 0 && enable != 1) return HC_ERR_INVALID_ARG;
    set_test_expire_waits(enable == 1);
    return HC_OK;
}

const char* hc_last_cuda_error(void) {
    return g_last_cuda_error == cudaSuccess ? "cudaSuccess" : cudaGetErrorName(g_last_cuda_error);
}

const char* hc_status_string(hc_status_t s) {
    switch (s) {
    case HC_OK: return "success";
    case HC_ERR_INVALID_ARG: return "invalid argument";
    case HC_ERR_UNSUPPORTED: return "unsupported combination";
    case HC_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case HC_ERR_SCRATCH: return "step-mode scratch missing or too small";
    case HC_ERR_CUDA: return "CUDA launch or query failed";
    case HC_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
    }
}

int hc_version(void) { return HC_VERSION; }

}  // extern "C"

// hc_trace.cpp -- tracing of libhc calls.
//
// NVTX ranges in the "libhc" domain, for Nsight tools: one per collective
// call (message = the entry point, category = algorithm and mode, payload =
// the element count) and one per step-mode kernel launch (payload = the
// launch's index in the call's plan, i.e. loop * steps_per_loop + step).
// With no tool attached a range costs one test of a function pointer.
//
// HC_LOG: when the environment variable HC_LOG is a nonzero integer, one
// line on stderr for every step-mode plan the library builds (the schedule,
// its steps per loop, the loop slicer's loops / chunk / tail and the number
// of launches, as the Pipeline article's OrchestrateLoop logs its loops
// before running them) and for the first fused call of every shape.  This
// is the per-collective breakdown the Ring vs RHD article describes
// (algorithm preparation, data slicing, transfer).
#include <nvtx3/nvToolsExt.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <set>
#include <tuple>

#include "hc_internal.h"

namespace hc {
namespace {

const char* algo_name(hc_algo_t a) {
    switch (a) {
    case HC_ALGO_RING: return "ring";
    case HC_ALGO_RHD: return "rhd";
    case HC_ALGO_PIPELINE: return "pipeline";
    case HC_ALGO_HIER: return "hier";
    default: return "?";
    }
}
const char* coll_name(hc_coll_t c) {
    switch (c) {
    case HC_COLL_ALLREDUCE: return "allreduce";
    case HC_COLL_REDUCE_SCATTER: return "reducescatter";
    case HC_COLL_ALLGATHER: return "allgather";
    case HC_COLL_BROADCAST: return "broadcast";
    default: return "?";
    }
}
const char* entry_name(hc_coll_t c) {
    switch (c) {
    case HC_COLL_ALLREDUCE: return "hc_allreduce";
    case HC_COLL_REDUCE_SCATTER: return "hc_reduce_scatter";
    case HC_COLL_ALLGATHER: return "hc_allgather";
    case HC_COLL_BROADCAST: return "hc_broadcast";
    default: return "hc_collective";
    }
}
const char* dtype_name(hc_dtype_t d) {
    return d == HC_INT32 ? "int32" : d == HC_FLOAT32 ? "float32" : "bfloat16";
}
const char* op_name(hc_op_t o) {
    return o == HC_SUM ? "sum" : o == HC_PROD ? "prod" : o == HC_MAX ? "max" : "min";
}

// The domain and its named categories (one per algorithm x mode), created
// on first use.
nvtxDomainHandle_t domain() {
    static nvtxDomainHandle_t d = [] {
        nvtxDomainHandle_t h = nvtxDomainCreateA("libhc");
        static const char* names[] = {"ring fused", "ring step", "rhd fused", "rhd step",
                                      "pipeline fused", "pipeline step", "hier fused", "hier step"};
        for (int i = 0; i < 8; i++) nvtxDomainNameCategoryA(h, (uint32_t)(i + 1), names[i]);
        return h;
    }();
    return d;
}

void push(const char* msg, uint32_t category, uint64_t payload) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.category = category;
    a.payloadType = NVTX_PAYLOAD_TYPE_UNSIGNED_INT64;
    a.payload.ullValue = payload;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = msg;
    nvtxDomainRangePushEx(domain(), &a);
}

bool read_log_env() {
    const char* v = std::getenv("HC_LOG");
    return v && std::atoi(v) != 0;
}

void log_line(const char* fmt, ...) {
    static std::mutex mu;  // one whole line at a time
    std::lock_guard<std::mutex> lock(mu);
    std::fputs("hc: ", stderr);
    va_list ap;
    va_start(ap, fmt);
    std::vfprintf(stderr, fmt, ap);
    va_end(ap);
    std::fputc('\n', stderr);
    std::fflush(stderr);
}

}  // namespace

uint32_t trace_category(hc_algo_t algo, hc_mode_t mode) {
    const int a = (algo >= HC_ALGO_RING && algo <= HC_ALGO_HIER) ? (int)algo : 0;
    return (uint32_t)(2 * a + (mode == HC_MODE_STEP ? 1 : 0) + 1);
}

TraceRange::TraceRange(hc_coll_t coll, uint32_t category, uint64_t payload) {
    push(entry_name(coll), category, payload);
}
TraceRange::TraceRange(const char* msg, uint32_t category, uint64_t payload) {
    push(msg, category, payload);
}
TraceRange::~TraceRange() { nvtxDomainRangePop(domain()); }

bool log_enabled() {
    static const bool on = read_log_env();
    return on;
}

void log_plan(hc_algo_t algo, hc_coll_t coll, int P, int p_intra, int64_t n, hc_dtype_t dt,
              int64_t loop_bytes, const Plan& plan) {
    if (!log_enabled()) return;
    log_line("plan %s %s P=%d ranks_per_server=%d n=%lld %s max_loop_bytes=%lld: "
             "segments=%d L=%lld steps_per_loop=%d loops=%d chunk=%lld tail=%lld launches=%zu",
             coll_name(coll), algo_name(algo), P, p_intra, (long long)n, dtype_name(dt),
             (long long)loop_bytes, plan.lay.S, (long long)plan.lay.L, plan.steps_per_loop,
             plan.sl.loops, (long long)plan.sl.chunk, (long long)plan.sl.tail,
             plan.launches.size());
}

void log_fused(const Prepared& c) {
    if (!log_enabled()) return;
    using Key = std::tuple<int, int, int, int, int64_t, int, int, bool>;
    static std::mutex mu;
    static std::set<Key> seen;
    {
        std::lock_guard<std::mutex> lock(mu);
        const Key k{(int)c.coll, (int)c.algo, c.P, c.p_intra, (int64_t)c.count, (int)c.dtype,
                    (int)c.op, c.host_buffers};
        if (seen.size() >= 4096 || !seen.insert(k).second) return;
    }
    log_line("fused %s %s P=%d ranks_per_server=%d n=%lld %s %s%s: segments=%d L=%lld launches=1",
             coll_name(c.coll), algo_name(c.algo), c.P, c.p_intra, (long long)c.count,
             dtype_name(c.dtype), op_name(c.op), c.host_buffers ? " host_buffers" : "", c.lay.S,
             (long long)c.lay.L);
}

}  // namespace hc

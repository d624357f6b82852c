// hc_internal.h -- types shared by the host scheduler (hc_sched.cpp), the
// C ABI (hc_api.cpp) and the kernels (hc_kernels.cu).  Not installed.
#pragma once

#include <cstddef>
#include <cstdint>
#include <memory>
#include <vector>

#include <cuda_runtime_api.h>

#include "../../include/hc.h"

namespace hc {

constexpr int kMaxRanks = HC_MAX_RANKS;
// Devices the per-device host caches (SM counts, device addresses of the
// library's __device__ variables) have room for; a higher ordinal is refused
// with HC_ERR_CUDA.
constexpr int kMaxDevices = 64;
constexpr int kVecBytes = 16;  // one vector = 16 bytes = 4 x 32-bit or 8 x bf16

// Buffer locations a step item can name, per rank.
enum Loc : uint8_t {
    LOC_ORIG = 0,   // the rank's input as handed in (send)
    LOC_WORK = 1,   // working / output buffer (recv, or scratch for out-of-place RS)
    LOC_FINAL = 2,  // ReduceScatter output segment (recv), global-indexed
    LOC_COUNT = 3
};

inline int elem_bytes(hc_dtype_t dt) { return dt == HC_BFLOAT16 ? 2 : 4; }

// ---------------------------------------------------------------------------
// Segment layout: S segments of stride L (a multiple of 16 bytes); segment k
// covers [min(kL, n), min((k+1)L, n)).
// ---------------------------------------------------------------------------
struct Layout {
    int S = 0;
    int64_t L = 0;
    int64_t n = 0;
    int A = 0;  // elements per 16-byte vector
    int64_t seg_lo(int k) const { int64_t v = (int64_t)k * L; return v < n ? v : n; }
    int64_t seg_hi(int k) const { int64_t v = (int64_t)(k + 1) * L; return v < n ? v : n; }
};

int num_segments(hc_algo_t algo, hc_coll_t coll, int P, int p_intra = 1);
Layout make_layout(hc_algo_t algo, hc_coll_t coll, int P, int64_t n, hc_dtype_t dt, int p_intra = 1);

struct Slicing {
    int64_t chunk = 0;  // elements per segment per loop
    int loops = 1;
    int64_t tail = 0;
};
Slicing make_slicing(hc_algo_t algo, int P, int p_intra, const Layout& lay, hc_dtype_t dt,
                     int64_t loop_bytes);

// ---------------------------------------------------------------------------
// Device step items.  An item computes, for every segment of its segment set
// and every element j of the launch's slice of that segment,
//     v = in[0][j] (+) in[1][j] (+) ... (+) in[cnt-1][j]      (left to right)
//     if acc >= 0:  v = acc[j] (+) v                           (received on the left)
//     out[o][j] = v  for every output o of both output sets
// A copy is an item with one input and no acc.  Rank sets are rotations:
// member i of (base, rot, mod, cnt) is rank base + (rot + i) % mod.  The
// second output set (out2_*, empty when out2_cnt is 0) holds the outputs of
// another copy of the same input block in the same step, merged into this
// item so that the block is read once (the Pipeline AllGather forwards a
// block to the next server and sends it to its own server's ranks).
// Segment set: seg_first + (i / seg_width) * seg_stride + (i % seg_width),
// i < seg_width * seg_reps.
// ---------------------------------------------------------------------------
struct DevItem {
    int16_t out_base, out_rot, out_mod, out_cnt;
    int16_t in_base, in_rot, in_mod, in_cnt;
    int16_t acc_rank;  // -1 = none
    uint8_t acc_loc, in_loc, out_loc;
    uint8_t early;     // 1: no launch of the call writes the inputs (out-of-place
                       // ranks' own inputs), so they may be loaded before the
                       // wait on the previous launch (see StepParams::early)
    int16_t seg_width, seg_reps;
    uint8_t once;      // 1: no other item of the launch reads this item's inputs or
                       // accumulator, so its loads may leave L2 first
    uint8_t keep;      // bit 0 / bit 1: a later launch of the call reads the block
                       // written to the first / second output set; the other
                       // outputs are final and their stores may leave L2 first
    int32_t seg_first, seg_stride;
    int32_t cta_begin;  // first CTA of this item in the launch grid
    int16_t out2_base, out2_rot, out2_mod, out2_cnt;
};
static_assert(sizeof(DevItem) == 48, "DevItem layout");

// Outputs of an item in both output sets.
inline int item_outputs(const DevItem& it) { return it.out_cnt + it.out2_cnt; }

// Kernel-parameter block of one step launch.  MAXI items at most.
template <int MAXI>
struct StepParams {
    uintptr_t base[LOC_COUNT][kMaxRanks];  // element 0 of each rank's global-indexed view
    int64_t L;        // segment stride (elements)
    int64_t n;        // elements per rank vector
    int64_t lo, hi;   // slice of every segment for this launch (relative to the segment start)
    int64_t vecs;     // vectors per segment slice: ceil((hi - lo) / A)
    int64_t tiles;    // TMA-staged step kernel: tiles of its tile size per segment slice
    unsigned long long wait_ns;  // TMA-staged step kernel: limit of the first mbarrier wait
    int* err;         // TMA-staged step kernel: device error flag (HC_ERR_TIMEOUT)
    int32_t hold;     // TMA-staged step kernel: wait-expiry test mode
    int32_t early;    // 1: not the call's first launch, so every kernel launched
                      // before this call has completed once this grid runs at all
                      // (each earlier launch of the call waited for its
                      // predecessor before letting its dependents start): items
                      // flagged `early` may load their inputs before the
                      // programmatic wait on the previous launch
    int32_t nitems;
    int32_t total_ctas;
    DevItem items[MAXI];
};

// One launch of a step-mode plan: items + the slice they act on.
struct PlanLaunch {
    int64_t lo = 0, hi = 0;  // slice relative to segment start
    std::vector<DevItem> items;
    int step = 0, loop = 0;
};

struct Plan {
    Layout lay;
    Slicing sl;
    int steps_per_loop = 0;
    std::vector<PlanLaunch> launches;
};

// Which buffers alias, per rank (step-mode planning).
struct Aliasing {
    bool orig_is_work[kMaxRanks];   // in place: send and working buffer coincide
    bool final_is_work[kMaxRanks];  // ReduceScatter in place: output segment is in the working buffer
};

// Build the step-mode plan (host only).  Returns false on bad arguments.
bool build_plan(hc_algo_t algo, hc_coll_t coll, int P, int p_intra, int root, int64_t n,
                hc_dtype_t dt, int64_t loop_bytes, const Aliasing& alias, Plan* out);

// Per-rank bytes sent over the whole schedule and steps per loop (host only).
bool schedule_traffic(hc_algo_t algo, hc_coll_t coll, int P, int p_intra, int root, int64_t n,
                      hc_dtype_t dt, int64_t loop_bytes, int* steps_per_loop,
                      unsigned long long* bytes_sent);

// Assign CTAs to the items of a launch; returns the grid size.
int assign_ctas(PlanLaunch& L, const Layout& lay, int threads, int max_ctas);

// ---------------------------------------------------------------------------
// Fused-mode launch description.
// ---------------------------------------------------------------------------
struct FusedArgs {
    hc_algo_t algo;
    hc_coll_t coll;
    hc_dtype_t dtype;
    hc_op_t op;
    int P;
    int p_intra;
    int64_t n;
    Layout lay;
    const void* const* send;  // host array of P device pointers (may be null for in-place AG)
    void* const* recv;
    bool ag_in_place[kMaxRanks];
    bool rs_in_place[kMaxRanks];
    int root;  // Broadcast root, -1 otherwise
    bool host_buffers;  // some buffers are page-locked host memory
};

// ---------------------------------------------------------------------------
// A validated collective call (hc_api.cpp): everything its launch needs, and
// the device byte ranges it reads and writes (for graph dependencies).
// ---------------------------------------------------------------------------
struct Interval {
    uintptr_t lo, hi;
};

struct Prepared {
    hc_coll_t coll = HC_COLL_ALLREDUCE;
    hc_algo_t algo = HC_ALGO_RING;
    hc_dtype_t dtype = HC_FLOAT32;
    hc_op_t op = HC_SUM;
    hc_mode_t mode = HC_MODE_FUSED;
    int P = 0;
    int p_intra = 1;
    int root = -1;  // Broadcast root
    int64_t loop_bytes = 0;
    size_t count = 0;
    bool empty = true;
    bool has_send = false;
    bool host_buffers = false;
    Layout lay;
    Aliasing al;
    bool rs_in_place[kMaxRanks] = {false};
    bool ag_in_place[kMaxRanks] = {false};
    uintptr_t send[kMaxRanks] = {0};
    uintptr_t recv[kMaxRanks] = {0};
    uintptr_t scratch = 0;
    std::shared_ptr<const Plan> plan;  // step mode (shared with the plan cache)
    std::vector<Interval> reads, writes;
};

// root: Broadcast root (-1 for the other collectives)
hc_status_t prepare(hc_coll_t coll, const void* const* send, void* const* recv, int P, size_t count,
                    hc_dtype_t dtype, hc_op_t op, hc_algo_t algo, const hc_opts_t* opts, int root,
                    Prepared* out);
hc_status_t execute(const Prepared& c, cudaStream_t stream);
// true when b must wait for a (a write of one overlaps a read or write of the other)
bool conflicts(const Prepared& a, const Prepared& b);

// ---------------------------------------------------------------------------
// Tracing (hc_trace.cpp): NVTX ranges in the "libhc" domain and HC_LOG lines.
// ---------------------------------------------------------------------------
uint32_t trace_category(hc_algo_t algo, hc_mode_t mode);
class TraceRange {  // pushes a range on construction, pops it on destruction
  public:
    TraceRange(hc_coll_t coll, uint32_t category, uint64_t payload);
    TraceRange(const char* msg, uint32_t category, uint64_t payload);
    ~TraceRange();
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};
bool log_enabled();  // HC_LOG is a nonzero integer (read once)
void log_plan(hc_algo_t algo, hc_coll_t coll, int P, int p_intra, int64_t n, hc_dtype_t dt,
              int64_t loop_bytes, const Plan& plan);
void log_fused(const Prepared& c);

// Kernel launchers (hc_kernels.cu).
cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream, int sm_count);
// Reads (and optionally clears) the device-side error flag of the TMA kernels.
cudaError_t read_device_error(bool clear, int* status);
// Switches the wait-expiry test mode of the TMA-staged kernels (hc_test_expire_waits).
void set_test_expire_waits(bool on);
// host_buffers: some buffers are page-locked host memory (plain loads and
// stores only, no bulk copies)
cudaError_t launch_step(const Plan& plan, int P, hc_dtype_t dt, hc_op_t op,
                        const uintptr_t (&base)[LOC_COUNT][kMaxRanks], cudaStream_t stream,
                        int sm_count, bool host_buffers);

}  // namespace hc

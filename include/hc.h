/*
 * hc.h -- C ABI of libhc: the data plane of HCCL-style AllReduce,
 * ReduceScatter and AllGather schedules (Ring, Recursive Halving-Doubling,
 * hierarchical Pipeline) for P virtual ranks whose buffers all live in the
 * memory of one GPU (sm_103a).
 *
 * Sources (page title, section):
 *  - "深入分析HCCL集合通信库中Ring AllReduce和Recursive Halving-Doubling…"
 *    (mhpn.cn, Ring vs RHD on Ascend): "AllReduce的数学抽象与问题定义"
 *    (definition Y[j] = sum_i X_i[j]), "Ring AllReduce带宽最优的环形流水线"
 *    (RingAllReduce(self, ring[], send_buf, recv_buf, elem_count, dtype, op,
 *    comm) and its reduce_op loop), "Recursive Halving-Doubling短消息场景的
 *    延迟优势", and "Ascend950的AIV/AICPU通信引擎与图模式" (HcclResult status
 *    convention of HcclGraphAddAllReduce).
 *  - HCCL topology / AllReduce / fault-recovery article (hwcomputing.csdn.net),
 *    "AllReduce算法实现" (Scatter-Reduce + AllGather, 128-byte chunking) and
 *    "梯度同步与计算重叠" (stream-ordered asynchronous collectives).
 *  - "HCCL RHD（Recursive Halving-Doubling）算法深度解析", "算法描述" and
 *    Table 1 (non-power-of-two fold, ReduceScatter keeping scatter order).
 *  - "HCCL Pipeline分级流水算法深度解析", "AllGather 算子的 Pipeline 时序编排",
 *    "Rank0 视角的传输任务编排" (LocalCopy only when input and output
 *    differ), "源码中的流水执行印证" (loops sized by a scratch limit, tail
 *    slice) and Table 1.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - P virtual ranks, 1 <= P <= HC_MAX_RANKS.  `send` and `recv` are host
 *    arrays of P device pointers (read during the call only; the library keeps
 *    no reference to them).  The caller owns every buffer and the scratch;
 *    the library allocates no device memory.
 *  - `count` is n, the number of elements of one rank's full vector, for all
 *    three collectives.  Segment k of a vector is [off_k, off_k + len_k) as
 *    returned by hc_segment_range(): L = ceil(n / S) rounded up to a multiple
 *    of 16 bytes, off_k = min(k L, n), len_k = min((k+1) L, n) - off_k, with
 *    S = P segments (S = 2^floor(log2 P) for the RHD AllReduce).  Trailing
 *    segments may be short or empty.
 *  - Every device pointer must be 16-byte aligned (HC_ERR_ALIGN otherwise).
 *    Buffers of different ranks must not overlap; a rank's send and recv are
 *    either disjoint or exactly "in place" as defined per collective.
 *  - Every call is asynchronous on `stream` (NULL = legacy default stream)
 *    and may be captured into a CUDA graph.  All validation happens before
 *    any launch: a non-HC_OK status means nothing was launched.  Faults of
 *    the kernels themselves surface at the next synchronisation.
 *  - count == 0 returns HC_OK and launches nothing.
 *  - Reduction semantics per element and per schedule step, acc (+) x:
 *      int32  sum/prod wrap modulo 2^32, max/min by signed compare;
 *      fp32   IEEE binary32 round-to-nearest-even, no FMA, no flush to zero;
 *      bf16   both operands widened to binary32, op applied, result rounded
 *             to bf16 (nearest even) after every step;
 *      max/min of fp32/bf16 follow IEEE 754 totalOrder (-0 < +0), so they are
 *             exact and independent of the schedule.
 *    Sum/prod of fp32/bf16 depend on association order; each (algo, mode)
 *    reproduces exactly the order its schedule implies:
 *      Ring      segment k: ((X_{k+1} (+) X_{k+2}) (+) ...) (+) X_k;
 *      RHD       folded pairs u_i = X_{2i} (+) X_{2i+1} (i < P - 2^floor(log2 P)),
 *                then a balanced pairwise tree over the 2^floor(log2 P)
 *                leaves in rank order (partner bit 0 first);
 *      Pipeline  segment (s,l): intra-server partials
 *                I_t = X_(t,l) (+) X_(t,l+1) (+) ... (rotated from l),
 *                then I_{s+1} (+) I_{s+2} (+) ... (+) I_s around the
 *                inter-server ring (rank = server * ranks_per_server + local).
 *  - Thread-safe: host threads may call every entry point concurrently, on
 *    the same or different streams.  The library's host-side caches (step
 *    plans, per-kernel attributes, SM counts) are guarded by locks.  Calls
 *    whose buffers overlap must still be ordered by the caller (one stream,
 *    or events), and a graph object must not be used from two threads at
 *    once.
 */
#ifndef HC_H
#define HC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HC_MAX_RANKS 64
#define HC_VERSION 1

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* hc_stream_t;

/* Status codes, after HcclResult / HCCL_SUCCESS. */
typedef enum {
    HC_OK = 0,
    HC_ERR_INVALID_ARG = 1,   /* null pointer, P out of range, overlap, bad enum value */
    HC_ERR_UNSUPPORTED = 2,   /* dtype x op or algo x option combination not provided */
    HC_ERR_ALIGN = 3,         /* a device pointer is not 16-byte aligned */
    HC_ERR_SCRATCH = 4,       /* step-mode scratch missing or too small */
    HC_ERR_CUDA = 5,          /* a CUDA launch or query failed */
    HC_ERR_TIMEOUT = 6        /* a bounded device-side wait gave up (see hc_device_status) */
} hc_status_t;

typedef enum { HC_INT32 = 0, HC_FLOAT32 = 1, HC_BFLOAT16 = 2 } hc_dtype_t;
typedef enum { HC_SUM = 0, HC_PROD = 1, HC_MAX = 2, HC_MIN = 3 } hc_op_t;
/*
 * HC_ALGO_HIER: the plain (non-pipelined) hierarchical AllReduce of the
 * Pipeline article's "与其它分级算法的关系" and the RHD article's
 * "耗时模型解读": an intra-server ReduceScatter (full mesh), an inter-server
 * RHD AllReduce among the ranks of equal local index, and an intra-server
 * AllGather (full mesh); ranks_per_server gives the server size.  AllReduce
 * only (the other collectives return HC_ERR_UNSUPPORTED).  Per element:
 * intra-server chains I_s = X_(s,l) (+) X_(s,l+1) (+) ... rotated from the
 * element's intra segment l, then the RHD tree over the servers (fold of
 * server pairs (2i, 2i+1), balanced pairwise tree).  Its layout has
 * ranks_per_server x 2^floor(log2 (P / ranks_per_server)) segments and is not
 * reported by hc_segment_range.
 */
typedef enum { HC_ALGO_RING = 0, HC_ALGO_RHD = 1, HC_ALGO_PIPELINE = 2, HC_ALGO_HIER = 3 } hc_algo_t;
typedef enum {
    HC_COLL_ALLREDUCE = 0,
    HC_COLL_REDUCE_SCATTER = 1,
    HC_COLL_ALLGATHER = 2,
    HC_COLL_BROADCAST = 3
} hc_coll_t;

/*
 * HC_MODE_FUSED: one kernel reads every rank's element once, reduces it in
 *   registers in the schedule's association order and writes every output
 *   (minimum traffic: AllReduce reads P n b and writes P n b bytes).
 * HC_MODE_STEP: one kernel launch per schedule step (and per loop), each a
 *   16-byte vectorised segment reduce / copy over all ranks, i.e. the steps
 *   run as the pages describe them, with the peers' buffers read directly.
 * Both modes give bit-identical results.
 */
typedef enum { HC_MODE_FUSED = 0, HC_MODE_STEP = 1 } hc_mode_t;

/*
 * Options; pass NULL for the defaults (fused, ranks_per_server 1, one loop,
 * no scratch, device buffers).  struct_size must be sizeof(hc_opts_t), or
 * offsetof(hc_opts_t, host_buffers) for callers built before that field
 * (host_buffers is then 0).
 *  ranks_per_server : Pipeline and hierarchical only: ranks per server
 *                     (p_intra); P must be a multiple of it;
 *                     rank = server * p_intra + local.
 *  max_loop_bytes   : step mode: byte limit per loop (the pages' scratch
 *                     limit maxTmpMemSize_); each segment is cut into slices
 *                     of c = align_down(max_loop_bytes / (P * slots * b),
 *                     128 / b) elements (slots = 1 Ring, ceil(P/2) RHD,
 *                     max(1, p_intra - 1) Pipeline and hierarchical) and the
 *                     schedule runs once
 *                     per slice; 0 = one loop.  Results do not depend on it.
 *  scratch          : step mode, out-of-place ReduceScatter only: device
 *                     memory of at least hc_scratch_bytes() bytes, 16-byte
 *                     aligned, holding the ranks' intermediate partial sums.
 *                     Its contents on entry are ignored and on exit undefined.
 *  host_buffers     : 0: send / recv are device memory (not checked).
 *                     1: each send / recv buffer may also be page-locked host
 *                     memory (cudaHostAlloc, cudaMallocHost or
 *                     cudaHostRegister) whose device address equals its host
 *                     address (unified addressing).  The kernels then read
 *                     and write that memory directly over the host link
 *                     (NVLink-C2C on Grace systems): no staging copies, and in
 *                     fused mode every input byte crosses the link once
 *                     towards the GPU and every output byte once back.  Each
 *                     non-empty buffer is checked with
 *                     cudaPointerGetAttributes: pageable (unregistered)
 *                     memory, or host memory mapped at another device
 *                     address, gives HC_ERR_INVALID_ARG and nothing is
 *                     launched.  Step mode is allowed but moves its working
 *                     traffic over the link as well.  The scratch stays
 *                     device memory.
 */
typedef struct {
    size_t struct_size;
    hc_mode_t mode;
    int ranks_per_server;
    size_t max_loop_bytes;
    void* scratch;
    size_t scratch_bytes;
    int host_buffers;
} hc_opts_t;

/*
 * AllReduce: recv[r][j] = (+)_i send[i][j] for every rank r and j < count.
 * ("AllReduce的数学抽象与问题定义"; Ring: "Ring AllReduce带宽最优的环形流水线";
 * RHD: RHD article "算法描述" / Table 1 Allreduce row; Pipeline: Pipeline
 * article Table 1 AllReduce row.)
 *  send[r] : device pointer, count elements of rank r's input.
 *  recv[r] : device pointer, count elements of rank r's output;
 *            recv[r] == send[r] means in place (send[r] is overwritten).
 */
hc_status_t hc_allreduce(const void* const* send, void* const* recv, int P, size_t count,
                         hc_dtype_t dtype, hc_op_t op, hc_algo_t algo,
                         const hc_opts_t* opts, hc_stream_t stream);

/*
 * ReduceScatter: recv[r][0 .. len_r) = segment r of (+)_i send[i], where
 * (off_r, len_r) = hc_segment_range(algo, HC_COLL_REDUCE_SCATTER, ...).
 * (Ring: reduce-scatter phase of "Ring AllReduce带宽最优的环形流水线"; RHD:
 * Table 1 ReduceScatter row, scatter order kept; Pipeline: Table 1
 * ReduceScatter row.)
 *  send[r] : count elements of rank r's input.
 *  recv[r] : len_r elements; recv[r] == send[r] + off_r means in place (then
 *            all of send[r] is used as working memory and overwritten).
 *  Step mode with any out-of-place rank needs opts->scratch.
 */
hc_status_t hc_reduce_scatter(const void* const* send, void* const* recv, int P, size_t count,
                              hc_dtype_t dtype, hc_op_t op, hc_algo_t algo,
                              const hc_opts_t* opts, hc_stream_t stream);

/*
 * Broadcast: recv[r][j] = root's vector[j] for every rank r and j < count
 * (RHD article, Table 1, Broadcast row: the root's parity decides whether the
 * even or the odd rank of each non-power-of-two part1 pair joins the
 * power-of-two block; the block spreads the data by distance halving and
 * each part1 member then sends it once to its pair partner; ceil(log2 P)
 * steps).  The segment layout is one segment, the whole vector.
 *  send    : device pointer to the root's count elements, or NULL when the
 *            data already sits in recv[root] (in place; also when send ==
 *            recv[root]).
 *  recv[r] : count elements of rank r's output.
 *  root    : 0 <= root < P.
 *  algo    : HC_ALGO_RHD (the pages describe no other broadcast);
 *            anything else returns HC_ERR_UNSUPPORTED.
 */
hc_status_t hc_broadcast(const void* send, void* const* recv, int P, size_t count,
                         hc_dtype_t dtype, int root, hc_algo_t algo, const hc_opts_t* opts,
                         hc_stream_t stream);

/*
 * ReduceScatter for callers that may not allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for callers such as a
 * plugin that a host framework hands only its input and output buffers
 * (the framework owns all device memory through its own pool), or a
 * latency-critical path that cannot afford cudaMalloc's implicit
 * synchronisation or its failure under memory pressure.
 *
 * It computes exactly what hc_reduce_scatter computes in step mode
 * (HC_MODE_STEP, same arguments and buffer conventions, bit-identical
 * results), but the working memory of out-of-place ranks is a fixed array of
 * HC_STATIC_SCRATCH_BYTES that the library places in the memory of every GPU
 * that loads it, held until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *  - Every argument is validated first, exactly as hc_reduce_scatter does,
 *    before the device is touched.  Work needing more than
 *    HC_STATIC_SCRATCH_BYTES (P * roundup(count * b, 256) bytes, see
 *    hc_scratch_bytes) is then rejected with HC_ERR_SCRATCH; nothing is
 *    launched.  A call whose ranks are all in place needs no scratch and
 *    never touches the array.
 *  - The first call on a device that needs the scratch, with that device
 *    current, looks up the array's device address (cudaGetSymbolAddress);
 *    make that first call before any stream capture.  Under lazy module
 *    loading (CUDA_MODULE_LOADING=LAZY, the runtime's default) the array is
 *    committed inside that lookup, so the first call can fail with
 *    HC_ERR_CUDA when the device cannot give it HC_STATIC_SCRATCH_BYTES at
 *    that moment; set CUDA_MODULE_LOADING=EAGER to commit it when the
 *    runtime initialises the device instead.  The address is looked up once
 *    per device ordinal: do not keep using the library across a
 *    cudaDeviceReset() of that device.
 *  - All calls share the one array and it keeps whatever the last call left
 *    there; nothing in it needs to start at zero, because every location is
 *    written before it is read within a call.  Calls that overlap on the GPU
 *    (different streams, or different host threads) race on the array:
 *    order them on one stream.
 */
#define HC_STATIC_SCRATCH_BYTES (32u << 20)
hc_status_t hc_reduce_scatter_static_scratch(const void* const* send, void* const* recv, int P,
                                             size_t count, hc_dtype_t dtype, hc_op_t op,
                                             hc_algo_t algo, int ranks_per_server,
                                             size_t max_loop_bytes, hc_stream_t stream);

/*
 * AllGather: recv[r][off_k .. off_k + len_k) = send[k][0 .. len_k) for every
 * rank r and segment k.  (Ring: all-gather phase; RHD: Table 1 AllGather row;
 * Pipeline: "AllGather 算子的 Pipeline 时序编排", LocalCopy of "Rank0 视角".)
 *  send    : NULL, or P pointers; send[k] holds len_k elements of segment k;
 *            send == NULL or send[k] == recv[k] + off_k means in place (the
 *            segment is already at its place in recv[k]).
 *  recv[r] : count elements.
 */
hc_status_t hc_allgather(const void* const* send, void* const* recv, int P, size_t count,
                         hc_dtype_t dtype, hc_algo_t algo,
                         const hc_opts_t* opts, hc_stream_t stream);

/*
 * Graph mode ("Ascend950的AIV/AICPU通信引擎与图模式" of the Ring vs RHD
 * article: HcclGraphAddAllReduce / HcclGraphBuild, whose build step analyses
 * the data dependencies between collectives, orders them and emits one task
 * list).  A graph is a list of collectives added once and replayed many
 * times with one launch:
 *  - hc_graph_add_* validate exactly like the eager entry points (same
 *    arguments and buffer conventions) and record the call; the device
 *    pointers and options are copied, the buffers must stay valid while the
 *    graph is used.  Nothing is launched.
 *  - Collective j depends on an earlier collective i when a device byte range
 *    written by one is read or written by the other; independent collectives
 *    may run concurrently.
 *  - hc_graph_build captures every collective's kernels (on a private stream)
 *    into one CUDA graph following those dependencies and instantiates it.
 *    Adding a collective after a build discards the built graph.
 *  - hc_graph_launch runs the built graph on `stream` (asynchronous); the
 *    results equal running the collectives eagerly in the order added.
 *  - hc_graph_info: collectives, dependency edges, kernel nodes (0 until built).
 * A graph is not thread-safe; destroy it with hc_graph_destroy.
 */
typedef struct hc_graph_s* hc_graph_t;
hc_status_t hc_graph_create(hc_graph_t* graph);
hc_status_t hc_graph_add_allreduce(hc_graph_t graph, const void* const* send, void* const* recv,
                                   int P, size_t count, hc_dtype_t dtype, hc_op_t op,
                                   hc_algo_t algo, const hc_opts_t* opts);
hc_status_t hc_graph_add_reduce_scatter(hc_graph_t graph, const void* const* send,
                                        void* const* recv, int P, size_t count, hc_dtype_t dtype,
                                        hc_op_t op, hc_algo_t algo, const hc_opts_t* opts);
hc_status_t hc_graph_add_allgather(hc_graph_t graph, const void* const* send, void* const* recv,
                                   int P, size_t count, hc_dtype_t dtype, hc_algo_t algo,
                                   const hc_opts_t* opts);
hc_status_t hc_graph_add_broadcast(hc_graph_t graph, const void* send, void* const* recv, int P,
                                   size_t count, hc_dtype_t dtype, int root, hc_algo_t algo,
                                   const hc_opts_t* opts);
hc_status_t hc_graph_build(hc_graph_t graph);
hc_status_t hc_graph_launch(hc_graph_t graph, hc_stream_t stream);
hc_status_t hc_graph_info(hc_graph_t graph, int* collectives, int* edges, int* kernels);
hc_status_t hc_graph_destroy(hc_graph_t graph);

/* Segment k's element range (see the layout rule above).  k < S, where
 * S = hc_num_segments(algo, coll, P). */
hc_status_t hc_segment_range(hc_algo_t algo, hc_coll_t coll, int P, size_t count,
                             hc_dtype_t dtype, int k, size_t* off, size_t* len);
int hc_num_segments(hc_algo_t algo, hc_coll_t coll, int P);

/* Scratch bytes a step-mode, out-of-place ReduceScatter needs. */
size_t hc_scratch_bytes(hc_algo_t algo, int P, size_t count, hc_dtype_t dtype);

/*
 * Schedule statistics (host only, no GPU needed; a Broadcast is counted
 * with root 0, every root giving the same counts).
 *  steps_per_loop : communication steps of one loop (Ring AllReduce 2(P-1),
 *                   RHD 2 ceil(log2 P), Pipeline 2 p_inter, ...)
 *  loops, chunk, tail : the loop slicer's result (elements per segment)
 *  launches_step  : kernels one step-mode call launches (in place)
 *  launches_fused : kernels one fused-mode call launches
 *  step_bytes     : bytes the step-mode kernels read + write (in place)
 *  fused_bytes    : bytes the fused kernel reads + writes (out of place)
 *  bytes_sent     : optional array of P: bytes each rank sends to other ranks
 *                   over the whole schedule (the pages' per-rank traffic)
 */
typedef struct {
    size_t struct_size;
    int steps_per_loop;
    int loops;
    size_t chunk;
    size_t tail;
    int launches_step;
    int launches_fused;
    unsigned long long step_bytes;
    unsigned long long fused_bytes;
} hc_stats_t;

hc_status_t hc_schedule_stats(hc_algo_t algo, hc_coll_t coll, int P, int ranks_per_server,
                              size_t count, hc_dtype_t dtype, size_t max_loop_bytes,
                              hc_stats_t* stats, unsigned long long* bytes_sent);

/*
 * Step-plan export for host-side checking (no GPU needed): the work each
 * step-mode launch performs, one record per (launch, item, segment).  With
 * cap == 0 or records == NULL only the number of records is returned in *n.
 * Locations: 0 = the rank's input (send), 1 = its working/output buffer
 * (recv, or the scratch for an out-of-place ReduceScatter), 2 = its
 * ReduceScatter output (recv).  Every record computes, for lo <= j < hi,
 *   out[o][j] = (acc (+)) in[0][j] (+) in[1][j] (+) ... for each o in outs.
 * `in_place` says which buffers alias (nonzero: every rank in place).
 * `root` is the Broadcast root (ignored by the other collectives).
 */
typedef struct {
    int32_t launch;
    int32_t seg;
    int64_t lo, hi;
    int32_t acc_rank;   /* -1: no left operand */
    int32_t acc_loc;
    int32_t in_loc;
    int32_t in_cnt;
    int32_t out_loc;
    int32_t out_cnt;
    int32_t in_ranks[HC_MAX_RANKS];
    int32_t out_ranks[HC_MAX_RANKS];
} hc_plan_record_t;

hc_status_t hc_step_plan(hc_algo_t algo, hc_coll_t coll, int P, int ranks_per_server,
                         size_t count, hc_dtype_t dtype, size_t max_loop_bytes, int in_place,
                         int root, hc_plan_record_t* records, size_t cap, size_t* n,
                         int* launches);

/*
 * Cost-model algorithm selection (the AllReduce article's cost model,
 * "AllReduce算法实现": T_Ring = 2(N-1)/N M/B + 2(N-1) L, choose the
 * cheapest; the alpha-beta-gamma tables of the RHD and Pipeline articles).
 * On one GB300 a schedule's cost is its kernel launches (alpha) and the
 * bytes its kernels move over the HBM bandwidth (beta; the reduction, gamma,
 * hides under the memory traffic).  Launches are queued asynchronously, so
 * the host's launch cost and the device time overlap:
 *   t = max(c_host + launches * alpha_host, t_device)
 *   step:  t_device = launches * (alpha_algo + a_rank * P) + step_bytes / (f_algo * B)
 *   fused: t_device = alpha_fused + r_algo * P + fused_bytes / (f_path * B)
 * with launches and bytes from hc_schedule_stats and, measured on GB300 for
 * a C caller: c_host = 0.55 us, alpha_host = 1.4 us per launch; the device
 * terms fitted to timed calls of every candidate (36 shapes): alpha_algo per
 * dependent launch 1.8 us (Ring), 2.0 us (RHD), 1.9 us (Pipeline), 2.6 us
 * (hierarchical), a_rank = 0.02 us; f_algo = 1.48 (Ring), 1.24 (RHD), 1.17
 * (Pipeline), 1.12 (hierarchical), above 1 where a step's outputs come back
 * from L2 as the next step's operands;
 * alpha_fused = 1.3 us, r_algo the per-rank cost of the schedule's
 * reduction in one block (Ring 0.064 us, RHD 0.057 below 16 ranks and 0.076
 * from 16, Pipeline 0.076, hierarchical 0.098, AllGather / Broadcast 0.042),
 * f_path = 1.03 (AllReduce / ReduceScatter up to 32 ranks, 0.99 above), 1.05
 * (AllGather / Broadcast below 16 ranks) or 1.09 (from 16, where each byte
 * read is written more often); B = 6800 GB/s, times 1.44 when the ranks'
 * vectors fit in L2 (P * count * element size <= 96 MiB: buffers that calls
 * on the same data keep resident).
 * Candidates: Ring and RHD; Pipeline and, for an AllReduce, the
 * hierarchical AllReduce when ranks_per_server > 1 divides P; Broadcast:
 * RHD only.  Between equal costs the lower device time wins, then the
 * earlier candidate (Ring, RHD, Pipeline, hierarchical).
 *  out_algo      : the cheapest schedule
 *  predicted_us  : its predicted time in microseconds (may be NULL)
 */
hc_status_t hc_select_algo(hc_coll_t coll, int P, int ranks_per_server, size_t count,
                           hc_dtype_t dtype, hc_mode_t mode, hc_algo_t* out_algo,
                           double* predicted_us);

/*
 * Device-side status of the kernels that wait on shared-memory barriers (the
 * TMA-staged kernels: fused AllReduce / ReduceScatter, and the step kernel's
 * launches of wide reduces and broadcasts).  Each such wait gives up after
 * about 2 s; the kernel then records HC_ERR_TIMEOUT here and returns instead
 * of hanging.
 * Returns HC_OK, HC_ERR_TIMEOUT, or HC_ERR_CUDA if the flag cannot be read.
 * Synchronises with the current device (it copies the flag to the host);
 * clear != 0 resets the flag.
 * A block whose wait gave up waits once more, also bounded, for the copies
 * into its own shared memory to land, and then exits without storing: the
 * outputs of the call that reported HC_ERR_TIMEOUT are undefined, and later
 * calls are unaffected.
 */
hc_status_t hc_device_status(int clear);

/*
 * Test hook for the path above (no counterpart on the pages).  enable = 1
 * switches every TMA-staged kernel launched from then on (any host
 * thread) into a mode in which the copies' shared-memory barrier waits for
 * one arrival more than the block makes before its first wait, and that
 * first wait gives up after 1 ms instead of 2 s.  Every copy still lands;
 * the first wait expires regardless, the block records HC_ERR_TIMEOUT, makes
 * the held arrival, waits (bounded) for its copies and exits without
 * storing.  Nothing hangs or faults.  enable = 0 restores normal operation.
 * Returns HC_ERR_INVALID_ARG for any other value.  Not for production use:
 * calls launched in this mode leave their outputs undefined.
 */
hc_status_t hc_test_expire_waits(int enable);

/* Name of the CUDA error (e.g. "cudaErrorInvalidValue") behind the last
 * HC_ERR_CUDA this host thread received; "cudaSuccess" if none. */
const char* hc_last_cuda_error(void);

const char* hc_status_string(hc_status_t status);
int hc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HC_H */

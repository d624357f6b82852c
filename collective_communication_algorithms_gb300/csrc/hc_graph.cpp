// hc_graph.cpp -- graph mode: a DAG of collectives built once and replayed
// with one launch ("Ascend950的AIV/AICPU通信引擎与图模式" of the Ring vs RHD
// article: HcclGraphAddAllReduce adds a collective to a graph,
// HcclGraphBuild analyses the data dependencies between them
// (GraphAnalyzeDeps), orders them (GraphScheduleOptimize) and emits the task
// list (GraphCodegen)).
//
// Here a node is a validated collective call (the same checks as the eager
// entry points).  Dependencies: node j waits for node i < j when one writes a
// device byte range the other reads or writes; independent nodes become
// parallel branches.  Build captures every node's kernel launches in one
// stream capture over private streams (one per lane of the DAG, joined by
// events) and instantiates the graph; launch replays it on the caller's
// stream with one call, so the per-launch host overhead of step mode and of
// chains of small collectives is paid once per build.
#include <algorithm>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "hc_internal.h"

using namespace hc;

struct hc_graph_s {
    std::vector<Prepared> nodes;
    std::vector<std::vector<int>> deps;  // deps[j]: nodes j waits for
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int kernels = 0;
};

namespace {

void release(hc_graph_s* g) {
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    g->exec = nullptr;
    g->graph = nullptr;
    g->kernels = 0;
}

hc_status_t add(hc_graph_t g, hc_coll_t coll, const void* const* send, void* const* recv, int P,
                size_t count, hc_dtype_t dtype, hc_op_t op, hc_algo_t algo, const hc_opts_t* opts,
                int root = -1) {
    if (!g) return HC_ERR_INVALID_ARG;
    Prepared c;
    const hc_status_t st = prepare(coll, send, recv, P, count, dtype, op, algo, opts, root, &c);
    if (st != HC_OK) return st;
    std::vector<int> d;
    for (int i = 0; i < (int)g->nodes.size(); i++)
        if (conflicts(g->nodes[i], c)) d.push_back(i);
    g->nodes.push_back(std::move(c));
    g->deps.push_back(std::move(d));
    release(g);  // a built graph no longer matches
    return HC_OK;
}

}  // namespace

extern "C" {

hc_status_t hc_graph_create(hc_graph_t* graph) {
    if (!graph) return HC_ERR_INVALID_ARG;
    *graph = new (std::nothrow) hc_graph_s();
    return *graph ? HC_OK : HC_ERR_INVALID_ARG;
}

hc_status_t hc_graph_add_allreduce(hc_graph_t g, const void* const* send, void* const* recv, int P,
                                   size_t count, hc_dtype_t dtype, hc_op_t op, hc_algo_t algo,
                                   const hc_opts_t* opts) {
    return add(g, HC_COLL_ALLREDUCE, send, recv, P, count, dtype, op, algo, opts);
}

hc_status_t hc_graph_add_reduce_scatter(hc_graph_t g, const void* const* send, void* const* recv,
                                        int P, size_t count, hc_dtype_t dtype, hc_op_t op,
                                        hc_algo_t algo, const hc_opts_t* opts) {
    return add(g, HC_COLL_REDUCE_SCATTER, send, recv, P, count, dtype, op, algo, opts);
}

hc_status_t hc_graph_add_allgather(hc_graph_t g, const void* const* send, void* const* recv, int P,
                                   size_t count, hc_dtype_t dtype, hc_algo_t algo,
                                   const hc_opts_t* opts) {
    return add(g, HC_COLL_ALLGATHER, send, recv, P, count, dtype, HC_SUM, algo, opts);
}

hc_status_t hc_graph_add_broadcast(hc_graph_t g, const void* send, void* const* recv, int P,
                                   size_t count, hc_dtype_t dtype, int root, hc_algo_t algo,
                                   const hc_opts_t* opts) {
    if (P < 1 || P > kMaxRanks) return HC_ERR_INVALID_ARG;
    const void* sendv[kMaxRanks] = {nullptr};
    if (root >= 0 && root < P) sendv[root] = send;
    return add(g, HC_COLL_BROADCAST, sendv, recv, P, count, dtype, HC_SUM, algo, opts, root);
}

hc_status_t hc_graph_build(hc_graph_t g) {
    if (!g) return HC_ERR_INVALID_ARG;
    release(g);
    const int N = (int)g->nodes.size();
    // Lanes: collective j continues the lane of its latest dependency when
    // no other collective has continued that one yet (it is then that lane's
    // last collective, so stream order adds no dependency the DAG lacks);
    // otherwise it opens a lane of its own.  Each lane is captured on its own
    // stream, so consecutive dependent collectives keep the programmatic
    // (PDL) edges between their launches, and independent ones become
    // parallel branches.
    std::vector<int> lane(N), tail;
    std::vector<char> continued(N, 0);
    for (int j = 0; j < N; j++) {
        int L = -1;
        if (!g->deps[j].empty()) {
            const int i = g->deps[j].back();
            if (!continued[i]) {
                continued[i] = 1;
                L = lane[i];
            }
        }
        if (L < 0) {
            L = (int)tail.size();
            tail.push_back(j);
        }
        lane[j] = L;
        tail[L] = j;
    }
    const int nl = std::max<int>(1, (int)tail.size());
    std::vector<cudaStream_t> st(nl, nullptr);
    std::vector<cudaEvent_t> done(N, nullptr);
    cudaEvent_t fork = nullptr;
    hc_status_t rc = HC_OK;
    auto ok = [&](cudaError_t e) {
        if (e != cudaSuccess && rc == HC_OK) rc = HC_ERR_CUDA;
        return rc == HC_OK;
    };
    for (int l = 0; l < nl && ok(cudaSuccess); l++) ok(cudaStreamCreateWithFlags(&st[l], cudaStreamNonBlocking));
    for (int j = 0; j < N && rc == HC_OK; j++) ok(cudaEventCreateWithFlags(&done[j], cudaEventDisableTiming));
    if (rc == HC_OK) ok(cudaEventCreateWithFlags(&fork, cudaEventDisableTiming));
    bool capturing = false;
    if (rc == HC_OK && ok(cudaStreamBeginCapture(st[0], cudaStreamCaptureModeThreadLocal))) {
        capturing = true;
        ok(cudaEventRecord(fork, st[0]));
        for (int l = 1; l < nl && rc == HC_OK; l++) ok(cudaStreamWaitEvent(st[l], fork, 0));
        for (int j = 0; j < N && rc == HC_OK; j++) {
            cudaStream_t s = st[lane[j]];
            for (int i : g->deps[j])
                if (lane[i] != lane[j] && !ok(cudaStreamWaitEvent(s, done[i], 0))) break;
            if (rc != HC_OK) break;
            const hc_status_t xs = execute(g->nodes[j], s);
            if (xs != HC_OK) {
                rc = xs;
                break;
            }
            ok(cudaEventRecord(done[j], s));
        }
        for (int l = 1; l < nl && rc == HC_OK; l++) ok(cudaStreamWaitEvent(st[0], done[tail[l]], 0));
    }
    if (capturing) {
        cudaGraph_t graph = nullptr;
        const cudaError_t ce = cudaStreamEndCapture(st[0], &graph);
        if (rc == HC_OK && (ce != cudaSuccess || !graph)) rc = HC_ERR_CUDA;
        if (rc == HC_OK) g->graph = graph;
        else if (graph) cudaGraphDestroy(graph);
    }
    if (rc == HC_OK) {
        size_t nn = 0;
        cudaGraphGetNodes(g->graph, nullptr, &nn);
        std::vector<cudaGraphNode_t> all(nn);
        if (nn) cudaGraphGetNodes(g->graph, all.data(), &nn);
        for (cudaGraphNode_t v : all) {
            cudaGraphNodeType t;
            if (cudaGraphNodeGetType(v, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) g->kernels++;
        }
        if (cudaGraphInstantiate(&g->exec, g->graph, 0) != cudaSuccess) rc = HC_ERR_CUDA;
    }
    if (fork) cudaEventDestroy(fork);
    for (cudaEvent_t e : done)
        if (e) cudaEventDestroy(e);
    for (cudaStream_t s : st)
        if (s) cudaStreamDestroy(s);
    if (rc != HC_OK) {
        cudaGetLastError();  // leave no pending error behind for the caller
        release(g);
    }
    return rc;
}

hc_status_t hc_graph_launch(hc_graph_t g, hc_stream_t stream) {
    if (!g) return HC_ERR_INVALID_ARG;
    if (!g->exec) return HC_ERR_INVALID_ARG;  // not built
    const hc::TraceRange range("hc_graph_launch", 0, (uint64_t)g->nodes.size());
    return cudaGraphLaunch(g->exec, (cudaStream_t)stream) == cudaSuccess ? HC_OK : HC_ERR_CUDA;
}

hc_status_t hc_graph_info(hc_graph_t g, int* nodes, int* edges, int* kernels) {
    if (!g) return HC_ERR_INVALID_ARG;
    int ne = 0;
    for (const auto& d : g->deps) ne += (int)d.size();
    if (nodes) *nodes = (int)g->nodes.size();
    if (edges) *edges = ne;
    if (kernels) *kernels = g->exec ? g->kernels : 0;
    return HC_OK;
}

hc_status_t hc_graph_destroy(hc_graph_t g) {
    if (!g) return HC_ERR_INVALID_ARG;
    release(g);
    delete g;
    return HC_OK;
}

}  // extern "C"

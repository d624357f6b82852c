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
// parallel branches.  Build captures each node's kernel launches into a
// child CUDA graph (stream capture on a private stream) and instantiates the
// whole DAG; launch replays it on the caller's stream with one call, so the
// per-launch host overhead of step mode and of chains of small collectives
// is paid once per build.
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
    cudaStream_t cs = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess) return HC_ERR_CUDA;
    e = cudaGraphCreate(&g->graph, 0);
    std::vector<cudaGraphNode_t> gn(g->nodes.size());
    hc_status_t st = e == cudaSuccess ? HC_OK : HC_ERR_CUDA;
    for (size_t j = 0; j < g->nodes.size() && st == HC_OK; j++) {
        cudaGraph_t child = nullptr;
        if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
            st = HC_ERR_CUDA;
            break;
        }
        const hc_status_t xs = execute(g->nodes[j], cs);
        const cudaError_t ce = cudaStreamEndCapture(cs, &child);
        if (xs != HC_OK || ce != cudaSuccess || !child) {
            if (child) cudaGraphDestroy(child);
            st = xs != HC_OK ? xs : HC_ERR_CUDA;
            break;
        }
        size_t nk = 0;
        cudaGraphGetNodes(child, nullptr, &nk);
        g->kernels += (int)nk;
        std::vector<cudaGraphNode_t> d;
        for (int i : g->deps[j]) d.push_back(gn[i]);
        e = cudaGraphAddChildGraphNode(&gn[j], g->graph, d.data(), d.size(), child);
        cudaGraphDestroy(child);
        if (e != cudaSuccess) st = HC_ERR_CUDA;
    }
    if (st == HC_OK && cudaGraphInstantiate(&g->exec, g->graph, 0) != cudaSuccess) st = HC_ERR_CUDA;
    cudaStreamDestroy(cs);
    if (st != HC_OK) release(g);
    return st;
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

// The fused train step captured once as a CUDA graph and replayed.
//
// Method: "Phase 2: Multi-Stream Graph Parallelism" runs the trainers' step
// as a captured CUDA graph; here the captured graph is one ofrl_train_step
// (relabel, V forward/backward, reduce + norms + Adam, with their
// programmatic dependent launches, cluster and cooperative attributes).  A
// replay costs one graph launch on the host instead of three or four kernel
// launches.  What changes from step to step is patched into the
// instantiated graph's kernel nodes before each replay: the relabel's step
// index, the V kernel's Q pointer, the auxiliary-source pointers, Adam's bias
// corrections and the fused kernel's grid-barrier target.  Each node's first
// arguments are the launch structs the kernels take (HerLaunch; VnetLaunch
// (+ the weight images, + the tensor maps of the layered path, whose second
// kernel reads no Q); ReduceLaunch, AdamLaunch, barrier, target; AdamLaunch),
// so the fields are patched in copies of the captured arguments.

#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "../../include/ofrl.h"

struct ofrl_step_graph {
    ofrl_ctx* ctx;
    ofrl_vnet* nets;          // caller's array: t advances here
    int32_t n_nets, n_aux;
    float beta1, beta2;
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    cudaGraphNode_t node[5];
    int n_nodes;              // kernels: relabel, V (1 or 2), reduce + Adam (1 or 2)
    // host I/O (ofrl_step_graph_create_io): Q copied in before the kernels,
    // loss and norms copied out after them (null nodes when not asked for)
    cudaGraphNode_t h2d_q, d2h_loss, d2h_norms;
    void* q_dev;
    const void* loss_dev;
    const void* norms_dev;
    size_t q_bytes, loss_bytes, norms_bytes;
    int red_node;             // index of the reduce node
    // the captured arguments of each node (copies patched before a replay)
    ofrl::HerLaunch her;
    ofrl::VnetLaunch vnet;
    const uint8_t* vnet_wimg;         // the tensor-core kernels' second argument
    ofrl::WideMaps* vnet_maps;        // the layered path's third argument (128-byte aligned copy)
    ofrl::ReduceLaunch red;
    ofrl::AdamLaunch red_adam;
    unsigned long long* bar;
    unsigned long long bar_target;
    ofrl::AdamLaunch adam;
    uint64_t barrier_arrivals;        // arrivals one replay adds (fused reduce + Adam)
};

using namespace ofrl;

namespace {

ofrl_status create_graph(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her, const ofrl_batch* batch,
                         const float* q, ofrl_vnet* nets, int32_t n_nets, const ofrl_opt* opt,
                         const float* const* aux_src, int32_t n_aux, float* v_out, float* pi_out,
                         int32_t* argmax_out, float* loss_out, float* norms_out, float* grad_out,
                         const float* q_host, float* loss_host, float* norms_host, ofrl_step_graph** out) {
    if (ctx == nullptr || out == nullptr || nets == nullptr || opt == nullptr) return OFRL_EINVAL;
    if (ctx->prof_events != nullptr) return OFRL_EINVAL;   // no profiling hooks inside a capture
    if ((q_host != nullptr && q == nullptr) || (loss_host != nullptr && loss_out == nullptr) ||
        (norms_host != nullptr && norms_out == nullptr) || her == nullptr)
        return OFRL_EINVAL;
    *out = nullptr;
    const size_t q_bytes = (size_t)her->batch * ctx->shape.num_actions * sizeof(float);
    const size_t loss_bytes = (size_t)n_nets * sizeof(float), norms_bytes = (size_t)n_nets * 5 * sizeof(float);
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return OFRL_ECUDA;
    std::vector<int32_t> t0(n_nets > 0 ? n_nets : 0);
    for (int k = 0; k < n_nets; ++k) t0[k] = nets[k].t;
    const uint64_t arrivals0 = ctx->barrier_arrivals;

    // capture one step (every argument check of ofrl_train_step applies)
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(st);
        return OFRL_ECUDA;
    }
    cudaError_t ecp = cudaSuccess;
    if (q_host != nullptr)
        ecp = cudaMemcpyAsync(const_cast<float*>(q), q_host, q_bytes, cudaMemcpyHostToDevice, st);
    ofrl_status s = ecp == cudaSuccess ? ofrl_train_step(ctx, replay, her, 0, batch, q, nets, n_nets, opt, aux_src,
                                                         n_aux, v_out, pi_out, argmax_out, loss_out, norms_out,
                                                         grad_out, st)
                                       : OFRL_ECUDA;
    if (s == OFRL_OK && loss_host != nullptr)
        ecp = cudaMemcpyAsync(loss_host, loss_out, loss_bytes, cudaMemcpyDeviceToHost, st);
    if (s == OFRL_OK && ecp == cudaSuccess && norms_host != nullptr)
        ecp = cudaMemcpyAsync(norms_host, norms_out, norms_bytes, cudaMemcpyDeviceToHost, st);
    if (s == OFRL_OK && ecp != cudaSuccess) s = OFRL_ECUDA;
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(st, &graph);
    cudaStreamDestroy(st);
    // the capture launched nothing: t and the barrier count are as before
    // (and the captured relabel has no kernel before it in the graph)
    for (int k = 0; k < n_nets; ++k) nets[k].t = t0[k];
    ctx->early_ok = 0;
    const uint64_t per_replay = ctx->barrier_arrivals - arrivals0;
    ctx->barrier_arrivals = arrivals0;
    if (s != OFRL_OK || ec != cudaSuccess || graph == nullptr) {
        if (graph) cudaGraphDestroy(graph);
        return s != OFRL_OK ? s : OFRL_ECUDA;
    }

    ofrl_step_graph* g = new (std::nothrow) ofrl_step_graph();
    if (g == nullptr) {
        cudaGraphDestroy(graph);
        return OFRL_ECUDA;
    }
    g->ctx = ctx;
    g->nets = nets;
    g->n_nets = n_nets;
    g->n_aux = n_aux;
    g->beta1 = opt->beta1;
    g->beta2 = opt->beta2;
    g->graph = graph;
    g->barrier_arrivals = per_replay;
    g->q_dev = const_cast<float*>(q);
    g->loss_dev = loss_out;
    g->norms_dev = norms_out;
    g->q_bytes = q_bytes;
    g->loss_bytes = loss_bytes;
    g->norms_bytes = norms_bytes;
    // the nodes in launch order (a captured stream is a chain): the Q copy,
    // the kernels, the loss and norms copies
    const int n_io = (q_host ? 1 : 0) + (loss_host ? 1 : 0) + (norms_host ? 1 : 0);
    size_t n = 0;
    cudaGraphGetNodes(graph, nullptr, &n);
    std::vector<cudaGraphNode_t> nodes(n);
    bool ok = (int)n >= 3 + n_io && (int)n <= 5 + n_io && cudaGraphGetNodes(graph, nodes.data(), &n) == cudaSuccess;
    // order by the chain: the node without dependencies first (the queries
    // take edge data: programmatic-launch edges carry it)
    std::vector<cudaGraphNode_t> chain;
    if (ok) {
        cudaGraphNode_t cur = nullptr;
        for (cudaGraphNode_t nd : nodes) {
            cudaGraphNode_t dep[8];
            cudaGraphEdgeData edge[8];
            size_t deps = 8;
            if (cudaGraphNodeGetDependencies(nd, dep, edge, &deps) != cudaSuccess) ok = false;
            else if (deps == 0) cur = nd;
        }
        while (ok && cur != nullptr && chain.size() < n) {
            chain.push_back(cur);
            cudaGraphNode_t next[8];
            cudaGraphEdgeData edge[8];
            size_t nd = 8;
            if (cudaGraphNodeGetDependentNodes(cur, next, edge, &nd) != cudaSuccess || nd > 1) break;
            cur = nd == 1 ? next[0] : nullptr;
        }
        ok = ok && chain.size() == n;
    }
    {
        size_t i = 0;
        if (ok && q_host != nullptr) g->h2d_q = chain[i++];
        const size_t kend = n - (loss_host ? 1 : 0) - (norms_host ? 1 : 0);
        int nk = 0;
        for (; ok && i < kend; ++i) {
            cudaGraphNodeType ty;
            ok = cudaGraphNodeGetType(chain[i], &ty) == cudaSuccess && ty == cudaGraphNodeTypeKernel;
            g->node[nk++] = chain[i];
        }
        if (ok && loss_host != nullptr) g->d2h_loss = chain[i++];
        if (ok && norms_host != nullptr) g->d2h_norms = chain[i++];
        for (cudaGraphNode_t io : {g->h2d_q, g->d2h_loss, g->d2h_norms}) {
            cudaGraphNodeType ty;
            if (ok && io != nullptr) ok = cudaGraphNodeGetType(io, &ty) == cudaSuccess && ty == cudaGraphNodeTypeMemcpy;
        }
        n = (size_t)nk;
    }
    g->n_nodes = (int)n;
    if (ok) {
        cudaKernelNodeParams p;
        ok = cudaGraphKernelNodeGetParams(g->node[0], &p) == cudaSuccess;
        if (ok) std::memcpy(&g->her, p.kernelParams[0], sizeof(HerLaunch));
        ok = ok && cudaGraphKernelNodeGetParams(g->node[1], &p) == cudaSuccess;
        if (ok) {
            std::memcpy(&g->vnet, p.kernelParams[0], sizeof(VnetLaunch));
            // the tensor-core kernels take the weight images as a second
            // argument, the layered path's first kernel its tensor maps as a third
            if (g->vnet.path == PATH_FUSED || g->vnet.path == PATH_LAYERED)
                std::memcpy(&g->vnet_wimg, p.kernelParams[1], sizeof(const uint8_t*));
            if (g->vnet.path == PATH_LAYERED) {
                g->vnet_maps = new (std::align_val_t(128), std::nothrow) WideMaps;
                if (g->vnet_maps == nullptr) ok = false;
                else std::memcpy(g->vnet_maps, p.kernelParams[2], sizeof(WideMaps));
            }
        }
        g->red_node = g->vnet.path == PATH_LAYERED ? 3 : 2;
        ok = ok && (int)n >= g->red_node + 1 && (int)n <= g->red_node + 2;
        ok = ok && cudaGraphKernelNodeGetParams(g->node[g->red_node], &p) == cudaSuccess;
        if (ok) {
            std::memcpy(&g->red, p.kernelParams[0], sizeof(ReduceLaunch));
            std::memcpy(&g->red_adam, p.kernelParams[1], sizeof(AdamLaunch));
            std::memcpy(&g->bar, p.kernelParams[2], sizeof(g->bar));
            std::memcpy(&g->bar_target, p.kernelParams[3], sizeof(g->bar_target));
        }
        if (ok && (int)n == g->red_node + 2) {
            ok = cudaGraphKernelNodeGetParams(g->node[g->red_node + 1], &p) == cudaSuccess;
            if (ok) std::memcpy(&g->adam, p.kernelParams[0], sizeof(AdamLaunch));
        }
    }
    ok = ok && cudaGraphInstantiate(&g->exec, graph, 0) == cudaSuccess;
    cudaGetLastError();   // no error of these queries stays behind for the caller
    if (!ok) {
        if (g->exec) cudaGraphExecDestroy(g->exec);
        cudaGraphDestroy(graph);
        if (g->vnet_maps) ::operator delete(g->vnet_maps, std::align_val_t(128));
        delete g;
        return OFRL_EUNSUPPORTED;
    }
    *out = g;
    return OFRL_OK;
}

cudaError_t set_args(ofrl_step_graph* g, int i, void** args) {
    cudaKernelNodeParams p;
    cudaError_t e = cudaGraphKernelNodeGetParams(g->node[i], &p);
    if (e != cudaSuccess) return e;
    p.kernelParams = args;
    p.extra = nullptr;
    return cudaGraphExecKernelNodeSetParams(g->exec, g->node[i], &p);
}

ofrl_status launch_graph(ofrl_step_graph* g, uint64_t step, const float* q, const float* const* aux_src,
                         const float* q_host, float* loss_host, float* norms_host, void* stream) {
    if (g == nullptr || step >= (1ull << 32)) return OFRL_EINVAL;
    if (g->n_aux > 0 && aux_src != nullptr)
        for (int i = 0; i < g->n_nets * g->n_aux; ++i)
            if (aux_src[i] == nullptr) return OFRL_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    g->ctx->early_ok = 0;
    // 1. relabel: the step index (and the Q pointer when the relabel stages Q
    // from host memory)
    g->her.step = step;
    if (q != nullptr && g->her.q_src != nullptr) g->her.q_src = q;
    void* a0[] = {&g->her};
    cudaError_t e = set_args(g, 0, a0);
    // 2. V: the Q pointer
    if (e == cudaSuccess && q != nullptr && g->her.q_src == nullptr && q != g->vnet.q) {
        g->vnet.q = q;
        void* a1[] = {&g->vnet, &g->vnet_wimg, g->vnet_maps};
        e = set_args(g, 1, a1);
    }
    // 3. reduce (+ Adam): sources, bias corrections, barrier target
    for (int k = 0; k < g->n_nets; ++k) {
        const int32_t t = g->nets[k].t + 1;
        float bc1, bc2;
        bias_corrections(g->beta1, g->beta2, t, &bc1, &bc2);
        g->red_adam.bc1[k] = g->adam.bc1[k] = bc1;
        g->red_adam.bc2[k] = g->adam.bc2[k] = bc2;
        if (aux_src != nullptr)
            for (int j = 0; j < g->n_aux; ++j) {
                const float* src = aux_src[k * g->n_aux + j];
                g->red.src[k][j + 1] = g->red_adam.src[k][j + 1] = g->adam.src[k][j + 1] = src;
            }
    }
    const unsigned long long base = g->ctx->barrier_arrivals;
    if (g->barrier_arrivals > 0) g->bar_target = base + g->barrier_arrivals;
    if (e == cudaSuccess) {
        void* a2[] = {&g->red, &g->red_adam, &g->bar, &g->bar_target};
        e = set_args(g, g->red_node, a2);
    }
    if (e == cudaSuccess && g->n_nodes == g->red_node + 2) {
        void* a3[] = {&g->adam};
        e = set_args(g, g->red_node + 1, a3);
    }
    // 4. host I/O: this step's host buffers
    if (e == cudaSuccess && g->h2d_q != nullptr && q_host != nullptr)
        e = cudaGraphExecMemcpyNodeSetParams1D(g->exec, g->h2d_q, g->q_dev, q_host, g->q_bytes,
                                               cudaMemcpyHostToDevice);
    if (e == cudaSuccess && g->d2h_loss != nullptr && loss_host != nullptr)
        e = cudaGraphExecMemcpyNodeSetParams1D(g->exec, g->d2h_loss, loss_host, g->loss_dev, g->loss_bytes,
                                               cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && g->d2h_norms != nullptr && norms_host != nullptr)
        e = cudaGraphExecMemcpyNodeSetParams1D(g->exec, g->d2h_norms, norms_host, g->norms_dev, g->norms_bytes,
                                               cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaGraphLaunch(g->exec, st);
    if (e != cudaSuccess) return OFRL_ECUDA;
    g->ctx->barrier_arrivals += g->barrier_arrivals;
    for (int k = 0; k < g->n_nets; ++k) g->nets[k].t += 1;
    return OFRL_OK;
}

}  // namespace

extern "C" ofrl_status ofrl_step_graph_create(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                                              const ofrl_batch* batch, const float* q, ofrl_vnet* nets,
                                              int32_t n_nets, const ofrl_opt* opt, const float* const* aux_src,
                                              int32_t n_aux, float* v_out, float* pi_out, int32_t* argmax_out,
                                              float* loss_out, float* norms_out, float* grad_out,
                                              ofrl_step_graph** out) {
    return create_graph(ctx, replay, her, batch, q, nets, n_nets, opt, aux_src, n_aux, v_out, pi_out, argmax_out,
                        loss_out, norms_out, grad_out, nullptr, nullptr, nullptr, out);
}

extern "C" ofrl_status ofrl_step_graph_create_io(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                                                 const ofrl_batch* batch, float* q, ofrl_vnet* nets, int32_t n_nets,
                                                 const ofrl_opt* opt, const float* const* aux_src, int32_t n_aux,
                                                 float* v_out, float* pi_out, int32_t* argmax_out, float* loss_out,
                                                 float* norms_out, float* grad_out, const float* q_host,
                                                 float* loss_host, float* norms_host, ofrl_step_graph** out) {
    return create_graph(ctx, replay, her, batch, q, nets, n_nets, opt, aux_src, n_aux, v_out, pi_out, argmax_out,
                        loss_out, norms_out, grad_out, q_host, loss_host, norms_host, out);
}

extern "C" ofrl_status ofrl_step_graph_launch(ofrl_step_graph* g, uint64_t step, const float* q,
                                              const float* const* aux_src, void* stream) {
    return launch_graph(g, step, q, aux_src, nullptr, nullptr, nullptr, stream);
}

extern "C" ofrl_status ofrl_step_graph_launch_io(ofrl_step_graph* g, uint64_t step, const float* q_host,
                                                 const float* const* aux_src, float* loss_host, float* norms_host,
                                                 void* stream) {
    return launch_graph(g, step, nullptr, aux_src, q_host, loss_host, norms_host, stream);
}

extern "C" ofrl_status ofrl_step_graph_destroy(ofrl_step_graph* g) {
    if (g == nullptr) return OFRL_OK;
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    if (g->vnet_maps) ::operator delete(g->vnet_maps, std::align_val_t(128));
    delete g;
    return OFRL_OK;
}

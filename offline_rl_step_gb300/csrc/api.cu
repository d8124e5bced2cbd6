// C ABI of the ofrl library: argument checks, the context, and the
// composition of the fused train step out of the device passes.
//
// Step order ("GPU IQL + HER Porting Plan", "Phase 3: Combined IQL + HER" and
// "IQL-augmented flow"; "Gradient Stability ...", "Proper design" pipeline):
//   her_relabel -> vnet_fwd_bwd (per network: V, loss, policy, per-tile
//   gradient partials) -> reduce_gram (primary gradient, Gram matrix of the
//   sources, budget coefficients, norms, loss) -> t += 1 -> adam.
// Nothing here allocates except ofrl_create; nothing synchronises the host
// except ofrl_poll_status and ofrl_destroy.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "common.cuh"
#include "tc_image.cuh"

using namespace ofrl;

namespace {

constexpr uint64_t kBarrierWaitNs = 1000000000ull;   // a CTA gives up at the grid barrier after 1 s

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool shape_ok(const ofrl_vshape* s) {
    if (s == nullptr) return false;
    if (s->state_dim < 1 || s->state_dim > kMaxStateDim) return false;
    if (s->num_actions < 1 || s->num_actions > kMaxActions) return false;
    if (s->prec != OFRL_PREC_FP32 && s->prec != OFRL_PREC_BF16) return false;
    return true;
}

bool hidden_supported(int h) { return h == 64 || h == 128 || h == 256; }

struct Layout {
    int64_t off_partials, off_tile_loss, off_g0, off_gram, off_scalars, off_counter, off_status, off_img, off_ximg,
        off_act[3], off_tvec, off_qbuf, off_barrier, total;
    int32_t max_tiles;
    int32_t tiles128;        // 128-row tiles of the tensor-core paths
    bool layered;            // the layered tensor-core path has its buffers
    int64_t P;
};

// The tensor-core paths: weight and state-tile images for every H (H = 64
// padded to 128 units); the layered path's activation images for H = 128 and
// 256 with S < 64.
bool tc_images(const ofrl_vshape* s) { return s->hidden == 64 || s->hidden == 128 || s->hidden == 256; }
int image_width(int hidden) { return hidden < 128 ? 128 : hidden; }
bool layered_possible(const ofrl_vshape* s) {
    return (s->hidden == 128 || s->hidden == 256) && s->state_dim < tc::KX;
}
int planes_of(const ofrl_vshape* s) { return s->prec == OFRL_PREC_BF16 ? 1 : 3; }

Layout layout_of(const ofrl_vshape* s, int32_t max_batch, int32_t max_nets) {
    Layout L;
    L.P = n_params_of(s->state_dim, s->hidden);
    const int tm = vnet_tile_rows(s->hidden);
    L.max_tiles = (int32_t)((max_batch + tm - 1) / tm);
    int64_t o = 0;
    auto take = [&](int64_t bytes) { const int64_t at = o; o = round_up(o + bytes, 256); return at; };
    L.off_partials = take((int64_t)max_nets * L.max_tiles * part_stride_of(L.P) * 4);
    L.off_tile_loss = take((int64_t)max_nets * L.max_tiles * 4);
    L.off_g0 = take((int64_t)max_nets * L.P * 4);
    L.off_gram = take((int64_t)max_nets * kMaxGramBlocks * kGramStride * 4);
    L.off_scalars = take((int64_t)max_nets * kScalars * 4);
    L.off_counter = take((int64_t)max_nets * 4);
    L.off_status = take((int64_t)OFRL_STAT_WORDS * 4);
    L.tiles128 = (int32_t)((max_batch + tc::TM - 1) / tc::TM);
    L.layered = layered_possible(s);
    L.off_img = take(tc_images(s) ? (int64_t)max_nets * tc::weight_image_bytes(image_width(s->hidden)) : 0);
    L.off_ximg = take(tc_images(s) ? (int64_t)L.tiles128 * tc::x_tile_bytes() : 0);
    for (int k = 0; k < 3; ++k)
        L.off_act[k] = take(L.layered ? (int64_t)max_nets * L.tiles128 * vnet_wide_act_bytes(s->hidden, planes_of(s))
                                      : 0);
    L.off_tvec = take(L.layered ? (int64_t)max_nets * L.tiles128 * vnet_wide_tvec_stride(s->hidden) * 4 : 0);
    L.off_qbuf = take((int64_t)max_batch * kMaxActions * 4);
    L.off_barrier = take(8);
    L.total = o;
    return L;
}

inline ofrl_status cuda_status(cudaError_t e) { return e == cudaSuccess ? OFRL_OK : OFRL_ECUDA; }

// Page-locked host memory (cudaHostAlloc / cudaHostRegister).
bool host_memory(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

ofrl_status check_ctx(const ofrl_ctx* ctx) {
    if (ctx == nullptr) return OFRL_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return OFRL_ECUDA;
    return dev == ctx->device ? OFRL_OK : OFRL_EINVAL;
}

ofrl_status check_replay(const ofrl_replay* r, const ofrl_her_cfg* h) {
    if (r == nullptr || h == nullptr) return OFRL_EINVAL;
    if (!r->states || !r->next_states || !r->actions || !r->rewards || !r->dones) return OFRL_EINVAL;
    if (r->capacity < 1 || r->capacity > INT32_MAX) return OFRL_EINVAL;
    if (r->state_dim < 1 || r->state_stride < r->state_dim || (r->state_stride & 3)) return OFRL_EINVAL;
    if (r->goal_dim < 1 || r->goal_dim > r->state_dim) return OFRL_EINVAL;
    if (r->state_dim > kMaxStateDim) return OFRL_EUNSUPPORTED;
    if (!aligned16(r->states) || !aligned16(r->next_states)) return OFRL_EINVAL;
    if (h->batch < 0 || h->her_count < 0 || h->her_count > h->batch) return OFRL_EINVAL;
    if (h->strategy != OFRL_HER_FINAL && h->strategy != OFRL_HER_FUTURE && h->strategy != OFRL_HER_RANDOM &&
        h->strategy != OFRL_HER_EPISODE)
        return OFRL_EINVAL;
    if (h->her_count > 0 && h->strategy != OFRL_HER_RANDOM) {
        if (r->episode_ends == nullptr || r->num_episodes < 1) return OFRL_EINVAL;
    }
    if (std::isnan(h->goal_threshold)) return OFRL_EINVAL;
    return OFRL_OK;
}

ofrl_status check_batch(const ofrl_batch* b, int state_dim) {
    if (b == nullptr) return OFRL_EINVAL;
    if (!b->states || !b->next_states || !b->actions || !b->rewards || !b->dones || !b->src_idx || !b->donor_idx)
        return OFRL_EINVAL;
    if (b->stride < ((state_dim + 3) & ~3) || (b->stride & 3)) return OFRL_EINVAL;
    if (!aligned16(b->states) || !aligned16(b->next_states)) return OFRL_EINVAL;
    return OFRL_OK;
}

ofrl_status check_opt(const ofrl_opt* o) {
    if (o == nullptr) return OFRL_EINVAL;
    if (!(o->max_grad_norm > 0.0f)) return OFRL_EINVAL;   // also rejects NaN
    if (!(o->beta1 >= 0.0f && o->beta1 < 1.0f) || !(o->beta2 >= 0.0f && o->beta2 < 1.0f)) return OFRL_EINVAL;
    if (!std::isfinite(o->lr) || !std::isfinite(o->eps) || !std::isfinite(o->weight_decay)) return OFRL_EINVAL;
    if (!(o->weight_clamp_max_abs >= 0.0f)) return OFRL_EINVAL;          // also rejects NaN
    if (o->sanitize_sources != 0 && o->sanitize_sources != 1) return OFRL_EINVAL;
    return OFRL_OK;
}

HerLaunch her_args(ofrl_ctx* ctx, const ofrl_replay* r, const ofrl_her_cfg* h, uint64_t step,
                   const ofrl_batch* out) {
    HerLaunch a;
    std::memset(&a, 0, sizeof(a));
    a.states = r->states;
    a.next_states = r->next_states;
    a.actions = r->actions;
    a.rewards = r->rewards;
    a.dones = r->dones;
    a.episode_ends = r->episode_ends;
    a.capacity = (int32_t)r->capacity;
    a.num_episodes = r->num_episodes;
    a.state_dim = r->state_dim;
    a.in_stride = r->state_stride;
    a.goal_dim = r->goal_dim;
    a.batch = h->batch;
    a.first_her = h->batch - h->her_count;
    a.strategy = h->strategy;
    a.threshold = h->goal_threshold;
    a.seed = h->seed;
    a.step = step;
    a.out_states = out->states;
    a.out_next_states = out->next_states;
    a.out_actions = out->actions;
    a.out_rewards = out->rewards;
    a.out_dones = out->dones;
    a.out_src = out->src_idx;
    a.out_donor = out->donor_idx;
    a.out_stride = out->stride;
    a.copy_cols = (r->state_dim + 3) & ~3;
    int rounds = 0;
    for (int64_t len = r->num_episodes; len > 16; len = (len + 15) / 16) ++rounds;
    a.search_rounds = rounds;
    a.status = ctx->ws.status;
    return a;
}

// Record the boundary event `which` of the current profiled step, if any.
inline void prof_mark(ofrl_ctx* ctx, int which, cudaStream_t st) {
    if (ctx->prof_events != nullptr && ctx->prof_count < ctx->prof_max)
        cudaEventRecord(ctx->prof_events[ctx->prof_count * (OFRL_PHASES + 1) + which], st);
}

void prof_release(ofrl_ctx* ctx) {
    if (ctx->prof_events == nullptr) return;
    for (int i = 0; i < ctx->prof_max * (OFRL_PHASES + 1); ++i)
        if (ctx->prof_events[i] != nullptr) cudaEventDestroy(ctx->prof_events[i]);
    delete[] ctx->prof_events;
    ctx->prof_events = nullptr;
    ctx->prof_max = ctx->prof_count = 0;
}

// The V forward/backward implementation a launch takes: the one the context
// asks for where it applies, else (PATH_AUTO) the fused tensor-core kernel
// for hidden 128, the layered one for hidden 256, the CUDA-core kernel
// otherwise.  Fills the layered path's fields of v.
int32_t choose_path(const ofrl_ctx* ctx, VnetLaunch& v) {
    if (ctx->maps != nullptr) {
        for (int k = 0; k < 3; ++k) v.act[k] = ctx->ws.act[k];
        v.tvec = ctx->ws.tvec;
        v.tvec_stride = ctx->tvec_stride;
        v.act_tiles = ctx->act_tiles;
        v.maps = ctx->maps;
        v.n_ranges = vnet_wide_ranges(v, ctx->num_sms);
        if (v.n_ranges > ctx->max_tiles) v.n_ranges = ctx->max_tiles;
    }
    const bool fused = vnet_tc_supported(v), layered = vnet_wide_supported(v);
    switch (ctx->vnet_path) {
        case PATH_SIMT: return PATH_SIMT;
        case PATH_FUSED: return fused ? PATH_FUSED : PATH_SIMT;
        case PATH_LAYERED: return layered ? PATH_LAYERED : PATH_SIMT;
        default: return fused ? PATH_FUSED : layered ? PATH_LAYERED : PATH_SIMT;
    }
}

// Rows per tile (entries of tile_loss) of the chosen path.
int path_tile_rows(const VnetLaunch& v) { return v.path == PATH_SIMT ? vnet_tile_rows(v.hidden) : tc::TM; }

// V forward/backward by v.path; all write the same gradient partials.
// `packed`: the weight images (and v.ximg, if set) were already written.
cudaError_t launch_vnet(ofrl_ctx* ctx, const VnetLaunch& v, bool packed, cudaStream_t st) {
    if (v.path == PATH_FUSED) {
        if (!packed) {
            const cudaError_t e = launch_vnet_tc_pack(v, ctx->ws.img, st);
            if (e != cudaSuccess) return e;
        }
        return launch_vnet_tc(v, ctx->ws.img, st);
    }
    if (v.path == PATH_LAYERED) {
        VnetLaunch w = v;
        if (!packed) {
            const cudaError_t e = launch_vnet_wide_pack(v, ctx->ws.img, ctx->ws.ximg, st);
            if (e != cudaSuccess) return e;
            w.ximg = ctx->ws.ximg;
        }
        return launch_vnet_wide(w, ctx->ws.img, st);
    }
    return launch_vnet_fwd_bwd(v, st);
}

// Gradient partials per network that launch_vnet leaves for n_tiles tiles:
// one per tile from the CUDA-core kernel, one per CTA from the fused
// tensor-core kernel, one per K-range from the layered one.
int vnet_parts(const VnetLaunch& v, int n_tiles) {
    if (v.path == PATH_FUSED) return vnet_tc_ctas(n_tiles, v.n_nets);
    if (v.path == PATH_LAYERED) return v.n_ranges;
    return n_tiles;
}

// Kernels a V forward/backward launch takes.
int vnet_kernels(const VnetLaunch& v) { return v.path == PATH_LAYERED ? 2 : 1; }

}  // namespace

void ofrl::bias_corrections(float beta1, float beta2, int32_t t, float* bc1, float* bc2) {
    *bc1 = (float)(1.0 - std::pow((double)beta1, (double)t));
    *bc2 = (float)(1.0 - std::pow((double)beta2, (double)t));
}

extern "C" {

int64_t ofrl_workspace_bytes(const ofrl_vshape* shape, int32_t max_batch, int32_t max_nets) {
    if (!shape_ok(shape) || !hidden_supported(shape->hidden) || max_batch < 1 || max_nets < 1 ||
        max_nets > kMaxNets)
        return -1;
    return layout_of(shape, max_batch, max_nets).total;
}

ofrl_status ofrl_create(const ofrl_vshape* shape, int32_t max_batch, int32_t max_nets, ofrl_ctx** out) {
    if (out == nullptr) return OFRL_EINVAL;
    *out = nullptr;
    if (!shape_ok(shape) || max_batch < 1 || max_nets < 1 || max_nets > kMaxNets) return OFRL_EINVAL;
    if (!hidden_supported(shape->hidden)) return OFRL_EUNSUPPORTED;
    ofrl_ctx* ctx = new (std::nothrow) ofrl_ctx;
    if (ctx == nullptr) return OFRL_ECUDA;
    std::memset(ctx, 0, sizeof(*ctx));
    if (cudaGetDevice(&ctx->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
        delete ctx;
        return OFRL_ECUDA;
    }
    const Layout L = layout_of(shape, max_batch, max_nets);
    ctx->shape = *shape;
    ctx->max_batch = max_batch;
    ctx->max_nets = max_nets;
    ctx->max_tiles = L.max_tiles;
    ctx->max_gram_blocks = kMaxGramBlocks;
    ctx->n_params = L.P;
    ctx->bytes = L.total;
    if (cudaMalloc(&ctx->base, (size_t)L.total) != cudaSuccess) {
        cudaGetLastError();
        delete ctx;
        return OFRL_ECUDA;
    }
    char* b = static_cast<char*>(ctx->base);
    ctx->ws.partials = reinterpret_cast<float*>(b + L.off_partials);
    ctx->ws.tile_loss = reinterpret_cast<float*>(b + L.off_tile_loss);
    ctx->ws.g0 = reinterpret_cast<float*>(b + L.off_g0);
    ctx->ws.gram_part = reinterpret_cast<float*>(b + L.off_gram);
    ctx->ws.scalars = reinterpret_cast<float*>(b + L.off_scalars);
    ctx->ws.counter = reinterpret_cast<unsigned int*>(b + L.off_counter);
    ctx->ws.status = reinterpret_cast<int32_t*>(b + L.off_status);
    ctx->ws.img = reinterpret_cast<uint8_t*>(b + L.off_img);
    ctx->ws.ximg = reinterpret_cast<uint8_t*>(b + L.off_ximg);
    for (int k = 0; k < 3; ++k) ctx->ws.act[k] = L.layered ? reinterpret_cast<uint8_t*>(b + L.off_act[k]) : nullptr;
    ctx->ws.tvec = L.layered ? reinterpret_cast<float*>(b + L.off_tvec) : nullptr;
    ctx->ws.qbuf = reinterpret_cast<float*>(b + L.off_qbuf);
    ctx->ws.barrier = reinterpret_cast<unsigned long long*>(b + L.off_barrier);
    ctx->barrier_arrivals = 0;
    ctx->barrier_wait_ns = kBarrierWaitNs;
    ctx->barrier_unreachable = 0;
    ctx->vnet_path = PATH_AUTO;
    ctx->early_ok = 0;
    ctx->early_stream = nullptr;
    ctx->act_tiles = L.tiles128;
    ctx->tvec_stride = L.layered ? vnet_wide_tvec_stride(shape->hidden) : 0;
    ctx->maps = nullptr;
    if (cudaMemset(ctx->base, 0, (size_t)L.total) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(ctx->base);
        delete ctx;
        return OFRL_ECUDA;
    }
    // tensor maps over the layered path's buffers; without them (no
    // tensor-map support in the driver) that path is unavailable
    if (L.layered) {
        WideMaps* m = new (std::align_val_t(128), std::nothrow) WideMaps;
        if (m != nullptr && vnet_wide_maps(m, shape->hidden, planes_of(shape), max_nets, L.tiles128, ctx->ws.act,
                                           ctx->ws.ximg, L.tiles128, ctx->ws.img) == cudaSuccess)
            ctx->maps = m;
        else if (m != nullptr)
            ::operator delete(m, std::align_val_t(128));
        cudaGetLastError();
    }
    *out = ctx;
    return OFRL_OK;
}

ofrl_status ofrl_destroy(ofrl_ctx* ctx) {
    if (ctx == nullptr) return OFRL_OK;
    const cudaError_t e1 = cudaDeviceSynchronize();
    prof_release(ctx);
    const cudaError_t e2 = cudaFree(ctx->base);
    if (ctx->maps != nullptr) ::operator delete(ctx->maps, std::align_val_t(128));
    delete ctx;
    return (e1 == cudaSuccess && e2 == cudaSuccess) ? OFRL_OK : OFRL_ECUDA;
}

ofrl_status ofrl_poll_status(ofrl_ctx* ctx, void* stream, int32_t* words_out) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    if (words_out == nullptr) return OFRL_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(words_out, ctx->ws.status, OFRL_STAT_WORDS * sizeof(int32_t),
                                    cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ctx->ws.status, 0, OFRL_STAT_WORDS * sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e);
}

const char* ofrl_status_string(ofrl_status s) {
    switch (s) {
        case OFRL_OK: return "OFRL_OK";
        case OFRL_EINVAL: return "OFRL_EINVAL: invalid argument";
        case OFRL_EUNSUPPORTED: return "OFRL_EUNSUPPORTED: unsupported configuration";
        case OFRL_ECUDA: return "OFRL_ECUDA: CUDA error";
        case OFRL_ETIMEOUT: return "OFRL_ETIMEOUT: bounded device wait gave up";
        default: return "unknown ofrl status";
    }
}

ofrl_status ofrl_her_relabel(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                             uint64_t step, const ofrl_batch* out, void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s == OFRL_OK) s = check_replay(replay, her);
    if (s == OFRL_OK) s = check_batch(out, replay->state_dim);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    if (step >= (1ull << 32)) return OFRL_EINVAL;
    if ((int64_t)her->batch >= (1ll << 31)) return OFRL_EINVAL;
    const HerLaunch a = her_args(ctx, replay, her, step, out);
    return cuda_status(launch_her_relabel(a, static_cast<cudaStream_t>(stream)));
}

ofrl_status ofrl_her_relabel_sources(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                                     uint64_t step, const int32_t* src_idx, const float* is_weights,
                                     const ofrl_batch* out, float* is_weights_out, void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s == OFRL_OK) s = check_replay(replay, her);
    if (s == OFRL_OK) s = check_batch(out, replay->state_dim);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    if (src_idx == nullptr || step >= (1ull << 32)) return OFRL_EINVAL;
    HerLaunch a = her_args(ctx, replay, her, step, out);
    a.src_in = src_idx;
    a.isw_in = is_weights;
    a.isw_out = is_weights_out;
    return cuda_status(launch_her_relabel(a, static_cast<cudaStream_t>(stream)));
}

ofrl_status ofrl_episode_ends_append(ofrl_ctx* ctx, const float* dones, int64_t first_index, int32_t n,
                                     int32_t* episode_ends, int32_t* num_episodes, int32_t max_episodes,
                                     void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    if (n < 0 || first_index < 0 || first_index + (int64_t)n > INT32_MAX || max_episodes < 0) return OFRL_EINVAL;
    if (n > 0 && (!dones || !episode_ends || !num_episodes)) return OFRL_EINVAL;
    return cuda_status(launch_episode_ends_append(dones, first_index, n, episode_ends, num_episodes, max_episodes,
                                                  ctx->ws.status, static_cast<cudaStream_t>(stream)));
}

namespace {

ofrl_status value_forward(ofrl_ctx* ctx, const float* params, const float* states, int32_t state_stride,
                          int32_t batch, const float* rewards, const float* dones, float gamma, float* v_out,
                          float* target_out, void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    const ofrl_vshape& sh = ctx->shape;
    if (!params || !states || (!v_out && !target_out)) return OFRL_EINVAL;
    if (batch < 1 || batch > ctx->max_batch || state_stride < sh.state_dim) return OFRL_EINVAL;
    VnetLaunch v;
    std::memset(&v, 0, sizeof(v));
    v.params[0] = params;
    v.n_nets = 1;
    v.state_dim = sh.state_dim;
    v.hidden = sh.hidden;
    v.num_actions = sh.num_actions;
    v.prec = sh.prec;
    v.states = states;
    v.stride = state_stride;
    v.batch = batch;
    v.v_out = v_out;
    v.rewards = rewards;
    v.dones = dones;
    v.gamma = gamma;
    v.target_out = target_out;
    v.status = ctx->ws.status;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the tensor cores where the context's step takes the fused kernel (and
    // the states meet its alignment), else the CUDA cores
    if (choose_path(ctx, v) == PATH_FUSED && ctx->ws.img != nullptr)
        return cuda_status(launch_vnet_tc_forward(v, ctx->ws.img, st));
    return cuda_status(launch_vnet_forward(v, st));
}

}  // namespace

ofrl_status ofrl_forward_values(ofrl_ctx* ctx, const float* params, const float* states, int32_t state_stride,
                                int32_t batch, float* v_out, void* stream) {
    if (v_out == nullptr) return OFRL_EINVAL;
    return value_forward(ctx, params, states, state_stride, batch, nullptr, nullptr, 0.0f, v_out, nullptr, stream);
}

ofrl_status ofrl_iql_target(ofrl_ctx* ctx, const float* params, const float* next_states, int32_t state_stride,
                            const float* rewards, const float* dones, int32_t batch, float gamma, float* v_next_out,
                            float* target_out, void* stream) {
    if (!rewards || !dones || !target_out) return OFRL_EINVAL;
    if (!(gamma >= 0.0f && gamma <= 1.0f)) return OFRL_EINVAL;
    return value_forward(ctx, params, next_states, state_stride, batch, rewards, dones, gamma, v_next_out,
                         target_out, stream);
}

ofrl_status ofrl_iql_value_fwd_bwd(ofrl_ctx* ctx, const float* params, const float* states,
                                   int32_t state_stride, int32_t batch, const float* q_taken, float tau,
                                   float* v_out, float* loss_out, float* grad_out, void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    const ofrl_vshape& sh = ctx->shape;
    if (!params || !states || !q_taken || !v_out || !loss_out || !grad_out) return OFRL_EINVAL;
    if (batch < 1 || batch > ctx->max_batch || state_stride < sh.state_dim) return OFRL_EINVAL;
    if (!(tau >= 0.0f && tau <= 1.0f)) return OFRL_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    VnetLaunch v;
    std::memset(&v, 0, sizeof(v));
    v.params[0] = params;
    v.tau[0] = tau;
    v.n_nets = 1;
    v.state_dim = sh.state_dim;
    v.hidden = sh.hidden;
    v.num_actions = sh.num_actions;
    v.prec = sh.prec;
    v.states = states;
    v.stride = state_stride;
    v.batch = batch;
    v.q_taken = q_taken;
    v.v_out = v_out;
    v.partials = ctx->ws.partials;
    v.tile_loss = ctx->ws.tile_loss;
    v.part_stride = part_stride_of(ctx->n_params);
    v.net_partial_stride = (int64_t)ctx->max_tiles * v.part_stride;
    v.net_tile_stride = ctx->max_tiles;
    v.status = ctx->ws.status;
    v.path = choose_path(ctx, v);
    const int tm = path_tile_rows(v);
    const int n_tiles = (batch + tm - 1) / tm;
    cudaError_t e = launch_vnet(ctx, v, false, st);
    if (e != cudaSuccess) return OFRL_ECUDA;

    ReduceLaunch r;
    std::memset(&r, 0, sizeof(r));
    r.n_nets = 1;
    r.P = ctx->n_params;
    r.n_tiles = n_tiles;
    r.n_parts = vnet_parts(v, n_tiles);
    r.partials = ctx->ws.partials;
    r.part_stride = v.part_stride;
    r.net_partial_stride = v.net_partial_stride;
    r.tile_loss = ctx->ws.tile_loss;
    r.net_tile_stride = ctx->max_tiles;
    r.inv_batch = 1.0f / (float)batch;
    r.g0_out[0] = grad_out;
    r.n_src = 0;
    r.max_grad_norm = INFINITY;
    r.gram_part = ctx->ws.gram_part;
    r.scalars = ctx->ws.scalars;
    r.counter = ctx->ws.counter;
    r.loss_out = loss_out;
    return cuda_status(launch_reduce_gram(r, st));
}

ofrl_status ofrl_expectile_loss(ofrl_ctx* ctx, const float* q_taken, const float* v, int32_t batch,
                                float tau, float* loss_out, float* dv_out, void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    if (!q_taken || !v || !loss_out || batch < 1) return OFRL_EINVAL;
    if (!(tau >= 0.0f && tau <= 1.0f)) return OFRL_EINVAL;
    return cuda_status(launch_expectile(q_taken, v, batch, tau, loss_out, dv_out,
                                        static_cast<cudaStream_t>(stream)));
}

ofrl_status ofrl_adv_weighted_policy(ofrl_ctx* ctx, const float* q, const float* v, int32_t batch,
                                     int32_t num_actions, float beta, float* pi_out, int32_t* argmax_out,
                                     void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    if (!q || !v || !pi_out || batch < 1 || num_actions < 1 || num_actions > kMaxActions) return OFRL_EINVAL;
    if (std::isnan(beta)) return OFRL_EINVAL;
    return cuda_status(launch_policy(q, v, batch, num_actions, beta, pi_out, argmax_out, 0, 1,
                                     static_cast<cudaStream_t>(stream)));
}

ofrl_status ofrl_budgeted_clip_saxpy(ofrl_ctx* ctx, const float* const* src, const float* budget_frac,
                                     const float* alpha, int32_t n_src, int64_t n, float max_grad_norm,
                                     float* grad_out, float* norms_out, void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    if (!src || !budget_frac || !alpha || !grad_out || n_src < 1 || n_src > kMaxSrc || n < 1) return OFRL_EINVAL;
    if (!(max_grad_norm > 0.0f)) return OFRL_EINVAL;
    for (int k = 0; k < n_src; ++k) {
        if (src[k] == nullptr || src[k] == grad_out) return OFRL_EINVAL;
        if (std::isnan(budget_frac[k]) || budget_frac[k] < 0.0f || std::isnan(alpha[k])) return OFRL_EINVAL;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ReduceLaunch r;
    std::memset(&r, 0, sizeof(r));
    r.n_nets = 1;
    r.P = n;
    r.inv_batch = 0.0f;
    for (int k = 0; k < n_src; ++k) {
        r.src[0][k] = src[k];
        r.budget[k] = budget_frac[k];
        r.alpha[k] = alpha[k];
    }
    r.n_src = n_src;
    r.max_grad_norm = max_grad_norm;
    r.gram_part = ctx->ws.gram_part;
    r.scalars = ctx->ws.scalars;
    r.counter = ctx->ws.counter;
    cudaError_t e = launch_reduce_gram(r, st);
    if (e != cudaSuccess) return OFRL_ECUDA;
    CombineLaunch c;
    std::memset(&c, 0, sizeof(c));
    c.n = n;
    for (int k = 0; k < n_src; ++k) c.src[k] = src[k];
    c.n_src = n_src;
    c.scalars = ctx->ws.scalars;
    c.out = grad_out;
    c.norms_out = norms_out;
    return cuda_status(launch_combine(c, st));
}

ofrl_status ofrl_target_ema(const float* params, float* target, int64_t n, float polyak, void* stream) {
    if (!params || !target || n < 1 || !(polyak >= 0.0f && polyak <= 1.0f)) return OFRL_EINVAL;
    return cuda_status(launch_target_ema(params, target, n, polyak, static_cast<cudaStream_t>(stream)));
}

ofrl_status ofrl_adam_step(ofrl_ctx* ctx, float* p, const float* g, float* m, float* v, int64_t n, int32_t t,
                           const ofrl_opt* opt, const float* grad_norm, void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s == OFRL_OK) s = check_opt(opt);
    if (s != OFRL_OK) return s;
    ctx->early_ok = 0;
    if (!p || !g || !m || !v || n < 1 || t < 1) return OFRL_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    AdamLaunch a;
    std::memset(&a, 0, sizeof(a));
    a.n_nets = 1;
    a.n = n;
    a.p[0] = p;
    a.m[0] = m;
    a.v[0] = v;
    a.src[0][0] = g;
    a.n_src = 1;
    a.lr[0] = opt->lr;
    bias_corrections(opt->beta1, opt->beta2, t, &a.bc1[0], &a.bc2[0]);
    a.beta1 = opt->beta1;
    a.beta2 = opt->beta2;
    a.eps = opt->eps;
    a.weight_decay = opt->weight_decay;
    a.max_grad_norm = opt->max_grad_norm;
    a.status = ctx->ws.status;
    a.clamp = opt->weight_clamp_max_abs;
    if (grad_norm == nullptr) {
        ReduceLaunch r;
        std::memset(&r, 0, sizeof(r));
        r.n_nets = 1;
        r.P = n;
        r.src[0][0] = g;
        r.n_src = 1;
        r.budget[0] = INFINITY;
        r.alpha[0] = 1.0f;
        r.max_grad_norm = 1.0f;
        r.gram_part = ctx->ws.gram_part;
        r.scalars = ctx->ws.scalars;
        r.counter = ctx->ws.counter;
        cudaError_t e = launch_reduce_gram(r, st);
        if (e != cudaSuccess) return OFRL_ECUDA;
        a.scalars = ctx->ws.scalars;
    } else {
        a.grad_norm = grad_norm;
    }
    return cuda_status(launch_adam(a, st));
}

int32_t ofrl_train_step_kernels(const ofrl_ctx* ctx, const ofrl_batch* batch, int32_t rows, int32_t n_nets) {
    if (ctx == nullptr || batch == nullptr || batch->states == nullptr) return 0;
    if (rows < 1 || rows > ctx->max_batch || n_nets < 1 || n_nets > ctx->max_nets) return 0;
    VnetLaunch v;
    std::memset(&v, 0, sizeof(v));
    v.n_nets = n_nets;
    v.state_dim = ctx->shape.state_dim;
    v.hidden = ctx->shape.hidden;
    v.prec = ctx->shape.prec;
    v.states = batch->states;
    v.stride = batch->stride;
    v.batch = rows;
    v.path = choose_path(ctx, v);
    const int tm = path_tile_rows(v);
    ReduceLaunch r;
    std::memset(&r, 0, sizeof(r));
    r.n_nets = n_nets;
    r.P = ctx->n_params;
    r.n_tiles = (rows + tm - 1) / tm;
    r.n_parts = vnet_parts(v, r.n_tiles);
    r.partials = ctx->ws.partials;
    return 1 + vnet_kernels(v) + (reduce_adam_fusable(r) ? 1 : 2);
}

ofrl_status ofrl_select_vnet_path(ofrl_ctx* ctx, int32_t path) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    const ofrl_vshape& sh = ctx->shape;
    switch (path) {
        case OFRL_VNET_AUTO:
        case OFRL_VNET_CUDA_CORES: break;
        case OFRL_VNET_TC_FUSED:
            if (sh.hidden > 128 || sh.state_dim > tc::KX) return OFRL_EUNSUPPORTED;
            break;
        case OFRL_VNET_TC_LAYERED:
            if (ctx->maps == nullptr) return OFRL_EUNSUPPORTED;
            break;
        default: return OFRL_EINVAL;
    }
    ctx->vnet_path = path;
    return OFRL_OK;
}

int32_t ofrl_vnet_path(const ofrl_ctx* ctx, int32_t n_nets) {
    if (ctx == nullptr || n_nets < 1 || n_nets > ctx->max_nets) return -1;
    // a train step's batch: 16-byte aligned rows (what ofrl_train_step requires)
    VnetLaunch v;
    std::memset(&v, 0, sizeof(v));
    v.n_nets = n_nets;
    v.state_dim = ctx->shape.state_dim;
    v.hidden = ctx->shape.hidden;
    v.prec = ctx->shape.prec;
    v.stride = (ctx->shape.state_dim + 3) & ~3;
    v.batch = ctx->max_batch;
    return choose_path(ctx, v);
}

ofrl_status ofrl_train_step(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her, uint64_t step,
                            const ofrl_batch* batch, const float* q, ofrl_vnet* nets, int32_t n_nets,
                            const ofrl_opt* opt, const float* const* aux_src, int32_t n_aux, float* v_out,
                            float* pi_out, int32_t* argmax_out, float* loss_out, float* norms_out,
                            float* grad_out, void* stream) {
    ofrl_status s = check_ctx(ctx);
    if (s == OFRL_OK) s = check_replay(replay, her);
    if (s == OFRL_OK) s = check_batch(batch, replay->state_dim);
    if (s == OFRL_OK) s = check_opt(opt);
    if (s != OFRL_OK) return s;
    const ofrl_vshape& sh = ctx->shape;
    if (replay->state_dim != sh.state_dim || q == nullptr || nets == nullptr) return OFRL_EINVAL;
    if (her->batch < 1 || her->batch > ctx->max_batch || step >= (1ull << 32)) return OFRL_EINVAL;
    if (n_nets < 1 || n_nets > ctx->max_nets || n_aux < 0 || n_aux > kMaxSrc - 1) return OFRL_EINVAL;
    if (n_aux > 0 && aux_src == nullptr) return OFRL_EINVAL;
    for (int k = 0; k < n_nets; ++k) {
        if (!nets[k].params || !nets[k].m || !nets[k].v || nets[k].t < 0) return OFRL_EINVAL;
        if (!(nets[k].tau >= 0.0f && nets[k].tau <= 1.0f)) return OFRL_EINVAL;
        if (nets[k].target != nullptr && !(nets[k].polyak >= 0.0f && nets[k].polyak <= 1.0f)) return OFRL_EINVAL;
        for (int j = 0; j < n_aux; ++j)
            if (aux_src[k * n_aux + j] == nullptr) return OFRL_EINVAL;
    }
    for (int j = 0; j <= n_aux; ++j)
        if (std::isnan(opt->budget[j]) || opt->budget[j] < 0.0f || std::isnan(opt->alpha[j])) return OFRL_EINVAL;
    if (pi_out != nullptr && std::isnan(opt->beta)) return OFRL_EINVAL;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t P = ctx->n_params;
    const int B = her->batch;

    // 2's arguments first: whether the tensor-core kernel runs decides what
    // the relabel launch also produces
    VnetLaunch v;
    std::memset(&v, 0, sizeof(v));
    for (int k = 0; k < n_nets; ++k) {
        v.params[k] = nets[k].params;
        v.tau[k] = nets[k].tau;
    }
    v.n_nets = n_nets;
    v.state_dim = sh.state_dim;
    v.hidden = sh.hidden;
    v.num_actions = sh.num_actions;
    v.prec = sh.prec;
    v.states = batch->states;
    v.stride = batch->stride;
    v.batch = B;
    v.q = q;
    v.actions = batch->actions;
    v.beta = opt->beta;
    v.v_out = v_out;
    v.pi_out = pi_out;
    v.argmax_out = pi_out != nullptr ? argmax_out : nullptr;
    v.partials = ctx->ws.partials;
    v.tile_loss = ctx->ws.tile_loss;
    v.part_stride = part_stride_of(P);
    v.net_partial_stride = (int64_t)ctx->max_tiles * v.part_stride;
    v.net_tile_stride = ctx->max_tiles;
    v.status = ctx->ws.status;
    v.path = choose_path(ctx, v);
    const bool tc_path = v.path == PATH_FUSED || v.path == PATH_LAYERED;

    // 1. HER relabel (+ state-tile images and packed weights for the tensor-core kernel)
    prof_mark(ctx, 0, st);
    HerLaunch ha = her_args(ctx, replay, her, step, batch);
    ha.early = ctx->early_ok && ctx->early_stream == stream ? 1 : 0;
    ctx->early_ok = 0;
    if (tc_path) {
        ha.ximg = ctx->ws.ximg;
        ha.img_planes = sh.prec == OFRL_PREC_BF16 ? 1 : 3;
        ha.img_rows = (B + tc::TM - 1) / tc::TM * tc::TM;
        ha.wimg = ctx->ws.img;
        ha.pack_hidden = sh.hidden;
        ha.pack_width = v.path == PATH_FUSED ? tc::HH : sh.hidden;
        ha.pack_nets = n_nets;
        for (int k = 0; k < n_nets; ++k) ha.pack_params[k] = nets[k].params;
        v.ximg = ctx->ws.ximg;
    }
    // Q in page-locked host memory: the relabel's row blocks, which run beside
    // the previous step's optimizer kernel, copy it into the workspace, and the
    // V kernel reads it there instead of across the host link
    if (host_memory(q)) {
        ha.q_src = q;
        ha.q_dst = ctx->ws.qbuf;
        ha.q_cols = sh.num_actions;
        v.q = ctx->ws.qbuf;
    }
    cudaError_t e = launch_her_relabel(ha, st);
    if (e != cudaSuccess) return OFRL_ECUDA;
    prof_mark(ctx, 1, st);

    // 2. V forward / loss / policy / backward partials, all networks in one grid
    e = launch_vnet(ctx, v, true, st);
    if (e != cudaSuccess) return OFRL_ECUDA;
    prof_mark(ctx, 2, st);

    // 3. primary gradient, Gram matrix, budget coefficients, norms, loss
    const int tm = path_tile_rows(v);
    ReduceLaunch r;
    std::memset(&r, 0, sizeof(r));
    r.n_nets = n_nets;
    r.P = P;
    r.n_tiles = (B + tm - 1) / tm;
    r.n_parts = vnet_parts(v, r.n_tiles);
    r.partials = ctx->ws.partials;
    r.part_stride = v.part_stride;
    r.net_partial_stride = v.net_partial_stride;
    r.tile_loss = ctx->ws.tile_loss;
    r.net_tile_stride = ctx->max_tiles;
    r.inv_batch = 1.0f / (float)B;
    for (int k = 0; k < n_nets; ++k) {
        r.g0_out[k] = grad_out != nullptr ? grad_out + (int64_t)k * P : ctx->ws.g0 + (int64_t)k * P;
        r.src[k][0] = r.g0_out[k];
        for (int j = 0; j < n_aux; ++j) r.src[k][j + 1] = aux_src[k * n_aux + j];
    }
    r.n_src = 1 + n_aux;
    for (int j = 0; j <= n_aux; ++j) {
        r.budget[j] = opt->budget[j];
        r.alpha[j] = opt->alpha[j];
    }
    r.max_grad_norm = opt->max_grad_norm;
    r.gram_part = ctx->ws.gram_part;
    r.scalars = ctx->ws.scalars;
    r.counter = ctx->ws.counter;
    r.norms_out = norms_out;
    r.loss_out = loss_out;
    r.sanitize = opt->sanitize_sources;
    r.status = ctx->ws.status;

    // 4. t += 1, then Adam with the safety clip
    AdamLaunch a;
    std::memset(&a, 0, sizeof(a));
    a.n_nets = n_nets;
    a.n = P;
    for (int k = 0; k < n_nets; ++k) {
        nets[k].t += 1;
        a.p[k] = nets[k].params;
        a.m[k] = nets[k].m;
        a.v[k] = nets[k].v;
        for (int j = 0; j <= n_aux; ++j) a.src[k][j] = r.src[k][j];
        a.lr[k] = opt->lr;
        bias_corrections(opt->beta1, opt->beta2, nets[k].t, &a.bc1[k], &a.bc2[k]);
        a.target[k] = nets[k].target;
        a.polyak[k] = nets[k].polyak;
    }
    a.sanitize = opt->sanitize_sources;
    a.clamp = opt->weight_clamp_max_abs;
    a.n_src = 1 + n_aux;
    a.scalars = ctx->ws.scalars;
    a.beta1 = opt->beta1;
    a.beta2 = opt->beta2;
    a.eps = opt->eps;
    a.weight_decay = opt->weight_decay;
    a.max_grad_norm = opt->max_grad_norm;
    a.status = ctx->ws.status;
    a.wait_ns = ctx->barrier_wait_ns;
    // 3 + 4 in one cooperative launch when its grid fits on the device
    // (a grid barrier between the reduce and Adam), else two launches
    if (reduce_adam_fusable(r)) {
        e = launch_reduce_adam(r, a, ctx->ws.barrier, ctx->barrier_arrivals + (ctx->barrier_unreachable ? 1u : 0u),
                               st);
        if (e != cudaSuccess) return OFRL_ECUDA;
        ctx->barrier_arrivals += (uint64_t)reduce_adam_blocks(r);
        prof_mark(ctx, 3, st);
    } else {
        e = launch_reduce_gram(r, st);
        if (e != cudaSuccess) return OFRL_ECUDA;
        prof_mark(ctx, 3, st);
        e = launch_adam(a, st);
        if (e != cudaSuccess) return OFRL_ECUDA;
    }
    prof_mark(ctx, 4, st);
    if (ctx->prof_events != nullptr && ctx->prof_count < ctx->prof_max) ctx->prof_count++;
    // the step ends with the optimizer kernel, which lets dependents launch
    // only after its own wait: the next step's relabel may start early
    ctx->early_ok = 1;
    ctx->early_stream = stream;
    return OFRL_OK;
}

ofrl_status ofrl_profile_begin(ofrl_ctx* ctx, int32_t max_steps) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    if (max_steps < 1) return OFRL_EINVAL;
    prof_release(ctx);
    const int n = max_steps * (OFRL_PHASES + 1);
    ctx->prof_events = new (std::nothrow) cudaEvent_t[n];
    if (ctx->prof_events == nullptr) return OFRL_ECUDA;
    for (int i = 0; i < n; ++i) ctx->prof_events[i] = nullptr;
    ctx->prof_max = max_steps;
    ctx->prof_count = 0;
    for (int i = 0; i < n; ++i) {
        if (cudaEventCreate(&ctx->prof_events[i]) != cudaSuccess) {
            prof_release(ctx);
            return OFRL_ECUDA;
        }
    }
    return OFRL_OK;
}

ofrl_status ofrl_profile_end(ofrl_ctx* ctx, float* phase_ms_out, int32_t* steps_out) {
    ofrl_status s = check_ctx(ctx);
    if (s != OFRL_OK) return s;
    if (phase_ms_out == nullptr || steps_out == nullptr) return OFRL_EINVAL;
    for (int p = 0; p < OFRL_PHASES; ++p) phase_ms_out[p] = 0.0f;
    *steps_out = ctx->prof_count;
    cudaError_t e = cudaSuccess;
    for (int k = 0; k < ctx->prof_count && e == cudaSuccess; ++k) {
        cudaEvent_t* ev = ctx->prof_events + k * (OFRL_PHASES + 1);
        e = cudaEventSynchronize(ev[OFRL_PHASES]);
        for (int p = 0; p < OFRL_PHASES && e == cudaSuccess; ++p) {
            float ms = 0.0f;
            e = cudaEventElapsedTime(&ms, ev[p], ev[p + 1]);
            phase_ms_out[p] += ms;
        }
    }
    prof_release(ctx);
    return cuda_status(e);
}

}  // extern "C"

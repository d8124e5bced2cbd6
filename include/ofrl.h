/*
 * ofrl.h -- C ABI of the GB300 (sm_103a) fused offline-RL train step:
 * HER batch relabel followed by an IQL value-network update with budgeted
 * per-source gradient clipping and Adam.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Pointers named in a comment as "device" are CUDA device pointers
 *    (or managed memory) on the current device; the caller owns every buffer.
 *    ofrl_train_step's q, loss_out and norms_out may also point into
 *    page-locked host memory (cudaHostAlloc / cudaHostRegister): the
 *    relabel launch then copies Q over the host link (NVLink-C2C on
 *    Grace-Blackwell) into the workspace while the previous step's
 *    optimizer kernel still runs, and the optimizer writes the loss and
 *    norms in place, instead of copies on the stream.
 *    The context owns only its workspace (gradient partials, reduction
 *    scratch, the status word), sized once at ofrl_create.  No call after
 *    ofrl_create allocates.
 *  - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL =
 *    the legacy default stream) and never synchronises the host, except
 *    ofrl_poll_status.
 *  - Shape, pointer-alignment and unsupported-configuration errors are
 *    detected on the host before anything is launched and return
 *    OFRL_EINVAL / OFRL_EUNSUPPORTED with nothing written.  A failed launch
 *    returns OFRL_ECUDA.  Anomalies only visible on the device (non-finite
 *    gradient elements skipped by Adam, out-of-range actions or indices) are
 *    counted in the context's status word, read by ofrl_poll_status.
 *  - Floating-point buffers are fp32, row-major.  Index buffers are int32.
 *  - Results are deterministic: no floating-point atomics; every reduction
 *    runs in a fixed order, so two identical calls give identical bits.
 *  - One context must not be used by two calls that overlap on the GPU
 *    (its workspace is shared by every call); use one context per stream.
 *
 * Notation: B batch, S state_dim, g goal_dim, H hidden, A num_actions,
 * P = H*S + H + H*H + H + H + 1 (V parameter count).  The flat V parameter
 * and gradient layout is W1[H,S], b1[H], W2[H,H], b2[H], W3[1,H], b3[1]
 * ("GPU IQL + HER Porting Plan", "CUDA Kernel: iql_value_kernel.cu",
 * parameter layout: w_v1, b_v1, w_v2, b_v2, w_vout, b_vout); every linear
 * layer computes y = x W^T + b.
 */
#ifndef OFRL_H
#define OFRL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ofrl_status;
enum {
    OFRL_OK = 0,
    OFRL_EINVAL = -1,        /* bad argument: null pointer, size, stride, alignment */
    OFRL_EUNSUPPORTED = -2,  /* valid request the library does not implement (e.g. H not in {64,128,256}) */
    OFRL_ECUDA = -3,         /* a CUDA runtime call or launch failed */
    OFRL_ETIMEOUT = -4       /* reserved: a bounded device-side wait gave up */
};

/* HER donor strategies ("GPU IQL + HER Porting Plan", "Donor Index
 * Generation"; the string map "final" / "future" / anything else -> Random
 * is in "Config Wiring" of the HER part).  EPISODE is named in "HER (CPU)"
 * item 5 without a definition: here, as in the HER paper's "episode"
 * strategy, the donor is uniform over the source's whole episode. */
enum { OFRL_HER_FINAL = 0, OFRL_HER_FUTURE = 1, OFRL_HER_RANDOM = 2, OFRL_HER_EPISODE = 3 };

/* GEMM operand precision.  FP32: fp32 operands and accumulation.  BF16:
 * GEMM operands rounded to bf16 (round-to-nearest-even), fp32 accumulation,
 * fp32 master weights, fp32 epilogues (the twin-network workload). */
enum { OFRL_PREC_FP32 = 0, OFRL_PREC_BF16 = 1 };

/* Device status word, read by ofrl_poll_status (counts since the last poll). */
enum {
    OFRL_STAT_NONFINITE_GRAD = 0,  /* gradient elements Adam skipped as non-finite */
    OFRL_STAT_BAD_ACTION = 1,      /* batch actions outside [0, A) (treated as action 0) */
    OFRL_STAT_BAD_INDEX = 2,       /* episode boundary lookups that fell outside the buffer */
    OFRL_STAT_TIMEOUT = 3,         /* bounded device waits that gave up */
    OFRL_STAT_SANITIZED = 4,       /* gradient-source elements counted as 0 (ofrl_opt.sanitize_sources) */
    OFRL_STAT_WORDS = 8
};

typedef struct ofrl_ctx ofrl_ctx;

/* Replay buffer, structure of arrays, all device, read only
 * ("GPU IQL + HER Porting Plan", "GPU PER buffer": states [capacity,
 * state_dim], next_states, actions, rewards, dones; "Episode Boundary
 * Tracking on GPU": an episode boundary array). */
typedef struct {
    const float* states;         /* [capacity, state_stride] */
    const float* next_states;    /* [capacity, state_stride] */
    const int32_t* actions;      /* [capacity] */
    const float* rewards;        /* [capacity] */
    const float* dones;          /* [capacity] */
    const int32_t* episode_ends; /* [num_episodes] exclusive ends, strictly ascending,
                                    last == capacity; needed by FINAL and FUTURE only */
    int64_t capacity;            /* 1 .. 2^31-1 transitions */
    int32_t num_episodes;
    int32_t state_dim;           /* S */
    int32_t state_stride;        /* row stride in floats, >= S, multiple of 4 (16-byte rows) */
    int32_t goal_dim;            /* g: the goal is the first g state elements, 1 <= g <= S */
} ofrl_replay;

/* HER batch assembly ("How HER Interacts with GPU PER"): rows
 * [0, batch - her_count) are normal rows, rows [batch - her_count, batch)
 * are relabelled.  her_count = floor(batch * her_ratio) is the caller's. */
typedef struct {
    int32_t batch;           /* B >= 1 */
    int32_t her_count;       /* 0 .. B */
    int32_t strategy;        /* OFRL_HER_* */
    float goal_threshold;    /* reward +1 if goal distance < threshold, else -0.01 (pages: 0.01) */
    uint64_t seed;           /* counter-based RNG key (SplitMix64, see ofrl_her_relabel) */
} ofrl_her_cfg;

/* Relabelled batch, all device, written by ofrl_her_relabel / ofrl_train_step. */
typedef struct {
    float* states;        /* [B, stride] */
    float* next_states;   /* [B, stride] */
    int32_t* actions;     /* [B] */
    float* rewards;       /* [B] */
    float* dones;         /* [B] */
    int32_t* src_idx;     /* [B] source transition of each row */
    int32_t* donor_idx;   /* [B] goal donor of each row, -1 for normal rows */
    int32_t stride;       /* row stride in floats, >= S, multiple of 4 */
} ofrl_batch;

/* V network shape. */
typedef struct {
    int32_t state_dim;    /* S, 1 .. 64 */
    int32_t hidden;       /* H, one of 64, 128, 256 */
    int32_t num_actions;  /* A, 1 .. 16 */
    int32_t prec;         /* OFRL_PREC_* */
} ofrl_vshape;

/* One V network's trainable state, device buffers of P floats.  `t` is
 * the Adam step counter (host side); ofrl_train_step increments it before
 * the Adam phase, so the first step runs with t = 1.  `target`: the
 * network's target copy ("GPU IQL + HER Porting Plan", "Rust Integration:
 * gpu_iql_trainer.rs", target_ema_update: EMA target update for the V
 * network, Polyak averaging; step 4 of "Where in the Training Loop IQL Gets
 * Called"), or NULL; when set, ofrl_train_step updates it in the Adam pass,
 * after the weights: target = (1 - polyak) target + polyak params. */
typedef struct {
    float* params;
    float* m;
    float* v;
    int32_t t;
    float tau;            /* expectile, 0 < tau < 1 */
    float* target;        /* device [P] or NULL */
    float polyak;         /* 0 <= polyak <= 1 (read when target != NULL) */
} ofrl_vnet;

/* Optimiser and policy hyper-parameters ("GPU IQL + HER Porting Plan",
 * IqlGpuConfig fields lr, beta1, beta2, epsilon, weight_decay,
 * max_grad_norm; beta is the advantage temperature). */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    float max_grad_norm;  /* > 0; +inf disables every clip */
    float beta;           /* advantage temperature */
    float budget[4];      /* budget fractions, primary first (pages: 0.70, 0.15, 0.10, 0.05) */
    float alpha[4];       /* SAXPY coefficient per source, primary first (1.0 each) */
    /* "DQN Backward-Path NaN Audit": a bound on |weight| applied in the Adam
     * kernel after each update (0 disables it) ... */
    float weight_clamp_max_abs;
    /* ... and the SAXPY's isfinite guard: 1 counts non-finite elements of
     * every gradient source as 0 (in the source norms, the Gram matrix and
     * the combination; counted in OFRL_STAT_SANITIZED); 0 leaves them. */
    int32_t sanitize_sources;
} ofrl_opt;

/* ---- context -------------------------------------------------------- */

/* Create a context for V networks of `shape`, batches up to max_batch rows
 * and up to max_nets (1 or 2) networks per step.  The only allocating call.
 * Binds to the current CUDA device.  Returns OFRL_EINVAL / OFRL_EUNSUPPORTED
 * for bad shapes, OFRL_ECUDA if allocation fails; *out is NULL on error. */
ofrl_status ofrl_create(const ofrl_vshape* shape, int32_t max_batch, int32_t max_nets,
                        ofrl_ctx** out);

/* Free the context (synchronises the device first).  NULL is a no-op. */
ofrl_status ofrl_destroy(ofrl_ctx* ctx);

/* Copy the device status word (OFRL_STAT_WORDS int32 counters) to the host
 * array `words_out` and clear it.  Synchronises `stream`. */
ofrl_status ofrl_poll_status(ofrl_ctx* ctx, void* stream, int32_t* words_out);

/* Human-readable name of a status code (static storage). */
const char* ofrl_status_string(ofrl_status s);

/* Number of bytes of device workspace ofrl_create reserves for these sizes. */
int64_t ofrl_workspace_bytes(const ofrl_vshape* shape, int32_t max_batch, int32_t max_nets);

/* ---- the hot-path operations ----------------------------------------- */

/* HER index sampling + gather + relabel ("GPU IQL + HER Porting Plan",
 * "CUDA Kernel: her_relabel_kernel.cu" and "Donor Index Generation").
 * For every row b: src = below(draw(seed, step*2^32 + 2b), capacity).  For a
 * HER row the donor is: FINAL episode_end(src) - 1; FUTURE src + 1 +
 * below(draw(seed, step*2^32 + 2b + 1), episode_end(src) - src - 1), or src
 * itself when src is its episode's last transition; RANDOM
 * below(draw(seed, ...2b + 1), capacity); EPISODE episode_start(src) +
 * below(draw(seed, ...2b + 1), episode_end(src) - episode_start(src)).
 * episode_end(i) is the first entry of episode_ends above i (binary search),
 * episode_start(i) the entry before it (0 for the first episode).  draw(k, n) is output n+1
 * of SplitMix64 seeded with k; below(r, n) = ((r >> 32) * n) >> 32.
 * Row output: states/next_states/action/reward/done of src; for HER rows the
 * first g elements of both states are replaced by next_states[donor, :g]
 * and the reward is +1.0f if the fp32 distance between next_states[src, :g]
 * and next_states[donor, :g] (summed in order without fused multiply-add,
 * IEEE sqrtf) is below goal_threshold, else -0.01f.  Columns
 * [S, stride) of the output rows are copied from the source rows.
 * Writes every field of `out`. */
ofrl_status ofrl_her_relabel(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                             uint64_t step, const ofrl_batch* out, void* stream);

/* The relabel with the caller's sources ("GPU IQL + HER Porting Plan", "How
 * HER Interacts with GPU PER": normal rows and the HER rows' sources come
 * from the PER sampler; the HER rows' importance weights are 1, no PER
 * bias).  src_idx: device [batch] source of every row (normal rows first,
 * then the her_count HER rows; outside [0, capacity) is clamped and counted
 * in OFRL_STAT_BAD_INDEX).  is_weights: device [batch] or NULL (weight 1).
 * is_weights_out: device [batch] or NULL: the normal rows' weights, 1 for
 * HER rows.  Donors, rewards and the copies as ofrl_her_relabel. */
ofrl_status ofrl_her_relabel_sources(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                                     uint64_t step, const int32_t* src_idx, const float* is_weights,
                                     const ofrl_batch* out, float* is_weights_out, void* stream);

/* Episode-boundary maintenance on the device ("GPU IQL + HER Porting
 * Plan", "Episode Boundary Tracking on GPU": each finished episode's end is
 * appended to a GPU-resident boundary array that grows as episodes
 * complete).  n new transitions were stored at buffer positions
 * first_index .. first_index + n - 1 with done flags dones[0 .. n) (device);
 * for every i with dones[i] != 0 the exclusive end first_index + i + 1 is
 * appended to episode_ends (device, max_episodes entries) after the
 * *num_episodes (device int32) already there, in ascending order, and
 * *num_episodes grows by their number.  Ends that do not fit are dropped and
 * counted in OFRL_STAT_BAD_INDEX.  first_index + n <= 2^31 - 1. */
ofrl_status ofrl_episode_ends_append(ofrl_ctx* ctx, const float* dones, int64_t first_index, int32_t n,
                                     int32_t* episode_ends, int32_t* num_episodes, int32_t max_episodes,
                                     void* stream);

/* V forward + expectile loss + V backward ("GPU IQL + HER Porting Plan",
 * "IQL (CPU)" items 1-2 and "CUDA Kernel: iql_value_kernel.cu").
 * states: device [batch, state_stride] (columns >= S ignored);
 * q_taken: device [batch], Q(s, a_taken); params: device [P].
 * Outputs (device): v_out [batch] = V(s); loss_out [1] =
 * mean(w (q - V)^2), w = tau if q - V >= 0 else 1 - tau; grad_out [P] =
 * dloss/dparams (overwritten, not accumulated).  batch <= max_batch. */
ofrl_status ofrl_iql_value_fwd_bwd(ofrl_ctx* ctx, const float* params, const float* states,
                                   int32_t state_stride, int32_t batch, const float* q_taken,
                                   float tau, float* v_out, float* loss_out, float* grad_out,
                                   void* stream);

/* V forward only, the network's value of each state ("GPU IQL + HER
 * Porting Plan", "Rust Integration: gpu_iql_trainer.rs", forward_values:
 * a forward-only pass of the V network, result kept on the device).
 * params: device [P] (the online or the target network); states: device
 * [batch, state_stride] (columns >= S ignored).  v_out: device [batch].
 * 1 <= batch <= max_batch; asynchronous on `stream`.  Runs on the tensor
 * cores (a weight-pack launch, then one CTA per 128-row tile: G1, h1, G2,
 * V) when ofrl_vnet_path(ctx, 1) is OFRL_VNET_TC_FUSED and the states are
 * 16-byte aligned with state_stride a multiple of 4; else on the CUDA
 * cores.  Uses the context's weight-image workspace, so calls on one
 * context must not overlap. */
ofrl_status ofrl_forward_values(ofrl_ctx* ctx, const float* params, const float* states,
                                int32_t state_stride, int32_t batch, float* v_out, void* stream);

/* IQL bootstrap target for the Q loss ("GPU IQL + HER Porting Plan", "IQL
 * modifies the target computation": r + gamma V(s') in place of the
 * max-over-actions target): target_out[b] = rewards[b] + gamma (1 - dones[b])
 * V(next_states[b]) with V from `params` (terminal rows bootstrap nothing).
 * rewards, dones: device [batch] (e.g. the relabelled batch's); v_next_out:
 * device [batch] or NULL, receives V(s').  gamma in [0, 1].  Same
 * implementation choice as ofrl_forward_values. */
ofrl_status ofrl_iql_target(ofrl_ctx* ctx, const float* params, const float* next_states,
                            int32_t state_stride, const float* rewards, const float* dones,
                            int32_t batch, float gamma, float* v_next_out, float* target_out,
                            void* stream);

/* Expectile loss alone ("IQL (CPU)" item 2): q_taken, v device [batch];
 * loss_out device [1] = mean(w d^2), d = q - v; dv_out device [batch] or
 * NULL: dloss/dv = -2 w d / batch.  batch >= 1. */
ofrl_status ofrl_expectile_loss(ofrl_ctx* ctx, const float* q_taken, const float* v,
                                int32_t batch, float tau, float* loss_out, float* dv_out,
                                void* stream);

/* Advantage-weighted policy ("IQL (CPU)" item 3): q device [batch,
 * num_actions], v device [batch]; pi_out device [batch, num_actions] =
 * softmax(beta * clamp(q - v, -10, 10)) with max-subtraction; argmax_out
 * device [batch] or NULL: lowest index of the row's largest pi. */
ofrl_status ofrl_adv_weighted_policy(ofrl_ctx* ctx, const float* q, const float* v,
                                     int32_t batch, int32_t num_actions, float beta,
                                     float* pi_out, int32_t* argmax_out, void* stream);

/* Budgeted clipped SAXPY ("Gradient Stability -- Multi-Task Gradient
 * Isolation + Full Spectral Norm", "Proper design" and Task 1 Step 5):
 * grad_out = sum_k alpha[k] * s_k * src[k], s_k = (n_k > c_k && n_k > 0) ?
 * c_k / n_k : 1, n_k = ||src[k]||, c_k = budget_frac[k] * max_grad_norm.
 * src: host array of n_src (1..4) device pointers to [n] floats (src[0] is
 * the primary); budget_frac, alpha: host arrays of n_src.  grad_out: device
 * [n] (may alias no source).  norms_out: device [n_src + 1] =
 * n_0 .. n_{n_src-1}, ||grad_out||. */
ofrl_status ofrl_budgeted_clip_saxpy(ofrl_ctx* ctx, const float* const* src,
                                     const float* budget_frac, const float* alpha,
                                     int32_t n_src, int64_t n, float max_grad_norm,
                                     float* grad_out, float* norms_out, void* stream);

/* Adam with the safety clip ("DQN Backward-Path NaN Audit", Adam kernel
 * findings; "GPU IQL + HER Porting Plan", "CUDA Kernel: iql_adam_kernel.cu"):
 * s = (n > mgn && n > 0) ? mgn / n : 1 with n = *grad_norm (device scalar,
 * or NULL to compute ||g|| here); per element g' = s * g[i]; a non-finite
 * g' leaves p, m, v unchanged and is counted in the status word; else
 * m = b1 m + (1-b1) g', v = b2 v + (1-b2) g'^2, p -= lr (m/(1-b1^t) /
 * (sqrt(v/(1-b2^t)) + eps) + weight_decay p), then p clamped to
 * [-w, w] with w = opt->weight_clamp_max_abs when w > 0.  t >= 1. */
ofrl_status ofrl_adam_step(ofrl_ctx* ctx, float* p, const float* g, float* m, float* v,
                           int64_t n, int32_t t, const ofrl_opt* opt, const float* grad_norm,
                           void* stream);

/* Polyak (EMA) update of a target network ("GPU IQL + HER Porting Plan",
 * "Rust Integration: gpu_iql_trainer.rs", target_ema_update):
 * target[i] = (1 - polyak) target[i] + polyak params[i], i < n.  Device
 * buffers; 0 <= polyak <= 1.  Needs no context. */
ofrl_status ofrl_target_ema(const float* params, float* target, int64_t n, float polyak, void* stream);

/* The fused train step: relabel -> per network {V fwd, expectile loss on
 * Q[b, action_b], policy, V bwd -> primary gradient g0; budgeted combine of
 * g0 (budget[0]) and the network's aux sources (budget[1..]); t += 1; Adam}.
 * q: device [B, A]; nets: host array of n_nets (1 or 2) networks sharing
 * the batch and Q; aux_src: host array of n_nets * n_aux device pointers
 * (network-major) to [P] floats, or NULL when n_aux == 0 (0..3).
 * Outputs (device, each may be NULL except batch): v_out [n_nets, B],
 * pi_out [n_nets, B, A], argmax_out [n_nets, B], loss_out [n_nets],
 * norms_out [n_nets, 5] (n_0..n_3 pre-clip source norms, 0 for absent
 * sources, then the combined norm), grad_out [n_nets, P] (the primary
 * gradient g0).  Increments nets[k].t on the host.
 * When the previous launch of this context on `stream` was a train step, the
 * relabel of this step's batch starts while that step's optimizer kernel
 * still runs (it reads only the replay buffer and, when q is in host memory,
 * q, and writes only the batch and the context's copy of q; the V kernel
 * still waits for both).  Writes to the replay buffer or q in between by
 * ordinary kernels or copies are ordered as usual; a kernel of the caller's
 * that lets its dependents launch early (programmatic dependent launch)
 * must not write them right before a step. */
ofrl_status ofrl_train_step(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                            uint64_t step, const ofrl_batch* batch, const float* q,
                            ofrl_vnet* nets, int32_t n_nets, const ofrl_opt* opt,
                            const float* const* aux_src, int32_t n_aux,
                            float* v_out, float* pi_out, int32_t* argmax_out, float* loss_out,
                            float* norms_out, float* grad_out, void* stream);

/* Kernel launches one ofrl_train_step on this context makes for `rows`
 * batch rows and n_nets networks writing into `batch` (no counterpart on the
 * pages: a planning aid for launch accounting and graph capture): relabel,
 * one V kernel (two on the layered tensor-core path), then reduce and Adam
 * as one cooperative launch when its grid fits on the device at once, else
 * two.  Returns 0 for invalid arguments.  Host only; launches nothing. */
int32_t ofrl_train_step_kernels(const ofrl_ctx* ctx, const ofrl_batch* batch, int32_t rows, int32_t n_nets);

/* ---- V forward/backward implementations --------------------------------
 * The batch x hidden GEMMs of the value network ("GPU IQL + HER Porting
 * Plan", "CUDA Kernel: iql_value_kernel.cu"; five GEMMs per network and
 * step) run in one of three ways, all with the same results to fp32
 * rounding (no counterpart on the pages, which use cuBLAS):
 *   TC_FUSED   H = 128, S <= 64: one CTA per 128-row tile runs all five
 *              GEMMs on the tensor cores (tcgen05, accumulators in TMEM);
 *   TC_LAYERED H = 128 or 256, S < 64: per tile the forward and the
 *              backward to dz1 on the tensor cores with operands streamed by
 *              TMA, then the weight gradients split over K-ranges of the
 *              batch (two kernels);
 *   CUDA_CORES every H in {64, 128, 256}.
 * AUTO (the default) takes TC_FUSED for H = 128, TC_LAYERED for H = 256 and
 * CUDA_CORES otherwise, falling back to CUDA_CORES where a choice does not
 * apply to a call (e.g. unaligned states in a standalone call).
 * ofrl_select_vnet_path sets the context's choice: OFRL_EUNSUPPORTED when
 * the shape (or the driver, for the layered path's tensor maps) does not
 * allow it, OFRL_EINVAL for an unknown value.  ofrl_vnet_path returns the
 * implementation a train step of n_nets networks takes (an OFRL_VNET_*
 * value, never AUTO), or -1 for invalid arguments.  Host only. */
enum { OFRL_VNET_AUTO = 0, OFRL_VNET_TC_FUSED = 1, OFRL_VNET_TC_LAYERED = 2, OFRL_VNET_CUDA_CORES = 3 };
ofrl_status ofrl_select_vnet_path(ofrl_ctx* ctx, int32_t path);
int32_t ofrl_vnet_path(const ofrl_ctx* ctx, int32_t n_nets);

/* ---- the step as a CUDA graph ------------------------------------------
 * "Phase 2: Multi-Stream Graph Parallelism" runs the trainers' step as a
 * captured CUDA graph.  ofrl_step_graph_create captures one ofrl_train_step
 * with these arguments (all of them checked as ofrl_train_step checks them;
 * nothing runs) and instantiates it.  ofrl_step_graph_launch replays it on
 * `stream` as the step `step`: the relabel uses `step`; q ([B, A], device
 * or, as for ofrl_train_step, page-locked host memory; NULL keeps the
 * previous one) and aux_src (host array of n_nets * n_aux
 * device pointers, or NULL to keep the previous ones) replace the captured
 * pointers; each network's t advances by one in the caller's `nets` array
 * (which must outlive the graph), exactly as ofrl_train_step would.  Every
 * other buffer is the one given at creation.  One graph launch on the host
 * per step.  The graph uses the context's workspace: do not interleave its
 * replays with other calls on the context from another stream.  Profiling
 * hooks (ofrl_profile_begin) must be off while creating one. */
typedef struct ofrl_step_graph ofrl_step_graph;
ofrl_status ofrl_step_graph_create(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                                   const ofrl_batch* batch, const float* q, ofrl_vnet* nets, int32_t n_nets,
                                   const ofrl_opt* opt, const float* const* aux_src, int32_t n_aux,
                                   float* v_out, float* pi_out, int32_t* argmax_out, float* loss_out,
                                   float* norms_out, float* grad_out, ofrl_step_graph** out);
ofrl_status ofrl_step_graph_launch(ofrl_step_graph* graph, uint64_t step, const float* q,
                                   const float* const* aux_src, void* stream);
ofrl_status ofrl_step_graph_destroy(ofrl_step_graph* graph);

/* The step graph with its host I/O inside (no counterpart on the pages): as
 * ofrl_step_graph_create, plus a copy of q_host (pinned host [B, A]) into
 * the device q before the kernels and copies of loss_out and norms_out into
 * loss_host ([n_nets]) and norms_host ([n_nets, 5]) after them, as nodes of
 * the graph; any of the three may be NULL (no copy).  Host buffers must be
 * page-locked (cudaHostAlloc / cudaHostRegister).  ofrl_step_graph_launch_io
 * replays it as step `step` with this step's host buffers (NULL keeps the
 * previous one): one graph launch does the copy-in, the step and the
 * copy-out.  The results are in the host buffers once `stream` has reached
 * the launch (synchronise or wait on an event).  ofrl_step_graph_destroy
 * releases it. */
ofrl_status ofrl_step_graph_create_io(ofrl_ctx* ctx, const ofrl_replay* replay, const ofrl_her_cfg* her,
                                      const ofrl_batch* batch, float* q, ofrl_vnet* nets, int32_t n_nets,
                                      const ofrl_opt* opt, const float* const* aux_src, int32_t n_aux,
                                      float* v_out, float* pi_out, int32_t* argmax_out, float* loss_out,
                                      float* norms_out, float* grad_out, const float* q_host, float* loss_host,
                                      float* norms_host, ofrl_step_graph** out);
ofrl_status ofrl_step_graph_launch_io(ofrl_step_graph* graph, uint64_t step, const float* q_host,
                                      const float* const* aux_src, float* loss_host, float* norms_host,
                                      void* stream);

/* ---- allocation-free variant (no counterpart in the method's pages) ---- */

/* Some callers may not allocate device memory: code whose GPU memory is
 * handed out by a host application's or framework's own pool (direct
 * cudaMalloc forbidden), code recorded into a CUDA graph under the global
 * capture mode (cudaMalloc is refused there), and latency-critical loops that
 * cannot take cudaMalloc's implicit device synchronisation.  ofrl_create
 * allocates, so they call the entry point below instead.
 *
 * Its scratch is one file-scope device array of OFRL_NOALLOC_SCRATCH_BYTES,
 * reserved in every GPU that loads this library until the library is
 * unloaded.  The first call made with a given device current looks up the
 * array's device address (cudaGetSymbolAddress) and keeps it; make that first
 * call before any stream capture.  All calls share the one array: two calls
 * whose kernels overlap on the GPU (different streams, or different host
 * threads) race and give wrong results, so serialise them (one stream). */
#define OFRL_NOALLOC_SCRATCH_BYTES (4u << 20)

/* Largest batch ofrl_iql_value_fwd_bwd_noalloc accepts for `shape` (what the
 * scratch array holds), or -1 for an unsupported shape. */
int64_t ofrl_noalloc_max_batch(const ofrl_vshape* shape);

/* Same computation, arguments and results as ofrl_iql_value_fwd_bwd (V
 * forward, expectile loss, V backward into grad_out), with `shape` in place
 * of a context.  Allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library call.  A batch above ofrl_noalloc_max_batch(shape) returns
 * OFRL_EINVAL before anything is launched; H outside {64, 128, 256} returns
 * OFRL_EUNSUPPORTED.  Asynchronous on `stream`. */
ofrl_status ofrl_iql_value_fwd_bwd_noalloc(const ofrl_vshape* shape, const float* params, const float* states,
                                           int32_t state_stride, int32_t batch, const float* q_taken, float tau,
                                           float* v_out, float* loss_out, float* grad_out, void* stream);

/* ---- measurement hooks (not part of the method) ----------------------- */

/* Phases of ofrl_train_step, in launch order. */
enum { OFRL_PHASE_RELABEL = 0, OFRL_PHASE_VNET = 1, OFRL_PHASE_REDUCE = 2, OFRL_PHASE_ADAM = 3,
       OFRL_PHASES = 4 };

/* Start recording per-phase device time of the next max_steps calls of
 * ofrl_train_step on this context: CUDA events recorded on the call's stream
 * around each phase (host-side event objects are created here; no device
 * memory is allocated).  A second begin replaces the first. */
ofrl_status ofrl_profile_begin(ofrl_ctx* ctx, int32_t max_steps);

/* Wait for the recorded events, write the summed time of each phase in
 * milliseconds to phase_ms_out[OFRL_PHASES] and the number of recorded steps
 * to *steps_out, and stop recording. */
ofrl_status ofrl_profile_end(ofrl_ctx* ctx, float* phase_ms_out, int32_t* steps_out);

#ifdef __cplusplus
}
#endif
#endif /* OFRL_H */

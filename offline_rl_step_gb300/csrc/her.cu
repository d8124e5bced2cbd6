// HER index sampling + gather + relabel.
//
// Method: "GPU IQL + HER Porting Plan", "CUDA Kernel: her_relabel_kernel.cu"
// (copy the source transition, overwrite the goal slice of state and
// next_state with the donor's achieved goal next_states[donor, :g], copy
// action and done, recompute the reward from the fp32 goal distance) and
// "Donor Index Generation" (Final / Future / Random).  The pages launch one
// warp per relabelled row and a separate donor kernel; here the index draw,
// the donor search and the row copy are one pass, and a row is moved by 16
// lanes with 16-byte loads and stores, so one warp moves two rows.  Random
// numbers come from a counter-based SplitMix64 instead of cuRAND, so any
// row's indices depend only on (seed, step, row).
//
// Memory-bound: per row 2 * copy_cols * 4 bytes gathered and written, plus
// g * 4 donor bytes and the scalars.  Source rows are whole 32-byte sectors
// when the row stride is a multiple of 8 floats.

#include "common.cuh"
#include "tc_image.cuh"

namespace ofrl {
namespace {

constexpr int kLanesPerRow = 16;
constexpr int kRelabelThreads = 256;
constexpr int kRowsPerBlock = kRelabelThreads / kLanesPerRow;
constexpr int kCappedBlocks = 4;   // relabel blocks per SM when the grid has slack (launch_her_relabel)
constexpr unsigned kFull = 0xffffffffu;

// First index k with ends[k] > i, found by the 16 lanes of a half-warp
// together: each round probes the last entry of 16 equal segments of the
// window and keeps the first segment that ends above i (a 16-ary search, so
// log16(n) rounds instead of log2(n) dependent loads).  `rounds` is the same
// for both half-warps, so every ballot is executed by the whole warp.
// Returns n when no entry is above i.
__device__ __forceinline__ int episode_search(const int32_t* __restrict__ ends, int n, int rounds, int i,
                                              int sub) {
    const int shift = threadIdx.x & 16;
    int lo = 0, len = n;
    for (int r = 0; r < rounds; ++r) {
        const int step = (len + kLanesPerRow - 1) / kLanesPerRow;
        const int p = lo + (sub + 1) * step - 1;
        const bool gt = len > kLanesPerRow && p < lo + len ? __ldg(ends + p) > i : true;
        const unsigned m = (__ballot_sync(kFull, gt) >> shift) & 0xFFFFu;
        if (len > kLanesPerRow) {
            const int f = __ffs(m) - 1;    // m != 0: the window's last segment always answers true
            const int nlo = lo + f * step;
            len = min(step, lo + len - nlo);
            lo = nlo;
        }
    }
    const bool gt = sub < len ? __ldg(ends + lo + sub) > i : true;
    const unsigned m = (__ballot_sync(kFull, gt) >> shift) & 0xFFFFu;
    const int f = __ffs(m) - 1;
    return f < len ? lo + f : lo + len;
}

// The relabelled rows are written, and (with random donors) the source rows
// gathered, once a step and read by no later kernel of the step:
// evict_first in L2, so they do not push out the state-tile images and
// gradient partials that the next kernels read.
__device__ __forceinline__ float4 ldg4_first(const float* p) {
    float4 v;
    asm volatile(
        "{\n\t.reg .b64 pol;\n\tcreatepolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ void st4_first(float* p, const float4& v) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\tcreatepolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, pol;\n\t}" ::"l"(p),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
        : "memory");
}

// put4 with the state-tile image kept in L2 (evict_last): the V kernel reads
// it next.
__device__ __forceinline__ void st8_keep(uint8_t* p, uint32_t lo, uint32_t hi) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\tcreatepolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
        "st.global.L2::cache_hint.v2.b32 [%0], {%1, %2}, pol;\n\t}" ::"l"(p),
        "r"(lo), "r"(hi)
        : "memory");
}
__device__ __forceinline__ void put4_keep(uint8_t* img, uint32_t plane, int np, int C, int r, int c,
                                          const float (&x)[4]) {
    const uint32_t o = tc::img_off(r, c, C);
    if (np == 3) {
        uint32_t a0, a1, a2, b0, b1, b2;
        tc::split3x2(x[0], x[1], a0, a1, a2);
        tc::split3x2(x[2], x[3], b0, b1, b2);
        st8_keep(img + o, a0, b0);
        st8_keep(img + plane + o, a1, b1);
        st8_keep(img + 2 * plane + o, a2, b2);
    } else {
        st8_keep(img + o, tc::pack_bf16x2(x[0], x[1]), tc::pack_bf16x2(x[2], x[3]));
    }
}

// Extra blocks of the relabel grid: W1 [H][S] -> [W x 64] image and
// W2 [H][H] -> [W x W] image of every network (W = pack_width >= H: units
// past H zero), img_planes planes.
__device__ void pack_weights(const HerLaunch& a) {
    const int S = a.state_dim, Hn = a.pack_hidden, H = a.pack_width, np = a.img_planes;
    const Offsets off = offsets_of(S, Hn);
    const int n1 = H * (tc::KX / 4), n2 = H * (H / 4);      // groups of 4 columns
    const int total = a.pack_nets * (n1 + n2);
    for (int e = (blockIdx.x - a.relabel_blocks) * blockDim.x + threadIdx.x; e < total;
         e += a.pack_blocks * blockDim.x) {
        const int net = e / (n1 + n2), f = e % (n1 + n2);
        const float* prm = a.pack_params[net];
        uint8_t* w1i = a.wimg + (int64_t)net * tc::weight_image_bytes(H);
        uint8_t* w2i = w1i + tc::w2_image_offset(H);
        const uint32_t plane1 = (uint32_t)(H * tc::KX * 2), plane2 = (uint32_t)(H * H * 2);
        float x[4];
        if (f < n1) {
            const int r = f / (tc::KX / 4), c = 4 * (f % (tc::KX / 4));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                x[j] = r < Hn && c + j < S ? __ldg(prm + off.w1 + (int64_t)r * S + c + j) : 0.0f;
            tc::put4(w1i, plane1, np, tc::KX, r, c, x);
        } else {
            const int g = f - n1, r = g / (H / 4), c = 4 * (g % (H / 4));
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = r < Hn && c + j < Hn ? __ldg(prm + off.w2 + (int64_t)r * Hn + c + j) : 0.0f;
            tc::put4(w2i, plane2, np, H, r, c, x);
        }
    }
}

template <bool STAGE_Q, bool RANDOM_DONORS>
__global__ void __launch_bounds__(kRelabelThreads) her_relabel_kernel(const HerLaunch a) {
    pdl_trigger();
    // The weight packing reads what the previous kernel (Adam) wrote.  The
    // rows read only the replay buffer: with `early` set (the previous kernel
    // on the stream is the optimizer of a train step, which lets dependents
    // launch only after everything before it, the V kernel included, has
    // completed) they run while that kernel still does.  The last row block
    // waits in any case, so this grid completes only after the previous one
    // did.
    const int rb = a.relabel_blocks;
    if (!a.early || (int)blockIdx.x >= rb - 1) pdl_wait();
    if ((int)blockIdx.x >= rb) {
        pack_weights(a);
        return;
    }
    // this block's rows of Q (one contiguous run of at most 16 x 16 floats)
    // from host memory: loaded here, stored into the device copy the V
    // kernel reads once the rows' own loads are done, so the host link's
    // latency overlaps them; 16-byte copies when the run is aligned
    float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
    float* q_to = nullptr;
    bool q_vec = false;
    if (STAGE_Q) {
        const int r0 = (rb - 1 - (int)blockIdx.x) * kRowsPerBlock;
        const int nr = min(kRowsPerBlock, a.batch - r0);
        if (nr > 0) {
            const int64_t e0 = (int64_t)r0 * a.q_cols;
            const int n = nr * a.q_cols;
            const float* qs = a.q_src + e0;
            float* qd = a.q_dst + e0;
            q_vec = ((reinterpret_cast<uintptr_t>(qs) | reinterpret_cast<uintptr_t>(qd)) & 15u) == 0 && (n & 3) == 0;
            const int i = (int)threadIdx.x;
            if (q_vec && i < n / 4) {
                qv = reinterpret_cast<const float4*>(qs)[i];
                q_to = qd + 4 * i;
            } else if (!q_vec && i < n) {
                qv.x = qs[i];
                q_to = qd + i;
            }
        }
    }
    const int sub = threadIdx.x & (kLanesPerRow - 1);
    // blocks in reverse row order: the HER rows (the last rows, with the
    // longest chain of dependent loads) are dispatched first
    const int row_raw = (rb - 1 - (int)blockIdx.x) * kRowsPerBlock + threadIdx.x / kLanesPerRow;
    const bool live = row_raw < a.batch;
    if (a.ximg != nullptr && row_raw >= a.batch && row_raw < a.img_rows) {
        // the last tile's rows past the batch: zero image rows
        const float z[4] = {0.f, 0.f, 0.f, 0.f};
        put4_keep(a.ximg + (int64_t)(row_raw / tc::TM) * a.img_planes * tc::kPlaneX, tc::kPlaneX, a.img_planes,
                  tc::KX, row_raw % tc::TM, 4 * sub, z);
    }
    const int row = live ? row_raw : a.batch - 1;   // dead half-warps shadow the last row, write nothing
    const uint64_t ctr = (a.step << 32) | ((uint64_t)row << 1);

    // 1. source index (drawn here, or the caller's), then the source rows'
    // loads go out at once
    int src = 0, bad = 0;
    if (sub == 0) {
        if (a.src_in != nullptr) {
            src = __ldg(a.src_in + row);
            if (src < 0 || src >= a.capacity) {   // flagged; the row stays inside the buffer
                src = src < 0 ? 0 : a.capacity - 1;
                bad = 1;
            }
        } else {
            src = (int)below(sm64_at(a.seed, ctr), (uint64_t)a.capacity);
        }
    }
    src = __shfl_sync(kFull, src, 0, kLanesPerRow);
    const int chunks = a.copy_cols >> 2;   // <= 16 (state_dim <= 64)
    const bool has = sub < chunks;
    float4 sv = make_float4(0.f, 0.f, 0.f, 0.f), nv = sv;
    if (has) {
        const float* sr = a.states + (int64_t)src * a.in_stride + 4 * sub;
        const float* nr = a.next_states + (int64_t)src * a.in_stride + 4 * sub;
        // evict_first on the gathers pays with 'random' donors (65,536 rows:
        // 96.3 -> 93.4 us a step) and costs with 'future' ones (two networks:
        // +0.9 us), so only the random strategy's instance marks them
        if constexpr (RANDOM_DONORS) {
            sv = ldg4_first(sr);
            nv = ldg4_first(nr);
        } else {
            sv = __ldg(reinterpret_cast<const float4*>(sr));
            nv = __ldg(reinterpret_cast<const float4*>(nr));
        }
    }
    int act = 0;
    float done = 0.0f, rew = 0.0f;
    if (sub == 0) {
        act = __ldg(a.actions + src);
        done = __ldg(a.dones + src);
        rew = __ldg(a.rewards + src);
    }

    // 2. donor (HER rows), overlapping the row loads
    const bool her = row >= a.first_her;
    int donor = -1;
    if (a.strategy == OFRL_HER_RANDOM) {
        if (sub == 0 && her) donor = (int)below(sm64_at(a.seed, ctr | 1ull), (uint64_t)a.capacity);
    } else if (__any_sync(kFull, live && her)) {   // warp-uniform: only warps holding a HER row search
        const int k = episode_search(a.episode_ends, a.num_episodes, a.search_rounds, src, sub);
        if (sub == 0 && her) {
            int end = k < a.num_episodes ? __ldg(a.episode_ends + k) : a.capacity;
            int start = k > 0 && k <= a.num_episodes ? __ldg(a.episode_ends + k - 1) : 0;
            if (k >= a.num_episodes || end > a.capacity || end <= src) {
                end = a.capacity;   // malformed boundaries: flagged; the donor stays inside the buffer
                bad = 1;
            }
            if (start > src || start < 0) {
                start = src;
                bad = 1;
            }
            if (a.strategy == OFRL_HER_FINAL) {
                donor = end - 1;
            } else if (a.strategy == OFRL_HER_EPISODE) {
                donor = start + (int)below(sm64_at(a.seed, ctr | 1ull), (uint64_t)(end - start));
            } else {
                const int lo = src + 1;
                donor = lo < end ? lo + (int)below(sm64_at(a.seed, ctr | 1ull), (uint64_t)(end - lo)) : src;
            }
        }
    }
    donor = __shfl_sync(kFull, donor, 0, kLanesPerRow);

    // 3. goal slice from the donor's next state; reward from the fp32 distance.
    // Every lane of a warp holding a HER row runs the shuffles (a normal row
    // beside it compares a row with itself and ignores the result).
    const bool goal_lane = has && 4 * sub < a.goal_dim;
    float4 gv = nv;
    if (goal_lane && donor >= 0)
        gv = __ldg(reinterpret_cast<const float4*>(a.next_states + (int64_t)donor * a.in_stride) + sub);
    // distance as the pages' kernel: float accumulator in order d = 0..g-1,
    // each product and sum rounded on its own (no FMA), IEEE sqrt
    float dsq = 0.0f;
    const bool any_her = __any_sync(kFull, donor >= 0);
    for (int c = 0; any_her && 4 * c < a.goal_dim; ++c) {
        const float av[4] = {__shfl_sync(kFull, nv.x, c, kLanesPerRow), __shfl_sync(kFull, nv.y, c, kLanesPerRow),
                             __shfl_sync(kFull, nv.z, c, kLanesPerRow), __shfl_sync(kFull, nv.w, c, kLanesPerRow)};
        const float bv[4] = {__shfl_sync(kFull, gv.x, c, kLanesPerRow), __shfl_sync(kFull, gv.y, c, kLanesPerRow),
                             __shfl_sync(kFull, gv.z, c, kLanesPerRow), __shfl_sync(kFull, gv.w, c, kLanesPerRow)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (4 * c + e < a.goal_dim) {
                const float diff = __fsub_rn(av[e], bv[e]);
                dsq = __fadd_rn(dsq, __fmul_rn(diff, diff));
            }
        }
    }
    const float r = __fsqrt_rn(dsq) < a.threshold ? 1.0f : -0.01f;
    if (goal_lane && donor >= 0) {
        const int base = 4 * sub;
        if (base + 0 < a.goal_dim) { sv.x = gv.x; nv.x = gv.x; }
        if (base + 1 < a.goal_dim) { sv.y = gv.y; nv.y = gv.y; }
        if (base + 2 < a.goal_dim) { sv.z = gv.z; nv.z = gv.z; }
        if (base + 3 < a.goal_dim) { sv.w = gv.w; nv.w = gv.w; }
    }
    if (STAGE_Q && q_to != nullptr) {
        if (q_vec) *reinterpret_cast<float4*>(q_to) = qv;
        else *q_to = qv.x;
    }
    if (!live) return;
    if (a.ximg != nullptr) {
        // the relabelled state, columns 4 sub .. 4 sub + 3, into this row's tile image
        float x[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (!has || 4 * sub + j >= a.state_dim) x[j] = tc::ones_column(4 * sub + j, a.state_dim) ? 1.0f : 0.0f;
        put4_keep(a.ximg + (int64_t)(row / tc::TM) * a.img_planes * tc::kPlaneX, tc::kPlaneX, a.img_planes, tc::KX,
                  row % tc::TM, 4 * sub, x);
    }
    if (has) {
        st4_first(a.out_states + (int64_t)row * a.out_stride + 4 * sub, sv);
        st4_first(a.out_next_states + (int64_t)row * a.out_stride + 4 * sub, nv);
    }
    if (sub == 0) {
        a.out_actions[row] = act;
        a.out_dones[row] = done;
        a.out_rewards[row] = donor >= 0 ? r : rew;
        a.out_src[row] = src;
        a.out_donor[row] = donor;
        if (a.isw_out != nullptr) a.isw_out[row] = her ? 1.0f : (a.isw_in != nullptr ? __ldg(a.isw_in + row) : 1.0f);
        if (bad) atomicAdd(a.status + OFRL_STAT_BAD_INDEX, 1);
    }
}

// Append the exclusive end (first_index + i + 1) of every transition i < n
// with dones[i] != 0 to episode_ends, in ascending order, after the
// *num_episodes entries already there ("GPU IQL + HER Porting Plan",
// "Episode Boundary Tracking on GPU": the experience kernel records each
// finished episode's end in a GPU-resident boundary array).  One CTA: thread
// t scans its contiguous share of the new transitions, a block-wide
// exclusive scan of the counts gives each thread its output position, so the
// array stays sorted (the pages' atomicAdd slot order would not).  Ends past
// max_episodes are dropped and counted as bad indices.
constexpr int kAppendThreads = 1024;
__global__ void __launch_bounds__(kAppendThreads) episode_ends_append_kernel(
    const float* __restrict__ dones, int64_t first_index, int32_t n, int32_t* __restrict__ ends,
    int32_t* __restrict__ count, int32_t max_ends, int32_t* __restrict__ status) {
    __shared__ int warp_tot[kAppendThreads / 32];
    __shared__ int base_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kAppendThreads - 1) / kAppendThreads;
    const int lo = tid * per < n ? tid * per : n;
    const int hi = lo + per < n ? lo + per : n;
    int c = 0;
    for (int i = lo; i < hi; ++i) c += __ldg(dones + i) != 0.0f;
    // inclusive scan inside the warp, then over the warp totals
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    if (tid == 0) base_s = *count;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    int pos = base_s + before + x - c;   // exclusive prefix of this thread
    int dropped = 0;
    for (int i = lo; i < hi; ++i) {
        if (__ldg(dones + i) != 0.0f) {
            if (pos < max_ends) ends[pos] = (int32_t)(first_index + i + 1);
            else ++dropped;
            ++pos;
        }
    }
    if (dropped) atomicAdd(status + OFRL_STAT_BAD_INDEX, dropped);
    if (tid == kAppendThreads - 1) {
        const int total = base_s + before + x;
        *count = total < max_ends ? total : max_ends;
    }
}

}  // namespace

cudaError_t launch_episode_ends_append(const float* dones, int64_t first_index, int32_t n, int32_t* episode_ends,
                                       int32_t* num_episodes, int32_t max_episodes, int32_t* status,
                                       cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    episode_ends_append_kernel<<<1, kAppendThreads, 0, st>>>(dones, first_index, n, episode_ends, num_episodes,
                                                             max_episodes, status);
    return cudaGetLastError();
}

cudaError_t launch_her_relabel(const HerLaunch& a_in, cudaStream_t st) {
    if (a_in.batch <= 0) return cudaSuccess;
    HerLaunch a = a_in;
    const int rows = a.ximg != nullptr ? a.img_rows : a.batch;
    a.relabel_blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    // the weight images grow with H^2: 48 blocks at H = 128
    a.pack_blocks = a.wimg != nullptr ? (a.pack_width > 128 ? 160 : 48) : 0;
    // Occupancy: when the rows run beside the previous step's optimizer kernel
    // (`early`) and the grid fits one wave of the SMs at full occupancy, it
    // has slack there; then each SM holds at most kCappedBlocks relabel blocks (by
    // asking for unused dynamic shared memory), leaving the optimizer more of
    // it (two networks: 35.0 -> 33.3 us a step; one network: unchanged).  A
    // larger grid keeps every slot (65,536 rows: 98.5 -> 100.2 us capped).
    static int sms = 0, smem_sm = 0, reserved = 0, full = 0;
    static bool configured = false;
    if (!configured) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        const int cap_bytes = smem_sm / kCappedBlocks - reserved;
        for (auto k : {her_relabel_kernel<false, false>, her_relabel_kernel<true, false>,
                       her_relabel_kernel<false, true>, her_relabel_kernel<true, true>}) {
            if (e == cudaSuccess) e = set_max_shared_carveout(k);
            if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, cap_bytes);
        }
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&full, her_relabel_kernel<false, false>, kRelabelThreads,
                                                              0);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int blocks = a.relabel_blocks + a.pack_blocks;
    const size_t smem = a.early && blocks <= full * sms ? (size_t)(smem_sm / kCappedBlocks - reserved) : 0;
    // Q staged from host memory: its own instance (the copy's registers
    // would lower the occupancy of the plain one)
    const bool rnd = a.strategy == OFRL_HER_RANDOM;
    const auto kern = a.q_src != nullptr ? (rnd ? her_relabel_kernel<true, true> : her_relabel_kernel<true, false>)
                                         : (rnd ? her_relabel_kernel<false, true> : her_relabel_kernel<false, false>);
    return launch_pdl(kern, dim3(blocks), dim3(kRelabelThreads), smem, st, a);
}

}  // namespace ofrl

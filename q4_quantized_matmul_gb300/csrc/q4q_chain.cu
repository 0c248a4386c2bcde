// q4q_chain.cu -- a chain of dependent Q4_0 projections of one token in one launch.
//
// A decode step runs its projections one after another, each reading what an
// earlier one wrote: the GPT-2 walkthrough's gpt2_eval goes through every layer's
// QKV projection (§3.2), output projection and MLP (§3.5), then the lm_head (§3.6),
// all of them ggml_mul_mat, as "llama.cpp 深度解读" §3 computes it (src1 rows
// quantized to Q8_0, sum_b fp32(d_w d_x) isum_b per output).  Launched one kernel
// per matrix, every small matrix pays a launch, its weights' first bytes and the
// wait for the previous kernel.  Here one persistent, co-resident grid walks the
// whole list ("links"):
//  * the producer warp of every CTA streams its units of link 0, 1, 2, ... through
//    the shared-memory ring without waiting for anything but free stages, so the
//    weights of the next links are in flight while the current one is computed;
//  * before link i reads its activations, every CTA has finished link i - 1: each
//    CTA adds 1 to done[i - 1] (release, after all its outputs of that link are
//    written) when it finishes its units of link i - 1, and the consumers wait for
//    done[i - 1] == gridDim.x (acquire) -- a bounded wait that gives up after the
//    time limit or as soon as another CTA raised the call's abort word;
//  * the activations are then loaded from L2 (they may have been written by another
//    CTA in this same launch), quantized to Q8_0 in shared memory exactly as the
//    GEMV does, and every unit's rows are dotted against them.
// The grid is launched cooperatively (every CTA resident at once, or the launch
// fails), so no CTA ever waits for one that has not started.
#include "q4q_gemv.cuh"

namespace q4q {
namespace {

constexpr int CHAIN_MAX = Q4Q_CHAIN_MAX;

struct ChainLink {
    const uint8_t* w;
    const float* x;
    float* dst;
    int ne00, nb, np, ne01, row_bytes;
    int G, n_units, lpr;
};

struct ChainParams {
    int n, S, stage_bytes, act_off, stage_off;
    unsigned int* done;          // [n] CTAs that finished link i (zero at launch)
    unsigned int* abort_word;    // raised by a CTA that gave up (zero at launch)
    uint64_t limit_ns;
    int fault;                   // test only: 1 = CTA 0 never reports link 0 finished
    ChainLink link[CHAIN_MAX];
};

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait for *ctr >= target (another CTA's release); false when the limit
// runs out or the call's abort word is raised.
__device__ __forceinline__ bool wait_count(const unsigned int* ctr, unsigned int target,
                                           const unsigned int* abort_word, uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t n = 1;; ++n) {
        if (ld_acquire(ctr) >= target) return true;
        if ((n & 15u) == 0u) {
            if (*reinterpret_cast<const volatile unsigned int*>(abort_word) != 0u) return false;
            const uint64_t t = global_timer_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > limit_ns) return false;
        }
    }
}

// The rows [r0, r0 + nr) of link L, staged at `stage`, against the link's
// quantized activations; LPR lanes per row (the link's np is a multiple of LPR).
template <int LPR>
__device__ __forceinline__ void chain_rows(const uint8_t* stage, const ChainLink& L, int r0, int nr,
                                           const uint4* quads, const float* dy, const int* sy8, int tid) {
    constexpr int RP = CONSUMERS / LPR;
    const int rr = tid / LPR, sl = tid % LPR;
    const int ppl = L.np / LPR;
    for (int j0 = 0; j0 < nr; j0 += RP) {
        const int j = j0 + rr;
        float acc = 0.0f;
        if (j < nr) {
            const uint8_t* rowp = stage + (size_t)j * L.row_bytes;
            for (int kk = 0; kk < ppl; ++kk) {
                const int pr = sl + kk * LPR;
                const PairActs a = load_pair_acts(quads, dy, sy8, L.np, L.nb, 0, pr);
                acc = pair_dot<WQ4_0>(rowp, pr, a, acc);
            }
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (j < nr && sl == 0) L.dst[r0 + j] = acc;
    }
}

__device__ __forceinline__ void give_up(volatile int* abort_flag, unsigned int* abort_word) {
    if (!*abort_flag) record_error(&g_gemv_status, DEV_TIMEOUT);
    *abort_flag = 1;
    atomicExch(abort_word, 1u);
}

__global__ void __launch_bounds__(THREADS, 2)
gemv_chain_kernel(const __grid_constant__ ChainParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);              // full[0..7], empty[8..15]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 128);
    uint8_t* stages = smem + p.stage_off;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grid = gridDim.x;
    const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[MAX_STAGES]);

    if (tid == 0) {
        for (int s = 0; s < p.S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, CONSUMERS / 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CONSUMERS / 32) {
        // ---------------- producer: every link's units, back to back
        if (lane == 0) {
            int k = 0;
            bool stop = false;
            for (int i = 0; i < p.n && !stop; ++i) {
                const ChainLink& L = p.link[i];
                for (int u = blockIdx.x; u < L.n_units; u += grid, ++k) {
                    const int s = k % p.S;
                    if (k >= p.S && !mbar_wait_until(empty0 + 8 * s, ((k / p.S) + 1) & 1, abort_flag, p.limit_ns)) {
                        if (!*abort_flag) give_up(abort_flag, p.abort_word);
                        stop = true;
                        break;
                    }
                    const int r0 = u * L.G;
                    const int nr = min(L.G, L.ne01 - r0);
                    const uint32_t bytes = (uint32_t)nr * (uint32_t)L.row_bytes;
                    mbar_arrive_expect_tx(full0 + 8 * s, bytes);
                    bulk_g2s(smem_u32(stages + (size_t)s * p.stage_bytes), L.w + (int64_t)r0 * L.row_bytes, bytes,
                             full0 + 8 * s);
                }
            }
            // every copy issued lands before the CTA can exit
            for (int k2 = max(0, k - p.S); k2 < k; ++k2)
                mbar_wait_bounded(full0 + 8 * (k2 % p.S), (uint32_t)((k2 / p.S) & 1), p.limit_ns);
        }
        return;
    }

    // ---------------- consumers
    __shared__ int go;
    const uint4* quads = reinterpret_cast<const uint4*>(smem + p.act_off);
    int k = 0;
    for (int i = 0; i < p.n; ++i) {
        const ChainLink& L = p.link[i];
        if (i > 0) {
            // link i - 1 finished in every CTA: its outputs (possibly this link's
            // input) are complete and visible
            if (tid == 0) {
                const bool ok = wait_count(p.done + (i - 1), (unsigned int)grid, p.abort_word, p.limit_ns);
                if (!ok) give_up(abort_flag, p.abort_word);
                go = ok ? 1 : 0;
            }
            consumer_sync();
            if (!go) break;
        }
        {
            ActDst<1> ad;
            ad.base[0] = smem_u32(smem);
            ad.q = (uint32_t)p.act_off;
            ad.d = (uint32_t)(p.act_off + L.np * 64);
            ad.s = (uint32_t)(ad.d + L.nb * 4);
            constexpr int U = 3;
            for (int m0 = 0; m0 < 4 * L.nb; m0 += CONSUMERS * U)
                quantize_acts<1, U, 1, true>(L.x, L.ne00, L.nb, L.np, m0, 4 * L.nb, ad, tid);
        }
        consumer_sync();
        const float* dy = reinterpret_cast<const float*>(smem + p.act_off + L.np * 64);
        const int* sy8 = reinterpret_cast<const int*>(smem + p.act_off + L.np * 64 + L.nb * 4);
        bool ok = true;
        for (int u = blockIdx.x; u < L.n_units; u += grid, ++k) {
            const int s = k % p.S;
            const uint32_t bar = full0 + 8 * s, par = (uint32_t)((k / p.S) & 1);
            int got = 1;
            if (lane == 0) {
                got = mbar_wait_until(bar, par, abort_flag, p.limit_ns) ? 1 : 0;
                if (!got) give_up(abort_flag, p.abort_word);
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) { ok = false; break; }
            mbar_try_wait(bar, par);       // per-lane acquire of the completed phase
            const uint8_t* stage = stages + (size_t)s * p.stage_bytes;
            const int r0 = u * L.G;
            const int nr = min(L.G, L.ne01 - r0);
            switch (L.lpr) {
                case 32: chain_rows<32>(stage, L, r0, nr, quads, dy, sy8, tid); break;
                case 16: chain_rows<16>(stage, L, r0, nr, quads, dy, sy8, tid); break;
                case 8:  chain_rows<8>(stage, L, r0, nr, quads, dy, sy8, tid); break;
                default: chain_rows<4>(stage, L, r0, nr, quads, dy, sy8, tid); break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // all of this CTA's outputs of link i are written (and its activations read)
        consumer_sync();
        if (!ok || *abort_flag) break;
        if (tid == 0 && !(p.fault && i == 0 && blockIdx.x == 0)) {
            __threadfence();
            atomicAdd(p.done + i, 1u);
        }
    }
}

bool plan_chain(const q4q_chain_link* links, int n, const DeviceInfo& info, ChainParams* p, size_t* smem) {
    int64_t act = 0, maxrow = 0;
    for (int i = 0; i < n; ++i) {
        const int64_t np = links[i].ne00 / 64, nb = links[i].ne00 / 32;
        act = std::max<int64_t>(act, np * 64 + nb * 8);
        maxrow = std::max<int64_t>(maxrow, nb * Q4_0_BYTES);
    }
    const int64_t head = 256;
    const int64_t act_bytes = (act + 127) / 128 * 128;
    const int64_t stage = std::max<int64_t>(16384, (maxrow + 127) / 128 * 128);
    // about 113 KB per CTA lets two CTAs share an SM (16 consumer warps), as the GEMV
    // does for its large matrices; otherwise one CTA with what fits
    int64_t S = (113 * 1024 - head - act_bytes) / stage;
    if (S < 3) S = (std::min<int64_t>(info.max_smem_optin, 227 * 1024) - 1024 - head - act_bytes) / stage;
    if (S < 2) return false;
    S = std::min<int64_t>(S, MAX_STAGES);
    p->n = n;
    p->S = (int)S;
    p->stage_bytes = (int)stage;
    p->act_off = (int)head;
    p->stage_off = (int)(head + act_bytes);
    *smem = (size_t)(head + act_bytes + S * stage);
    return true;
}

// Units of each link for a grid of `grid` CTAs: about two per CTA where the rows
// allow, at most one stage each.
void plan_links(const q4q_chain_link* links, int n, int grid, ChainParams* p) {
    for (int i = 0; i < n; ++i) {
        ChainLink& L = p->link[i];
        L.w = static_cast<const uint8_t*>(links[i].src0);
        L.x = links[i].src1;
        L.dst = links[i].dst;
        L.ne00 = (int)links[i].ne00;
        L.nb = L.ne00 / QK;
        L.np = L.nb / 2;
        L.ne01 = (int)links[i].ne01;
        L.row_bytes = L.nb * Q4_0_BYTES;
        int64_t G = (links[i].ne01 + 2 * (int64_t)grid - 1) / (2 * (int64_t)grid);
        G = std::max<int64_t>(1, std::min<int64_t>(G, p->stage_bytes / L.row_bytes));
        L.G = (int)G;
        L.n_units = (int)((links[i].ne01 + G - 1) / G);
        L.lpr = 4;
        for (int c : {32, 16, 8})
            if (L.np % c == 0) { L.lpr = c; break; }
    }
}

}  // namespace

unsigned int chain_take_device_status() { return take_gemv_status_word(); }

size_t chain_workspace_bytes(int n) { return ((size_t)(n + 1) * 4 + 255) / 256 * 256; }

q4q_status chain_check(const q4q_chain_link* links, int n) {
    for (int i = 0; i < n; ++i) {
        const q4q_chain_link& l = links[i];
        if (l.ne00 <= 0 || l.ne00 % 256 != 0 || l.ne00 >= (1 << 20) || l.ne01 <= 0 || l.ne01 >= (1ll << 31))
            return Q4Q_ERR_SHAPE;
        if (!l.src0 || !l.src1 || !l.dst) return Q4Q_ERR_NULL;
        if (!aligned(l.src0, 16) || !aligned(l.src1, 16) || !aligned(l.dst, 4)) return Q4Q_ERR_ALIGN;
    }
    return Q4Q_OK;
}

q4q_status chain_launch(const q4q_chain_link* links, int n, void* workspace, cudaStream_t stream,
                        const DeviceInfo& info, const KernelDebug* dbg) {
    static std::mutex mu;
    static std::map<std::pair<int, size_t>, int> resident;
    ChainParams p{};
    size_t smem = 0;
    if (!plan_chain(links, n, info, &p, &smem)) return Q4Q_ERR_SHAPE;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto key = std::make_pair(info.device, smem);
        auto it = resident.find(key);
        if (it == resident.end()) {
            if (cudaFuncSetAttribute(gemv_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                    cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_chain_kernel, THREADS, smem) !=
                    cudaSuccess) {
                (void)cudaGetLastError();
                return Q4Q_ERR_CUDA;
            }
            resident[key] = per_sm;
        } else {
            per_sm = it->second;
        }
    }
    if (per_sm <= 0) return Q4Q_ERR_CUDA;
    const int grid = per_sm * info.sm_count;
    plan_links(links, n, grid, &p);
    p.done = static_cast<unsigned int*>(workspace);
    p.abort_word = p.done + n;
    p.limit_ns = dbg ? dbg->limit_ns : WAIT_LIMIT_NS;
    p.fault = dbg ? dbg->fault : 0;
    if (cudaMemsetAsync(workspace, 0, (size_t)(n + 1) * 4, stream) != cudaSuccess) return Q4Q_ERR_CUDA;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemv_chain_kernel, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4Q_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace q4q

using namespace q4q;

extern "C" q4q_status q4q_mul_mat_chain_workspace_size(int n, size_t* bytes) {
    if (!bytes) return Q4Q_ERR_NULL;
    if (n < 1 || n > Q4Q_CHAIN_MAX) return Q4Q_ERR_ARG;
    *bytes = chain_workspace_bytes(n);
    return Q4Q_OK;
}

extern "C" q4q_status q4q_mul_mat_chain(const q4q_chain_link* links, int n, int64_t ne11, void* workspace,
                                        size_t workspace_bytes, unsigned int flags, q4q_stream_t stream) {
    if (n < 1 || n > Q4Q_CHAIN_MAX || flags != 0u) return Q4Q_ERR_ARG;
    if (!links) return Q4Q_ERR_NULL;
    if (ne11 != 1) return Q4Q_ERR_SHAPE;
    q4q_status st = chain_check(links, n);
    if (st != Q4Q_OK) return st;
    if (workspace_bytes < chain_workspace_bytes(n)) return Q4Q_ERR_WORKSPACE;
    if (!workspace) return Q4Q_ERR_NULL;
    if (!aligned(workspace, 4)) return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    return chain_launch(links, n, workspace, (cudaStream_t)stream, info, nullptr);
}

// Two-level state passing for the tensor-core path: the states entering the segments of long sequences, computed
// before the fused kernel runs so that its chunk-to-chunk state chain restarts at every segment start.
//
// The state recurrence of the SSD scan is linear, S_t = exp(dt_t A) S_{t-1} + dt_t B_t x_t^T, so it regroups
// over any run of tokens ("Accelerating Mamba2 with Kernel Fusion", state passing step): the state after a block
// of tokens is exp(L_blk) S_before + s_blk with
//   L_blk = sum over the block of dt_t A                                (log of the block's decay)
//   s_blk = sum over the block of exp(cs_end - cs_t) dt_t B_t x_t^T     (cs: inclusive cumsum of dt A)
// This file computes (s_blk, L_blk) for the blocks that precede each sequence's last segment, all blocks in
// parallel, and then chains the block aggregates into the segment entering states.
//
// Block kernel (tcgen05 / TMA). A work unit is (sequence, block of `blk` chunks, `hs` heads of one group). The
// block's chunks are walked from the last to the first; for each chunk and head the decay to the block end folds
// into the x rows, X'_t = w_t x_t with w_t = exp(after + cs_end(c) - cs_t) dt_t, where cs is the chunk-local
// cumsum and `after` the summed dt A of the block's later chunks (so every weight is at most dt_t and the
// exponent never grows), and one accumulator per head in TMEM collects s_blk = sum_c B_c^T X'_c over the whole
// block. Warp roles (512 threads):
//   warp 0       TMA: per chunk the B tile (two 64-column halves), per head the x tile into an 8-deep ring
//   warp 1       TMEM allocator + single-thread tcgen05.mma issuer (M = 128 d_state rows, N = 64, K = 128 tokens)
//   warps 2, 3   B tile halves bf16 -> fp16 in place (fp16 inputs pass straight through)
//   warps 4-7    weight tables, item j by warp 4 + (j mod 4): dt, the chunk cumsum (4 tokens a lane), the
//                within-chunk weights exp(cs_end - cs_t) dt_t and the chunk's summed dt A, into a ring of its own
//   warps 8-11   X' = exp(after) w o x to fp16 in place in the x slot (the MMA's B operand there) for the heads of
//                even index, 12-15 for the odd ones (hs is even, so a warpgroup sees every chunk of its heads, in
//                order, and keeps their running `after`); at the unit end these heads' accumulators and block
//                decays to global memory
// Combine kernel (SIMT): per sequence, head and state element, S <- exp(L_k) S + s_blk_k from the initial state
// over the blocks, storing S at each segment start.
#include <cuda.h>
#include <stddef.h>

#include <type_traits>

#include "sm100_ptx.cuh"
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kQ = 128, kP = 64, kN = 128;
constexpr int kThreadsB = 512;
constexpr int kXR = 8;             // x ring depth (even: each X' warpgroup owns every other slot)
constexpr int kTB = 4;             // weight tables per table warp
constexpr uint32_t kTile = 16384;  // [128 rows x 128 B] 128B-swizzled 16-bit tile
constexpr float kLog2e = 1.4426950408889634f;

struct __align__(1024) SmemB {
    uint8_t b[2][2][kTile];   // per chunk stage: B n[0,64), B n[64,128)
    uint8_t x[kXR][kTile];    // per (chunk, head) item: the x tile, then X' in its place
    float wt[4][kTB][kQ];     // per weight-table warp, a ring of kTB: an item's within-chunk weights
    float tot[4][kTB];        // beside each table: the chunk's summed dt A (log2 units)
    uint64_t b_full[2], b_conv[2], b_empty[2], x_full[kXR], x_conv[kXR], x_empty[kXR];
    uint64_t t_full[4][kTB], t_empty[4][kTB];
    uint64_t acc_full, acc_empty, drain;
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(offsetof(SmemB, x) % 1024 == 0 && offsetof(SmemB, wt) % 16 == 0, "swizzled tiles are 1024-aligned");
static_assert(kXR == 8, "a chunk's items fill consecutive slots for every hs in {2, 4, 8}; X' warpgroup w fills "
                         "the slots of parity w");
static_assert(sizeof(SmemB) + 1024 <= 227 * 1024, "shared memory of one CTA");

__device__ __forceinline__ float ex2f(float v) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// Packed fp32 pair product (one instruction, each lane rounded as a scalar fmul).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}
template <typename IO> __device__ __forceinline__ float2 unpack2(uint32_t v);
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t v) {
    return __half22float2(*reinterpret_cast<__half2 *>(&v));
}
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&v));
}

__device__ __noinline__ void seg_pipe_timeout(int32_t *abort_flag, WsHeader *hdr, uint32_t epoch) {
    *reinterpret_cast<volatile int32_t *>(abort_flag) = 1;
    report_error(hdr, epoch, DEV_PIPE, 0, 0, WAIT_PIPE);
}

// Bounded wait on an intra-CTA mbarrier phase; on timeout it records the error and raises the CTA's abort flag,
// after which every other wait gives up at once.
__device__ __noinline__ bool seg_wait_slow(uint64_t *bar, uint32_t parity, int32_t *abort_flag, WsHeader *hdr,
                                           uint32_t epoch) {
    const uint64_t t0 = globaltimer();
    const uint64_t limit = 4 * (hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs) + 100000000ull;
    for (uint32_t it = 0; it < kMaxSpinIters; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 15u) {
            if (*reinterpret_cast<volatile int32_t *>(abort_flag)) return false;
            if (globaltimer() - t0 > limit) break;
        }
    }
    seg_pipe_timeout(abort_flag, hdr, epoch);
    return false;
}
__device__ __forceinline__ bool seg_wait(uint64_t *bar, uint32_t parity, int32_t *abort_flag, WsHeader *hdr,
                                         uint32_t epoch) {
    return mbar_try_wait(bar, parity) || seg_wait_slow(bar, parity, abort_flag, hdr, epoch);
}

// Opt-in timeline trace (build with -DSSD_TRACE): in CTA 0 lane 0 of every warp records (SM clock, tag).
#ifdef SSD_TRACE
constexpr int kSegTraceRoles = 16, kSegTraceN = 4096;
__device__ unsigned long long g_seg_trace[kSegTraceRoles][kSegTraceN][2];
__device__ unsigned int g_seg_trace_n[kSegTraceRoles];
// (one record stream per warp, written by its lane 0 with a register counter; the counts at the end)
#define STRACE(role, ev, item)                                                                         \
    do {                                                                                               \
        if (blockIdx.x == 0 && trace_i < kSegTraceN) {                                                 \
            g_seg_trace[role][trace_i][0] = clock64();                                                 \
            g_seg_trace[role][trace_i][1] = ((unsigned long long)(ev) << 32) | (unsigned int)(item);   \
        }                                                                                              \
        ++trace_i;                                                                                     \
    } while (0)
#else
#define STRACE(role, ev, item) \
    do {                       \
    } while (0)
#endif

struct Unit {
    int64_t s, k, h0, g;
};
__device__ __forceinline__ Unit unit_of(const Params &p, const SegPlan &sp, int64_t u) {
    const int64_t slices = p.H / sp.hs;
    Unit r;
    r.h0 = (u % slices) * sp.hs;
    r.g = r.h0 / p.heads_per_group;
    r.k = (u / slices) % sp.nblk;
    r.s = u / (slices * sp.nblk);
    return r;
}

template <typename IO>
__global__ void __launch_bounds__(kThreadsB, 1)
    block_state_kernel(const Params p, const SegPlan sp, const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ CUtensorMap map_b) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    SmemB &sm = *reinterpret_cast<SmemB *>(smem_raw + pad);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WsHeader *hdr = p.hdr;
    const uint32_t epoch = ld_relaxed_gpu(&hdr->epoch) + 1u;
    constexpr bool kBf16 = !std::is_same<IO, __half>::value;
    int32_t *abort_flag = &sm.abort;
    const int hs = sp.hs;
    const int64_t units = p.nseq * sp.nblk * (p.H / hs);
    const int64_t blk = sp.blk;
    unsigned int trace_i = 0;  // per-thread trace record counter (trace builds)
    (void)trace_i;
// whole-warp waits are warp-uniform; WAIT1 is the wait of one issuing lane
#define WAITW(bar, par) __all_sync(0xffffffffu, seg_wait((bar), (par), abort_flag, hdr, epoch))
#define WAIT1(bar, par) seg_wait((bar), (par), abort_flag, hdr, epoch)

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.b_full[i], 1);
            mbar_init(&sm.b_conv[i], 2);  // warps 2 and 3, one half each
            mbar_init(&sm.b_empty[i], 1);
        }
        for (int i = 0; i < kXR; ++i) {
            mbar_init(&sm.x_full[i], 1);    // the TMA's bytes
            mbar_init(&sm.x_conv[i], 128);  // X' written in place by the item's warpgroup
            mbar_init(&sm.x_empty[i], 1);   // the MMA has read X'
        }
        // A table warp's items are not consecutive in the x ring, so it cannot use the ring's barriers: a parity
        // wait there could pass on a phase two items early. Each table warp fills a ring of its own instead, in its
        // own item order.
        for (int t = 0; t < 4; ++t)
            for (int j = 0; j < kTB; ++j) {
                mbar_init(&sm.t_full[t][j], 1);
                mbar_init(&sm.t_empty[t][j], 128);
            }
        mbar_init(&sm.acc_full, 1);
        mbar_init(&sm.acc_empty, 256);
        mbar_init(&sm.drain, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&map_x);
            prefetch_tensormap(&map_b);
            uint32_t bc = 0, xc = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < units; u += gridDim.x) {
                const Unit un = unit_of(p, sp, u);
                for (int64_t ci = 0; ok && ci < blk; ++ci) {
                    const int64_t c = un.k * blk + blk - 1 - ci;
                    const int row0 = (int)(un.s * p.L + c * kQ);
                    const uint32_t st = bc & 1;
                    if (!WAIT1(&sm.b_empty[st], ((bc >> 1) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
#ifdef SSD_BOUNDS_CHECK
                    // the tile's rows and group inside the tensor (a failed check skips the copies; the pipeline then
                    // times out and the launch reports the error)
                    if (row0 < 0 || row0 + kQ > p.batch * p.L || un.g >= p.G || un.h0 + hs > p.H) {
                        bounds_hit(hdr, SITE_SEG_TMA, row0);
                        ok = false;
                        break;
                    }
#endif
                    mbar_arrive_expect_tx(&sm.b_full[st], 2 * kTile);
                    tma_load_4d(sm.b[st][0], &map_b, &sm.b_full[st], 0, (int)un.g, row0, 0);
                    tma_load_4d(sm.b[st][1], &map_b, &sm.b_full[st], 64, (int)un.g, row0, 0);
                    STRACE(0, 1, bc);
                    ++bc;
                    for (int hh = 0; hh < hs; ++hh) {
                        const uint32_t k = xc % kXR;
                        if (!WAIT1(&sm.x_empty[k], ((xc / kXR) & 1) ^ 1)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&sm.x_full[k], kTile);
                        tma_load_4d(sm.x[k], &map_x, &sm.x_full[k], 0, (int)(un.h0 + hh), row0, 0);
                        STRACE(0, 2, xc);
                        ++xc;
                    }
                }
            }
            // the copies issued last into every stage and slot have landed before the CTA exits (a consumer that
            // gave up early may not have waited for them)
            for (uint32_t j = 0; j < 2 && j < bc; ++j) {
                const uint32_t b = bc - 1 - j;
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&sm.b_full[b & 1], (b >> 1) & 1) && globaltimer() - t0 < 100000000ull) {
                }
            }
            for (uint32_t j = 0; j < (uint32_t)kXR && j < xc; ++j) {
                const uint32_t x = xc - 1 - j;
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&sm.x_full[x % kXR], (x / kXR) & 1) && globaltimer() - t0 < 100000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (warp-uniform waits) and one elected lane issues the MMAs and commits: a
        // burst issued this way completes sooner than one lane's.
        {
            constexpr uint32_t idST = idesc_f16_f32(128, 64, true, true) & ~(0x3Fu << 17);  // N set per MMA
            const bool leader = elect_one();
            uint32_t bc = 0, uc = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < units; u += gridDim.x, ++uc) {
                if (!WAITW(&sm.acc_empty, (uc & 1) ^ 1)) break;  // the last unit's accumulators have been read
                tc_fence_after();
                if (lane == 0) STRACE(1, 1, uc);
                for (int64_t ci = 0; ok && ci < blk; ++ci, ++bc) {
                    const uint32_t st = bc & 1;
                    if (!WAITW(&sm.b_conv[st], (bc >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) STRACE(1, 4, bc);
                    // every item of the chunk first, then all their MMAs in one burst: any wait or bookkeeping
                    // between two MMAs leaves the tensor pipe idle (it takes about 50 cycles for one)
                    const uint32_t j0 = bc * (uint32_t)hs;  // first item of the chunk in this CTA
                    for (int hh = 0; hh < hs && ok; ++hh)
                        if (!WAITW(&sm.x_conv[(j0 + hh) % kXR], ((j0 + hh) / kXR) & 1)) ok = false;
                    if (!ok) break;
                    if (lane == 0) STRACE(1, 5, j0);
                    tc_fence_after();
                    uint64_t da[8];
#pragma unroll
                    for (uint32_t s = 0; s < 8; ++s) da[s] = desc_sw128(smem_u32(sm.b[st][0]), kTile, 1024) + 128 * s;
                    if (leader) {
                        // up to four heads per MMA: their X' tiles sit in consecutive slots (a chunk's items start on
                        // a multiple of hs, and hs divides the ring), the slot stride is the B operand's stride
                        // between 64-column atoms, and their accumulators are adjacent in TMEM (N = 64 per head)
                        for (int g = 0; g < hs; g += 4) {
                            const int nh = hs - g < 4 ? hs - g : 4;
                            const uint32_t id = idST | ((uint32_t)(64 * nh) >> 3 << 17);
                            const uint64_t dxs = desc_sw128(smem_u32(sm.x[(j0 + g) % kXR]), kTile, 1024);
                            const uint32_t d = tmem + 64 * g;
                            // K step s: 16 tokens = 2048 bytes further
                            mma_ss(d, da[0], dxs, id, ci > 0);
#pragma unroll
                            for (uint32_t s = 1; s < 8; ++s) mma_ss(d, da[s], dxs + 128 * s, id, 1);
                        }
                        for (int hh = 0; hh < hs; ++hh) mma_commit(&sm.x_empty[(j0 + hh) % kXR]);
                        mma_commit(&sm.b_empty[st]);
                    }
                    __syncwarp();
                    if (lane == 0) STRACE(1, 2, j0);
                }
                if (leader) mma_commit(&sm.acc_full);
                __syncwarp();
            }
            // every MMA issued above completes before TMEM is released
            if (leader) {
                mma_commit(&sm.drain);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&sm.drain, 0) && globaltimer() - t0 < 1000000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------------------ B conversion (one half per warp)
        const int half = warp - 2;
        uint32_t bc = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; ok && u < units; u += gridDim.x) {
            for (int64_t ci = 0; ci < blk; ++ci, ++bc) {
                const uint32_t st = bc & 1;
                if (!WAITW(&sm.b_full[st], (bc >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) STRACE(warp, 1, bc);
                if constexpr (kBf16) {
                    uint8_t *t = sm.b[st][half];
#pragma unroll 1
                    for (int r = lane; r < kQ; r += 32) {
                        // row r: its 8 16-byte chunks in place (the swizzle is kept), visited in an order rotated by
                        // the row so that the 8 lanes of a quarter-warp hit 8 different bank groups
                        uint4 v[8];
#pragma unroll
                        for (int lc = 0; lc < 8; ++lc)
                            v[lc] = *reinterpret_cast<const uint4 *>(t + r * 128 + ((lc ^ (r & 7)) << 4));
#pragma unroll
                        for (int lc = 0; lc < 8; ++lc) {
                            uint32_t *wv = reinterpret_cast<uint32_t *>(&v[lc]);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = unpack2<IO>(wv[e]);
                                wv[e] = pack_h2(f.x, f.y);
                            }
                            *reinterpret_cast<uint4 *>(t + r * 128 + ((lc ^ (r & 7)) << 4)) = v[lc];
                        }
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sm.b_conv[st]);
                    STRACE(warp, 2, bc);
                }
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------ weight tables (item j: warp 4 + j mod 4)
        // Per item (chunk ci of the block, walked from the last, head hh): dt = softplus(dt_raw + dt_bias), lane l
        // holding tokens 4 l .. 4 l + 3; cs = chunk-local inclusive cumsum of dt A (log2 units); the weights
        // exp2(cs_end - cs_t) dt_t and the total cs_end into the warp's ring slot r mod kTB, r = j / 4.
        const int tw = warp - 4;
        const IO *dtr = static_cast<const IO *>(p.dt_raw);
        uint32_t xc = 0;  // items before this unit (the unit's items are xc .. xc + blk hs - 1)
        bool ok = true;
        const int64_t nitems = blk * hs;
        for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
            const Unit un = unit_of(p, sp, u);
            // lane hh < hs holds head hh's dt_bias and A log2(e) (broadcast per item by shuffles)
            const float lb = lane < hs ? p.dt_bias[un.h0 + lane] : 0.f;
            const float la = lane < hs ? p.A[un.h0 + lane] * kLog2e : 0.f;
            auto load_raw = [&](int64_t jj, float (&r)[4]) {  // dt_raw of this lane's 4 tokens for local item jj
                const int64_t c = un.k * blk + blk - 1 - jj / hs, hh = jj % hs;
                const int64_t row = un.s * p.L + c * kQ + 4 * lane;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    r[e] = jj < nitems ? to_f32(*chk(dtr, (row + e) * p.H + un.h0 + hh, 1, p.batch * p.L * p.H, hdr,
                                                     SITE_SEG_DT))
                                       : 0.f;
            };
            int64_t jj = (int64_t)((tw - (int)(xc & 3u)) & 3);  // this warp's first local item in the unit
            float raw[4], nxt[4];
            load_raw(jj, raw);
            for (; jj < nitems; jj += 4) {
                load_raw(jj + 4, nxt);  // one item ahead
                const uint32_t j = xc + (uint32_t)jj, r = j >> 2;
                const int hh = (int)(jj % hs);
                const float bias = __shfl_sync(0xffffffffu, lb, hh), Al = __shfl_sync(0xffffffffu, la, hh);
                float dt[4], cum[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dt[e] = softplus_f32(raw[e] + bias);
                    cum[e] = fmaf(dt[e], Al, e ? cum[e - 1] : 0.f);
                }
                float incl = cum[3];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const float excl = incl - cum[3];
                const float end = __shfl_sync(0xffffffffu, incl, 31);
                const float base = end - excl;
                const float4 wv = make_float4(ex2f(base - cum[0]) * dt[0], ex2f(base - cum[1]) * dt[1],
                                              ex2f(base - cum[2]) * dt[2], ex2f(base - cum[3]) * dt[3]);
                if (lane == 0) STRACE(warp, 1, r);
                if (ok && !WAITW(&sm.t_empty[tw][r % kTB], ((r / kTB) & 1) ^ 1)) ok = false;  // slot read
                if (lane == 0) STRACE(warp, 2, r);
                *reinterpret_cast<float4 *>(&sm.wt[tw][r % kTB][4 * lane]) = wv;
                if (lane == 0) sm.tot[tw][r % kTB] = end;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.t_full[tw][r % kTB]);
#pragma unroll
                for (int e = 0; e < 4; ++e) raw[e] = nxt[e];
            }
            xc += (uint32_t)nitems;
        }
    } else {
        // ------------------------------------------------------------ X' warpgroups (w = 0: even items, 1: odd)
        // After a failed wait the loops still run to their ends, with no more waiting, so that every warp meets the
        // same barriers; the error is recorded and the results are discarded by the host.
        const int w = (warp - 8) >> 2;
        const int i = tid - 256 - 128 * w;  // token row of the chunk, and TMEM lane (d_state row) in the epilogue
        const uint32_t lrow = (uint32_t)(32 * (warp & 3)) << 16;
        const int nmine = hs / 2;  // heads w, w + 2, ... of every unit (hs is even)
        uint32_t xc = 0, uc = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++uc) {
            const Unit un = unit_of(p, sp, u);
            float after[4] = {0.f, 0.f, 0.f, 0.f};  // per own head: summed dt A (log2) of the chunks already done
            for (uint32_t xj = xc + (uint32_t)w; xj < xc + (uint32_t)(blk * hs); xj += 2) {
                const uint32_t xk = xj % kXR;
                const uint32_t t = xj & 3, r = xj >> 2;  // the item's table: warp t, its r-th item
                const int m = (int)((xj - xc) % (uint32_t)hs) >> 1;  // this warpgroup's head index
                if (lane == 0) STRACE(warp, 2, xj);
                if (ok && !WAITW(&sm.x_full[xk], (xj / kXR) & 1)) ok = false;
                if (ok && !WAITW(&sm.t_full[t][r % kTB], (r / kTB) & 1)) ok = false;
                if (lane == 0) STRACE(warp, 3, xj);
                float am = after[0];
#pragma unroll
                for (int e = 1; e < 4; ++e) am = m == e ? after[e] : am;
                const float wt = sm.wt[t][r % kTB][i] * ex2f(am), end = sm.tot[t][r % kTB];
#pragma unroll
                for (int e = 0; e < 4; ++e) after[e] += m == e ? end : 0.f;
                uint8_t *xr = sm.x[xk] + i * 128;
                // X' in place (same 16-byte positions: the swizzle carries over); the 8 chunks of the row are read
                // first, in an order rotated by the row so that the 8 threads of a quarter-warp hit 8 bank groups
                uint4 a[8];
#pragma unroll
                for (int lc = 0; lc < 8; ++lc) a[lc] = *reinterpret_cast<const uint4 *>(xr + ((lc ^ (i & 7)) << 4));
                mbar_arrive(&sm.t_empty[t][r % kTB]);  // the weight is in a register
                const float2 w2 = make_float2(wt, wt);
#pragma unroll
                for (int lc = 0; lc < 8; ++lc) {
                    uint32_t *av = reinterpret_cast<uint32_t *>(&a[lc]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = fmul2(unpack2<IO>(av[e]), w2);
                        av[e] = pack_h2(f.x, f.y);
                    }
                    *reinterpret_cast<uint4 *>(xr + ((lc ^ (i & 7)) << 4)) = a[lc];
                }
                fence_proxy_async_smem();
                mbar_arrive(&sm.x_conv[xk]);
                if (lane == 0) STRACE(warp, 4, xj);
            }
            xc += (uint32_t)(blk * hs);
            // epilogue: the heads of this warpgroup's parity, accumulator row i (d_state index) to s_blk [.., P, N]
            if (ok && !WAITW(&sm.acc_full, uc & 1)) ok = false;
            tc_fence_after();
            if (lane == 0) STRACE(warp, 5, uc);
            const int64_t base = (un.s * sp.nblk + un.k) * p.H;
            for (int m = 0; m < nmine; ++m) {
                const int hh = w + 2 * m;
                float *dst = chk(sp.blk_s, (base + un.h0 + hh) * (int64_t)(kP * kN) + i, (kP - 1) * kN + 1,
                                 p.nseq * sp.nblk * p.H * kP * kN, hdr, SITE_SEG_BLK);
                if (i == 0) {  // the block decay of this head
                    float am = after[0];
#pragma unroll
                    for (int e = 1; e < 4; ++e) am = m == e ? after[e] : am;
                    *chk(sp.blk_L, base + un.h0 + hh, 1, p.nseq * sp.nblk * p.H, hdr, SITE_SEG_DECAY) = am;
                }
#pragma unroll 1
                for (int pc = 0; pc < 4; ++pc) {
                    uint32_t r[16];
                    tmem_ld16(tmem + lrow + 64 * hh + 16 * pc, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) __stcg(dst + (16 * pc + e) * kN, __uint_as_float(r[e]));
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.acc_empty);
            if (lane == 0) STRACE(warp, 6, uc);
        }
    }
#undef WAITW
#undef WAIT1
#ifdef SSD_TRACE
    if (blockIdx.x == 0 && lane == 0) g_seg_trace_n[warp] = trace_i;
#endif

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// S <- exp2(L_k) S + s_blk_k over each sequence's blocks from its initial state; S stored at every segment start.
// Block (x, y): state elements 1024 x .. 1024 x + 1023 of the (sequence, head) pairs y, y + gridDim.y, ..., four
// consecutive ones a thread (16-byte loads and stores); the loads of eight blocks are issued before their FMAs, so
// the chain over the blocks waits for memory once per eight. (One element a thread left 4 waves of CTAs at 4 per
// SM: 17.6 us on the 16K-token layer in 8 segments.)
template <typename ST>
__global__ void __launch_bounds__(256) combine_kernel(const Params p, const SegPlan sp) {
    constexpr int64_t pn = kP * kN;
    const int pe = (blockIdx.x * 256 + threadIdx.x) * 4;
    const int bps = (int)(p.seg_chunks / sp.blk);  // blocks per segment
    const int nblk = (int)sp.nblk;
    const ST *init = static_cast<const ST *>(p.init);
    float *out = const_cast<float *>(p.seg_states);
    const int64_t nblk_el = p.nseq * sp.nblk * p.H;  // extents (bounds-checked builds)
    for (int64_t sh = blockIdx.y; sh < p.nseq * p.H; sh += gridDim.y) {
        const int64_t s = sh / p.H, h = sh % p.H;
        float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
        if (init) {  // scalar loads: the caller's initial states carry no alignment promise beyond the element's
            const ST *i0 = chk(init, sh * pn + pe, 4, p.nseq * p.H * pn, p.hdr, SITE_SEG_INIT);
            S = make_float4(to_f32(i0[0]), to_f32(i0[1]), to_f32(i0[2]), to_f32(i0[3]));
        }
        const int64_t b0 = s * sp.nblk * p.H + h;  // block k of this pair: b0 + k H
        float *o = out + (s * (p.nseg - 1) * p.H + h) * pn + pe;  // segment g + 1: o + g H pn
        int seg = 0, kk = 0;
        for (int k0 = 0; k0 < nblk; k0 += 8) {
            float4 v[8];
            float a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t bk = b0 + (int64_t)(k0 + j) * p.H;
                const bool in = k0 + j < nblk;
                v[j] = in ? __ldcs(reinterpret_cast<const float4 *>(
                                chk(sp.blk_s, bk * pn + pe, 4, nblk_el * pn, p.hdr, SITE_SEG_BLK)))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
                a[j] = in ? __ldg(chk(sp.blk_L, bk, 1, nblk_el, p.hdr, SITE_SEG_DECAY)) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (k0 + j >= nblk) break;
                const float e = exp2f(a[j]);
                S = make_float4(fmaf(e, S.x, v[j].x), fmaf(e, S.y, v[j].y), fmaf(e, S.z, v[j].z), fmaf(e, S.w, v[j].w));
                if (++kk == bps) {
                    kk = 0;
                    *reinterpret_cast<float4 *>(chk(o, (int64_t)seg * p.H * pn, 4,
                                                    p.nseq * (p.nseg - 1) * p.H * pn - ((o - out)), p.hdr,
                                                    SITE_SEG_STATE)) = S;
                    ++seg;
                }
            }
        }
    }
}

// 4-D map over a [1, T, mid, inner] 16-bit tensor, box [1, 128 rows, 1, 64 inner], 128B swizzle.
bool make_map4(CUtensorMap *m, const void *base, bool bf16, int64_t inner, int64_t mid, int64_t T, int64_t ld) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)mid, (cuuint64_t)T, 1};
    const cuuint64_t strides[3] = {(cuuint64_t)(inner * 2), (cuuint64_t)(ld * 2), (cuuint64_t)(ld * T * 2)};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kQ, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(base),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename IO>
cudaError_t launch_blocks(const Params &p, const SegPlan &sp, int sms, cudaStream_t stream) {
    CUtensorMap mx, mb;
    const bool bf = !std::is_same<IO, __half>::value;
    const int64_t T = p.batch * p.L;
    if (!make_map4(&mx, p.x, bf, kP, p.H, T, p.x_ld) || !make_map4(&mb, p.B, bf, kN, p.G, T, p.bc_ld))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(SmemB) + 1024;
    auto k = block_state_kernel<IO>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t units = p.nseq * sp.nblk * (p.H / sp.hs);
    k<<<(unsigned)std::min<int64_t>(units, sms), kThreadsB, smem, stream>>>(p, sp, mx, mb);
    return cudaGetLastError();
}

}  // namespace

// Segments and blocks for a regular batch, or nseg = 1 (one chain per sequence). The fused kernel is bounded by
// the larger of two times: its per-head cadence spread over the SMs (about 2.3 us per head and chunk) and the
// serial state chain of a sequence (about 2.4 us per chunk to chunk hop). Two-level passing costs a block pass
// over most of x (about 0.9 us per head and chunk on an SM) and two more launches, so it is taken only where the
// launch is long (at least 256 heads x chunks per SM) and the chain is at least 1.5 times the cadence time, or,
// on shorter launches with fp32 states (a hop of about 3 us: flag, then data), at least 2.2 times (the 8K-token
// batch-1 layer: 4 segments of 16 chunks, 0.168 against 0.193 ms; the 130M-shaped batch, at 2.1 times, is 8 %
// slower segmented), and with fp16 states at least 1.8 times (the 16K-token layer, at 1.98: 8 segments of 16
// chunks with per-head flags, 0.279 against 0.293 ms; the 130M-shaped batch, at 1.67, 6-22 % slower);
// segments are then cut so that a segment's chain takes at most half the cadence time, rounded up to a multiple
// of 8 chunks (measured on the 2.7B-shaped 256K-token sequence with fp32 states: 4
// segments of 512 chunks 3.55 ms, 5 of 410 3.70, 6 of 342 3.64, 8 of 256 3.74, 2 of 1024 3.74). A segment with
// no block length in [min(segment, 8), 32] keeps one chain. A block holds at least
// min(segment, 8) chunks, so that its
// aggregate (32 KB a head) costs at most a quarter of the x it reads; among such blocks and the head counts per
// unit (2, 4 or 8 dividing the heads per group: a chunk's heads then fill consecutive ring slots and share MMAs
// of up to N = 256, and each X' warpgroup owns half of them; groups of an odd number of heads keep one chain per
// sequence), the first pair, by more heads then longer blocks, that gives every SM two block units, else the pair
// with the most units.
SegChoice choose_segments(int64_t nseq, int64_t nc, int64_t H, int64_t G, int sms, int64_t forced, bool fp32_states) {
    SegChoice r{1, nc, 0, 0, 1};
    if (nseq < 1 || nc < 2 || sms < 1) return r;
    int64_t seg;
    if (forced >= 0) {
        if (forced == 0 || forced >= nc) return r;
        seg = forced;
    } else {
        const double per_sm = (double)nseq * (double)nc * (double)H / sms, cadence_us = per_sm * 2.3;
        // long launches: a chain at least 1.5 x the cadence time; shorter ones (the block pass and two more
        // launches weigh more) only with fp32 states, whose hop (flag, then data) costs about 3 us, and a chain at
        // least 2.2 x the cadence time
        const bool long_launch = per_sm >= 256.0 && (double)nc * 2.4 >= 1.5 * cadence_us;
        const bool short_fp32 = per_sm < 256.0 && fp32_states && (double)nc * 3.0 >= 2.2 * cadence_us;
        // shorter fp16 launches: their segmented chains take per-head flags (plain halves, no tagged words)
        const bool short_fp16 = per_sm < 256.0 && !fp32_states && (double)nc * 2.4 >= 1.8 * cadence_us;
        if (!long_launch && !short_fp32 && !short_fp16) return r;
        // fp16 states: segments half as long (their chains run with per-head flags, which want many of them)
        const int64_t seg_max = (int64_t)(cadence_us / ((fp32_states ? 2.0 : 4.0) * 2.4));
        if (seg_max >= nc || seg_max < 8) return r;
        const int64_t nseg0 = (nc + seg_max - 1) / seg_max;
        seg = (nc + nseg0 - 1) / nseg0;
        seg = (seg + 7) / 8 * 8;  // a multiple of 8: blocks of 8 chunks always divide it
    }
    r.nseg = (nc + seg - 1) / seg;
    if (r.nseg < 2) return SegChoice{1, nc, 0, 0, 1};
    r.seg_chunks = seg;
    const int64_t hpg = H / G, min_blk = std::min<int64_t>(seg, 8);
    int64_t best_units = -1;
    bool found = false;
    if (hpg % 2) return SegChoice{1, nc, 0, 0, 1};  // the block kernel takes an even number of heads
    for (int hs = 8; hs >= 2 && !found; hs /= 2) {
        if (hpg % hs) continue;
        for (int64_t blk = std::min<int64_t>(32, seg); blk >= min_blk; --blk) {
            if (seg % blk) continue;
            const int64_t units = nseq * (r.nseg - 1) * (seg / blk) * (H / hs);
            if (units >= 2 * (int64_t)sms) {
                r.hs = hs;
                r.blk = blk;
                found = true;
                break;
            }
            if (units > best_units) {
                best_units = units;
                r.hs = hs;
                r.blk = blk;
            }
        }
    }
    if (r.blk < 1) return SegChoice{1, nc, 0, 0, 1};  // no divisor of the segment in [min_blk, 32]: one chain
    r.nblk = (r.nseg - 1) * (seg / r.blk);
    return r;
}

cudaError_t launch_segstate(const Params &p, const SegPlan &sp, int io_dtype, int state_dtype, int sms,
                            cudaStream_t stream) {
    if (p.nseg < 2 || sp.nblk < 1 || (sp.hs != 2 && sp.hs != 4 && sp.hs != 8) || p.H % sp.hs ||
        p.heads_per_group % sp.hs || p.seg_chunks % sp.blk)
        return cudaErrorInvalidValue;
    cudaError_t e = io_dtype == 1 ? launch_blocks<__nv_bfloat16>(p, sp, sms, stream)
                                  : launch_blocks<__half>(p, sp, sms, stream);
    if (e != cudaSuccess) return e;
    const dim3 grid(kP * kN / 1024, (unsigned)std::min<int64_t>(p.nseq * p.H, 65535));
    if (state_dtype == 0)
        combine_kernel<float><<<grid, 256, 0, stream>>>(p, sp);
    else
        combine_kernel<__half><<<grid, 256, 0, stream>>>(p, sp);
    return cudaGetLastError();
}

}  // namespace ssd

#ifdef SSD_TRACE
extern "C" __attribute__((visibility("default"))) int ssd_seg_trace_read(unsigned long long *dst, unsigned int *counts) {
    if (cudaMemcpyFromSymbol(counts, ssd::g_seg_trace_n, sizeof(ssd::g_seg_trace_n)) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(dst, ssd::g_seg_trace, sizeof(ssd::g_seg_trace)) != cudaSuccess) return -1;
    static const unsigned int zero[ssd::kSegTraceRoles] = {};
    return cudaMemcpyToSymbol(ssd::g_seg_trace_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}
#endif

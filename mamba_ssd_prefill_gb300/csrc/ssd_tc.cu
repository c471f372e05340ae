// Tensor-core (tcgen05 / TMEM / TMA) kernel of the fused SSD prefill forward,
// bf16 or fp16 I/O, headdim P = 64, d_state N = 128, chunk Q = 128.
//
// One persistent CTA per SM pulls work units (chunk c, batch b, group g, slice
// of `hs` heads of that group) from an atomic ticket in chunk-major order and
// runs the five SSD steps of "Accelerating Mamba2 with Kernel Fusion" (chunk
// cumsum, BMM, chunk state, state passing, chunk scan) for them:
//
//   CB      = C_c B_c^T                       (tcgen05, once per unit, TMEM)
//   P       = CB o exp(segsum(dt*A)) o dt_j   (+ D on the diagonal; fp16 in TMEM)
//   y_intra = P x_c                           (tcgen05, A operand from TMEM)
//   s_c     = B_c^T (exp(cs_last - cs_j) dt_j x_j)   (decay applied to x, the
//                                             inner dimension of the contraction)
//   S_c+1   = exp(cs_last) S_c + s_c          (flag-ordered chain across CTAs)
//   y       = y_intra + exp(cs_i) C_c S_c     (tcgen05 C.S, fused epilogue)
//
// Warp roles (352 threads):
//   warp 0      unit loader (tickets, dt_raw, B/C tiles by TMA), up to two units ahead
//   warp 10     x-tile loader (one TMA per head)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2-5   "math": X_s (and the x tile to fp16), decay mask P -> TMEM, epilogue
//               y = y_intra + exp(cs) y_inter staged in shared memory, TMA-stored
//   warps 6-9   "chain": state passing (wait flag, S_in, S_out, publish), S_in
//               -> shared memory as the C.S operand, final states
// All MMA operands are fp16 (bf16 inputs are converted on chip; the contractions
// with P, X_s and S need fp16's 11-bit significand to hold 1e-2).
//
// TMEM (512 columns): CB [0,128), P / y_inter x2 [128,256), y_intra x2
// [256,384), chunk state s x2 [384,512).
#include <cuda.h>

#include <type_traits>

#include "sm100_ptx.cuh"
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kQ = 128;
constexpr int kP = 64;
constexpr int kN = 128;
constexpr int kMaxHs = 8;
constexpr int kThreads = 352;
constexpr int kXWarp = 10;  // x-tile loader warp
constexpr uint32_t kTile = 16384;  // [128 rows x 128 B] 128B-swizzled 16-bit tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kColCB = 0, kColP = 128, kColYI = 256, kColS = 384;
constexpr uint32_t kBarMath = 1;  // named barrier of the math warpgroup (0 is __syncthreads)

struct Sched {
    int32_t valid, s, c, g, h0, rows, row0, last;  // row0: the chunk's first token on the packed token axis
};

struct __align__(1024) Smem {
    uint8_t bc[2][4][kTile];   // per unit stage: B n[0,64), B n[64,128), C n[0,64), C n[64,128)
    uint8_t x[2][kTile];       // per head buffer: x tile (fp16 after conversion)
    uint8_t xs[2][kTile];      // per head buffer: X_s, then S_in (fp16, C.S operand)
    uint8_t xhalo[2][384];     // fused convolution: the 3 raw x rows before the chunk, dense [3][64] 16-bit
    float4 xtap[2][kP];        // fused convolution: the head's taps per x channel (tap 3 on the current token)
    float xbias[2][kP];        //                    and its bias
    float cs2[2][kMaxHs][kQ];  // raw dt_raw from the producer, then log2(e) * cumsum(dt*A)
    float dt[2][kMaxHs][kQ];   // dt
    float wt[2][kMaxHs][kQ];   // exp(cs_anchor(j) - cs_j) dt_j, anchor(j) = last row of j's 32-row block
    float dskip[2][kMaxHs];    // D of the unit's heads (0 when absent)
    Sched sched[2];
    uint64_t sched_full[2], bc_full[2], bc_conv[2], bc_empty[2], cb_full, cb_empty, unit_go;
    uint64_t x_full[2], x_empty[2], p_full[2], mma1[2], s_free[2], sin_full[2], mma2[2], drain;
    uint32_t tmem_base;
    int32_t abort;
};

// Opt-in timeline trace (build with -DSSD_TRACE): CTA 0 records (%globaltimer, tag) per role.
#ifdef SSD_TRACE
constexpr int kTraceN = 8192;
__device__ unsigned long long g_trace[4][kTraceN][2];
__device__ unsigned int g_trace_n[4];
// one tracing thread per role keeps its own counter (no atomics: recording must not perturb the timeline)
#define TRACE(role, tag)                                                                   \
    do {                                                                                   \
        if (blockIdx.x == 0 && trace_i < kTraceN) {                                        \
            g_trace[role][trace_i][0] = globaltimer();                                     \
            g_trace[role][trace_i][1] = (unsigned long long)(tag);                         \
            ++trace_i;                                                                     \
            g_trace_n[role] = trace_i;                                                     \
        }                                                                                  \
    } while (0)
#else
#define TRACE(role, tag) \
    do {                 \
    } while (0)
#endif

__device__ __forceinline__ float ex2(float v) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Plain C++ shared-memory vector accesses, so the compiler can batch and overlap them; their
// ordering against TMA, tensor-core reads and barriers comes from those operations' volatile asm
// (memory clobbers) and from the proxy fences.
__device__ __forceinline__ uint4 lds128(const void *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ void sts128(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <typename IO> __device__ __forceinline__ uint32_t pack_io(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack_io<__half>(float lo, float hi) { return pack_f16(lo, hi); }
template <> __device__ __forceinline__ uint32_t pack_io<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <typename IO> __device__ __forceinline__ float2 unpack_io(uint32_t v);
template <> __device__ __forceinline__ float2 unpack_io<__half>(uint32_t v) {
    return __half22float2(*reinterpret_cast<__half2 *>(&v));
}
template <> __device__ __forceinline__ float2 unpack_io<__nv_bfloat16>(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&v));
}
__device__ __forceinline__ float2 unpack_f16(uint32_t v) { return __half22float2(*reinterpret_cast<__half2 *>(&v)); }

// ---------------------------------------------------------------- fused depthwise convolution (width 4)
// SiLU with one special-function op: v sigmoid(v) = h + h tanh(h) with h = v / 2, tanh by tanh.approx.f32 (the
// form of the separate conv kernel, so both paths round alike).
__device__ __forceinline__ float silu_fast(float v) {
    const float h = 0.5f * v;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

// The 3 raw inputs before token row0 of channels ch, ch + 1 (h[j] = token row0 - 3 + j): the rows themselves inside
// the sequence (which starts at token tok0), else the conv cache of sequence s, else zeros.
template <typename IO>
__device__ __forceinline__ void conv_halo(const Params &p, int64_t s, int64_t tok0, int64_t row0, int64_t ch,
                                          float (&h)[3][2]) {
    const IO *xraw = static_cast<const IO *>(p.x);
    const IO *st = static_cast<const IO *>(p.conv_state);
    const int64_t nx = p.batch * p.L * p.x_ld, nst = p.nseq * p.x_ld * 3;  // extents (bounds-checked builds)
    (void)nx;
    (void)nst;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int64_t tok = row0 - 3 + j;
        if (tok >= tok0) {
            const float2 f = unpack_io<IO>(
                *reinterpret_cast<const uint32_t *>(chk(xraw, tok * p.x_ld + ch, 2, nx, p.hdr, SITE_CONV_IN)));
            h[j][0] = f.x;
            h[j][1] = f.y;
        } else if (st) {
            h[j][0] = to_f32(*chk(st, (s * p.x_ld + ch) * 3 + 3 + (tok - tok0), 1, nst, p.hdr, SITE_CONV_STATE));
            h[j][1] = to_f32(*chk(st, (s * p.x_ld + ch + 1) * 3 + 3 + (tok - tok0), 1, nst, p.hdr, SITE_CONV_STATE));
        } else {
            h[j][0] = h[j][1] = 0.f;
        }
    }
}

// Causal width-4 convolution in place over a [128 rows x 64 channels] 128B-swizzled 16-bit tile (1024-aligned); lane
// owns channels 2 lane, 2 lane + 1 and walks the rows with the last 3 inputs in registers; results are fp16.
template <typename IO>
__device__ __forceinline__ void conv_tile(uint8_t *tile, const float4 w0, const float4 w1, float b0, float b1,
                                          float (&h)[3][2], bool silu, int lane) {
    const int lc = lane >> 2, wo = (lane & 3) * 4;
#pragma unroll 1
    for (int r0 = 0; r0 < kQ; r0 += 8) {
        uint32_t raw[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) raw[u] = *reinterpret_cast<const uint32_t *>(tile + (r0 + u) * 128 + ((lc ^ u) << 4) + wo);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float2 v = unpack_io<IO>(raw[u]);
            float o0 = fmaf(w0.w, v.x, fmaf(w0.z, h[2][0], fmaf(w0.y, h[1][0], fmaf(w0.x, h[0][0], b0))));
            float o1 = fmaf(w1.w, v.y, fmaf(w1.z, h[2][1], fmaf(w1.y, h[1][1], fmaf(w1.x, h[0][1], b1))));
            if (silu) {
                o0 = silu_fast(o0);
                o1 = silu_fast(o1);
            }
            *reinterpret_cast<uint32_t *>(tile + (r0 + u) * 128 + ((lc ^ u) << 4) + wo) = pack_f16(o0, o1);
            h[0][0] = h[1][0];
            h[0][1] = h[1][1];
            h[1][0] = h[2][0];
            h[1][1] = h[2][1];
            h[2][0] = v.x;
            h[2][1] = v.y;
        }
    }
}

__device__ __noinline__ void chain_timeout(WsHeader *hdr, uint32_t epoch, uint32_t chunk) {
    report_error(hdr, epoch, DEV_TIMEOUT, 0, chunk, WAIT_CHAIN);
}

// fp16 state ring vector: two 8-byte words, each two fp16 values and a 32-bit tag, each word single-copy atomic
// (aligned, relaxed, gpu scope).
__device__ __forceinline__ ulonglong2 ld_ring(const ulonglong2 *p) {
    ulonglong2 r;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(r.x), "=l"(r.y) : "l"(p) : "memory");
    return r;
}
__device__ __forceinline__ void st_ring(ulonglong2 *p, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

// Bounded wait until both words of the ring vector *p carry the tag `want` (the producer writes this vector of a
// row last). On timeout records SSD_ERR_TIMEOUT and returns false; returns false at once when another CTA aborted
// the launch. Out of line: it is the slow path.
__device__ __noinline__ bool wait_ring(const ulonglong2 *p, uint32_t want, uint32_t epoch, WsHeader *hdr,
                                       uint64_t limit_ns, uint32_t chunk) {
    const uint64_t t0 = globaltimer();
    uint32_t sleep_ns = 16;
    for (uint32_t it = 0; it < kMaxSpinIters; ++it) {
        const ulonglong2 v = ld_ring(p);
        if ((uint32_t)(v.x >> 32) == want && (uint32_t)(v.y >> 32) == want) return true;
        if ((it & 7u) == 7u) {
            if (aborted(hdr, epoch)) return false;
            if (globaltimer() - t0 > limit_ns) break;
        }
        __nanosleep(sleep_ns);
        if (sleep_ns < 64) sleep_ns += 16;
    }
    chain_timeout(hdr, epoch, chunk);
    return false;
}

// Bounded wait until *tag == want (acquire). On timeout records SSD_ERR_TIMEOUT and returns false;
// returns false at once when another CTA aborted the launch. Out of line: it is the slow path.
__device__ __noinline__ bool wait_tag(const uint64_t *tag, uint64_t want, uint32_t epoch, WsHeader *hdr,
                                         uint64_t limit_ns, uint32_t chunk) {
    const uint64_t t0 = globaltimer();
    uint32_t sleep_ns = 20;
    for (uint32_t it = 0; it < kMaxSpinIters; ++it) {
        if (ld_acquire_u64(tag) == want) return true;
        if ((it & 7u) == 7u) {
            if (aborted(hdr, epoch)) return false;
            if (globaltimer() - t0 > limit_ns) break;
        }
        __nanosleep(sleep_ns);
        if (sleep_ns < 160) sleep_ns += 20;
    }
    chain_timeout(hdr, epoch, chunk);
    return false;
}

__device__ __noinline__ void pipe_timeout(Smem &sm, WsHeader *hdr, uint32_t epoch) {
    *reinterpret_cast<volatile int32_t *>(&sm.abort) = 1;
    report_error(hdr, epoch, DEV_PIPE, 0, 0, WAIT_PIPE);
}

// Bounded wait on an intra-CTA mbarrier phase. On timeout (a broken pipeline)
// it records the error, raises the CTA abort flag and returns false; every
// other wait then gives up too and the CTA drains to its teardown. Its limit
// is four times the state-passing limit plus 100 ms: a pipeline stage may
// legitimately sit behind one full state-passing wait, which must time out
// (and report itself) first. Only the first probe is inline: the polling loop
// is one out-of-line copy, so the hot code of every role stays small.
__device__ __noinline__ bool bwait_slow(uint64_t *bar, uint32_t parity, Smem &sm, WsHeader *hdr, uint32_t epoch) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; it < kMaxSpinIters; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 15u) {
            if (*reinterpret_cast<volatile int32_t *>(&sm.abort)) return false;
            const uint64_t limit = 4 * (hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs) + 100000000ull;
            if (globaltimer() - t0 > limit) break;
        }
    }
    pipe_timeout(sm, hdr, epoch);
    return false;
}
__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t parity, Smem &sm, WsHeader *hdr, uint32_t epoch) {
    return mbar_try_wait(bar, parity) || bwait_slow(bar, parity, sm, hdr, epoch);
}

template <typename IO, typename ST, bool CONV>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const Params p, const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_b,
              const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_y,
              const __grid_constant__ CUtensorMap map_xh, const int hs) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base (128B-swizzle atoms). Computed as smem_raw + pad, not through an integer
    // round trip, so the compiler keeps the shared address space and emits LDS/STS for every access.
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw + pad);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WsHeader *hdr = p.hdr;
    const uint32_t epoch = ld_relaxed_gpu(&hdr->epoch) + 1u;
    constexpr bool kBf16 = sizeof(IO) == 2 && !std::is_same<IO, __half>::value;
    unsigned int trace_i = 0;  // per-thread trace record counter (SSD_TRACE builds)
    (void)trace_i;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.sched_full[i], 1);
            mbar_init(&sm.bc_full[i], 1);
            mbar_init(&sm.bc_conv[i], 1);
            mbar_init(&sm.bc_empty[i], 1);
            mbar_init(&sm.x_full[i], 1);
            mbar_init(&sm.x_empty[i], 1);
            mbar_init(&sm.p_full[i], 1);
            mbar_init(&sm.mma1[i], 1);
            mbar_init(&sm.s_free[i], 128);   // every chain thread arrives
            mbar_init(&sm.sin_full[i], 128);
            mbar_init(&sm.mma2[i], 1);
        }
        mbar_init(&sm.cb_full, 1);
        mbar_init(&sm.unit_go, 1);
        mbar_init(&sm.cb_empty, 1);
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
    const int64_t slices = p.heads_per_group / hs;

    if (warp == 0) {
        // ------------------------------------------------------------ unit loader
        // Per unit: ticket, dt_raw rows, B/C tiles by TMA; and, for the unit requested one iteration earlier
        // (so its TMA latency is already behind it), the bf16 -> fp16 conversion of B/C in place (same 16-bit
        // positions, same swizzle) and the chunk cumsum tables of its heads. Tickets are fetched one unit ahead,
        // or, when the state chain bounds the launch (few units per chunk index), only once the unit before is
        // three heads from its end: a ticket taken early sits on a CTA that is busy for a whole unit more, and
        // the chain reaching that chunk waits for it; late tickets follow the order in which CTAs free up.
        if (lane == 0) {
            prefetch_tensormap(&map_b);
            prefetch_tensormap(&map_c);
        }
        const IO *dtr = static_cast<const IO *>(p.dt_raw);
        int armed_bc = 0;  // for the drain at teardown
        uint32_t bc_par[2] = {0, 0};
        uint32_t t = 0;
        if (lane == 0) t = atomicAdd(&hdr->ticket, 1u);
        t = __shfl_sync(0xffffffffu, t, 0);
        Sched prev{0, 0, 0, 0, 0, 0, 0, 0};
        const uint32_t total = total_units(p, (uint32_t)(p.G * slices));
        const bool late = p.tc_late_ticket != 0;
        const int64_t ndt = p.batch * p.L * p.H;  // dt_raw extent (bounds-checked builds)
#ifdef SSD_BOUNDS_CHECK
        const int64_t probe = hdr->bounds_probe ? ndt : 0;  // test hook: plant the dt rows one extent further
#else
        const int64_t probe = 0;
#endif
        bool ok = true;
        // conversion + tables of the unit in stage uu (whose tiles were requested earlier)
        auto finish = [&](uint32_t vv, const Sched &sc) -> bool {
            const uint32_t uu = vv & 1;
            if (!bwait(&sm.bc_full[uu], (vv >> 1) & 1, sm, hdr, epoch)) return false;
            if constexpr (CONV) {  // B, C: the raw tiles convolved in place (fp16 out), halo from the rows or the cache
                const int64_t tok0 = sc.row0 - (int64_t)sc.c * kQ;
#pragma unroll 1
                for (int t = 0; t < 4; ++t) {
                    const int64_t ch = p.conv_hp + (t >= 2 ? p.G * kN : 0) + (int64_t)sc.g * kN + (t & 1) * 64 + 2 * lane;
                    const float4 w0 = *reinterpret_cast<const float4 *>(p.conv_w + ch * 4);
                    const float4 w1 = *reinterpret_cast<const float4 *>(p.conv_w + (ch + 1) * 4);
                    const float b0 = p.conv_b ? p.conv_b[ch] : 0.f, b1 = p.conv_b ? p.conv_b[ch + 1] : 0.f;
                    float hv[3][2];
                    conv_halo<IO>(p, sc.s, tok0, sc.row0, ch, hv);
                    conv_tile<IO>(sm.bc[uu][t], w0, w1, b0, b1, hv, p.conv_silu != 0, lane);
                }
            } else if (kBf16) {
#pragma unroll 1
                for (int it = 0; it < 16; ++it) {  // 4 tiles x 4 rows per lane
                    const int row = lane + 32 * (it & 3);
                    uint8_t *base = sm.bc[uu][it >> 2] + row * 128;
                    uint4 w[8];
                    // chunk order rotated by row: the lanes of a quarter-warp hit 8 different bank groups
#pragma unroll
                    for (int lc = 0; lc < 8; ++lc) w[lc] = lds128(base + ((lc ^ (row & 7)) << 4));
#pragma unroll
                    for (int lc = 0; lc < 8; ++lc) {
                        uint32_t *wv = reinterpret_cast<uint32_t *>(&w[lc]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_io<IO>(wv[e]);
                            wv[e] = pack_f16(f.x, f.y);
                        }
                        sts128(base + ((lc ^ (row & 7)) << 4), w[lc]);
                    }
                }
            }
            // chunk cumsum: dt = softplus(dt_raw + dt_bias) (0 past the sequence end), inclusive scan of
            // dt*A over the 128 rows; this lane owns rows 4*lane .. 4*lane+3
#pragma unroll 1
            for (int hh = 0; hh < kMaxHs; ++hh) {
                if (hh < hs) {
                    const int h = sc.h0 + hh;
                    const float bias = p.dt_bias[h], Ah = p.A[h];
                    float dtv[4], cum[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int row = 4 * lane + jj;
                        dtv[jj] = row < sc.rows ? softplus_f32(sm.cs2[uu][hh][row] + bias) : 0.f;
                        cum[jj] = dtv[jj] * Ah + (jj ? cum[jj - 1] : 0.f);
                    }
                    float incl = cum[3];
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float w = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += w;
                    }
                    const float excl = incl - cum[3];
                    float cs2v[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) cs2v[jj] = (excl + cum[jj]) * kLog2e;
                    // anchor of these rows' 32-row block: its last row, owned by lane (lane | 7), jj = 3
                    const float anchor = __shfl_sync(0xffffffffu, cs2v[3], lane | 7);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int row = 4 * lane + jj;
                        sm.cs2[uu][hh][row] = cs2v[jj];
                        sm.dt[uu][hh][row] = dtv[jj];
                        sm.wt[uu][hh][row] = ex2(anchor - cs2v[jj]) * dtv[jj];
                    }
                    if (lane == 0) sm.dskip[uu][hh] = p.D ? p.D[h] : 0.f;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.bc_conv[uu]);
            TRACE(0, (2u << 24) | vv);
            return true;
        };
        for (uint32_t v = 0; ok; ++v) {
            const uint32_t u = v & 1, nn = v >> 1;
            uint32_t t_next = 0;
            if (!late && lane == 0 && t < total) t_next = atomicAdd(&hdr->ticket, 1u);  // in flight meanwhile
            // the previous unit first: the MMA issuer frees stage u (unit v-2's last C.S) only after it
            // has seen unit v-1 converted
            if (v > 0 && !finish(v - 1, prev)) break;
            if (late && v > 0) {  // the ticket only now that the unit before it is three heads from its end
                if (!bwait(&sm.unit_go, (v - 1) & 1, sm, hdr, epoch)) break;
                if (lane == 0) t = atomicAdd(&hdr->ticket, 1u);
                t = __shfl_sync(0xffffffffu, t, 0);
            }
            if (t >= total) {
                if (!bwait(&sm.bc_empty[u], (nn & 1) ^ 1, sm, hdr, epoch)) break;
                if (lane == 0) {
                    sm.sched[u].valid = 0;
                    mbar_arrive(&sm.sched_full[u]);
                    mbar_arrive(&sm.bc_conv[u]);
                }
                break;
            }
            if (!bwait(&sm.bc_empty[u], (nn & 1) ^ 1, sm, hdr, epoch)) break;
            TRACE(0, (1u << 24) | v);
            const SeqChunk sq = seq_chunk(p, t / (p.G * slices));
            const int64_t r = t % (p.G * slices);
            const int64_t c = sq.c;
            const int64_t g = r / slices;
            const int64_t h0 = g * p.heads_per_group + (r % slices) * hs;
            const int64_t row0 = sq.tok0 + c * kQ;
            const int rows = (int)((sq.len - c * kQ) < kQ ? (sq.len - c * kQ) : kQ);
            const int last = c == (sq.len + kQ - 1) / kQ - 1;
            // dt_raw rows 4*lane .. 4*lane+3 of the unit's heads, every load in flight at once
            float raw[4][kMaxHs];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int i = 4 * lane + jj;
#pragma unroll
                for (int hh = 0; hh < kMaxHs; ++hh) {
                    raw[jj][hh] = 0.f;
                    if (hh < hs && i < rows)
                        raw[jj][hh] = to_f32(*chk(dtr, (row0 + i) * p.H + h0 + hh + probe, 1, ndt, hdr, SITE_TC_DT));
                }
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int hh = 0; hh < kMaxHs; ++hh)
                    if (hh < hs) sm.cs2[u][hh][4 * lane + jj] = raw[jj][hh];
            const Sched cur{1, (int32_t)sq.s, (int32_t)c, (int32_t)g, (int32_t)h0, rows, (int32_t)row0, last};
            __syncwarp();
            if (lane == 0) {
                sm.sched[u] = cur;
                mbar_arrive(&sm.sched_full[u]);
                mbar_arrive_expect_tx(&sm.bc_full[u], 4 * kTile);
                tma_load_4d(sm.bc[u][0], &map_b, &sm.bc_full[u], 0, (int)g, (int)row0, 0);
                tma_load_4d(sm.bc[u][1], &map_b, &sm.bc_full[u], 64, (int)g, (int)row0, 0);
                tma_load_4d(sm.bc[u][2], &map_c, &sm.bc_full[u], 0, (int)g, (int)row0, 0);
                tma_load_4d(sm.bc[u][3], &map_c, &sm.bc_full[u], 64, (int)g, (int)row0, 0);
                armed_bc |= 1 << u;
                bc_par[u] = nn & 1;
            }
            prev = cur;
            if (!late) t = __shfl_sync(0xffffffffu, t_next, 0);
        }
        // teardown: make sure no TMA write into this CTA's shared memory is still in flight
        if (lane == 0 && *reinterpret_cast<volatile int32_t *>(&sm.abort)) {
            for (int u = 0; u < 2; ++u)
                if (armed_bc & (1 << u)) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(&sm.bc_full[u], bc_par[u]) && globaltimer() - t0 < 100000000ull) {
                    }
                }
        }
        __syncwarp();
    } else if (warp == kXWarp) {
        // ------------------------------------------------------------ x loader
        // One TMA per head into the 2-deep x ring (lane 0). With the fused convolution it also brings the 3 raw rows
        // before the chunk: by TMA inside the sequence, else written by the lanes from the conv cache (or zeros).
        if (lane == 0) {
            prefetch_tensormap(&map_x);
            if (CONV) prefetch_tensormap(&map_xh);
        }
        uint32_t hc = 0;
        int armed_x = 0;
        uint32_t x_par[2] = {0, 0};
        for (uint32_t v = 0;; ++v) {
            const uint32_t u = v & 1;
            if (!bwait(&sm.sched_full[u], (v >> 1) & 1, sm, hdr, epoch)) break;
            const Sched sc = sm.sched[u];
            if (!sc.valid) break;
            bool ok = true;
            for (int hh = 0; hh < hs; ++hh, ++hc) {
                const uint32_t k = hc & 1, n = hc >> 1;
                if (!bwait(&sm.x_empty[k], (n & 1) ^ 1, sm, hdr, epoch)) {
                    ok = false;
                    break;
                }
                const bool halo_tma = CONV && sc.c > 0;
                if (CONV) {  // the head's taps and bias, read by the math warps as broadcasts
                    const int64_t ch0 = (int64_t)(sc.h0 + hh) * kP;
                    for (int e = lane; e < kP; e += 32) {
                        sm.xtap[k][e] = *reinterpret_cast<const float4 *>(p.conv_w + (ch0 + e) * 4);
                        sm.xbias[k][e] = p.conv_b ? p.conv_b[ch0 + e] : 0.f;
                    }
                }
                if (CONV && sc.c == 0) {  // the sequence starts here: its conv cache (or zeros) before it
                    const IO *st = static_cast<const IO *>(p.conv_state);
                    IO *dst = reinterpret_cast<IO *>(sm.xhalo[k]);
                    for (int e = lane; e < 3 * kP; e += 32) {
                        const int r = e / kP, pc = e % kP;
                        const int64_t ch = (int64_t)(sc.h0 + hh) * kP + pc;
                        dst[r * kP + pc] = st ? *chk(st, ((int64_t)sc.s * p.x_ld + ch) * 3 + r, 1, p.nseq * p.x_ld * 3, hdr,
                                                     SITE_CONV_STATE)
                                              : from_f32<IO>(0.f);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.x_full[k], kTile + (halo_tma ? 3 * kP * 2 : 0));
                    tma_load_4d(sm.x[k], &map_x, &sm.x_full[k], 0, sc.h0 + hh, sc.row0, 0);
                    if (halo_tma) tma_load_4d(sm.xhalo[k], &map_xh, &sm.x_full[k], 0, sc.h0 + hh, sc.row0 - 3, 0);
                    armed_x |= 1 << k;
                    x_par[k] = n & 1;
                }
            }
            if (!ok) break;
        }
        if (lane == 0 && *reinterpret_cast<volatile int32_t *>(&sm.abort)) {
            for (int k = 0; k < 2; ++k)
                if (armed_x & (1 << k)) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(&sm.x_full[k], x_par[k]) && globaltimer() - t0 < 100000000ull) {
                    }
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Event driven: heads h are numbered across units (unit h / hs). For each head it issues
        // MMA1 (P.x and the chunk state) once P is in TMEM, and C.S once the entering state is in
        // shared memory, whichever is ready first, C.S preferred (the epilogue waits on it). CB of a
        // unit goes out before the unit's first MMA1.
        if (lane == 0) {
            constexpr uint32_t idCB = idesc_f16_f32(128, 128, false, false);
            constexpr uint32_t idPX = idesc_f16_f32(128, 64, false, true);
            constexpr uint32_t idST = idesc_f16_f32(128, 64, true, true);
            constexpr uint32_t idCS = idesc_f16_f32(128, 64, false, true);
            const uint32_t uhs = (uint32_t)hs;
            uint32_t v_cb = 0;                // next unit whose CB is due
            uint32_t h1 = 0, h2 = 0;          // next head for MMA1 / for C.S (h2 <= h1)
            uint32_t end_heads = 0xffffffffu; // total heads, once the end-of-work unit is seen
            uint64_t idle_since = globaltimer();
            const uint64_t limit = 4 * (hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs) + 100000000ull;
            for (uint32_t spin = 0;; ++spin) {
                bool progress = false;
                // C.S of head h2: y_inter = C . S_in
                if (h2 < h1 && mbar_try_wait_ns(&sm.sin_full[h2 & 1], (h2 >> 1) & 1, 64)) {
                    const uint32_t k = h2 & 1, vu = h2 / uhs, u = vu & 1;
                    tc_fence_after();
                    const uint32_t ca = smem_u32(sm.bc[u][2]), sa = smem_u32(sm.xs[k]);
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t off = (uint32_t)(s >> 2) * kTile + (uint32_t)(s & 3) * 32;
                        mma_ss(tmem + kColP + 64 * k, desc_sw128(ca + off, 16, 1024),
                               desc_sw128(sa + 2048 * s, 8192, 1024), idCS, s > 0);
                    }
                    mma_commit(&sm.mma2[k]);
                    if (h2 % uhs == uhs - 1) mma_commit(&sm.bc_empty[u]);  // last reader of the unit's B/C
                    TRACE(1, (3u << 24) | h2);
                    ++h2;
                    progress = true;
                }
                if (end_heads != 0xffffffffu && h2 == end_heads) break;
                // CB of unit v_cb, due when MMA1 has reached its first head
                if (end_heads == 0xffffffffu && h1 == v_cb * uhs &&
                    mbar_test_wait(&sm.bc_conv[v_cb & 1], (v_cb >> 1) & 1)) {
                    const uint32_t u = v_cb & 1;
                    if (!*reinterpret_cast<volatile int32_t *>(&sm.sched[u].valid)) {
                        end_heads = v_cb * uhs;
                        progress = true;
                    } else if (mbar_test_wait(&sm.cb_empty, (v_cb & 1) ^ 1)) {
                        tc_fence_after();
                        const uint32_t ba = smem_u32(sm.bc[u][0]), ca = smem_u32(sm.bc[u][2]);
#pragma unroll
                        for (int s = 0; s < 8; ++s) {
                            const uint32_t off = (uint32_t)(s >> 2) * kTile + (uint32_t)(s & 3) * 32;
                            mma_ss(tmem + kColCB, desc_sw128(ca + off, 16, 1024), desc_sw128(ba + off, 16, 1024),
                                   idCB, s > 0);
                        }
                        mma_commit(&sm.cb_full);
                        TRACE(1, (1u << 24) | v_cb);
                        ++v_cb;
                        progress = true;
                    }
                }
                // MMA1 of head h1: y_intra = P . x and s = B^T . X_s
                if (h1 < v_cb * uhs && mbar_try_wait_ns(&sm.p_full[h1 & 1], (h1 >> 1) & 1, 64) &&
                    mbar_test_wait(&sm.s_free[h1 & 1], ((h1 >> 1) & 1) ^ 1)) {
                    const uint32_t k = h1 & 1, u = (h1 / uhs) & 1;
                    tc_fence_after();
                    const uint32_t ba = smem_u32(sm.bc[u][0]);
                    const uint32_t xa = smem_u32(sm.x[k]), xsa = smem_u32(sm.xs[k]);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma_ts(tmem + kColYI + 64 * k, tmem + kColP + 64 * k + 8 * s,
                               desc_sw128(xa + 2048 * s, 8192, 1024), idPX, s > 0);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma_ss(tmem + kColS + 64 * k, desc_sw128(ba + 2048 * s, kTile, 1024),
                               desc_sw128(xsa + 2048 * s, 8192, 1024), idST, s > 0);
                    mma_commit(&sm.mma1[k]);
                    mma_commit(&sm.x_empty[k]);
                    TRACE(1, (2u << 24) | h1);
                    ++h1;
                    progress = true;
                }
                if (progress) {
                    idle_since = globaltimer();
                } else if ((spin & 15u) == 15u) {
                    if (*reinterpret_cast<volatile int32_t *>(&sm.abort)) break;
                    if (globaltimer() - idle_since > limit) {
                        pipe_timeout(sm, hdr, epoch);
                        break;
                    }
                }
            }
            // drain: every MMA issued above has completed before TMEM is released
            mma_commit(&sm.drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(&sm.drain, 0) && globaltimer() - t0 < 1000000000ull) {
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ math warpgroup
        const int q = warp & 3;              // TMEM lane quarter of this warp
        const int i = 32 * q + lane;         // tile row (token within the chunk) owned by this thread
        const uint32_t lrow = (uint32_t)(32 * q) << 16;
        const bool leader = warp == 2 && lane == 0;
        if (lane == 0) prefetch_tensormap(&map_y);
        uint32_t hc = 0;
        bool pend = false;
        uint32_t pk = 0, pn = 0;
        float pecs = 0.f;
        int ph = 0, prow = 0, pvr = 0;  // y of the pending head: head, first token of this warp's rows, valid rows
        IO *yg = static_cast<IO *>(p.y);
        bool ok = true;
        // y = y_intra + exp(cs_i) y_inter of the pending head, staged in its C.S operand tile (free once C.S
        // has completed) with the operand's 128B swizzle, then one TMA store per warp of its 32 rows; the
        // store clips rows past the sequence end.
        auto epilogue = [&]() -> bool {
            if (!bwait(&sm.mma2[pk], pn & 1, sm, hdr, epoch)) return false;
            if (leader) TRACE(2, (6u << 24) | (pn * 2 + pk));
            tc_fence_after();
            uint8_t *yrow = sm.xs[pk] + i * 128;
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                uint32_t a[16], c2[16];
                tmem_ld16(tmem + lrow + kColYI + 64 * pk + 16 * m, a);
                tmem_ld16(tmem + lrow + kColP + 64 * pk + 16 * m, c2);
                tmem_ld_wait();
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float y0 = __uint_as_float(a[2 * e]) + pecs * __uint_as_float(c2[2 * e]);
                    const float y1 = __uint_as_float(a[2 * e + 1]) + pecs * __uint_as_float(c2[2 * e + 1]);
                    o[e] = pack_io<IO>(y0, y1);
                }
                sts128(yrow + (((2 * m) ^ (i & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
                sts128(yrow + (((2 * m + 1) ^ (i & 7)) << 4), make_uint4(o[4], o[5], o[6], o[7]));
            }
            if (pvr >= 32) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_4d(&map_y, sm.xs[pk] + 32 * q * 128, 0, ph, prow, 0);
                    bulk_commit();
                }
            } else if (lane < pvr) {  // ragged last chunk: the valid rows one by one (the next sequence follows)
                uint4 *dst = reinterpret_cast<uint4 *>(
                    chk(yg, ((int64_t)(prow + lane) * p.H + ph) * kP, kP, p.batch * p.L * p.H * kP, hdr, SITE_TC_Y));
#pragma unroll
                for (int lc = 0; lc < 8; ++lc) dst[lc] = lds128(yrow + ((lc ^ (i & 7)) << 4));
            }
            if (leader) TRACE(2, (7u << 24) | (pn * 2 + pk));
            return true;
        };
        for (uint32_t v = 0; ok; ++v) {
            const uint32_t u = v & 1, nn = v >> 1;
            if (!bwait(&sm.bc_conv[u], nn & 1, sm, hdr, epoch)) {
                ok = false;
                break;
            }
            const Sched sc = sm.sched[u];
            if (!sc.valid) break;
            if (leader) TRACE(2, (1u << 24) | v);

            // (3) per head: X_s, P, then the previous head's epilogue
            for (int hh = 0; hh < hs; ++hh, ++hc) {
                const uint32_t k = hc & 1, n = hc >> 1;
                const int h = sc.h0 + hh;
                if (!bwait(&sm.x_full[k], n & 1, sm, hdr, epoch)) {
                    ok = false;
                    break;
                }
                if (leader) TRACE(2, (2u << 24) | hc);
                if (lane == 0) bulk_wait_read0();  // this warp's y store from xs[k] (two heads back) has read it
                __syncwarp();
                const float cs2i = sm.cs2[u][hh][i];
                const float xscale = ex2(sm.cs2[u][hh][kQ - 1] - cs2i) * sm.dt[u][hh][i];
                if constexpr (CONV) {
                    // row i of x convolved from the raw rows i-3 .. i (rows before the chunk from the halo), then,
                    // once every row has been read, written back as fp16 together with X_s
                    uint32_t xo[kP / 2], so[kP / 2];
#pragma unroll
                    for (int lc = 0; lc < 8; ++lc) {
                        uint4 rr[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int r = i - 3 + j;
                            rr[j] = r >= 0 ? lds128(sm.x[k] + r * 128 + ((lc ^ (r & 7)) << 4))
                                           : lds128(sm.xhalo[k] + (r + 3) * 128 + lc * 16);
                        }
                        const float4 bb0 = reinterpret_cast<const float4 *>(sm.xbias[k])[2 * lc];
                        const float4 bb1 = reinterpret_cast<const float4 *>(sm.xbias[k])[2 * lc + 1];
                        const float bias8[8] = {bb0.x, bb0.y, bb0.z, bb0.w, bb1.x, bb1.y, bb1.z, bb1.w};
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {  // channel pairs of this 16-byte chunk
                            float o[2];
#pragma unroll
                            for (int c2 = 0; c2 < 2; ++c2) {
                                const int e = 2 * e2 + c2;
                                const float4 tw = sm.xtap[k][8 * lc + e];
                                float in[4];
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const uint32_t wv = reinterpret_cast<const uint32_t *>(&rr[j])[e2];
                                    const float2 f = unpack_io<IO>(wv);
                                    in[j] = c2 ? f.y : f.x;
                                }
                                float acc = fmaf(tw.w, in[3], fmaf(tw.z, in[2], fmaf(tw.y, in[1], fmaf(tw.x, in[0], bias8[e]))));
                                o[c2] = p.conv_silu ? silu_fast(acc) : acc;
                            }
                            xo[4 * lc + e2] = pack_f16(o[0], o[1]);
                            so[4 * lc + e2] = pack_f16(o[0] * xscale, o[1] * xscale);
                        }
                    }
                    bar_sync(kBarMath, 128);  // every thread has read its raw rows: the tile may be overwritten
                    uint8_t *xr = sm.x[k] + i * 128;
                    uint8_t *sr = sm.xs[k] + i * 128;
#pragma unroll
                    for (int lc = 0; lc < 8; ++lc) {
                        const int off = (lc ^ (i & 7)) << 4;
                        sts128(xr + off, make_uint4(xo[4 * lc], xo[4 * lc + 1], xo[4 * lc + 2], xo[4 * lc + 3]));
                        sts128(sr + off, make_uint4(so[4 * lc], so[4 * lc + 1], so[4 * lc + 2], so[4 * lc + 3]));
                    }
                } else {
                    uint8_t *xr = sm.x[k] + i * 128;
                    uint8_t *sr = sm.xs[k] + i * 128;
                    uint4 w[8];
#pragma unroll
                    for (int lc = 0; lc < 8; ++lc) w[lc] = lds128(xr + ((lc ^ (i & 7)) << 4));
#pragma unroll
                    for (int lc = 0; lc < 8; ++lc) {
                        const int off = (lc ^ (i & 7)) << 4;
                        uint32_t *wv = reinterpret_cast<uint32_t *>(&w[lc]);
                        uint4 s4;
                        uint32_t *sv = reinterpret_cast<uint32_t *>(&s4);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_io<IO>(wv[e]);
                            sv[e] = pack_f16(f.x * xscale, f.y * xscale);
                            if (kBf16) wv[e] = pack_f16(f.x, f.y);
                        }
                        if (kBf16) sts128(xr + off, w[lc]);
                        sts128(sr + off, s4);
                    }
                }
                if (leader) TRACE(2, (8u << 24) | hc);
                fence_proxy_async_smem();
                if (leader) TRACE(2, (5u << 24) | hc);
                if (hh == 0) {
                    if (!bwait(&sm.cb_full, v & 1, sm, hdr, epoch)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                // P = CB o decay o dt (+ D on the diagonal), masked above the diagonal, fp16 into TMEM
                const float Dh = sm.dskip[u][hh];
                const float *cs2r = sm.cs2[u][hh];
                const float *dtr = sm.dt[u][hh];
                const float *wtr = sm.wt[u][hh];
                // One 32-column block of CB per iteration (rolled: keeps the hot code small). Blocks above
                // the diagonal block are zero. Elsewhere exp(cs_i - cs_j) = exp(cs_i - cs_a) exp(cs_a - cs_j)
                // with a the block's last row: below the diagonal block both factors are <= 1; in the
                // diagonal block the first is >= 1, so it is used only while the block's whole decay range
                // keeps it <= 2^100 (warp-uniform test), else the diagonal block takes exp directly. The
                // shared-memory tables are read before the TMEM load so their latency overlaps it.
#pragma unroll 1
                for (int J = 0; J < 4; ++J) {
                    uint32_t pk16[16];
                    if (J > q) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) pk16[e] = 0u;
                    } else {
                        const bool diag = J == q;
                        const float ca = cs2r[32 * J + 31];
                        const bool fac = !diag || cs2r[32 * J] - ca <= 100.f;
                        float4 t1[8], t2[8];
                        const float4 *s1 = reinterpret_cast<const float4 *>((fac ? wtr : cs2r) + 32 * J);
#pragma unroll
                        for (int e = 0; e < 8; ++e) t1[e] = s1[e];
                        if (!fac) {
                            const float4 *d4 = reinterpret_cast<const float4 *>(dtr + 32 * J);
#pragma unroll
                            for (int e = 0; e < 8; ++e) t2[e] = d4[e];
                        }
                        const float ui = ex2(cs2i - ca);
                        uint32_t cb[32];
                        tmem_ld16(tmem + lrow + kColCB + 32 * J, *reinterpret_cast<uint32_t(*)[16]>(&cb[0]));
                        tmem_ld16(tmem + lrow + kColCB + 32 * J + 16, *reinterpret_cast<uint32_t(*)[16]>(&cb[16]));
                        tmem_ld_wait();
                        if (leader) TRACE(2, ((9u + J) << 24) | hc);
                        if (fac) {
                            const int lim = diag ? i : (1 << 30);  // columns j < lim are kept; j == i also takes D
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j0 = 32 * J + 4 * e;
                                float v0 = __uint_as_float(cb[4 * e]) * ui * t1[e].x;
                                float v1 = __uint_as_float(cb[4 * e + 1]) * ui * t1[e].y;
                                float v2 = __uint_as_float(cb[4 * e + 2]) * ui * t1[e].z;
                                float v3 = __uint_as_float(cb[4 * e + 3]) * ui * t1[e].w;
                                v0 = j0 < lim ? v0 : (j0 == i ? v0 + Dh : 0.f);
                                v1 = j0 + 1 < lim ? v1 : (j0 + 1 == i ? v1 + Dh : 0.f);
                                v2 = j0 + 2 < lim ? v2 : (j0 + 2 == i ? v2 + Dh : 0.f);
                                v3 = j0 + 3 < lim ? v3 : (j0 + 3 == i ? v3 + Dh : 0.f);
                                pk16[2 * e] = pack_f16(v0, v1);
                                pk16[2 * e + 1] = pack_f16(v2, v3);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float4 cv = t1[e], dv = t2[e];
                                const int j0 = 32 * J + 4 * e;
                                float v0 = __uint_as_float(cb[4 * e]) * ex2(cs2i - cv.x) * dv.x;
                                float v1 = __uint_as_float(cb[4 * e + 1]) * ex2(cs2i - cv.y) * dv.y;
                                float v2 = __uint_as_float(cb[4 * e + 2]) * ex2(cs2i - cv.z) * dv.z;
                                float v3 = __uint_as_float(cb[4 * e + 3]) * ex2(cs2i - cv.w) * dv.w;
                                v0 = j0 < i ? v0 : (j0 == i ? v0 + Dh : 0.f);
                                v1 = j0 + 1 < i ? v1 : (j0 + 1 == i ? v1 + Dh : 0.f);
                                v2 = j0 + 2 < i ? v2 : (j0 + 2 == i ? v2 + Dh : 0.f);
                                v3 = j0 + 3 < i ? v3 : (j0 + 3 == i ? v3 + Dh : 0.f);
                                pk16[2 * e] = pack_f16(v0, v1);
                                pk16[2 * e + 1] = pack_f16(v2, v3);
                            }
                        }
                    }
                    tmem_st16(tmem + lrow + kColP + 64 * k + 16 * J, pk16);
                }
                tmem_st_wait();
                if (leader) TRACE(2, (13u << 24) | hc);
                tc_fence_before();
                bar_sync(kBarMath, 128);
                if (leader) TRACE(2, (14u << 24) | hc);
                if (leader) {
                    mbar_arrive(&sm.p_full[k]);
                    if (hh == hs - 1) mbar_arrive(&sm.cb_empty);
                    if (hh == (hs > 3 ? hs - 3 : 0)) mbar_arrive(&sm.unit_go);  // late tickets: the next unit
                    TRACE(2, (3u << 24) | hc);
                }
                if (pend && !epilogue()) {
                    ok = false;
                    break;
                }
                pend = true;
                pk = k;
                pn = n;
                pecs = ex2(cs2i);
                ph = h;
                prow = sc.row0 + 32 * q;
                pvr = sc.rows - 32 * q;
            }
        }
        if (ok && pend) epilogue();
        if (lane == 0) bulk_wait0();  // every y store of this warp has completed
        __syncwarp();
    } else {
        // ------------------------------------------------------------ chain warpgroup
        // Thread n owns d_state row n of every state and passes it to the next chunk through a 2-slot ring per
        // chain, with no CTA barrier on either side of a hop:
        //  - fp32 states: the row, then its own release flag (a 64-bit tag epoch:chunk); after each publish the
        //    next head's row is prefetched when its flag is already visible;
        //  - fp16 states: every 8-byte ring word carries two values and the 32-bit tag epoch * 4 + (chunk mod 4)
        //    (a slot only has to tell chunk c from c - 2, its previous occupant, and from older launches). An aligned
        //    8-byte access is single-copy atomic, so a word with the expected tag holds this launch's values for
        //    that chunk: the data is its own flag (no release, no flag load), which shortens the serial chain of
        //    hops by a round trip. (fp32 rows would need 128 registers in flight this way.)
        const int q = warp & 3;
        const int nrow = 32 * q + lane;  // state row (d_state index) owned by this thread
        const uint32_t lrow = (uint32_t)(32 * q) << 16;
        const uint64_t limit = hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs;
        const int64_t skip = hdr->skip_publish - 1;
        const ST *init = static_cast<const ST *>(p.init);
        ST *fin = static_cast<ST *>(p.final_states);
        uint64_t *tags = reinterpret_cast<uint64_t *>(p.flags);  // [chain][slot][row]
        constexpr bool kTagged = sizeof(ST) == 2;
        float S[kP];          // entering state of the current head (fp32)
        bool have_S = false;  // the current head's entering state is (being) loaded into registers
        Sched sc;
        uint32_t v = 0;
        int hh = 0;
        auto enter_unit = [&](uint32_t vv) -> bool {
            const uint32_t uu = vv & 1;
            if (!bwait(&sm.bc_conv[uu], (vv >> 1) & 1, sm, hdr, epoch)) return false;
            sc = sm.sched[uu];
            return sc.valid != 0;
        };
        ulonglong2 *ringv = static_cast<ulonglong2 *>(p.ring);  // fp16: [chain][slot][P / 4 vectors][row]
        const int64_t nvec = p.ring_bytes / 16, nstate = p.nseq * p.H * kP * kN;  // extents (bounds-checked builds)
        // row nrow of a slot: 16 vectors kN apart (checked as one span)
        auto vrow_of = [&](int64_t chain, int c) {
            return chk(ringv, (chain * 2 + (c & 1)) * (int64_t)(kP / 4 * kN) + nrow, (kP / 4 - 1) * kN + 1, nvec, hdr,
                       SITE_TC_RING);
        };
        auto vtag = [&](int c) { return (epoch << 2) | (uint32_t)(c & 3); };
        // fp16: the tagged row of chunk c as loaded, and whether any of its words is stale
        uint64_t raw[kTagged ? kP / 2 : 1];
        auto issue_tagged = [&](int64_t chain, int c) {
            const ulonglong2 *src = vrow_of(chain, c);
#pragma unroll
            for (int j = 0; j < (kTagged ? kP / 4 : 0); ++j) {
                const ulonglong2 t = ld_ring(src + j * kN);
                raw[2 * j] = t.x;
                raw[2 * j + 1] = t.y;
            }
        };
        auto stale = [&](uint32_t want) {
            uint32_t bad = 0;
#pragma unroll
            for (int w = 0; w < (kTagged ? kP / 2 : 0); ++w) bad |= (uint32_t)(raw[w] >> 32) ^ want;
            return bad != 0;
        };
        // Row nrow of the state entering chunk c > 0 of `chain`, from the ring (the caller has seen its tag).
        auto load_ring = [&](int64_t chain, int c) {
            if (sizeof(ST) == 4) {
                const float4 *src = chk(reinterpret_cast<const float4 *>(p.ring),
                                        (chain * 2 + (c & 1)) * (int64_t)(kP / 4 * kN) + nrow, (kP / 4 - 1) * kN + 1,
                                        nvec, hdr, SITE_TC_RING);
#pragma unroll
                for (int m = 0; m < kP / 4; ++m) {
                    const float4 f = __ldcg(src + m * kN);
                    S[4 * m] = f.x;
                    S[4 * m + 1] = f.y;
                    S[4 * m + 2] = f.z;
                    S[4 * m + 3] = f.w;
                }
            }
        };
        auto tag_of = [&](int64_t chain, int c) {
            return chk(tags, (chain * 2 + (c & 1)) * kN + nrow, 1, p.flag_count, hdr, SITE_TC_FLAG);
        };
        auto want_of = [&](int c) { return ((uint64_t)epoch << 32) | (uint32_t)c; };
        // Prefetch (fp32 states): load the entering state now when its producer's tag is already visible.
        auto prefetch = [&](int64_t chain, int c) -> bool {
            if (kTagged || c == 0 || ld_acquire_u64(tag_of(chain, c)) != want_of(c)) return false;
            load_ring(chain, c);
            return true;
        };
        bool more = enter_unit(0);
        int64_t chain = 0;
        int c = 0;
        if (more) {
            chain = (int64_t)sc.s * p.H + sc.h0;
            c = sc.c;
        }
        uint32_t hc = 0;
        while (more) {
            const uint32_t k = hc & 1, n = hc >> 1;
            // state entering the chunk
            auto fetch_S = [&]() {
                if (!have_S) {
                    if (c == 0) {
#pragma unroll
                        for (int pp = 0; pp < kP; ++pp)
                            S[pp] = init ? to_f32(*chk(init, (chain * kP + pp) * kN + nrow, 1, nstate, hdr, SITE_TC_INIT)) : 0.f;
                    } else if (kTagged) {
                        const uint32_t want = vtag(c);
                        issue_tagged(chain, c);
                        bool ok = !stale(want);
                        while (!ok) {  // not yet published, or only partly visible: wait on the row's last vector, reload
                            if (aborted(hdr, epoch) ||
                                !wait_ring(vrow_of(chain, c) + (kP / 4 - 1) * kN, want, epoch, hdr, limit, (uint32_t)c))
                                break;
                            issue_tagged(chain, c);
                            ok = !stale(want);
                        }
                        if (ok) {
#pragma unroll
                            for (int w = 0; w < (kTagged ? kP / 2 : 0); ++w) {
                                const float2 f = unpack_f16((uint32_t)raw[w]);
                                S[2 * w] = f.x;
                                S[2 * w + 1] = f.y;
                            }
                        } else {  // the error is recorded; carry on with zeros so the CTA drains
#pragma unroll
                            for (int pp = 0; pp < kP; ++pp) S[pp] = 0.f;
                        }
                    } else if ((ld_acquire_u64(tag_of(chain, c)) == want_of(c) ||
                                (!aborted(hdr, epoch) && wait_tag(tag_of(chain, c), want_of(c), epoch, hdr, limit, (uint32_t)c)))) {
                        load_ring(chain, c);
                    } else {  // the error is recorded; carry on with zeros so the CTA drains
#pragma unroll
                        for (int pp = 0; pp < kP; ++pp) S[pp] = 0.f;
                    }
                }
            };
            // fp16 states fetch (and, if need be, wait for) the entering row before s_c is read, so no wait is a
            // call with s_c's 64 registers live; fp32 states free s_c's TMEM columns first
            if (kTagged) fetch_S();
            // chunk state s_c from TMEM
            if (!bwait(&sm.mma1[k], n & 1, sm, hdr, epoch)) break;
            tc_fence_after();
            float s[kP];
            {
                uint32_t r[4][16];
#pragma unroll
                for (int m = 0; m < 4; ++m) tmem_ld16(tmem + lrow + kColS + 64 * k + 16 * m, r[m]);
                tmem_ld_wait();
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int e = 0; e < 16; ++e) s[16 * m + e] = __uint_as_float(r[m][e]);
            }
            tc_fence_before();
            mbar_arrive(&sm.s_free[k]);
            if (warp == 6 && lane == 0) TRACE(3, (1u << 24) | hc);
            const float a = ex2(sm.cs2[v & 1][hh][kQ - 1]);  // decay across the chunk
            if (!kTagged) fetch_S();
            // state leaving the chunk: S_out = a S_in + s (kept in s[])
#pragma unroll
            for (int pp = 0; pp < kP; ++pp) s[pp] = fmaf(a, S[pp], s[pp]);
            const bool publish = !sc.last && c != skip;
            if (sc.last) {
                if (fin) {
#pragma unroll
                    for (int pp = 0; pp < kP; ++pp)
                        *chk(fin, (chain * kP + pp) * kN + nrow, 1, nstate, hdr, SITE_TC_FINAL) = from_f32<ST>(s[pp]);
                }
            } else if (publish) {
                if (sizeof(ST) == 4) {
                    float4 *dst = chk(reinterpret_cast<float4 *>(p.ring),
                                      (chain * 2 + ((c + 1) & 1)) * (int64_t)(kP / 4 * kN) + nrow, (kP / 4 - 1) * kN + 1,
                                      nvec, hdr, SITE_TC_RING);
#pragma unroll
                    for (int m = 0; m < kP / 4; ++m)
                        __stcg(dst + m * kN, make_float4(s[4 * m], s[4 * m + 1], s[4 * m + 2], s[4 * m + 3]));
                } else {  // tagged words, the last vector last
                    ulonglong2 *dst = vrow_of(chain, c + 1);
                    const uint64_t tg = (uint64_t)vtag(c + 1) << 32;
#pragma unroll
                    for (int j = 0; j < kP / 4; ++j)
                        st_ring(dst + j * kN, tg | pack_f16(s[4 * j], s[4 * j + 1]), tg | pack_f16(s[4 * j + 2], s[4 * j + 3]));
                }
            }
            // S_in (fp16) -> the C.S operand: K-row nrow of a [128 x 64] MN-major 128B-swizzled tile
            {
                uint8_t *row = sm.xs[k] + nrow * 128;
#pragma unroll
                for (int lc = 0; lc < 8; ++lc)
                    sts128(row + ((lc ^ (nrow & 7)) << 4),
                           make_uint4(pack_f16(S[8 * lc], S[8 * lc + 1]), pack_f16(S[8 * lc + 2], S[8 * lc + 3]),
                                      pack_f16(S[8 * lc + 4], S[8 * lc + 5]), pack_f16(S[8 * lc + 6], S[8 * lc + 7])));
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.sin_full[k]);
            if (warp == 6 && lane == 0) TRACE(3, (3u << 24) | hc);
            // publish this head's row (the release orders the row's stores before the tag), then move to
            // the next head and prefetch its entering state
            if (publish && !kTagged)
                st_release_u64(tags + (chain * 2 + ((c + 1) & 1)) * kN + nrow,
                               ((uint64_t)epoch << 32) | (uint32_t)(c + 1));
            ++hc;
            if (hh + 1 < hs) {
                ++hh;
                ++chain;
            } else {
                ++v;
                hh = 0;
                more = enter_unit(v);
                if (!more) break;
                chain = (int64_t)sc.s * p.H + sc.h0;
                c = sc.c;
            }
            have_S = prefetch(chain, c);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0) {
        __threadfence();
        const uint32_t d = atomicAdd(&hdr->done, 1u);
        if (d == gridDim.x - 1) {
            hdr->ticket = 0;
            hdr->done = 0;
            __threadfence();
            st_relaxed_gpu(&hdr->epoch, epoch);
        }
    }
}

// ---------------------------------------------------------------------- host
// 4-D map over a [1, T, mid, inner] 16-bit tensor (all sequences on one packed token axis of T tokens),
// box = [1, box_rows, 1, 64 inner], 128B swizzle. Rows past T read as zeros; a chunk's rows past its own
// sequence read the next sequence and are masked by dt = 0.
bool make_map(CUtensorMap *m, const void *base, bool bf16, int64_t inner, int64_t mid, int64_t T, int64_t ld,
              uint32_t box_rows, bool swizzle = true) {
    const int64_t L = T, batch = 1;
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)mid, (cuuint64_t)L, (cuuint64_t)batch};
    // ld: elements from one token to the next (inner * mid when packed, more when a slice of wider rows)
    const cuuint64_t strides[3] = {(cuuint64_t)(inner * 2), (cuuint64_t)(ld * 2), (cuuint64_t)(ld * L * 2)};
    const cuuint32_t box[4] = {64, 1, box_rows, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
               const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename IO, typename ST, bool CONV>
cudaError_t launch_t(const Params &p, int hs, int sms, cudaStream_t stream) {
    CUtensorMap mx, mb, mc, my, mxh;
    const bool bf = !std::is_same<IO, __half>::value;
    const int64_t T = p.batch * p.L;
    if (!make_map(&mx, p.x, bf, kP, p.H, T, p.x_ld, kQ) || !make_map(&mb, p.B, bf, kN, p.G, T, p.bc_ld, kQ) ||
        !make_map(&mc, p.C, bf, kN, p.G, T, p.bc_ld, kQ) || !make_map(&my, p.y, bf, kP, p.H, T, p.H * kP, 32))
        return cudaErrorInvalidValue;
    if (CONV ? !make_map(&mxh, p.x, bf, kP, p.H, T, p.x_ld, 3, false) : false) return cudaErrorInvalidValue;
    if (!CONV) mxh = mx;
    const size_t smem = sizeof(Smem) + 1024;
    auto k = tc_kernel<IO, ST, CONV>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = p.ctab ? (int64_t)sms : std::min<int64_t>((int64_t)p.total_units, (int64_t)sms);
    k<<<(unsigned)grid, kThreads, smem, stream>>>(p, mx, mb, mc, my, mxh, hs);
    return cudaGetLastError();
}

}  // namespace

// Any chunk size that is a multiple of 128 runs in 128-token chunks: the chunked result is exact for every
// chunk size (only its rounding differs), so a larger requested chunk is served by passing states more often.
bool tc_supports(int64_t P, int64_t N, int64_t Q, int io_dtype) {
    return P == kP && N == kN && Q % kQ == 0 && (io_dtype == 1 || io_dtype == 2);
}

int64_t tc_chunk() { return kQ; }

size_t tc_flag_bytes(int64_t chains) { return (size_t)chains * 2 * kN * sizeof(uint64_t); }

// Per chain 2 slots of P x N states: fp32 values (flagged), or fp16 values in tagged 8-byte words (two values and
// a 32-bit tag): 4 bytes per element either way.
size_t tc_ring_bytes(int64_t chains, int64_t P, int64_t N, int state_dtype) {
    (void)state_dtype;
    return (size_t)chains * 2 * (size_t)(P * N) * 4;
}

// Late tickets pay where few units share a chunk index, so that the state chain bounds the launch (measured on
// GB300: -13 % at L = 256K and -6 % at L = 16K with 10-16 units per chunk index, -7 % on the 130M-shaped batch
// with 32; +17-24 % at batch 8-32 with 80 and more, where the loads then exposed at every unit boundary cost more
// than the chain).
bool tc_late_ticket(int64_t units_per_chunk, int sms) { return units_per_chunk * 4 <= sms; }

uint32_t tc_total_units(int64_t batch, int64_t H, int64_t G, int64_t nc, int hs) {
    (void)G;
    return (uint32_t)(nc * batch * (H / hs));
}

// Heads per work unit: the largest divisor of heads-per-group (<= 8) that still leaves at least six units per
// SM; small problems fall back to 1. More heads per unit share one C.B^T and one B/C load; more units spread the
// chunk-serial state chain over more SMs (measured on GB300: the 130M-shaped batch runs 3 heads per unit 7-9 %
// faster than 4 with late tickets; 4 beat 8 by 8-9 % where 8 left 2.5-4 units per SM; 8 beat 4 by 8 % at 33 units
// per SM).
int tc_heads_per_unit(int64_t batch, int64_t H, int64_t G, int64_t nc, int sms) {
    const int64_t hpg = H / G;
    for (int d = kMaxHs; d >= 1; --d)
        if (hpg % d == 0 && nc * batch * (H / d) >= 6 * (int64_t)sms) return d;
    return 1;
}

template <bool CONV>
cudaError_t launch_any(const Params &p, int io_dtype, int state_dtype, int hs, int sms, cudaStream_t stream) {
    if (io_dtype == 1)
        return state_dtype == 0 ? launch_t<__nv_bfloat16, float, CONV>(p, hs, sms, stream)
                                : launch_t<__nv_bfloat16, __half, CONV>(p, hs, sms, stream);
    return state_dtype == 0 ? launch_t<__half, float, CONV>(p, hs, sms, stream)
                            : launch_t<__half, __half, CONV>(p, hs, sms, stream);
}

cudaError_t launch_tc(Params p, int io_dtype, int state_dtype, int hs, int sms, cudaStream_t stream) {
    return p.conv_w ? launch_any<true>(p, io_dtype, state_dtype, hs, sms, stream)
                    : launch_any<false>(p, io_dtype, state_dtype, hs, sms, stream);
}

}  // namespace ssd

#ifdef SSD_TRACE
extern "C" __attribute__((visibility("default"))) int ssd_trace_read(unsigned long long *dst, unsigned int *counts) {
    if (cudaMemcpyFromSymbol(counts, ssd::g_trace_n, sizeof(ssd::g_trace_n)) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(dst, ssd::g_trace, sizeof(ssd::g_trace)) != cudaSuccess) return -1;
    static const unsigned int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(ssd::g_trace_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}
#endif

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
//   y       = y_intra + exp(cs_i) C_c S_c     (tcgen05 C.S, fused epilogue; D x enters through P's diagonal)
//
// Warp roles (512 threads, four warpgroups); every per-head phase has warps of
// its own, so the phases of consecutive heads overlap:
//   warp 0       unit loader: tickets, B/C tiles by TMA, their bf16 -> fp16 conversion one unit behind
//   warp 1       TMEM allocator + tcgen05.mma issuer (one elected lane) of C.B^T and of each head's P.x and chunk state
//   warp 2       x loader: per head one TMA of the x tile into a 3-deep ring, and the head's chunk cumsum tables
//   warp 3       tcgen05.mma issuer (one elected lane) of each head's C.S
//   warps 4-7    P: the decay-masked C.B^T of each head, fp16 into TMEM; then the head's X_s = w o x (and x to
//                fp16), both before the head's first MMAs
//   warps 8-11   epilogue after the head's C.S, staged in the head's x slot (x is no longer needed then) and
//                sent by TMA stores
//   warps 12-15  chain: state passing, S_in -> shared memory as the C.S operand, final states
// All MMA operands are fp16 (bf16 inputs are converted on chip; the contractions
// with P, X_s and S need fp16's 11-bit significand to hold 1e-2).
//
// TMEM (512 columns): CB [0,128), P x2 [128,256), y_intra x2 [256,384), and x2 [384,512) the chunk state s,
// which C.S overwrites with y_inter once the chain has read it.
#include <cuda.h>
#include <stddef.h>

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
constexpr int kThreads = 512;
constexpr uint32_t kTile = 16384;  // [128 rows x 128 B] 128B-swizzled 16-bit tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kColCB = 0, kColP = 128, kColYI = 256, kColS = 384;
constexpr uint32_t kBarE = 1;  // named barrier of the P / X_s warpgroup (0 is __syncthreads)

struct Sched {
    int32_t valid, s, c, g, h0, rows, row0, last;  // row0: the chunk's first token on the packed token axis
};

// Per head, beside its x tile: the chunk cumsum tables and what the consumers need to know about the head.
// 16-byte aligned: the tables are written and read as float4 vectors in every slot.
struct __align__(16) HeadTab {
    float cs2[kQ];  // log2(e) * chunk-local inclusive cumsum of dt*A
    float wt[kQ];   // exp(cs_anchor(j) - cs_j) dt_j, anchor(j) = last row of j's 32-row block
    float dt[kQ];   // dt (0 past the sequence end)
    int32_t valid;  // 0: no more work (end marker)
    int32_t h, hh, v, c, s, row0, rows, last;
    float dskip;  // D of the head (0 when absent)
};

template <bool CONV>
struct __align__(128) ConvStage {  // fused convolution: per x slot the 3 raw rows before the chunk (a TMA
                                   // destination: 128-byte aligned), the head's taps and bias
    uint8_t halo[3][384];
    float4 tap[3][kP];
    float bias[3][kP];
};
template <>
struct ConvStage<false> {};

template <bool CONV>
struct __align__(1024) Smem {
    uint8_t bc[2][4][kTile];  // per unit stage: B n[0,64), B n[64,128), C n[0,64), C n[64,128)
    uint8_t x[3][kTile];      // per head slot: x tile (fp16 after conversion), then S_in (fp16, C.S operand),
                              // then the head's staged y
    uint8_t xs[2][kTile];     // per head buffer: X_s
    HeadTab tab[4];           // head h's tables in slot h mod 4 (one more than the x slots: the x loader fills
                              // a head's table while it still waits for the head's x slot)
    ConvStage<CONV> cv;
    Sched sched[2];
    uint64_t sched_full[2], bc_full[2], bc_conv[2], bc_empty[2], cb_full, cb_empty, unit_go;
    uint64_t tab_full[4];  // head h's table written (slot h mod 4)
    uint64_t x_full[3], x_empty[3], xs_full[2], p_full[2], mma1[2], acc_free[2], sin_full[2], mma2[2], drain[2];
    uint32_t tmem_base;
    int32_t abort;
};

static_assert(sizeof(HeadTab) % 16 == 0, "every table slot starts on a 16-byte boundary");
static_assert(offsetof(Smem<false>, x) % 1024 == 0 && offsetof(Smem<false>, xs) % 1024 == 0 &&
                  offsetof(Smem<true>, x) % 1024 == 0 && offsetof(Smem<true>, xs) % 1024 == 0,
              "128B-swizzled tiles start on 1024-byte boundaries");
static_assert(offsetof(Smem<false>, tab) % 16 == 0 && offsetof(Smem<true>, tab) % 16 == 0,
              "vector-accessed tables start on 16-byte boundaries");
static_assert(offsetof(Smem<true>, cv) % 128 == 0 && offsetof(ConvStage<true>, halo) % 128 == 0 &&
                  sizeof(ConvStage<true>::halo[0]) % 128 == 0 && offsetof(ConvStage<true>, tap) % 16 == 0 &&
                  offsetof(ConvStage<true>, bias) % 16 == 0,
              "TMA destinations start on 128-byte boundaries, vector-accessed arrays on 16-byte ones");
static_assert(sizeof(Smem<true>) + 1024 <= 227 * 1024, "shared memory of one CTA");

// Opt-in timeline trace (build with -DSSD_TRACE): in CTA 0 lane 0 of every warp records (SM clock, tag).
#ifdef SSD_TRACE
constexpr int kTraceRoles = 16, kTraceN = 4096;  // one record stream per warp (lane 0)
__device__ unsigned long long g_trace[kTraceRoles][kTraceN][2];
__device__ unsigned int g_trace_n[kTraceRoles];
#define TRACE(role, ev, head)                                                                          \
    do {                                                                                               \
        if (blockIdx.x == 0 && trace_i < kTraceN) {                                                    \
            g_trace[role][trace_i][0] = clock64();  /* SM cycles: every record comes from one SM */     \
            g_trace[role][trace_i][1] = ((unsigned long long)(ev) << 32) | (unsigned)(head);           \
            g_trace_n[role] = ++trace_i;                                                               \
        }                                                                                              \
    } while (0)
#else
#define TRACE(role, ev, head) \
    do {                      \
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

// Packed fp32 pairs (one instruction for both lanes of the pair; each lane rounded as a scalar fmul / fmaf).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
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
__device__ __forceinline__ float2 f2(uint32_t lo, uint32_t hi) {
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

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

__device__ __noinline__ void pipe_timeout(int32_t *abort_flag, WsHeader *hdr, uint32_t epoch) {
    *reinterpret_cast<volatile int32_t *>(abort_flag) = 1;
    report_error(hdr, epoch, DEV_PIPE, 0, 0, WAIT_PIPE);
}

// Bounded wait on an intra-CTA mbarrier phase. On timeout (a broken pipeline)
// it records the error, raises the CTA abort flag and returns false; every
// other wait then gives up too and the CTA drains to its teardown. Its limit
// is four times the state-passing limit plus 100 ms: a pipeline stage may
// legitimately sit behind one full state-passing wait, which must time out
// (and report itself) first. Only the first probe is inline: the polling loop
// is one out-of-line copy, so the hot code of every role stays small.
__device__ __noinline__ bool bwait_slow(uint64_t *bar, uint32_t parity, int32_t *abort_flag, WsHeader *hdr,
                                        uint32_t epoch) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; it < kMaxSpinIters; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 15u) {
            if (*reinterpret_cast<volatile int32_t *>(abort_flag)) return false;
            const uint64_t limit = 4 * (hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs) + 100000000ull;
            if (globaltimer() - t0 > limit) break;
        }
    }
    pipe_timeout(abort_flag, hdr, epoch);
    return false;
}
__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t parity, int32_t *abort_flag, WsHeader *hdr,
                                      uint32_t epoch) {
    return mbar_try_wait(bar, parity) || bwait_slow(bar, parity, abort_flag, hdr, epoch);
}

// 16 final-state values of one d_state row (columns p .. p + 15, kN apart from index `base`), in the state dtype.
// Out of line: it runs at a sequence's last chunk only, so it is kept out of the chain's hot code.
template <typename ST>
__device__ __noinline__ void store_final16(ST *fin, int64_t base, int64_t n, WsHeader *hdr, float4 a, float4 b,
                                           float4 c, float4 d) {
    (void)n;
    (void)hdr;
    const float o[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
    for (int e = 0; e < 16; ++e) *chk(fin, base + (int64_t)e * kN, 1, n, hdr, SITE_TC_FINAL) = from_f32<ST>(o[e]);
}

// softplus out of line: the per-head table code stays small in the instruction cache.
__device__ __noinline__ float softplus_ool(float v) { return softplus_f32(v); }

// The diagonal 32-column block of P with exp taken per element (decay ranges too wide for the rank-1 split): CB
// from TMEM, exp(cs_i - cs_j) dt_j, D on the diagonal, the causal mask (a NaN or inf past the diagonal included),
// fp16 into TMEM. Out of line: it is the rare path, kept away from the hot code. Warp-collective.
__device__ __noinline__ void p_block_exact(uint32_t cb_col, uint32_t p_col, const float *cs2, const float *dt,
                                           float cs2i, float dskip) {
    const int lane = threadIdx.x & 31;
    uint32_t cb[32];
    tmem_ld16(cb_col, *reinterpret_cast<uint32_t(*)[16]>(&cb[0]));
    tmem_ld16(cb_col + 16, *reinterpret_cast<uint32_t(*)[16]>(&cb[16]));
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        pk[e] = pack_f16(__uint_as_float(cb[2 * e]) * ex2(cs2i - cs2[2 * e]) * dt[2 * e] + (2 * e == lane ? dskip : 0.f),
                         __uint_as_float(cb[2 * e + 1]) * ex2(cs2i - cs2[2 * e + 1]) * dt[2 * e + 1] +
                             (2 * e + 1 == lane ? dskip : 0.f)) &
                ((2 * e <= lane ? 0x0000ffffu : 0u) | (2 * e + 1 <= lane ? 0xffff0000u : 0u));
    tmem_st16(p_col, pk);
}

// HF: fp32 states published behind one release flag per head, stored by the C.S warp (a separate instantiation,
// so that the kernel without it keeps its own code).
template <typename IO, typename ST, bool CONV, bool HF>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const Params p, const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_b,
              const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_y,
              const __grid_constant__ CUtensorMap map_xh, const int hs) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base (128B-swizzle atoms). Computed as smem_raw + pad, not through an integer
    // round trip, so the compiler keeps the shared address space and emits LDS/STS for every access.
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    Smem<CONV> &sm = *reinterpret_cast<Smem<CONV> *>(smem_raw + pad);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WsHeader *hdr = p.hdr;
    const uint32_t epoch = ld_relaxed_gpu(&hdr->epoch) + 1u;
    constexpr bool kBf16 = sizeof(IO) == 2 && !std::is_same<IO, __half>::value;
    int32_t *abort_flag = &sm.abort;
    unsigned int trace_i = 0;  // per-thread trace record counter (trace builds)
    (void)trace_i;
// Waits of whole warps are made warp-uniform (a timeout or abort seen by some lanes only must not leave the others
// in a warp-collective instruction).
#define BWAIT(bar, par) __all_sync(0xffffffffu, bwait((bar), (par), abort_flag, hdr, epoch))

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.sched_full[i], 1);
            mbar_init(&sm.bc_full[i], 1);
            mbar_init(&sm.bc_conv[i], 1);
            mbar_init(&sm.bc_empty[i], 1);
            mbar_init(&sm.xs_full[i], 128);   // every X_s / epilogue thread arrives
            mbar_init(&sm.p_full[i], 128);    // every P thread arrives
            mbar_init(&sm.mma1[i], 1);
            mbar_init(&sm.acc_free[i], 128);  // every X_s / epilogue thread arrives
            mbar_init(&sm.sin_full[i], 128);  // every chain thread arrives
            mbar_init(&sm.mma2[i], 1);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(&sm.x_full[i], CONV ? 2 : 1);  // the TMA's arrive (with its bytes); with the convolution
                                                     // also the arrive after the taps and the halo
            mbar_init(&sm.x_empty[i], 4);  // one lane per epilogue warp, after its y store has read the slot
        }
        for (int i = 0; i < 4; ++i) mbar_init(&sm.tab_full[i], 1);
        mbar_init(&sm.cb_full, 1);
        mbar_init(&sm.cb_empty, 128);
        mbar_init(&sm.unit_go, 128);
        mbar_init(&sm.drain[0], 1);
        mbar_init(&sm.drain[1], 1);
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
        // Per unit: ticket, B/C tiles by TMA; and, for the unit requested one iteration earlier (so its TMA latency
        // is already behind it), the bf16 -> fp16 conversion of B/C in place (same 16-bit positions, same swizzle),
        // or with the fused convolution the B/C columns convolved in place. Tickets are fetched one unit ahead, or,
        // when the state chain bounds the launch (few units per chunk index), only once the unit before is three
        // heads from its end: a ticket taken early sits on a CTA that is busy for a whole unit more, and the chain
        // reaching that chunk waits for it; late tickets follow the order in which CTAs free up.
        if (lane == 0) {
            prefetch_tensormap(&map_b);
            prefetch_tensormap(&map_c);
        }
        int armed_bc = 0;  // for the drain at teardown
        uint32_t bc_par[2] = {0, 0};
        uint32_t t = 0;
        if (lane == 0) t = atomicAdd(&hdr->ticket, 1u);
        t = __shfl_sync(0xffffffffu, t, 0);
        Sched prev{0, 0, 0, 0, 0, 0, 0, 0};
        const uint32_t total = total_units(p, (uint32_t)(p.G * slices));
        const bool late = p.tc_late_ticket != 0;
        auto finish = [&](uint32_t vv, const Sched &sc) -> bool {
            const uint32_t uu = vv & 1;
            if (!BWAIT(&sm.bc_full[uu], (vv >> 1) & 1)) return false;
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
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.bc_conv[uu]);
                TRACE(warp, 2, vv);
            }
            return true;
        };
        for (uint32_t v = 0;; ++v) {
            const uint32_t u = v & 1, nn = v >> 1;
            uint32_t t_next = 0;
            if (!late && lane == 0 && t < total) t_next = atomicAdd(&hdr->ticket, 1u);  // in flight meanwhile
            // the previous unit first: the MMA issuer frees stage u (unit v-2's last C.S) only after it
            // has seen unit v-1 converted
            if (v > 0 && !finish(v - 1, prev)) break;
            if (late && v > 0) {  // the ticket only now that the unit before it is three heads from its end
                if (!BWAIT(&sm.unit_go, (v - 1) & 1)) break;
                if (lane == 0) t = atomicAdd(&hdr->ticket, 1u);
                t = __shfl_sync(0xffffffffu, t, 0);
            }
            if (!BWAIT(&sm.bc_empty[u], (nn & 1) ^ 1)) break;
            if (t >= total) {
                if (lane == 0) {
                    sm.sched[u].valid = 0;
                    mbar_arrive(&sm.sched_full[u]);
                    mbar_arrive(&sm.bc_conv[u]);
                }
                break;
            }
            const SeqChunk sq = seq_chunk(p, t / (p.G * slices));
            const int64_t r = t % (p.G * slices);
            const int64_t c = sq.c;
            const int64_t g = r / slices;
            const int64_t h0 = g * p.heads_per_group + (r % slices) * hs;
            const int64_t row0 = sq.tok0 + c * kQ;
            const int rows = (int)((sq.len - c * kQ) < kQ ? (sq.len - c * kQ) : kQ);
            const int last = c == (sq.len + kQ - 1) / kQ - 1;
            const Sched cur{1, (int32_t)sq.s, (int32_t)c, (int32_t)g, (int32_t)h0, rows, (int32_t)row0, last};
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
                TRACE(warp, 1, v);
            }
            __syncwarp();
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
    } else if (warp == 2) {
        // ------------------------------------------------------------ x loader
        // Per head: the x tile by one TMA into the 3-deep ring (and, with the fused convolution, the 3 raw rows
        // before the chunk and the head's taps), then the head's chunk cumsum: dt = softplus(dt_raw + dt_bias)
        // (0 past the sequence end), inclusive scan of dt*A over the 128 rows, into the slot's tables. The end of
        // the work goes to the consumers as a table with valid = 0.
        if (lane == 0) {
            prefetch_tensormap(&map_x);
            if (CONV) prefetch_tensormap(&map_xh);
        }
        const IO *dtr = static_cast<const IO *>(p.dt_raw);
        const int64_t ndt = p.batch * p.L * p.H;  // dt_raw extent (bounds-checked builds)
#ifdef SSD_BOUNDS_CHECK
        const int64_t probe = hdr->bounds_probe ? ndt : 0;  // test hook: plant the dt rows one extent further
#else
        const int64_t probe = 0;
#endif
        uint32_t hc = 0;
        int armed_x = 0;
        uint32_t x_par[3] = {0, 0, 0};
        bool done = false;
        for (uint32_t v = 0; !done; ++v) {
            const uint32_t u = v & 1;
            if (!BWAIT(&sm.sched_full[u], (v >> 1) & 1)) break;
            const Sched sc = sm.sched[u];
            const int nh = sc.valid ? hs : 1;
            // dt_raw rows 4*lane .. 4*lane+3 of every head of the unit, all loads in flight at once (one memory
            // latency per unit rather than per head)
            float raw[4][kMaxHs];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int i = 4 * lane + jj;
#pragma unroll
                for (int hh = 0; hh < kMaxHs; ++hh)
                    raw[jj][hh] = sc.valid && hh < hs && i < sc.rows
                                      ? to_f32(*chk(dtr, (sc.row0 + i) * p.H + sc.h0 + hh + probe, 1, ndt, hdr, SITE_TC_DT))
                                      : 0.f;
            }
            // the unit's per-head parameters, lane hh holding head h0 + hh's (broadcast per head by shuffles)
            const bool own = sc.valid && lane < hs;
            const float u_bias = own ? p.dt_bias[sc.h0 + lane] : 0.f, u_A = own ? p.A[sc.h0 + lane] : 0.f;
            const float u_D = own && p.D ? p.D[sc.h0 + lane] : 0.f;
            for (int hh = 0; hh < nh; ++hh, ++hc) {
                const uint32_t k = hc % 3, n = hc / 3;
                HeadTab &tb = sm.tab[hc % 4];  // last read by head hc - 4, whose slot's wait passed a head ago
                if (!sc.valid) {
                    if (!BWAIT(&sm.x_empty[k], (n & 1) ^ 1)) {
                        done = true;
                        break;
                    }
                    if (lane == 0) {
                        tb.valid = 0;
                        mbar_arrive(&sm.tab_full[hc % 4]);
                        mbar_arrive(&sm.x_full[k]);
                        if (CONV) mbar_arrive(&sm.x_full[k]);
                    }
                    done = true;
                    break;
                }
                const int h = sc.h0 + hh;
                // the head's table first, while the x slot may still be in use (its barrier is already in this
                // head's phase: the phase before completed when head hc - 3's tile landed)
                float rh[4];  // this head's column of raw (a register select: hh is not a compile-time index)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    rh[jj] = raw[jj][0];
#pragma unroll
                    for (int e = 1; e < kMaxHs; ++e) rh[jj] = hh == e ? raw[jj][e] : rh[jj];
                }
                const float bias = __shfl_sync(0xffffffffu, u_bias, hh), Ah = __shfl_sync(0xffffffffu, u_A, hh);
                const float dskip = __shfl_sync(0xffffffffu, u_D, hh);
                float dtv[4], cum[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    dtv[jj] = 4 * lane + jj < sc.rows ? softplus_ool(rh[jj] + bias) : 0.f;
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
                reinterpret_cast<float4 *>(tb.cs2)[lane] = make_float4(cs2v[0], cs2v[1], cs2v[2], cs2v[3]);
                reinterpret_cast<float4 *>(tb.dt)[lane] = make_float4(dtv[0], dtv[1], dtv[2], dtv[3]);
                reinterpret_cast<float4 *>(tb.wt)[lane] =
                    make_float4(ex2(anchor - cs2v[0]) * dtv[0], ex2(anchor - cs2v[1]) * dtv[1],
                                ex2(anchor - cs2v[2]) * dtv[2], ex2(anchor - cs2v[3]) * dtv[3]);
                if (lane == 0) {
                    tb.valid = 1;
                    tb.h = h;
                    tb.hh = hh;
                    tb.v = (int32_t)v;
                    tb.c = sc.c;
                    tb.s = sc.s;
                    tb.row0 = sc.row0;
                    tb.rows = sc.rows;
                    tb.last = sc.last;
                    tb.dskip = dskip;
                }
                __syncwarp();
                if (lane == 0) {  // the table's readers that need no x (P, C.S, chain) start from here
                    mbar_arrive(&sm.tab_full[hc % 4]);
                    TRACE(warp, 2, hc);
                }
                if (!BWAIT(&sm.x_empty[k], (n & 1) ^ 1)) {
                    done = true;
                    break;
                }
                const bool halo_tma = CONV && sc.c > 0;
                if (lane == 0) {
                    TRACE(warp, 1, hc);
                    mbar_arrive_expect_tx(&sm.x_full[k], kTile + (halo_tma ? 3 * kP * 2 : 0));
                    tma_load_4d(sm.x[k], &map_x, &sm.x_full[k], 0, h, sc.row0, 0);
                    if constexpr (CONV) {
                        if (halo_tma) tma_load_4d(sm.cv.halo[k], &map_xh, &sm.x_full[k], 0, h, sc.row0 - 3, 0);
                    }
                    armed_x |= 1 << k;
                    x_par[k] = n & 1;
                }
                if constexpr (CONV) {  // the head's taps and bias (read as broadcasts), the cache before a sequence
                    const int64_t ch0 = (int64_t)h * kP;
                    for (int e = lane; e < kP; e += 32) {
                        sm.cv.tap[k][e] = *reinterpret_cast<const float4 *>(p.conv_w + (ch0 + e) * 4);
                        sm.cv.bias[k][e] = p.conv_b ? p.conv_b[ch0 + e] : 0.f;
                    }
                    if (sc.c == 0) {
                        const IO *st = static_cast<const IO *>(p.conv_state);
                        IO *dst = reinterpret_cast<IO *>(sm.cv.halo[k]);
                        for (int e = lane; e < 3 * kP; e += 32) {
                            const int r = e / kP, pc = e % kP;
                            dst[r * kP + pc] = st ? *chk(st, ((int64_t)sc.s * p.x_ld + ch0 + pc) * 3 + r, 1,
                                                         p.nseq * p.x_ld * 3, hdr, SITE_CONV_STATE)
                                                  : from_f32<IO>(0.f);
                        }
                    }
                }
                if constexpr (CONV) {  // with the convolution the slot's taps and halo are part of what is announced
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.x_full[k]);
                }
            }
        }
        if (lane == 0 && *reinterpret_cast<volatile int32_t *>(&sm.abort)) {
            for (int k = 0; k < 3; ++k)
                if (armed_x & (1 << k)) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(&sm.x_full[k], x_par[k]) && globaltimer() - t0 < 100000000ull) {
                    }
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer: CB and MMA1
        // Event driven: heads h are numbered across units (unit h / hs). For each head it issues MMA1 (P.x and
        // the chunk state) once P, X_s and the head's accumulators are ready; CB of a unit goes out before the
        // unit's first MMA1. The whole warp runs the loop on warp-uniform values (every barrier test is made
        // uniform across the lanes) and one elected lane issues each burst with its K steps unrolled: issued this
        // way a burst completes in about half the time of one lane's rolled loop (16 MMAs: ~810 against ~1750
        // cycles), and the burst is on every head's critical path.
        {
            constexpr uint32_t idCB = idesc_f16_f32(128, 128, false, false);
            constexpr uint32_t idPX = idesc_f16_f32(128, 64, false, true);
            constexpr uint32_t idST = idesc_f16_f32(128, 64, true, true);
            const uint32_t uhs = (uint32_t)hs;
            const bool leader = elect_one();
            uint32_t v_cb = 0;  // next unit whose CB is due
            uint32_t h1 = 0;    // next head for MMA1
            uint64_t idle_since = 0;
            uint32_t idle = 0;
            const uint64_t limit = 4 * (hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs) + 100000000ull;
            auto ready = [&](uint64_t *bar, uint32_t par) { return __all_sync(0xffffffffu, mbar_test_wait(bar, par)); };
            // Every barrier is polled without suspending (a thread suspended on one barrier does not wake for
            // another); an idle round sleeps a few tens of ns, and the clock is read once per 256 idle rounds.
            for (;;) {
                bool progress = false;
                // CB of unit v_cb, due when MMA1 has reached its first head and the P warps are done with the last
                if (h1 == v_cb * uhs && ready(&sm.bc_conv[v_cb & 1], (v_cb >> 1) & 1)) {
                    const uint32_t u = v_cb & 1;
                    if (!__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int32_t *>(&sm.sched[u].valid), 0))
                        break;  // no more work
                    if (ready(&sm.cb_empty, (v_cb & 1) ^ 1)) {
                        tc_fence_after();
                        const uint64_t da = desc_sw128(smem_u32(sm.bc[u][2]), 16, 1024);
                        const uint64_t db = desc_sw128(smem_u32(sm.bc[u][0]), 16, 1024);
                        if (leader) {
#pragma unroll
                            for (uint32_t s = 0; s < 8; ++s) {  // K step s: 16-bit tile s / 4, 32-byte column s % 4
                                const uint64_t off = (s >> 2) * (kTile >> 4) + (s & 3) * 2;
                                mma_ss(tmem + kColCB, da + off, db + off, idCB, s > 0);
                            }
                            mma_commit(&sm.cb_full);
                        }
                        __syncwarp();
                        if (lane == 0) TRACE(warp, 1, v_cb);
                        ++v_cb;
                        progress = true;
                    }
                }
                // MMA1 of head h1: y_intra = P . x and s = B^T . X_s
                if (h1 < v_cb * uhs) {
                    const uint32_t k = h1 & 1, n = h1 >> 1;
                    if (ready(&sm.p_full[k], n & 1) && ready(&sm.xs_full[k], n & 1) &&
                        ready(&sm.acc_free[k], (n & 1) ^ 1)) {
                        const uint32_t u = (h1 / uhs) & 1;
                        tc_fence_after();
                        const uint64_t dx = desc_sw128(smem_u32(sm.x[h1 % 3]), 8192, 1024);
                        const uint64_t dbt = desc_sw128(smem_u32(sm.bc[u][0]), kTile, 1024);
                        const uint64_t dxs = desc_sw128(smem_u32(sm.xs[k]), 8192, 1024);
                        if (leader) {
#pragma unroll
                            for (uint32_t s = 0; s < 8; ++s)  // K step s: 16 rows = 2048 bytes further
                                mma_ts(tmem + kColYI + 64 * k, tmem + kColP + 64 * k + 8 * s, dx + 128 * s, idPX, s > 0);
#pragma unroll
                            for (uint32_t s = 0; s < 8; ++s)
                                mma_ss(tmem + kColS + 64 * k, dbt + 128 * s, dxs + 128 * s, idST, s > 0);
                            mma_commit(&sm.mma1[k]);
                        }
                        __syncwarp();
                        if (lane == 0) TRACE(warp, 2, h1);
                        ++h1;
                        progress = true;
                    }
                }
                if (progress) {
                    idle = 0;
                } else {
                    if ((++idle & 255u) == 0) {
                        if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int32_t *>(&sm.abort), 0)) break;
                        const uint64_t now = __shfl_sync(0xffffffffu, globaltimer(), 0);
                        if (idle == 256u) {
                            idle_since = now;
                        } else if (now - idle_since > limit) {
                            if (lane == 0) pipe_timeout(abort_flag, hdr, epoch);
                            break;
                        }
                    }
                    __nanosleep(32);
                }
            }
            // drain: every MMA issued above has completed before TMEM is released
            if (leader) {
                mma_commit(&sm.drain[0]);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&sm.drain[0], 0) && globaltimer() - t0 < 1000000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------------------ MMA issuer: C.S
        // Per head, once the chain has put the entering state into shared memory: y_inter = C . S_in into the
        // columns of the head's chunk state (already read by the chain). Issued apart from MMA1 so that neither
        // waits behind the other's issue; like MMA1, by one elected lane of the whole warp, K steps unrolled.
        // With fp32 states and per-head flags (HF) this warp also publishes the head's leaving state:
        // every chain thread stored its row before arriving on sin_full (release, CTA scope), this warp's wait
        // acquires them, and one release store of the head's flag at GPU scope (cumulative: it orders the rows
        // this warp has observed) publishes the whole state, right after C.S is issued. The chain threads then
        // never wait on a release fence (about half a microsecond a head), at the price of a later publish.
        {
            constexpr uint32_t idCS = idesc_f16_f32(128, 64, false, true);
            const bool leader = elect_one();
            const int64_t skip = hdr->skip_publish - 1;
            uint64_t *flags = reinterpret_cast<uint64_t *>(p.flags);  // [chain][slot][row]: row 0's place per head
            (void)skip;
            (void)flags;
            for (uint32_t h2 = 0;; ++h2) {
                const uint32_t k3 = h2 % 3, k = h2 & 1;
                if (!BWAIT(&sm.tab_full[h2 % 4], (h2 / 4) & 1)) break;
                const int32_t valid = sm.tab[h2 % 4].valid, last_of_unit = sm.tab[h2 % 4].hh == hs - 1;
                if (!valid) break;
                if (!BWAIT(&sm.sin_full[k], (h2 >> 1) & 1)) break;
                const uint32_t u = (h2 / (uint32_t)hs) & 1;
                tc_fence_after();
                const uint64_t da = desc_sw128(smem_u32(sm.bc[u][2]), 16, 1024);
                const uint64_t db = desc_sw128(smem_u32(sm.x[k3]), 8192, 1024);
                if (leader) {
#pragma unroll
                    for (uint32_t s = 0; s < 8; ++s)
                        mma_ss(tmem + kColS + 64 * k, da + (s >> 2) * (kTile >> 4) + (s & 3) * 2, db + 128 * s, idCS,
                               s > 0);
                    mma_commit(&sm.mma2[k]);
                    if (last_of_unit) mma_commit(&sm.bc_empty[u]);  // last reader of the unit's B/C
                }
                __syncwarp();
                if constexpr (HF) {
                    const HeadTab &tb = sm.tab[h2 % 4];
                    const int c = tb.c;
                    // no publish after the last chunk of a sequence or of a segment
                    if (lane == 0 && !tb.last && c != skip && !(p.nseg > 1 && (c + 1) % p.seg_chunks == 0))
                        st_release_u64(chk(flags, (chain_of(p, tb.s, c, tb.h) * 2 + ((c + 1) & 1)) * kN, 1,
                                           p.flag_count, hdr, SITE_TC_FLAG),
                                       ((uint64_t)epoch << 32) | (uint32_t)(c + 1));
                    __syncwarp();
                }
                if (lane == 0) TRACE(warp, 3, h2);
            }
            if (leader) {
                mma_commit(&sm.drain[1]);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&sm.drain[1], 0) && globaltimer() - t0 < 1000000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ P / X_s warpgroup
        // Per head P, then X_s. P = CB o decay o dt, masked above the diagonal, fp16 into the head's P slot. One 32-column block of CB
        // per step. Blocks above the diagonal block stay zero: they are written once here, and nothing else writes
        // the P columns. Below the diagonal block exp(cs_i - cs_j) = exp(cs_i - cs_a) exp(cs_a - cs_j) with a the
        // block's last row, both factors <= 1 (the semiseparable off-diagonal blocks are low rank). In the
        // diagonal block the first factor is >= 1, so the split is used only while the block's whole decay range
        // keeps it <= 2^100 (warp-uniform test), else exp is taken per element; the mask then clears every column
        // past the row's own (an inf or NaN there included) by bit masks on the packed halves.
        // X_s = exp(cs_last - cs_j) dt_j x_j (and the x tile to fp16 in place) into the head's X_s buffer, once
        // the x tile has landed.
        const int q = warp & 3;       // TMEM lane quarter of this warp
        const int i = 32 * q + lane;  // tile row (token within the chunk) owned by this thread
        const uint32_t lrow = (uint32_t)(32 * q) << 16;
        {
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
            for (int k = 0; k < 2; ++k)
                for (int J = q + 1; J < 4; ++J) tmem_st16(tmem + lrow + kColP + 64 * k + 16 * J, z);
            tmem_st_wait();
        }
        // diagonal-block masks: keep columns e <= lane (low half of pair m: column 2m, high half: 2m + 1)
        uint32_t dmask[16];
#pragma unroll
        for (int m = 0; m < 16; ++m)
            dmask[m] = (2 * m <= lane ? 0x0000ffffu : 0u) | (2 * m + 1 <= lane ? 0xffff0000u : 0u);
        for (uint32_t hc = 0;; ++hc) {
            const uint32_t k3 = hc % 3, n3 = hc / 3, k2 = hc & 1, n2 = hc >> 1;
            if (!BWAIT(&sm.tab_full[hc % 4], (hc / 4) & 1)) break;  // the head's table (its x tile is not needed)
            const HeadTab &tb = sm.tab[hc % 4];
            if (!tb.valid) break;
            if (!BWAIT(&sm.mma1[k2], (n2 & 1) ^ 1)) break;  // P slot and X_s buffer free: MMA1 of head hc - 2 done
            if (tb.hh == 0 && !BWAIT(&sm.cb_full, tb.v & 1)) break;
            tc_fence_after();
            if (lane == 0) TRACE(warp, 1, hc);
            const float cs2i = tb.cs2[i];
            const uint32_t pcol = tmem + lrow + kColP + 64 * k2;
            const float dk = tb.dskip;
            const float4 dadd = make_float4((lane & 3) == 0 ? dk : 0.f, (lane & 3) == 1 ? dk : 0.f,
                                            (lane & 3) == 2 ? dk : 0.f, (lane & 3) == 3 ? dk : 0.f);
#pragma unroll 1
            for (int J = 0; J <= q; ++J) {
                const float ca = tb.cs2[32 * J + 31];
                const bool diag = J == q;
                if (diag && tb.cs2[32 * J] - ca > 100.f) {  // rare: decay range too wide for the split
                    p_block_exact(tmem + lrow + kColCB + 32 * J, pcol + 16 * J, tb.cs2 + 32 * J, tb.dt + 32 * J, cs2i,
                                  tb.dskip);
                    continue;
                }
                const int ed = diag ? lane >> 2 : -1;  // the 4-column group holding this row's diagonal element
                float4 t1[8];
                const float4 *s1 = reinterpret_cast<const float4 *>(tb.wt + 32 * J);
#pragma unroll
                for (int e = 0; e < 8; ++e) t1[e] = s1[e];
                const float ui = ex2(cs2i - ca);
                uint32_t cb[32];
                tmem_ld16(tmem + lrow + kColCB + 32 * J, *reinterpret_cast<uint32_t(*)[16]>(&cb[0]));
                tmem_ld16(tmem + lrow + kColCB + 32 * J + 16, *reinterpret_cast<uint32_t(*)[16]>(&cb[16]));
                tmem_ld_wait();
                uint32_t pk[16];
                const float2 uu = make_float2(ui, ui);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float2 a = fmul2(fmul2(f2(cb[4 * e], cb[4 * e + 1]), make_float2(t1[e].x, t1[e].y)), uu);
                    float2 b = fmul2(fmul2(f2(cb[4 * e + 2], cb[4 * e + 3]), make_float2(t1[e].z, t1[e].w)), uu);
                    if (e == ed) {  // D x_i enters y through P's diagonal (added before the fp16 rounding)
                        a.x += dadd.x;
                        a.y += dadd.y;
                        b.x += dadd.z;
                        b.y += dadd.w;
                    }
                    pk[2 * e] = pack_f16(a.x, a.y);
                    pk[2 * e + 1] = pack_f16(b.x, b.y);
                }
                if (diag) {
#pragma unroll
                    for (int m = 0; m < 16; ++m) pk[m] &= dmask[m];
                }
                tmem_st16(pcol + 16 * J, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_full[k2]);
            if (lane == 0) TRACE(warp, 2, hc);
            if (tb.hh == hs - 1) mbar_arrive(&sm.cb_empty);
            if (tb.hh == (hs > 3 ? hs - 3 : 0)) mbar_arrive(&sm.unit_go);  // late tickets: the next unit
            // X_s of the same head (x tile landed; its buffer was released with the P slot, by MMA1 two heads back)
            if (!BWAIT(&sm.x_full[k3], n3 & 1)) break;
            if (lane == 0) TRACE(warp, 6, hc);
            const float xscale = ex2(tb.cs2[kQ - 1] - tb.cs2[i]) * tb.dt[i];
            uint8_t *xr = sm.x[k3] + i * 128;
            uint8_t *sr = sm.xs[k2] + i * 128;
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
                        rr[j] = r >= 0 ? lds128(sm.x[k3] + r * 128 + ((lc ^ (r & 7)) << 4))
                                       : lds128(sm.cv.halo[k3] + (r + 3) * 128 + lc * 16);
                    }
                    const float4 bb0 = reinterpret_cast<const float4 *>(sm.cv.bias[k3])[2 * lc];
                    const float4 bb1 = reinterpret_cast<const float4 *>(sm.cv.bias[k3])[2 * lc + 1];
                    const float bias8[8] = {bb0.x, bb0.y, bb0.z, bb0.w, bb1.x, bb1.y, bb1.z, bb1.w};
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {  // channel pairs of this 16-byte chunk
                        float o[2];
#pragma unroll
                        for (int c2 = 0; c2 < 2; ++c2) {
                            const int e = 2 * e2 + c2;
                            const float4 tw = sm.cv.tap[k3][8 * lc + e];
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
                bar_sync(kBarE, 128);  // every thread has read its raw rows: the tile may be overwritten
#pragma unroll
                for (int lc = 0; lc < 8; ++lc) {
                    const int off = (lc ^ (i & 7)) << 4;
                    sts128(xr + off, make_uint4(xo[4 * lc], xo[4 * lc + 1], xo[4 * lc + 2], xo[4 * lc + 3]));
                    sts128(sr + off, make_uint4(so[4 * lc], so[4 * lc + 1], so[4 * lc + 2], so[4 * lc + 3]));
                }
            } else {
                const float2 xs2 = make_float2(xscale, xscale);
#pragma unroll 2
                for (int lc = 0; lc < 8; ++lc) {
                    const int off = (lc ^ (i & 7)) << 4;
                    uint4 w = lds128(xr + off);
                    uint32_t *wv = reinterpret_cast<uint32_t *>(&w);
                    uint4 s4;
                    uint32_t *sv = reinterpret_cast<uint32_t *>(&s4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = unpack_io<IO>(wv[e]);
                        const float2 sc = fmul2(f, xs2);
                        sv[e] = pack_f16(sc.x, sc.y);
                        if (kBf16) wv[e] = pack_f16(f.x, f.y);
                    }
                    if (kBf16) sts128(xr + off, w);
                    sts128(sr + off, s4);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.xs_full[k2]);
            if (lane == 0) TRACE(warp, 7, hc);
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ epilogue warpgroup
        // Per head, after its C.S: y = y_intra + exp(cs_i) y_inter (D x is in y_intra through P's diagonal),
        // staged in the head's x slot in the y map's 128B swizzle and sent by one TMA store per warp (32 rows);
        // the store clips rows past the sequence end. These warps do nothing else, so that no other phase of a
        // later head waits behind an epilogue (X_s of head h + 2 once did, and the chain of waits MMA1 -> chain ->
        // C.S -> epilogue -> X_s paced every head).
        const int q = warp & 3;
        const int i = 32 * q + lane;
        const uint32_t lrow = (uint32_t)(32 * q) << 16;
        if (lane == 0) prefetch_tensormap(&map_y);
        IO *yg = static_cast<IO *>(p.y);
        auto epilogue = [&](uint32_t hp) -> bool {
            const uint32_t k2 = hp & 1, n2 = hp >> 1, k3 = hp % 3;
            if (!BWAIT(&sm.mma2[k2], n2 & 1)) return false;
            tc_fence_after();
            if (lane == 0) TRACE(warp, 3, hp);
            const HeadTab &tb = sm.tab[hp % 4];
            const float ecs = ex2(tb.cs2[i]);
            uint8_t *row = sm.x[k3] + i * 128;  // y row i, staged in the head's x slot (C.S has read S_in there)
            const float2 e2 = make_float2(ecs, ecs);
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {  // columns 16 m .. 16 m + 15: 16-byte chunks 2 m, 2 m + 1 of the row
                uint32_t a[16], c2[16];
                tmem_ld16(tmem + lrow + kColYI + 64 * k2 + 16 * m, a);
                tmem_ld16(tmem + lrow + kColS + 64 * k2 + 16 * m, c2);
                const int o0 = ((2 * m) ^ (i & 7)) << 4, o1 = ((2 * m + 1) ^ (i & 7)) << 4;
                tmem_ld_wait();
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 y = ffma2(e2, f2(c2[2 * e], c2[2 * e + 1]), f2(a[2 * e], a[2 * e + 1]));
                    o[e] = pack_io<IO>(y.x, y.y);
                }
                sts128(row + o0, make_uint4(o[0], o[1], o[2], o[3]));
                sts128(row + o1, make_uint4(o[4], o[5], o[6], o[7]));
            }
            tc_fence_before();
            mbar_arrive(&sm.acc_free[k2]);  // y_intra and y_inter of this slot have been read
            if (lane == 0) TRACE(warp, 5, hp);
            const int vr = tb.rows - 32 * q, ph = tb.h, prow = tb.row0 + 32 * q;
            if (vr >= 32) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_4d(&map_y, sm.x[k3] + 32 * q * 128, 0, ph, prow, 0);
                    bulk_commit();
                    TRACE(warp, 6, hp);
                    bulk_wait_read0();  // the store has read the slot
                    mbar_arrive(&sm.x_empty[k3]);
                }
            } else {
                if (lane < vr) {  // ragged last chunk: the valid rows one by one (the next sequence follows)
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        chk(yg, ((int64_t)(prow + lane) * p.H + ph) * kP, kP, p.batch * p.L * p.H * kP, hdr, SITE_TC_Y));
#pragma unroll
                    for (int lc = 0; lc < 8; ++lc) dst[lc] = lds128(row + ((lc ^ (i & 7)) << 4));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.x_empty[k3]);
            }
            __syncwarp();
            if (lane == 0) TRACE(warp, 4, hp);
            return true;
        };
        bool ok = true;
        for (uint32_t hc = 0;; ++hc) {
            if (!BWAIT(&sm.tab_full[hc % 4], (hc / 4) & 1)) {
                ok = false;
                break;
            }
            if (!sm.tab[hc % 4].valid) break;
            if (!epilogue(hc)) {
                ok = false;
                break;
            }
        }
        (void)ok;
        if (lane == 0) bulk_wait0();  // every y store of this warp has completed
        __syncwarp();
    } else if (warp >= 12) {
        // ------------------------------------------------------------ chain warpgroup
        // Thread n owns d_state row n of every state and passes it to the next chunk through a 2-slot ring per
        // chain, with no CTA barrier on either side of a hop:
        //  - fp32 states: the row, then its release flag (a 64-bit tag epoch:chunk): per row, by its thread, or
        //    (HF) one per head, by the C.S warp once all 128 rows are stored;
        //  - fp16 states: every 8-byte ring word carries two values and the 32-bit tag epoch * 1024 + (chunk mod
        //    1024). A slot can still hold any earlier chunk of its chain that a unit in flight has not yet
        //    overwritten; at most two tickets per CTA are unfinished, so those chunks lie fewer than 2 x SMs
        //    (< 1024) indices back, and the chunk field tells them apart. An aligned 8-byte access is single-copy
        //    atomic, so a word with the expected tag holds this launch's values for that chunk: the data is its
        //    own flag (no release, no flag load), which shortens the serial chain of hops by a round trip.
        // The entering row is fetched (and, if need be, awaited) first; then s_c is read from TMEM in four pieces
        // of 16 columns, each combined, published and written to the C.S operand at once.
        const int q = warp & 3;
        const int nrow = 32 * q + lane;  // state row (d_state index) owned by this thread
        const uint32_t lrow = (uint32_t)(32 * q) << 16;
        const uint64_t limit = hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs;
        const int64_t skip = hdr->skip_publish - 1;
        const ST *init = static_cast<const ST *>(p.init);
        ST *fin = static_cast<ST *>(p.final_states);
        uint64_t *tags = reinterpret_cast<uint64_t *>(p.flags);  // [chain][slot][row]
        constexpr bool kTagged = sizeof(ST) == 2 && !HF;  // fp16 states in tagged words
        constexpr bool kPlain16 = sizeof(ST) == 2 && HF;  // fp16 states as plain halves behind the head's flag
        ulonglong2 *ringv = static_cast<ulonglong2 *>(p.ring);  // fp16: [chain][slot][P / 4 vectors][row]
        const int64_t nvec = p.ring_bytes / 16, nstate = p.nseq * p.H * kP * kN;  // extents (bounds-checked builds)
        // row nrow of a slot: 16 vectors kN apart (checked as one span)
        auto vrow_of = [&](int64_t chain, int c) {
            return chk(ringv, (chain * 2 + (c & 1)) * (int64_t)(kP / 4 * kN) + nrow, (kP / 4 - 1) * kN + 1, nvec, hdr,
                       SITE_TC_RING);
        };
        auto vtag = [&](int c) { return (epoch << 10) | (uint32_t)(c & 1023); };
        auto tag_of = [&](int64_t chain, int c) {  // fp32: the row's flag, or with HF the head's (row 0's place)
            return chk(tags, (chain * 2 + (c & 1)) * kN + (HF ? 0 : nrow), 1, p.flag_count, hdr, SITE_TC_FLAG);
        };
        auto want_of = [&](int c) { return ((uint64_t)epoch << 32) | (uint32_t)c; };
        float S[kP];  // entering state of the current head (fp32)
        for (uint32_t hc = 0;; ++hc) {
            const uint32_t k2 = hc & 1, n2 = hc >> 1;
            if (!BWAIT(&sm.tab_full[hc % 4], (hc / 4) & 1)) break;  // the head's table (its x tile is not needed)
            const HeadTab &tb = sm.tab[hc % 4];
            if (!tb.valid) break;
            const int64_t chain = (int64_t)tb.s * p.H + tb.h;  // (sequence, head): initial and final states
            const int c = tb.c;
            const int64_t rchain = chain_of(p, tb.s, c, tb.h);  // the state chain through the ring
            const bool last = tb.last != 0;
            const bool seg_start = p.nseg > 1 && c > 0 && c % p.seg_chunks == 0;
            if (lane == 0) TRACE(warp, 1, hc);
            // state entering the chunk
            if (c == 0) {
#pragma unroll
                for (int pp = 0; pp < kP; ++pp)
                    S[pp] = init ? to_f32(*chk(init, (chain * kP + pp) * kN + nrow, 1, nstate, hdr, SITE_TC_INIT)) : 0.f;
            } else if (seg_start) {  // the segment's entering state, computed before this launch
                const int64_t base = ((tb.s * (p.nseg - 1) + c / p.seg_chunks - 1) * p.H + tb.h) * kP * kN + nrow;
#pragma unroll
                for (int pp = 0; pp < kP; ++pp)
                    S[pp] = __ldcg(chk(p.seg_states, base + pp * kN, 1, p.nseq * (p.nseg - 1) * p.H * kP * kN, hdr,
                                       SITE_TC_INIT));
            } else if (kTagged) {
                const uint32_t want = vtag(c);
                uint64_t raw[kTagged ? kP / 2 : 1];
                auto issue = [&]() {
                    const ulonglong2 *src = vrow_of(rchain, c);
#pragma unroll
                    for (int j = 0; j < (kTagged ? kP / 4 : 0); ++j) {
                        const ulonglong2 t = ld_ring(src + j * kN);
                        raw[2 * j] = t.x;
                        raw[2 * j + 1] = t.y;
                    }
                };
                auto stale = [&]() {
                    uint32_t bad = 0;
#pragma unroll
                    for (int w = 0; w < (kTagged ? kP / 2 : 0); ++w) bad |= (uint32_t)(raw[w] >> 32) ^ want;
                    return bad != 0;
                };
                issue();
                bool ok = !stale();
                while (!ok) {  // not yet published, or only partly visible: wait on the row's last vector, reload
                    if (aborted(hdr, epoch) ||
                        !wait_ring(vrow_of(rchain, c) + (kP / 4 - 1) * kN, want, epoch, hdr, limit, (uint32_t)c))
                        break;
                    issue();
                    ok = !stale();
                }
#pragma unroll
                for (int w = 0; w < (kTagged ? kP / 2 : 0); ++w) {  // zeros after a recorded error: the CTA drains
                    const float2 f = ok ? unpack_f16((uint32_t)raw[w]) : make_float2(0.f, 0.f);
                    S[2 * w] = f.x;
                    S[2 * w + 1] = f.y;
                }
            } else if (ld_acquire_u64(tag_of(rchain, c)) == want_of(c) ||
                       (!aborted(hdr, epoch) && wait_tag(tag_of(rchain, c), want_of(c), epoch, hdr, limit, (uint32_t)c))) {
                if constexpr (kPlain16) {  // 8 vectors of 8 halves, kN apart
                    const uint4 *src = chk(reinterpret_cast<const uint4 *>(p.ring),
                                           (rchain * 2 + (c & 1)) * (int64_t)(kP / 8 * kN) + nrow,
                                           (kP / 8 - 1) * kN + 1, nvec, hdr, SITE_TC_RING);
#pragma unroll
                    for (int m = 0; m < kP / 8; ++m) {
                        const uint4 v = __ldcg(src + m * kN);
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_f16(w4[e]);
                            S[8 * m + 2 * e] = f.x;
                            S[8 * m + 2 * e + 1] = f.y;
                        }
                    }
                } else {
                    const float4 *src = chk(reinterpret_cast<const float4 *>(p.ring),
                                            (rchain * 2 + (c & 1)) * (int64_t)(kP / 4 * kN) + nrow,
                                            (kP / 4 - 1) * kN + 1, nvec, hdr, SITE_TC_RING);
#pragma unroll
                    for (int m = 0; m < kP / 4; ++m) {
                        const float4 f = __ldcg(src + m * kN);
                        S[4 * m] = f.x;
                        S[4 * m + 1] = f.y;
                        S[4 * m + 2] = f.z;
                        S[4 * m + 3] = f.w;
                    }
                }
            } else {  // the error is recorded; carry on with zeros so the CTA drains
#pragma unroll
                for (int pp = 0; pp < kP; ++pp) S[pp] = 0.f;
            }
            // chunk state s_c from TMEM, in pieces of 16 columns: S_out = a S_in + s_c, published; S_in to the
            // C.S operand (K-row nrow of a [128 x 64] MN-major 128B-swizzled tile)
            if (lane == 0) TRACE(warp, 2, hc);
            if (!BWAIT(&sm.mma1[k2], n2 & 1)) break;
            tc_fence_after();
            if (lane == 0) TRACE(warp, 3, hc);
            const float a = ex2(tb.cs2[kQ - 1]);  // decay across the chunk
            // no publish after the last chunk of a sequence or of a segment (the next segment starts from its own
            // entering state)
            const bool publish = !last && c != skip && !(p.nseg > 1 && (c + 1) % p.seg_chunks == 0);
            uint8_t *srow = sm.x[hc % 3] + nrow * 128;  // the x tile is dead once MMA1 has read it
            float4 *dst32 = nullptr;
            ulonglong2 *dst16 = nullptr;
            uint4 *dsth = nullptr;
            if (publish) {
                if (kTagged)
                    dst16 = vrow_of(rchain, c + 1);
                else if (kPlain16)
                    dsth = chk(reinterpret_cast<uint4 *>(p.ring),
                               (rchain * 2 + ((c + 1) & 1)) * (int64_t)(kP / 8 * kN) + nrow, (kP / 8 - 1) * kN + 1,
                               nvec, hdr, SITE_TC_RING);
                else
                    dst32 = chk(reinterpret_cast<float4 *>(p.ring),
                                (rchain * 2 + ((c + 1) & 1)) * (int64_t)(kP / 4 * kN) + nrow, (kP / 4 - 1) * kN + 1,
                                nvec, hdr, SITE_TC_RING);
            }
            const uint64_t tg = (uint64_t)vtag(c + 1) << 32;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint32_t r[16];
                tmem_ld16(tmem + lrow + kColS + 64 * k2 + 16 * m, r);
                tmem_ld_wait();
                if (m == 1 && lane == 0) TRACE(warp, 5, hc);
                float o[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e] = fmaf(a, S[16 * m + e], __uint_as_float(r[e]));
                if (last) {
                    if (fin)
                        store_final16<ST>(fin, (chain * kP + 16 * m) * kN + nrow, nstate, hdr,
                                          make_float4(o[0], o[1], o[2], o[3]), make_float4(o[4], o[5], o[6], o[7]),
                                          make_float4(o[8], o[9], o[10], o[11]), make_float4(o[12], o[13], o[14], o[15]));
                } else if (publish) {
                    if (kTagged) {  // tagged words, the row's last vector last
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            st_ring(dst16 + (4 * m + j) * kN, tg | pack_f16(o[4 * j], o[4 * j + 1]),
                                    tg | pack_f16(o[4 * j + 2], o[4 * j + 3]));
                    } else if (kPlain16) {
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            __stcg(dsth + (2 * m + j) * kN,
                                   make_uint4(pack_f16(o[8 * j], o[8 * j + 1]), pack_f16(o[8 * j + 2], o[8 * j + 3]),
                                              pack_f16(o[8 * j + 4], o[8 * j + 5]), pack_f16(o[8 * j + 6], o[8 * j + 7])));
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            __stcg(dst32 + (4 * m + j) * kN, make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]));
                    }
                }
#pragma unroll
                for (int lc = 2 * m; lc < 2 * m + 2; ++lc)
                    sts128(srow + ((lc ^ (nrow & 7)) << 4),
                           make_uint4(pack_f16(S[8 * lc], S[8 * lc + 1]), pack_f16(S[8 * lc + 2], S[8 * lc + 3]),
                                      pack_f16(S[8 * lc + 4], S[8 * lc + 5]), pack_f16(S[8 * lc + 6], S[8 * lc + 7])));
            }
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive(&sm.sin_full[k2]);
            if (lane == 0) TRACE(warp, 4, hc);
            // per-row flags: publish this head's row (the release orders the row's stores before the tag)
            if (publish && !kTagged && !HF) st_release_u64(tag_of(rchain, c + 1), want_of(c + 1));
        }
    }
#undef BWAIT

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

template <typename IO, typename ST, bool CONV, bool HF>
cudaError_t launch_t(const Params &p, int hs, int sms, cudaStream_t stream) {
    CUtensorMap mx, mb, mc, my, mxh;
    const bool bf = !std::is_same<IO, __half>::value;
    const int64_t T = p.batch * p.L;
    if (!make_map(&mx, p.x, bf, kP, p.H, T, p.x_ld, kQ) || !make_map(&mb, p.B, bf, kN, p.G, T, p.bc_ld, kQ) ||
        !make_map(&mc, p.C, bf, kN, p.G, T, p.bc_ld, kQ) || !make_map(&my, p.y, bf, kP, p.H, T, p.H * kP, 32))
        return cudaErrorInvalidValue;
    if (CONV ? !make_map(&mxh, p.x, bf, kP, p.H, T, p.x_ld, 3, false) : false) return cudaErrorInvalidValue;
    if (!CONV) mxh = mx;
    const size_t smem = sizeof(Smem<CONV>) + 1024;
    auto k = tc_kernel<IO, ST, CONV, HF>;
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

// Late tickets pay where few units share a chunk index, so that the state chain bounds the launch; where many
// units share one, the loads then exposed at every unit boundary cost more than the chain.
bool tc_late_ticket(int64_t units_per_chunk, int sms) { return units_per_chunk * 4 <= sms; }

// One release flag per head, stored by the C.S warp after all rows, frees the chain threads of a release fence
// every head (fp32 states) or of tagged ring words (fp16 states, then plain halves), but publishes a head's state
// later (once its C.S is issued). That pays only where a chunk's successor starts well after it: early tickets and
// many head chains per chunk position (the 2.7B layer at batch 8: fp32 -12 %, fp16 -20 %; batch 32 fp32 -5 %; the
// 256K-token layer with fp16 states in 8 segments, 640 chains, -4 %); with fp32 states in 4 segments (320 chains)
// that layer lost 12 %, late-ticket launches 10-30 % (same-box A/B).
bool tc_head_flags(int64_t chains_per_position, bool late_ticket, int sms) {
    return !late_ticket && chains_per_position >= 3 * (int64_t)sms;
}

uint32_t tc_total_units(int64_t batch, int64_t H, int64_t G, int64_t nc, int hs) {
    (void)G;
    return (uint32_t)(nc * batch * (H / hs));
}

// Heads per work unit: the largest divisor of heads-per-group (<= 8) that still leaves at least six units per
// SM; small problems fall back to 1. More heads per unit share one C.B^T and one B/C load; more units spread the
// chunk-serial state chain over more SMs.
int tc_heads_per_unit(int64_t batch, int64_t H, int64_t G, int64_t nc, int sms) {
    const int64_t hpg = H / G;
    for (int d = kMaxHs; d >= 1; --d)
        if (hpg % d == 0 && nc * batch * (H / d) >= 6 * (int64_t)sms) return d;
    return 1;
}

// fp32 states: per-head flags where the plan chose them (not with the fused convolution)
template <typename IO, bool CONV>
cudaError_t launch_f32(const Params &p, int hs, int sms, cudaStream_t stream) {
    if constexpr (!CONV) {
        if (p.tc_head_flags) return launch_t<IO, float, CONV, true>(p, hs, sms, stream);
    }
    return launch_t<IO, float, CONV, false>(p, hs, sms, stream);
}

// fp16 states: plain halves behind per-head flags where asked (not with the fused convolution), else tagged words
template <typename IO, bool CONV>
cudaError_t launch_f16(const Params &p, int hs, int sms, cudaStream_t stream) {
    if constexpr (!CONV) {
        if (p.tc_head_flags) return launch_t<IO, __half, CONV, true>(p, hs, sms, stream);
    }
    return launch_t<IO, __half, CONV, false>(p, hs, sms, stream);
}

template <bool CONV>
cudaError_t launch_any(const Params &p, int io_dtype, int state_dtype, int hs, int sms, cudaStream_t stream) {
    if (io_dtype == 1)
        return state_dtype == 0 ? launch_f32<__nv_bfloat16, CONV>(p, hs, sms, stream)
                                : launch_f16<__nv_bfloat16, CONV>(p, hs, sms, stream);
    return state_dtype == 0 ? launch_f32<__half, CONV>(p, hs, sms, stream) : launch_f16<__half, CONV>(p, hs, sms, stream);
}

cudaError_t launch_tc(Params p, int io_dtype, int state_dtype, int hs, int sms, cudaStream_t stream) {
    if (hs < 1 || hs > kMaxHs || p.heads_per_group % hs) return cudaErrorInvalidValue;
    return p.conv_w ? launch_any<true>(p, io_dtype, state_dtype, hs, sms, stream)
                    : launch_any<false>(p, io_dtype, state_dtype, hs, sms, stream);
}

}  // namespace ssd

#ifdef SSD_TRACE
extern "C" __attribute__((visibility("default"))) int ssd_trace_read(unsigned long long *dst, unsigned int *counts) {
    if (cudaMemcpyFromSymbol(counts, ssd::g_trace_n, sizeof(ssd::g_trace_n)) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(dst, ssd::g_trace, sizeof(ssd::g_trace)) != cudaSuccess) return -1;
    static const unsigned int zero[ssd::kTraceRoles] = {};
    return cudaMemcpyToSymbol(ssd::g_trace_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}
#endif

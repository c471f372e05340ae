// Shared device-side definitions of the SSD prefill library: workspace header,
// kernel parameters, scheduling and flag helpers, dtype conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

// ---------------------------------------------------------------------------
// Workspace. The header sits at offset 0; the per-chain flags and the state
// ring follow at offsets the host computes (see ssd_api.cu).
//
// Epochs make the flags self-clearing: launch k (k = 1, 2, ...) reads
// epoch = header.epoch + 1, tags every flag it publishes with that value and,
// in the last CTA to finish, stores it back into header.epoch. A flag is
// "set" for this launch only when it equals this launch's epoch.
// ---------------------------------------------------------------------------
struct WsHeader {
    uint32_t epoch;       // epoch of the last finished launch
    uint32_t ticket;      // persistent-grid work counter (reset by the last CTA)
    uint32_t done;        // CTAs finished (reset by the last CTA)
    uint32_t status;      // first device error of any launch since the last check
    uint32_t abort;       // == epoch when this launch gave up: waiters bail out
    uint32_t err_unit;    // unit (ticket) that recorded the error
    uint32_t err_chunk;   // chunk index of that unit
    uint32_t err_where;   // which wait gave up (WAIT_* below)
    uint64_t timeout_ns;  // limit of every device wait, 0 = default
    int64_t skip_publish; // test hook: 1 + chunk whose publish is skipped (0 = off, the zero-filled state)
    uint32_t bounds_probe;  // test hook of bounds-checked builds: 1 = one checked index is planted one past its end
    uint32_t err_index_lo, err_index_hi;  // bounds-checked builds: the first rejected index
    uint32_t pad[49];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s
constexpr uint32_t kMaxSpinIters = 1u << 26;           // hard cap besides the clock

enum WaitSite : uint32_t {
    WAIT_CHAIN = 1,   // state-passing flag of the previous chunk
    WAIT_PIPE = 2,    // intra-CTA mbarrier (tensor-core kernel)
};

enum DevStatus : uint32_t { DEV_OK = 0, DEV_BAD_SEQLENS = 1, DEV_TIMEOUT = 5, DEV_PIPE = 6, DEV_BOUNDS = 7 };

// Access sites of the bounds-checked builds (recorded in err_where with DEV_BOUNDS).
enum BoundsSite : uint32_t {
    SITE_TC_DT = 101, SITE_TC_Y = 102, SITE_TC_INIT = 103, SITE_TC_FINAL = 104, SITE_TC_RING = 105, SITE_TC_FLAG = 106,
    SITE_SIMT_IN = 111, SITE_SIMT_Y = 112, SITE_SIMT_INIT = 113, SITE_SIMT_FINAL = 114, SITE_SIMT_RING = 115,
    SITE_SIMT_FLAG = 116,
    SITE_STEP_IN = 121, SITE_STEP_Y = 122, SITE_STEP_STATE = 123,
    SITE_CONV_IN = 131, SITE_CONV_OUT = 132, SITE_CONV_STATE = 133,
    SITE_SEG_DT = 141, SITE_SEG_BLK = 142, SITE_SEG_DECAY = 143, SITE_SEG_STATE = 144, SITE_SEG_INIT = 145,
    SITE_SEG_TMA = 146,
};

// Parameters common to the kernels. Element strides are implied by the packed
// layouts documented in ssd.h. Tokens are addressed on one packed axis: a
// regular batch is nseq = batch sequences of L tokens each (token s*L + t), a
// variable-length batch has its sequences at the offsets cu[s] .. cu[s+1].
// Chunks never straddle two sequences: chunk c of sequence s starts at token
// offset(s) + c*Q, and the last chunk of a sequence may be ragged.
struct Params {
    const void *x;
    const void *dt_raw;
    const float *dt_bias;
    const float *A;
    const void *B;
    const void *C;
    const float *D;     // may be null
    const void *init;   // may be null
    void *y;
    void *final_states; // may be null
    WsHeader *hdr;
    uint64_t *flags;    // state-passing tags, [chain][ring slot] (per state row too in the tensor-core kernel)
    void *ring;         // state ring, layout per kernel
    int64_t batch, L, H, P, N, G, Q, nc;
    int64_t heads_per_group;
    uint32_t total_units;  // regular batches; variable-length: *vtot chunk pairs times the units per chunk pair
    int64_t nseq;          // sequences (= batch for a regular batch)
    int64_t x_ld, bc_ld;   // elements from one token to the next in x (packed: H*P) and in B, C (packed: G*N)
    // Depthwise convolution (width 4) fused in front (tensor-core kernel): x, B, C are then slices of the raw rows
    // [tokens, Dc = x_ld] starting at channels 0, conv_hp and conv_hp + G*N.
    const float *conv_w;     // [Dc, 4], tap 3 on the current token
    const float *conv_b;     // [Dc] or null
    const void *conv_state;  // [nseq, Dc, 3] inputs before each sequence (I/O dtype), or null (zeros)
    int64_t conv_hp;         // H * P
    int conv_silu;
    const int32_t *cu;     // variable-length: token offsets [nseq + 1]; null for a regular batch
    const int2 *ctab;      // variable-length: (sequence, chunk) of each chunk pair, chunk-major
    const uint32_t *vtot;  // variable-length: number of chunk pairs (written by the planning kernel)
    int tc_late_ticket;    // tensor-core kernel: take each next ticket only when the unit before it nears its end
    int tc_head_flags;     // tensor-core kernel, fp32 states: one release flag per head (by the C.S warp), not per row
    int64_t ring_bytes, flag_count;  // extents of the ring and the flags (bounds-checked builds compare with them)
    // Two-level state passing (tensor-core kernel, regular batches): with nseg > 1 every sequence is cut into nseg
    // segments of seg_chunks chunks (the last one shorter or equal), the chunk-to-chunk state chain restarts at
    // every segment, and the state entering segment k >= 1 is read from seg_states [nseq][nseg - 1][H][P][N]
    // (fp32), computed beforehand from block aggregates. nseg <= 1: one chain per sequence.
    int64_t nseg, seg_chunks;
    const float *seg_states;
};

// Causal depthwise convolution over the packed token axis (nseq sequences of L tokens, D channels).
struct ConvParams {
    const void *in;       // [nseq * L, D] raw inputs
    const float *w;       // [D, k] taps (tap k - 1 on the current token)
    const float *bias;    // [D] or null
    const void *state;    // [nseq, D, k - 1] inputs before each sequence, or null (zeros)
    void *out;            // [nseq * L, D]
    void *state_out;      // [nseq, D, k - 1] the last k - 1 inputs of each sequence, or null; may alias state
    int64_t T, L, D, nseq;
    int k, silu;
    WsHeader *hdr;        // for the bounds-checked builds' reports (may be null: not checked)
};

// Chunk pair cp (one chunk of one sequence) in chunk-major order -> sequence, chunk, first token, length.
struct SeqChunk {
    int64_t s, c, tok0, len;
};
__device__ __forceinline__ SeqChunk seq_chunk(const Params &p, int64_t cp) {
    SeqChunk r;
    if (p.ctab) {
        const int2 e = p.ctab[cp];
        r.s = e.x;
        r.c = e.y;
        r.tok0 = p.cu[r.s];
        r.len = p.cu[r.s + 1] - r.tok0;
    } else if (p.nseg > 1) {
        // position-major over the (sequence, segment) chains, so that the segments of one sequence run side by
        // side; only each sequence's last segment can be shorter (last_len chunks)
        const int64_t nvs = p.nseq * p.nseg, last_len = p.nc - (p.nseg - 1) * p.seg_chunks;
        int64_t pos, k;
        if (cp < last_len * nvs) {
            pos = cp / nvs;
            r.s = (cp % nvs) / p.nseg;
            k = (cp % nvs) % p.nseg;
        } else {
            const int64_t m = p.nseq * (p.nseg - 1), q = cp - last_len * nvs;
            pos = last_len + q / m;
            r.s = (q % m) / (p.nseg - 1);
            k = (q % m) % (p.nseg - 1);
        }
        r.c = k * p.seg_chunks + pos;
        r.tok0 = r.s * p.L;
        r.len = p.L;
    } else {
        r.s = cp % p.nseq;
        r.c = cp / p.nseq;
        r.tok0 = r.s * p.L;
        r.len = p.L;
    }
    return r;
}
// Index of the state chain of chunk c of sequence s, head h: one per (sequence, head), or with two-level state
// passing one per (sequence, segment, head).
__device__ __forceinline__ int64_t chain_of(const Params &p, int64_t s, int64_t c, int64_t h) {
    return p.nseg > 1 ? (s * p.nseg + c / p.seg_chunks) * p.H + h : s * p.H + h;
}
// Chunk pairs of this launch (regular batches know it on the host; variable-length ones read the device count).
__device__ __forceinline__ uint32_t total_units(const Params &p, uint32_t units_per_pair) {
    return p.ctab ? *p.vtot * units_per_pair : p.total_units;
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t chain_tag(uint32_t epoch, int64_t chunk) {
    return ((uint64_t)epoch << 32) | (uint32_t)chunk;
}

// ---------------------------------------------------------------------------
// Small PTX helpers (hand-written; no library code).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Record the first device error and raise this launch's abort flag.
__device__ __forceinline__ void report_error(WsHeader *hdr, uint32_t epoch, uint32_t code, uint32_t unit,
                                             uint32_t chunk, uint32_t where) {
    if (atomicCAS(&hdr->status, 0u, code) == 0u) {
        hdr->err_unit = unit;
        hdr->err_chunk = chunk;
        hdr->err_where = where;
    }
    __threadfence();
    st_relaxed_gpu(&hdr->abort, epoch);
}

__device__ __forceinline__ bool aborted(const WsHeader *hdr, uint32_t epoch) {
    return ld_relaxed_gpu(&hdr->abort) == epoch;
}

// Bounds-checked builds (-DSSD_BOUNDS_CHECK), the stand-in for a memory checker: a checked access goes through
// chk(), which compares the element index and the access's span with the buffer's extent. Outside it, the first
// such access records DEV_BOUNDS, the site and the index in the workspace header, and the access is redirected to
// the buffer's first element, so nothing outside the buffers is touched and ssd_fwd_check reports it. Release
// builds compile chk() to the plain address.
#ifdef SSD_BOUNDS_CHECK
static __device__ __noinline__ void bounds_hit(WsHeader *hdr, uint32_t site, int64_t idx) {
    if (hdr && atomicCAS(&hdr->status, 0u, (uint32_t)DEV_BOUNDS) == 0u) {
        hdr->err_where = site;
        hdr->err_index_lo = (uint32_t)idx;
        hdr->err_index_hi = (uint32_t)((uint64_t)idx >> 32);
    }
}
template <typename T>
__device__ __forceinline__ T *chk(T *base, int64_t idx, int64_t span, int64_t n, WsHeader *hdr, uint32_t site) {
    if (idx >= 0 && idx + span <= n) return base + idx;
    bounds_hit(hdr, site, idx);
    return base;
}
#else
template <typename T>
__device__ __forceinline__ T *chk(T *base, int64_t idx, int64_t, int64_t, WsHeader *, uint32_t) {
    return base + idx;
}
#endif

// Bounded wait until *tag == want (acquire). Returns false (after recording
// a timeout) when the limit passes or another CTA aborted the launch.
__device__ __forceinline__ bool wait_flag(const uint64_t *tag, uint64_t want, uint32_t epoch, WsHeader *hdr,
                                          uint64_t limit_ns, uint32_t unit, uint32_t chunk) {
    if (ld_acquire_u64(tag) == want) return true;
    const uint64_t t0 = globaltimer();
    uint32_t sleep_ns = 20;
    for (uint32_t it = 0; it < kMaxSpinIters; ++it) {
        if (ld_acquire_u64(tag) == want) return true;
        if ((it & 7u) == 7u) {
            if (aborted(hdr, epoch)) return false;
            if (globaltimer() - t0 > limit_ns) break;
        }
        __nanosleep(sleep_ns);
        if (sleep_ns < 200) sleep_ns += 20;
    }
    report_error(hdr, epoch, DEV_TIMEOUT, unit, chunk, WAIT_CHAIN);
    return false;
}

// ---------------------------------------------------------------------------
// Element conversion.
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// softplus(v) = log(1 + e^v); above 20 it equals v to fp32 precision.
__device__ __forceinline__ float softplus_f32(float v) { return v > 20.f ? v : log1pf(expf(v)); }

}  // namespace ssd

// The C ABI declared in include/ssd.h: argument checks, workspace layout,
// kernel selection and launch. Host code only.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "../../include/ssd.h"
#include "ssd_internal.h"

namespace ssd {

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;  // benign race: every caller stores the same pointer
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

namespace {
// heads per unit, late ticket, SIMT two pass, conv TMA, chunks per segment
std::atomic<int> g_knob[6] = {{-1}, {-1}, {-1}, {-1}, {-1}, {-1}};
}  // namespace

Knobs knobs() {
    return Knobs{g_knob[0].load(std::memory_order_relaxed), g_knob[1].load(std::memory_order_relaxed),
                 g_knob[2].load(std::memory_order_relaxed), g_knob[3].load(std::memory_order_relaxed),
                 g_knob[4].load(std::memory_order_relaxed), g_knob[5].load(std::memory_order_relaxed)};
}

}  // namespace ssd

namespace {

using ssd::Params;
using ssd::WsHeader;

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0 = not queried yet (threads that race store the same value)

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < kMaxDevices) {
        const int c = g_sm_count[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t elem_size(int dt) { return dt == SSD_F32 ? 4 : 2; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Plan {
    int kernel = 0;          // SSD_KERNEL_SIMT / _TC / _STEP
    int64_t nc = 0;          // chunks per sequence (regular) or the bound ceil(T / exec_chunk) (variable-length)
    int64_t exec_chunk = 0;  // tokens per state-passing step in the chosen kernel
    int64_t nseq = 0;        // sequences: batch (regular) or the cu_seqlens count (variable-length)
    bool varlen = false;
    int heads_per_unit = 1;  // TC only
    bool late_ticket = false;  // TC only: next ticket taken when the unit before it nears its end
    bool head_flags = false;   // TC only, fp32 states: one release flag per head
    uint32_t total_units = 0;
    ssd::SegChoice seg{1, 0, 0, 0, 1};  // TC only, regular batches: two-level state passing when seg.nseg > 1
    size_t flags_off = 0, ring_off = 0, tab_off = 0, seg_off = 0, blk_s_off = 0, blk_L_off = 0, bytes = 0;
};

// Variable-length tables after the ring: chunk pairs (int2), then four uint32 arrays of nc + 2 (histogram of
// chunks per sequence, its suffix sums, fill counters, chunk starts) and the chunk-pair count.
size_t varlen_table_bytes(int64_t nc, int64_t nseq) {
    return align_up(sizeof(int32_t) * 2 * (size_t)(nc + nseq), 256) + sizeof(uint32_t) * (4 * (size_t)(nc + 2) + 1);
}

// Validate the problem and lay out the workspace. No CUDA calls except the
// SM count used to size the tensor-core work units. nseq < 0: a regular batch.
ssd_status_t plan(const ssd_problem_t *pr, int64_t nseq, Plan *out, bool segments = true) {
    if (!pr || !out) return SSD_ERR_INVALID_ARG;
    if (pr->reserved != 0) return SSD_ERR_INVALID_ARG;
    if (pr->batch < 0 || pr->seqlen < 0 || pr->nheads < 1 || pr->headdim < 1 || pr->dstate < 1 ||
        pr->ngroups < 1 || pr->chunk_size < 1)
        return SSD_ERR_INVALID_ARG;
    if (pr->nheads % pr->ngroups) return SSD_ERR_INVALID_ARG;
    if (pr->io_dtype < SSD_F32 || pr->io_dtype > SSD_F16) return SSD_ERR_INVALID_ARG;
    if (pr->state_dtype != SSD_F32 && pr->state_dtype != SSD_F16) return SSD_ERR_INVALID_ARG;
    if (pr->kernel < SSD_KERNEL_AUTO || pr->kernel > SSD_KERNEL_STEP) return SSD_ERR_INVALID_ARG;
    const bool varlen = nseq >= 0;
    if (varlen && (pr->batch != 1 || nseq > INT32_MAX || pr->seqlen > INT32_MAX)) return SSD_ERR_INVALID_ARG;
    // keep every element index comfortably inside int64
    const double tok = (double)pr->batch * (double)pr->seqlen;
    const double seqs = varlen ? (double)nseq : (double)pr->batch;
    if (tok * (double)pr->nheads * (double)pr->headdim > 4e18 || tok * (double)pr->ngroups * (double)pr->dstate > 4e18 ||
        seqs * pr->nheads * pr->headdim * pr->dstate > 4e18)
        return SSD_ERR_INVALID_ARG;

    Plan pl;
    pl.varlen = varlen;
    pl.nseq = varlen ? nseq : pr->batch;
    const bool tc_ok = ssd::tc_supports(pr->headdim, pr->dstate, pr->chunk_size, pr->io_dtype);
    const bool simt_ok = ssd::simt_smem_bytes(pr->headdim, pr->dstate) <= 227u * 1024u;
    if (pr->kernel == SSD_KERNEL_STEP || (pr->kernel == SSD_KERNEL_AUTO && !varlen && pr->seqlen == 1)) {
        if (varlen || pr->seqlen > 1) return SSD_ERR_UNSUPPORTED;
        pl.kernel = SSD_KERNEL_STEP;
    } else if (pr->kernel == SSD_KERNEL_TC) {
        if (!tc_ok) return SSD_ERR_UNSUPPORTED;
        pl.kernel = SSD_KERNEL_TC;
    } else if (pr->kernel == SSD_KERNEL_SIMT) {
        if (!simt_ok) return SSD_ERR_UNSUPPORTED;
        pl.kernel = SSD_KERNEL_SIMT;
    } else {
        if (tc_ok)
            pl.kernel = SSD_KERNEL_TC;
        else if (simt_ok)
            pl.kernel = SSD_KERNEL_SIMT;
        else
            return SSD_ERR_UNSUPPORTED;
    }
    pl.exec_chunk = pl.kernel == SSD_KERNEL_TC ? ssd::tc_chunk() : pr->chunk_size;
    if (pl.kernel == SSD_KERNEL_STEP) {  // no inter-CTA state passing: the workspace is its header only
        pl.nc = pr->seqlen;
        pl.flags_off = pl.ring_off = pl.tab_off = pl.bytes = sizeof(WsHeader);
        *out = pl;
        return SSD_OK;
    }
    // regular: chunks per sequence; variable-length: no sequence has more than ceil(T / chunk)
    pl.nc = (pr->seqlen + pl.exec_chunk - 1) / pl.exec_chunk;
    int64_t chains = pl.nseq * pr->nheads;
    double units;
    if (pl.kernel == SSD_KERNEL_TC) {
        if (!varlen && segments) {
            // test hook: forced chunks per segment (0: off)
            const int forced = ssd::knobs().tc_segment_chunks;
            pl.seg = ssd::choose_segments(pl.nseq, pl.nc, pr->nheads, pr->ngroups, std::max(1, sm_count()), forced,
                                          pr->state_dtype == SSD_F32);
            chains *= pl.seg.nseg;  // one state chain per (sequence, segment, head)
        }
        // for a variable-length batch the chunk count is only bounded here (pairs <= nc + nseq); it sizes the units
        const int64_t pairs = varlen ? pl.nc + pl.nseq : pl.nc * pr->batch;
        pl.heads_per_unit = ssd::tc_heads_per_unit(1, pr->nheads, pr->ngroups, pairs, std::max(1, sm_count()));
        const ssd::Knobs kn = ssd::knobs();
        // test hook: forced heads per work unit (used when it divides nheads / ngroups)
        if (kn.tc_heads_per_unit >= 1 && (pr->nheads / pr->ngroups) % kn.tc_heads_per_unit == 0)
            pl.heads_per_unit = kn.tc_heads_per_unit;
        units = (double)pairs * (double)(pr->nheads / pl.heads_per_unit);
        pl.late_ticket = ssd::tc_late_ticket(pl.nseq * pl.seg.nseg * (pr->nheads / pl.heads_per_unit),
                                             std::max(1, sm_count()));
        // test hook: forced early (0) or late (1) tickets
        if (kn.tc_late_ticket >= 0) pl.late_ticket = kn.tc_late_ticket == 1;
        pl.head_flags = ssd::tc_head_flags(pl.nseq * pl.seg.nseg * pr->nheads, pl.late_ticket, std::max(1, sm_count()));
        if (kn.tc_head_flags >= 0) pl.head_flags = kn.tc_head_flags == 1;  // test hook
    } else {
        units = (double)(varlen ? pl.nc + pl.nseq : pl.nc * pr->batch) * (double)pr->nheads;
    }
    if (units >= 4.0e9) return SSD_ERR_UNSUPPORTED;
    pl.total_units = varlen ? 0u : (uint32_t)units;
    pl.flags_off = sizeof(WsHeader);
    const size_t flag_bytes = pl.kernel == SSD_KERNEL_TC ? ssd::tc_flag_bytes(chains) : sizeof(uint64_t) * 2 * (size_t)chains;
    pl.ring_off = align_up(pl.flags_off + flag_bytes, 256);
    size_t ring;
    if (pl.kernel == SSD_KERNEL_TC)
        ring = ssd::tc_ring_bytes(chains, pr->headdim, pr->dstate, pr->state_dtype);
    else
        ring = (size_t)chains * 2 * (size_t)(pr->headdim * pr->dstate) * elem_size(pr->state_dtype);
    pl.tab_off = align_up(pl.ring_off + ring, 256);
    pl.seg_off = align_up(pl.tab_off + (varlen ? varlen_table_bytes(pl.nc, pl.nseq) : 0), 256);
    pl.blk_s_off = pl.blk_L_off = pl.bytes = pl.seg_off;
    if (pl.seg.nseg > 1) {  // segment entering states, block aggregates and block decays (fp32)
        const size_t st = (size_t)(pr->headdim * pr->dstate) * 4;
        pl.blk_s_off = align_up(pl.seg_off + (size_t)(pl.nseq * (pl.seg.nseg - 1) * pr->nheads) * st, 256);
        pl.blk_L_off = align_up(pl.blk_s_off + (size_t)(pl.nseq * pl.seg.nblk * pr->nheads) * st, 256);
        pl.bytes = align_up(pl.blk_L_off + (size_t)(pl.nseq * pl.seg.nblk * pr->nheads) * 4, 256);
    }
    *out = pl;
    return SSD_OK;
}

// Argument checks and launch shared by the regular and the variable-length entry points.
// x_ld, bc_ld: elements from one token to the next in x and in B, C (0: packed).
ssd_status_t run(const ssd_problem_t *prob, int64_t nseq, const int32_t *cu_seqlens, const void *x, const void *dt_raw,
                 const float *dt_bias, const float *A, const void *B, const void *C, const float *D,
                 const void *init_states, void *y, void *final_states, void *workspace, size_t workspace_bytes,
                 void *stream, int64_t x_ld = 0, int64_t bc_ld = 0, const ssd::Params *conv = nullptr) {
    Plan pl;
    ssd_status_t st = plan(prob, nseq, &pl);
    if (st != SSD_OK) return st;
    const ssd_problem_t &pr = *prob;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t es = elem_size(pr.io_dtype);
    const size_t ses = elem_size(pr.state_dtype);
    const bool tokens = pr.batch > 0 && pr.seqlen > 0;
    if (!dt_bias || !A) return SSD_ERR_INVALID_ARG;
    if (!aligned(dt_bias, 4) || !aligned(A, 4) || (D && !aligned(D, 4))) return SSD_ERR_INVALID_ARG;
    if (init_states && !aligned(init_states, 16)) return SSD_ERR_INVALID_ARG;
    if (final_states && !aligned(final_states, 16)) return SSD_ERR_INVALID_ARG;
    if (pl.varlen && pl.nseq > 0 && (!cu_seqlens || !aligned(cu_seqlens, 4))) return SSD_ERR_INVALID_ARG;
    if (tokens) {
        if (!x || !dt_raw || !B || !C || !y) return SSD_ERR_INVALID_ARG;
        if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16) || !aligned(dt_raw, es))
            return SSD_ERR_INVALID_ARG;
    }
    if (pl.nseq == 0) return SSD_OK;
    if (pr.seqlen == 0) {  // nothing to scan: every final state is the initial one
        if (!final_states) return SSD_OK;
        const size_t n = (size_t)(pl.nseq * pr.nheads * pr.headdim * pr.dstate) * ses;
        const cudaError_t e = init_states ? cudaMemcpyAsync(final_states, init_states, n, cudaMemcpyDeviceToDevice, s)
                                          : cudaMemsetAsync(final_states, 0, n, s);
        return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    }
    if (workspace_bytes < pl.bytes) {  // too small for two-level state passing: one state chain per sequence
        Plan one;
        if (plan(prob, nseq, &one, false) == SSD_OK && workspace_bytes >= one.bytes) pl = one;
    }
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < pl.bytes) return SSD_ERR_WORKSPACE;
    const int sms = sm_count();
    if (sms <= 0) return SSD_ERR_CUDA;

    Params p;
    memset(&p, 0, sizeof(p));
    p.x = x;
    p.dt_raw = dt_raw;
    p.dt_bias = dt_bias;
    p.A = A;
    p.B = B;
    p.C = C;
    p.D = D;
    p.init = init_states;
    p.y = y;
    p.final_states = final_states;
    char *ws = static_cast<char *>(workspace);
    p.hdr = reinterpret_cast<WsHeader *>(ws);
    p.flags = reinterpret_cast<uint64_t *>(ws + pl.flags_off);
    p.ring = ws + pl.ring_off;
    p.batch = pr.batch;
    p.L = pr.seqlen;
    p.H = pr.nheads;
    p.P = pr.headdim;
    p.N = pr.dstate;
    p.G = pr.ngroups;
    p.Q = pl.exec_chunk;
    p.nc = pl.nc;
    p.heads_per_group = pr.nheads / pr.ngroups;
    p.total_units = pl.total_units;
    p.nseq = pl.nseq;
    p.ring_bytes = (int64_t)(pl.tab_off - pl.ring_off);
    p.flag_count = (int64_t)((pl.ring_off - pl.flags_off) / sizeof(uint64_t));
    p.tc_late_ticket = pl.late_ticket ? 1 : 0;
    p.tc_head_flags = pl.head_flags ? 1 : 0;
    p.x_ld = x_ld ? x_ld : pr.nheads * pr.headdim;
    p.bc_ld = bc_ld ? bc_ld : pr.ngroups * pr.dstate;
    ssd::SegPlan sp{pl.seg.blk, pl.seg.nblk, pl.seg.hs, reinterpret_cast<float *>(ws + pl.blk_s_off),
                    reinterpret_cast<float *>(ws + pl.blk_L_off)};
    // two-level state passing (not with the fused convolution: the block kernel reads x as stored)
    const bool seg = pl.seg.nseg > 1 && !conv;
    p.nseg = seg ? pl.seg.nseg : 1;
    p.seg_chunks = seg ? pl.seg.seg_chunks : pl.nc;
    p.seg_states = seg ? reinterpret_cast<const float *>(ws + pl.seg_off) : nullptr;
    if (conv) {  // convolution fused into the tensor-core kernel: x, B, C are slices of the raw rows
        p.conv_w = conv->conv_w;
        p.conv_b = conv->conv_b;
        p.conv_state = conv->conv_state;
        p.conv_hp = conv->conv_hp;
        p.conv_silu = conv->conv_silu;
    }

    cudaError_t e = cudaSuccess;
    if (pl.varlen) {
        // chunk-major (sequence, chunk) table from cu_seqlens, on the device
        char *tab = ws + pl.tab_off;
        int2 *ctab = reinterpret_cast<int2 *>(tab);
        uint32_t *scratch = reinterpret_cast<uint32_t *>(tab + align_up(sizeof(int32_t) * 2 * (size_t)(pl.nc + pl.nseq), 256));
        p.cu = cu_seqlens;
        p.ctab = ctab;
        p.vtot = scratch + 4 * (size_t)(pl.nc + 2);
        e = ssd::launch_varlen_plan(p, scratch, ses, s);
        if (e != cudaSuccess) return SSD_ERR_CUDA;
    }
    if (pl.kernel == SSD_KERNEL_STEP)
        e = ssd::launch_step(p, pr.io_dtype, pr.state_dtype, sms, s);
    else if (pl.kernel == SSD_KERNEL_TC) {
        if (seg) e = ssd::launch_segstate(p, sp, pr.io_dtype, pr.state_dtype, sms, s);
        if (e == cudaSuccess) e = ssd::launch_tc(p, pr.io_dtype, pr.state_dtype, pl.heads_per_unit, sms, s);
    }
    else
        e = ssd::launch_simt(p, pr.io_dtype, pr.state_dtype, sms, s);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

namespace ssd {
ssd_status_t workspace_bytes(const ssd_problem_t *prob, bool segments, size_t *bytes) {
    Plan pl;
    const ssd_status_t st = plan(prob, -1, &pl, segments);
    if (st == SSD_OK) *bytes = pl.bytes;
    return st;
}
}  // namespace ssd

extern "C" {

SSD_API ssd_status_t ssd_fwd_workspace_size(const ssd_problem_t *prob, size_t *bytes) {
    if (!bytes) return SSD_ERR_INVALID_ARG;
    Plan pl;
    const ssd_status_t st = plan(prob, -1, &pl);
    if (st != SSD_OK) return st;
    *bytes = pl.bytes;
    return SSD_OK;
}

SSD_API int ssd_fwd_kernel_for(const ssd_problem_t *prob) {
    Plan pl;
    const ssd_status_t st = plan(prob, -1, &pl);
    return st == SSD_OK ? pl.kernel : -(int)st;
}

SSD_API ssd_status_t ssd_fwd_plan(const ssd_problem_t *prob, ssd_plan_t *out) {
    if (!out) return SSD_ERR_INVALID_ARG;
    Plan pl;
    const ssd_status_t st = plan(prob, -1, &pl);
    if (st != SSD_OK) return st;
    const bool tokens = prob->batch > 0 && prob->seqlen > 0;
    out->kernel = pl.kernel;
    out->segments = pl.seg.nseg;
    out->segment_chunks = pl.seg.nseg > 1 ? pl.seg.seg_chunks : pl.nc;
    out->launches = !tokens ? 0 : (pl.seg.nseg > 1 ? 3 : 1);
    out->workspace_bytes = pl.bytes;
    out->head_flags = pl.kernel == SSD_KERNEL_TC && pl.head_flags ? 1 : 0;
    out->reserved = 0;
    return SSD_OK;
}

SSD_API ssd_status_t ssd_fwd(const ssd_problem_t *prob, const void *x, const void *dt_raw, const float *dt_bias,
                             const float *A, const void *B, const void *C, const float *D, const void *init_states,
                             void *y, void *final_states, void *workspace, size_t workspace_bytes, void *stream) {
    return run(prob, -1, nullptr, x, dt_raw, dt_bias, A, B, C, D, init_states, y, final_states, workspace,
               workspace_bytes, stream);
}

SSD_API ssd_status_t ssd_fwd_varlen_workspace_size(const ssd_problem_t *prob, int64_t nseq, size_t *bytes) {
    if (!bytes || nseq < 0) return SSD_ERR_INVALID_ARG;
    Plan pl;
    const ssd_status_t st = plan(prob, nseq, &pl);
    if (st != SSD_OK) return st;
    *bytes = pl.bytes;
    return SSD_OK;
}

SSD_API ssd_status_t ssd_fwd_varlen(const ssd_problem_t *prob, const int32_t *cu_seqlens, int64_t nseq, const void *x,
                                    const void *dt_raw, const float *dt_bias, const float *A, const void *B,
                                    const void *C, const float *D, const void *init_states, void *y,
                                    void *final_states, void *workspace, size_t workspace_bytes, void *stream) {
    if (nseq < 0) return SSD_ERR_INVALID_ARG;
    return run(prob, nseq, cu_seqlens, x, dt_raw, dt_bias, A, B, C, D, init_states, y, final_states, workspace,
               workspace_bytes, stream);
}

SSD_API ssd_status_t ssd_fwd_conv(const ssd_problem_t *prob, int32_t conv_width, int32_t activation, const void *xbc,
                                  const float *conv_weight, const float *conv_bias, const void *conv_state,
                                  void *conv_state_out, void *xbc_out, const void *dt_raw, const float *dt_bias,
                                  const float *A, const float *D, const void *init_states, void *y, void *final_states,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    if (!prob) return SSD_ERR_INVALID_ARG;
    const ssd_problem_t &pr = *prob;
    if (conv_width < 1 || conv_width > 8 || (activation != SSD_ACT_NONE && activation != SSD_ACT_SILU))
        return SSD_ERR_INVALID_ARG;
    Plan pl;
    ssd_status_t st = plan(prob, -1, &pl);  // the SSD problem checks
    if (st != SSD_OK) return st;
    const size_t es = elem_size(pr.io_dtype);
    const int64_t hp = pr.nheads * pr.headdim, gn = pr.ngroups * pr.dstate, ch = hp + 2 * gn;
    const int64_t vec = 16 / (int64_t)es;  // x, B, C are 16-byte aligned slices of the convolved rows
    if (hp % vec || gn % vec) return SSD_ERR_INVALID_ARG;
    const bool tokens = pr.batch > 0 && pr.seqlen > 0;
    if (!conv_weight || !aligned(conv_weight, 4) || (conv_bias && !aligned(conv_bias, 4))) return SSD_ERR_INVALID_ARG;
    if (tokens && (!xbc || !aligned(xbc, 16) || (xbc_out && (!aligned(xbc_out, 16) || xbc == xbc_out))))
        return SSD_ERR_INVALID_ARG;
    if ((conv_state && !aligned(conv_state, es)) || (conv_state_out && !aligned(conv_state_out, es)))
        return SSD_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return SSD_ERR_CUDA;
    ssd::ConvParams c;
    memset(&c, 0, sizeof(c));
    c.hdr = static_cast<WsHeader *>(workspace);
    c.in = xbc;
    c.w = conv_weight;
    c.bias = conv_bias;
    c.state = conv_state;
    c.out = xbc_out;
    c.state_out = conv_state_out;
    c.T = pr.batch * pr.seqlen;
    c.L = pr.seqlen;
    c.D = ch;
    c.nseq = pr.batch;
    c.k = conv_width;
    c.silu = activation == SSD_ACT_SILU;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const char *xb = static_cast<const char *>(xbc);
    if (!xbc_out && tokens) {
        // fused: the tensor-core kernel convolves the raw rows as it loads them (no activation buffer)
        if (pl.kernel != SSD_KERNEL_TC || conv_width != 4 || !aligned(conv_weight, 16) ||
            (conv_bias && !aligned(conv_bias, 16)))
            return SSD_ERR_UNSUPPORTED;
        ssd::Params cv;
        memset(&cv, 0, sizeof(cv));
        cv.conv_w = conv_weight;
        cv.conv_b = conv_bias;
        cv.conv_state = conv_state;
        cv.conv_hp = hp;
        cv.conv_silu = activation == SSD_ACT_SILU;
        st = run(prob, -1, nullptr, xb, dt_raw, dt_bias, A, xb + hp * es, xb + (hp + gn) * es, D, init_states, y,
                 final_states, workspace, workspace_bytes, stream, ch, ch, &cv);
        if (st != SSD_OK) return st;
        c.T = 0;  // the cache only, after the kernel that reads the cache given on entry
        return ssd::launch_conv(c, pr.io_dtype, sms, s) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    }
    if (ssd::launch_conv(c, pr.io_dtype, sms, s) != cudaSuccess) return SSD_ERR_CUDA;
    const char *xo = static_cast<const char *>(xbc_out);
    return run(prob, -1, nullptr, xo, dt_raw, dt_bias, A, xo ? xo + hp * es : nullptr, xo ? xo + (hp + gn) * es : nullptr, D,
               init_states, y, final_states, workspace, workspace_bytes, stream, ch, ch);
}

SSD_API ssd_status_t ssd_fwd_check(void *workspace, void *stream) {
    if (!workspace || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
    uint32_t status = 0;
    WsHeader *hdr = static_cast<WsHeader *>(workspace);
    if (cudaMemcpy(&status, &hdr->status, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess) return SSD_ERR_CUDA;
    if (status == 0) return SSD_OK;
    if (cudaMemset(&hdr->status, 0, sizeof(status)) != cudaSuccess) return SSD_ERR_CUDA;
    if (status == ssd::DEV_TIMEOUT) return SSD_ERR_TIMEOUT;
    if (status == ssd::DEV_BAD_SEQLENS) return SSD_ERR_INVALID_ARG;
    return SSD_ERR_DEVICE;  // DEV_PIPE, or DEV_BOUNDS from a bounds-checked build
}

SSD_API ssd_status_t ssd_debug_set(void *workspace, uint64_t timeout_ns, int64_t skip_publish, void *stream) {
    if (!workspace || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SSD_ERR_CUDA;
    WsHeader *hdr = static_cast<WsHeader *>(workspace);
    if (cudaMemcpy(&hdr->timeout_ns, &timeout_ns, sizeof(timeout_ns), cudaMemcpyHostToDevice) != cudaSuccess)
        return SSD_ERR_CUDA;
    const int64_t stored = skip_publish < 0 ? 0 : skip_publish + 1;  // 0 = off (zero-filled workspace)
    if (cudaMemcpy(&hdr->skip_publish, &stored, sizeof(stored), cudaMemcpyHostToDevice) != cudaSuccess)
        return SSD_ERR_CUDA;
    const uint32_t probe = skip_publish == -2 ? 1u : 0u;  // bounds-checked builds: plant one index past its end
    if (cudaMemcpy(&hdr->bounds_probe, &probe, sizeof(probe), cudaMemcpyHostToDevice) != cudaSuccess)
        return SSD_ERR_CUDA;
    return SSD_OK;
}

SSD_API ssd_status_t ssd_debug_knobs(int32_t tc_heads_per_unit, int32_t tc_late_ticket, int32_t simt_two_pass,
                                     int32_t conv_tma, int32_t tc_segment_chunks, int32_t tc_head_flags) {
    if (tc_heads_per_unit != -1 && (tc_heads_per_unit < 1 || tc_heads_per_unit > 8)) return SSD_ERR_INVALID_ARG;
    if (tc_late_ticket < -1 || tc_late_ticket > 1 || simt_two_pass < -1 || simt_two_pass > 1 || conv_tma < -1 ||
        conv_tma > 1 || tc_segment_chunks < -1 || tc_head_flags < -1 || tc_head_flags > 1)
        return SSD_ERR_INVALID_ARG;
    ssd::g_knob[5].store(tc_head_flags, std::memory_order_relaxed);
    ssd::g_knob[4].store(tc_segment_chunks, std::memory_order_relaxed);
    ssd::g_knob[0].store(tc_heads_per_unit, std::memory_order_relaxed);
    ssd::g_knob[1].store(tc_late_ticket, std::memory_order_relaxed);
    ssd::g_knob[2].store(simt_two_pass, std::memory_order_relaxed);
    ssd::g_knob[3].store(conv_tma, std::memory_order_relaxed);
    return SSD_OK;
}

SSD_API const char *ssd_status_string(ssd_status_t status) {
    switch (status) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported problem (no kernel instance)";
        case SSD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case SSD_ERR_CUDA: return "CUDA runtime error";
        case SSD_ERR_TIMEOUT: return "device wait timed out (state passing)";
        case SSD_ERR_DEVICE: return "device pipeline error";
    }
    return "unknown status";
}

SSD_API int ssd_version(void) { return 10100; }

}  // extern "C"

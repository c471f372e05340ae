// ssd_fwd_host: the SSD prefill forward on host-resident tensors, streamed
// through the GPU in pieces so that the host<->device copies overlap the
// computation.
//
// The batch is cut along its tokens at multiples of the chunk size, every
// piece holding the same token range of all sequences: the states leaving one
// piece are the states entering the next, which is the chunked scan's own
// state passing ("Mamba hardware-aware algorithms", structured state space
// duality: the final state of a prefix is the initial state of the rest), so
// the pieces compute the same chunks, in the same order and precision, as one
// call would, and each piece keeps the whole batch's parallelism. The states
// run through one device buffer in place; a piece's rows of x, dt_raw, B, C
// and y are strided in host memory (one row range per sequence) and move by
// 2-D copies.
//
// Three device slots hold a piece's inputs and outputs. For piece k in slot
// k % 3: its inputs are copied in on the library's upload stream once piece
// k - 3 has been computed, it is computed on the caller's stream once they
// are in and piece k - 3's outputs are out, and its outputs are copied out on
// the download stream. So the upload of piece k + 1, the computation of piece
// k and the download of piece k - 1 run at once (on GB300 the host link then
// carries about 340 GB/s both ways together, against 210 and 190 GB/s for one
// direction alone). A slot is busy from its upload to its download, so with
// two slots the slots, not the link, would pace the pieces. The two copy streams are created once per device and kept
// for the life of the process.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/ssd.h"

namespace {

constexpr int kMaxDevices = 64;
// The library's piece count: about 256 MiB of copies (up and down) per piece, from 8 to 32 pieces. Measured on
// GB300: the 256K-token layer (6.5 GB of copies) 23.4 ms with 8 pieces, 22.4 with 16, 22.2 with 32, 22.9 with 64;
// batch 8 of the 2.7B layer (1.4 GB) 5.07 ms with 8, 5.03 with 16, 5.56 with 32; 4 to 8 pieces were best on the
// smaller launches, where fewer pieces leave too little to overlap.
constexpr int kMinPieces = 8, kMaxPieces = 32;
constexpr size_t kPieceBytes = size_t(256) << 20;
constexpr int kSlots = 3;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }
size_t esize(int dt) { return dt == SSD_F32 ? 4 : 2; }

std::mutex g_streams_mu;
cudaStream_t g_up[kMaxDevices], g_down[kMaxDevices];

// The upload and download streams of the current device (created on first use).
bool copy_streams(cudaStream_t *up, cudaStream_t *down) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_streams_mu);
    if (!g_up[dev]) {
        cudaStream_t a = nullptr, b = nullptr;
        if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess) return false;
        if (cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(a);
            return false;
        }
        g_up[dev] = a;
        g_down[dev] = b;
    }
    *up = g_up[dev];
    *down = g_down[dev];
    return true;
}

// How a problem is cut and where the pieces live in the scratch. Piece k holds chunks [first(k), first(k + 1)) of
// every sequence: the first and the last piece `edge` chunks, the ones between `mid` chunks (the last of them
// possibly fewer). Short end pieces shorten the pipeline's fill (the first upload, before any computation) and
// drain (the last computation and download, after every other copy).
struct HostPlan {
    int64_t nc = 0;       // chunks per sequence
    int64_t edge = 0;     // chunks of the first and the last piece
    int64_t mid = 0;      // chunks of each piece between them
    int64_t pieces = 0;
    int64_t chunk = 0;    // tokens per chunk
    ssd_problem_t sub{};  // the largest piece: [batch, tokens of `mid` chunks]
    size_t ws = 0;        // workspace bytes of the largest piece (at offset 0 of the scratch)
    size_t bx = 0, bdt = 0, bbc = 0;  // per-slot bytes of x (and y), dt_raw, B (and C)
    size_t slot = 0;      // bytes of one slot (kSlots of them)
    size_t state_off = 0; // the states carried from piece to piece, [batch, H, P, N]
    size_t bytes = 0;     // total scratch
};

ssd_status_t host_plan(const ssd_problem_t *prob, int32_t pieces, HostPlan *out) {
    if (!prob || !out || pieces < 0) return SSD_ERR_INVALID_ARG;
    const ssd_problem_t &pr = *prob;
    size_t probe = 0;
    ssd_status_t st = ssd_fwd_workspace_size(prob, &probe);  // every problem check of ssd_fwd
    if (st != SSD_OK) return st;
    HostPlan hp;
    const size_t es = esize(pr.io_dtype), ses = esize(pr.state_dtype);
    const size_t states = align256((size_t)(pr.batch * pr.nheads * pr.headdim * pr.dstate) * ses);
    if (pr.batch == 0 || pr.seqlen == 0) {  // nothing to stream: only final = init (or zeros)
        hp.bytes = states;
        *out = hp;
        return SSD_OK;
    }
    const int64_t nc = (pr.seqlen + pr.chunk_size - 1) / pr.chunk_size;
    int64_t want = pieces;
    if (!want) {  // x, dt_raw, B, C up, y down, for the whole batch
        const size_t copied = (size_t)(pr.batch * pr.seqlen) *
                              (size_t)(2 * pr.nheads * pr.headdim + pr.nheads + 2 * pr.ngroups * pr.dstate) * es;
        const int64_t by_size = (int64_t)((copied + kPieceBytes - 1) / kPieceBytes);
        want = by_size < kMinPieces ? kMinPieces : (by_size > kMaxPieces ? kMaxPieces : by_size);
    }
    const int64_t n = want < nc ? want : nc;
    const int64_t even = (nc + n - 1) / n;  // chunks per piece of an even cut
    hp.nc = nc;
    hp.chunk = pr.chunk_size;
    hp.edge = hp.mid = even;
    // From 8 pieces on, end pieces of a quarter of the even size and the rest shared out evenly (measured on GB300
    // at 8 pieces: 3 % faster on the 130M-shaped batch, equal at L = 16K and batch 8; with 4 pieces the two middle
    // pieces grew too large to overlap, up to 10 % slower, so fewer pieces are cut evenly).
    if (n >= 8 && even >= 4) {
        hp.edge = even / 4;
        hp.mid = (nc - 2 * hp.edge + n - 3) / (n - 2);
        hp.pieces = 2 + (nc - 2 * hp.edge + hp.mid - 1) / hp.mid;
    } else {
        hp.pieces = (nc + even - 1) / even;
    }
    const int64_t big = (hp.mid > hp.edge ? hp.mid : hp.edge) * pr.chunk_size;
    hp.sub = pr;
    hp.sub.seqlen = big < pr.seqlen ? big : pr.seqlen;
    st = ssd_fwd_workspace_size(&hp.sub, &hp.ws);
    if (st != SSD_OK) return st;
    const int64_t T = hp.sub.batch * hp.sub.seqlen;  // tokens of the largest piece
    hp.bx = align256((size_t)(T * pr.nheads * pr.headdim) * es);
    hp.bdt = align256((size_t)(T * pr.nheads) * es);
    hp.bbc = align256((size_t)(T * pr.ngroups * pr.dstate) * es);
    hp.slot = 2 * hp.bx + hp.bdt + 2 * hp.bbc;  // x, y, dt, B, C
    hp.ws = align256(hp.ws);
    hp.state_off = hp.ws + kSlots * hp.slot;
    hp.bytes = hp.state_off + states;
    *out = hp;
    return SSD_OK;
}

// First chunk of piece k (k = pieces: the end).
int64_t piece_first(const HostPlan &hp, int64_t k) {
    if (k <= 0) return 0;
    if (k >= hp.pieces) return hp.nc;
    if (hp.edge == hp.mid) return k * hp.mid;
    if (k == hp.pieces - 1) return hp.nc - hp.edge;
    return hp.edge + (k - 1) * hp.mid;
}

}  // namespace

extern "C" {

SSD_API ssd_status_t ssd_fwd_host_scratch_size(const ssd_problem_t *prob, int32_t pieces, size_t *bytes) {
    if (!bytes) return SSD_ERR_INVALID_ARG;
    HostPlan hp;
    const ssd_status_t st = host_plan(prob, pieces, &hp);
    if (st != SSD_OK) return st;
    *bytes = hp.bytes;
    return SSD_OK;
}

SSD_API ssd_status_t ssd_fwd_host(const ssd_problem_t *prob, int32_t pieces, const void *x, const void *dt_raw,
                                  const float *dt_bias, const float *A, const void *B, const void *C, const float *D,
                                  const void *init_states, void *y, void *final_states, void *scratch,
                                  size_t scratch_bytes, void *stream) {
    HostPlan hp;
    ssd_status_t st = host_plan(prob, pieces, &hp);
    if (st != SSD_OK) return st;
    const ssd_problem_t &pr = *prob;
    if (hp.pieces == 0 && (!final_states || pr.batch == 0)) return SSD_OK;  // nothing to compute or write
    if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 255) || scratch_bytes < hp.bytes) return SSD_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t es = esize(pr.io_dtype), ses = esize(pr.state_dtype);
    const size_t state1 = (size_t)(pr.nheads * pr.headdim * pr.dstate) * ses;
    char *sc = static_cast<char *>(scratch);
    if (hp.pieces == 0) {  // no tokens: the final states are the initial ones (or zeros)
        const size_t n = (size_t)pr.batch * state1;
        cudaError_t e = init_states ? cudaMemcpyAsync(final_states, init_states, n, cudaMemcpyHostToHost, s)
                                    : cudaMemsetAsync(sc, 0, n, s);
        if (e == cudaSuccess && !init_states) e = cudaMemcpyAsync(final_states, sc, n, cudaMemcpyDeviceToHost, s);
        return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    }
    if (!x || !dt_raw || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    cudaStream_t up = nullptr, down = nullptr;
    if (!copy_streams(&up, &down)) return SSD_ERR_CUDA;

    // events: start, and per slot inputs-in / computed / outputs-out
    constexpr int kEv = 1 + 3 * kSlots;
    cudaEvent_t ev[kEv] = {};
    for (int i = 0; i < kEv; ++i)
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            return SSD_ERR_CUDA;
        }
    cudaEvent_t ev_start = ev[0], *ev_in = ev + 1, *ev_comp = ev + 1 + kSlots, *ev_out = ev + 1 + 2 * kSlots;
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t r) {
        if (e == cudaSuccess) e = r;
        return e == cudaSuccess;
    };
    // the copies come after whatever the caller queued on `stream` before (it may have written the inputs or
    // still use the scratch)
    ok(cudaEventRecord(ev_start, s));
    ok(cudaStreamWaitEvent(up, ev_start, 0));
    ok(cudaStreamWaitEvent(down, ev_start, 0));
    const char *hx = static_cast<const char *>(x), *hdt = static_cast<const char *>(dt_raw);
    const char *hb = static_cast<const char *>(B), *hc = static_cast<const char *>(C);
    char *hy = static_cast<char *>(y), *hfin = static_cast<char *>(final_states);
    char *state = sc + hp.state_off;
    const size_t states = (size_t)pr.batch * state1;
    // per token, the bytes of a row of x (and y), dt_raw, B (and C)
    const size_t rx = (size_t)(pr.nheads * pr.headdim) * es, rdt = (size_t)pr.nheads * es,
                 rbc = (size_t)(pr.ngroups * pr.dstate) * es;
    const size_t L = (size_t)pr.seqlen, nb = (size_t)pr.batch;
    if (init_states) ok(cudaMemcpyAsync(state, init_states, states, cudaMemcpyHostToDevice, up));
    for (int64_t k = 0; k < hp.pieces && e == cudaSuccess; ++k) {
        const int u = (int)(k % kSlots);
        char *slot = sc + hp.ws + (size_t)u * hp.slot;
        char *dx = slot, *dy = dx + hp.bx, *ddt = dy + hp.bx, *dB = ddt + hp.bdt, *dC = dB + hp.bbc;
        const size_t t0 = (size_t)(piece_first(hp, k) * hp.chunk);
        const size_t t1 = (size_t)(piece_first(hp, k + 1) * hp.chunk);
        const size_t n = (t1 < L ? t1 : L) - t0;  // tokens of the piece
        ssd_problem_t sub = pr;
        sub.seqlen = (int64_t)n;
        // inputs of piece k into slot u, once piece k - kSlots (same slot) has been computed: per sequence, rows
        // t0 .. t0 + n of [L] rows, packed to [n] rows
        if (k >= kSlots) ok(cudaStreamWaitEvent(up, ev_comp[u], 0));
        ok(cudaMemcpy2DAsync(dx, n * rx, hx + t0 * rx, L * rx, n * rx, nb, cudaMemcpyHostToDevice, up));
        ok(cudaMemcpy2DAsync(ddt, n * rdt, hdt + t0 * rdt, L * rdt, n * rdt, nb, cudaMemcpyHostToDevice, up));
        ok(cudaMemcpy2DAsync(dB, n * rbc, hb + t0 * rbc, L * rbc, n * rbc, nb, cudaMemcpyHostToDevice, up));
        ok(cudaMemcpy2DAsync(dC, n * rbc, hc + t0 * rbc, L * rbc, n * rbc, nb, cudaMemcpyHostToDevice, up));
        ok(cudaEventRecord(ev_in[u], up));
        // compute piece k on the caller's stream once its inputs are in and piece k - kSlots's outputs are out;
        // the states run through `state` in place (none on entry to the first piece without initial states)
        ok(cudaStreamWaitEvent(s, ev_in[u], 0));
        if (k >= kSlots) ok(cudaStreamWaitEvent(s, ev_out[u], 0));
        if (e != cudaSuccess) break;
        const void *init_d = (k == 0 && !init_states) ? nullptr : state;
        st = ssd_fwd(&sub, dx, ddt, dt_bias, A, dB, dC, D, init_d, dy, state, sc, hp.ws, stream);
        if (st != SSD_OK) break;
        ok(cudaEventRecord(ev_comp[u], s));
        // outputs of piece k back to the host
        ok(cudaStreamWaitEvent(down, ev_comp[u], 0));
        ok(cudaMemcpy2DAsync(hy + t0 * rx, L * rx, dy, n * rx, n * rx, nb, cudaMemcpyDeviceToHost, down));
        if (hfin && k == hp.pieces - 1) ok(cudaMemcpyAsync(hfin, state, states, cudaMemcpyDeviceToHost, down));
        ok(cudaEventRecord(ev_out[u], down));
    }
    // later work on `stream` comes after every copy queued above, on any path (the events are re-recorded at the
    // copy streams' ends)
    cudaError_t e2 = cudaEventRecord(ev_in[0], up);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, ev_in[0], 0);
    if (e2 == cudaSuccess) e2 = cudaEventRecord(ev_out[0], down);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, ev_out[0], 0);
    ok(e2);
    for (int i = 0; i < kEv; ++i) cudaEventDestroy(ev[i]);
    if (st != SSD_OK) return st;
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"

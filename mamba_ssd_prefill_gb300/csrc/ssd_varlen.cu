// Planning kernel of a variable-length batch: from the device array cu_seqlens
// (sequence s holds tokens cu[s] .. cu[s+1] of the packed token axis) it builds
// the chunk-major table of (sequence, chunk) pairs that the prefill kernels
// take tickets from, so that chunk c of every sequence comes before chunk c+1
// of any (every state wait then targets a lower ticket that a running CTA
// holds, as in a regular batch). Sequences restart the recurrence from their
// own initial state (a second kernel copies the initial state of the empty
// ones to their final state); this is the varlen form of the chunked scan in
// "Mamba hardware-aware algorithms" (pseudo chunks that never cross a sequence
// boundary), with chunks aligned to each sequence's start.
//
// One CTA: a counting sort of the sequences by chunk count (descending), so the
// sequences that reach chunk c are a prefix of that order and a sequence's
// slot is the same in every chunk: pair index = start[c] + rank(s), with
// start[c] = sum over c' < c of #{s : nc_s > c'}. Cost O(nseq + chunks). Bad
// offsets (not starting at 0, decreasing, or not ending at the token count) are
// reported in the workspace header and no work is scheduled.
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 1024;

// Block-wide exclusive prefix sum of a[0, n) in place (reverse = suffix sums: a[i] = sum over j > i).
__device__ void block_scan(uint32_t *a, int64_t n, bool reverse, uint32_t *part) {
    const int tid = threadIdx.x;
    const int64_t seg = (n + kThreads - 1) / kThreads;
    const int64_t lo = tid * seg, hi = lo + seg < n ? lo + seg : n;
    uint32_t sum = 0;
    for (int64_t i = lo; i < hi; ++i) sum += a[reverse ? n - 1 - i : i];
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        uint32_t run = 0;
        for (int k = 0; k < kThreads; ++k) {
            const uint32_t v = part[k];
            part[k] = run;
            run += v;
        }
    }
    __syncthreads();
    uint32_t run = part[tid];
    for (int64_t i = lo; i < hi; ++i) {
        const int64_t j = reverse ? n - 1 - i : i;
        const uint32_t v = a[j];
        a[j] = run;
        run += v;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) varlen_plan_kernel(Params p, uint32_t *scratch) {
    __shared__ uint32_t part[kThreads];
    __shared__ int bad;
    const int tid = threadIdx.x;
    const int64_t M = p.nc + 2;  // chunk counts 0 .. nc (+1 spare)
    uint32_t *hist = scratch, *base = scratch + M, *fill = scratch + 2 * M, *start = scratch + 3 * M;
    uint32_t *vtot = scratch + 4 * M;
    WsHeader *hdr = p.hdr;
    const int64_t T = p.batch * p.L;
    if (tid == 0) bad = 0;
    for (int64_t i = tid; i < M; i += kThreads) hist[i] = fill[i] = 0;
    __syncthreads();
    for (int64_t s = tid; s < p.nseq; s += kThreads) {
        const int64_t a = p.cu[s], b = p.cu[s + 1];
        if (a > b || b > T || (s == 0 && a != 0) || (s == p.nseq - 1 && b != T)) {
            bad = 1;
            continue;
        }
        atomicAdd(&hist[(b - a + p.Q - 1) / p.Q], 1u);
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            atomicCAS(&hdr->status, 0u, (uint32_t)DEV_BAD_SEQLENS);
            *vtot = 0;
        }
        return;
    }
    // base[v] = #{s : nc_s > v}: the rank of the first sequence with nc_s = v, and the sequences that reach chunk v
    for (int64_t i = tid; i < M; i += kThreads) base[i] = hist[i];
    __syncthreads();
    block_scan(base, M, true, part);
    // start[c] = sum over c' < c of base[c']: the first pair index of chunk c
    for (int64_t i = tid; i < M; i += kThreads) start[i] = base[i];
    __syncthreads();
    block_scan(start, M, false, part);
    if (tid == 0) *vtot = start[p.nc];
    // pairs: sequence s takes the same rank in every chunk it reaches
    for (int64_t s = tid; s < p.nseq; s += kThreads) {
        const int64_t len = p.cu[s + 1] - p.cu[s];
        const int64_t nc = (len + p.Q - 1) / p.Q;
        const uint32_t rank = base[nc] + atomicAdd(&fill[nc], 1u);
        int2 *ctab = const_cast<int2 *>(p.ctab);  // written here, read-only for the prefill kernels
        for (int64_t c = 0; c < nc; ++c) ctab[start[c] + rank] = make_int2((int)s, (int)c);
    }
}

// Sequences of length 0 have no chunk: their final state is the initial one (or zero). One CTA per sequence;
// the CTAs of non-empty sequences return at once. Copies in 2-byte words (a sequence's states are
// H * P * N elements of 2 or 4 bytes).
__global__ void __launch_bounds__(256) varlen_empty_kernel(Params p, int state_bytes) {
    const int64_t s = blockIdx.x;
    if (p.cu[s + 1] != p.cu[s]) return;
    const int64_t words = p.H * p.P * p.N * state_bytes / 2;
    uint16_t *dst = static_cast<uint16_t *>(p.final_states) + s * words;
    const uint16_t *src = p.init ? static_cast<const uint16_t *>(p.init) + s * words : nullptr;
    if (src == dst) return;
    for (int64_t i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src ? src[i] : (uint16_t)0;
}

}  // namespace

cudaError_t launch_varlen_plan(const Params &p, uint32_t *scratch, size_t state_bytes, cudaStream_t stream) {
    varlen_plan_kernel<<<1, kThreads, 0, stream>>>(p, scratch);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !p.final_states || p.nseq == 0) return e;
    varlen_empty_kernel<<<(unsigned)p.nseq, 256, 0, stream>>>(p, (int)state_bytes);
    return cudaGetLastError();
}

}  // namespace ssd

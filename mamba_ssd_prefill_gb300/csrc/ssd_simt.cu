// fp32 SIMT kernel of the fused SSD prefill forward.
//
// Used for fp32 I/O (where tensor-core TF32 would not hold the fp32 accuracy
// bound) and for shapes the tensor-core kernel has no instance for. One work
// unit is (chunk c, batch b, head h); units are handed out by an atomic ticket
// in chunk-major order, so a unit only ever waits on a lower ticket that a
// running CTA already holds (deadlock-free without co-residency).
//
// Per unit: wait for the state entering chunk c (the chain's 64-bit tag
// epoch:c in a 2-slot ring), then walk the chunk in 32-token sub-chunks with the running state
// in shared memory, doing the five SSD steps of "Accelerating Mamba2 with
// Kernel Fusion" (chunk cumsum, BMM, chunk state, state passing, chunk scan)
// at sub-chunk granularity, then publish the state leaving chunk c.
//
// With few chains (fewer than the resident CTAs) the chain's hops bound the launch, and each hop
// would carry the whole chunk's work. There the unit runs in two passes: first the chunk state from
// a zero state, s_c, and the chunk's decay a (no wait needed), then the wait, S_out = a S_in + s_c
// published at once, and only then the pass that produces y from S_in. A hop then costs the wait,
// one multiply-add per state element and the publish.
#include <stdlib.h>

#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kSub = 32;  // tokens per sub-chunk (one warp-wide cumsum)

template <typename IO, typename ST>
__global__ void __launch_bounds__(kThreads, 3) simt_kernel(Params p, int two_pass) {
    extern __shared__ float4 smem_f4[];
    float *smem = reinterpret_cast<float *>(smem_f4);
    const int P = (int)p.P, N = (int)p.N, NB = N + 1;  // padded B/C rows avoid bank conflicts
    float *S = smem;              // [N][P] running state
    float *xs = S + N * P;        // [kSub][P]
    float *Bs = xs + kSub * P;    // [kSub][N+1]
    float *Cs = Bs + kSub * NB;   // [kSub][N+1]
    float *Pm = Cs + kSub * NB;   // [kSub][kSub] masked, decayed C.B^T * dt
    float *cs = Pm + kSub * kSub; // [kSub] inclusive cumsum of dt*A
    float *dts = cs + kSub;       // [kSub] dt
    float *wj = dts + kSub;       // [kSub] exp(cs_last - cs_j) * dt_j
    float *ecs = wj + kSub;       // [kSub] exp(cs_i)
    __shared__ uint32_t s_ticket;
    __shared__ int s_ok;

    const int tid = threadIdx.x;
    WsHeader *hdr = p.hdr;
    const uint32_t epoch = ld_relaxed_gpu(&hdr->epoch) + 1u;
    const uint64_t limit = hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs;
    const int64_t skip = hdr->skip_publish - 1;  // -1: no chunk skipped
    const uint32_t total = total_units(p, (uint32_t)p.H);
    const IO *x = static_cast<const IO *>(p.x);
    const IO *dtr = static_cast<const IO *>(p.dt_raw);
    const IO *Bg = static_cast<const IO *>(p.B);
    const IO *Cg = static_cast<const IO *>(p.C);
    IO *y = static_cast<IO *>(p.y);
    const ST *init = static_cast<const ST *>(p.init);
    ST *fin = static_cast<ST *>(p.final_states);
    ST *ring = static_cast<ST *>(p.ring);

    for (;;) {
        if (tid == 0) s_ticket = atomicAdd(&hdr->ticket, 1u);
        __syncthreads();
        const uint32_t t = s_ticket;
        __syncthreads();
        if (t >= total) break;
        const SeqChunk sq = seq_chunk(p, t / p.H);
        const int64_t c = sq.c, h = t % p.H;
        const int64_t g = h / p.heads_per_group;
        const int64_t chain = sq.s * p.H + h;
        const bool last = c == (sq.len + p.Q - 1) / p.Q - 1;
        const float Ah = p.A[h], bias = p.dt_bias[h], Dh = p.D ? p.D[h] : 0.f;
        // extents of the checked accesses (bounds-checked builds)
        const int64_t Tt = p.batch * p.L, nstate = p.nseq * p.H * P * N;
        (void)Tt;
        (void)nstate;

        // tokens [c0, c1) of the packed token axis
        const int64_t c0 = sq.tok0 + c * p.Q, end = sq.tok0 + sq.len, c1 = (c0 + p.Q < end) ? c0 + p.Q : end;
        // step 1 of a sub-chunk (dt = softplus(dt_raw + bias), inclusive cumsum of dt*A; rows >= T: dt = 0) and
        // its x and B rows (and C rows when y is computed)
        auto load_sub = [&](int64_t s0, int T, bool with_c) {
            if (tid < 32) {
                float dtv = 0.f;
                if (tid < T) dtv = softplus_f32(to_f32(*chk(dtr, (s0 + tid) * p.H + h, 1, Tt * p.H, hdr, SITE_SIMT_IN)) + bias);
                float sc = dtv * Ah;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float u = __shfl_up_sync(0xffffffffu, sc, o);
                    if (tid >= o) sc += u;
                }
                const float last = __shfl_sync(0xffffffffu, sc, 31);
                cs[tid] = sc;
                dts[tid] = dtv;
                wj[tid] = expf(last - sc) * dtv;
                ecs[tid] = expf(sc);
            }
            for (int e = tid; e < kSub * P; e += kThreads) {
                const int r = e / P, q = e % P;
                xs[e] = r < T ? to_f32(*chk(x, (s0 + r) * p.x_ld + h * P + q, 1, Tt * p.x_ld, hdr, SITE_SIMT_IN)) : 0.f;
            }
            for (int e = tid; e < kSub * N; e += kThreads) {
                const int r = e / N, q = e % N;
                const int64_t off = (s0 + r) * p.bc_ld + g * N + q;
                Bs[r * NB + q] = r < T ? to_f32(*chk(Bg, off, 1, Tt * p.bc_ld, hdr, SITE_SIMT_IN)) : 0.f;
                if (with_c) Cs[r * NB + q] = r < T ? to_f32(*chk(Cg, off, 1, Tt * p.bc_ld, hdr, SITE_SIMT_IN)) : 0.f;
            }
            __syncthreads();
        };
        // steps 3 + 4 (chunk state, state passing) over a sub-chunk: S = exp(cs_last) S + sum_j w_j x_j (outer) B_j.
        // Where N and P are multiples of 4, a thread owns 4 x 4 blocks of S (4 state rows n, 4 columns q): per token
        // one 16-byte x load and 4 B loads feed 16 multiply-adds, against two loads per multiply-add otherwise.
        auto advance = [&](int T) {
            const float decay = ecs[kSub - 1];
            if ((N & 3) == 0 && (P & 3) == 0) {
                const int qb_n = P / 4;
                for (int blk = tid; blk < (N / 4) * qb_n; blk += kThreads) {
                    const int q0 = 4 * (blk % qb_n), n0 = 4 * (blk / qb_n);
                    float acc[4][4] = {};
                    for (int j = 0; j < T; ++j) {
                        const float4 xv = *reinterpret_cast<const float4 *>(xs + j * P + q0);
                        const float w = wj[j];
                        const float xw[4] = {w * xv.x, w * xv.y, w * xv.z, w * xv.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float b = Bs[j * NB + n0 + k];
#pragma unroll
                            for (int l = 0; l < 4; ++l) acc[k][l] = fmaf(xw[l], b, acc[k][l]);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float4 *row = reinterpret_cast<float4 *>(S + (n0 + k) * P + q0);
                        const float4 sv = *row;
                        *row = make_float4(fmaf(decay, sv.x, acc[k][0]), fmaf(decay, sv.y, acc[k][1]),
                                           fmaf(decay, sv.z, acc[k][2]), fmaf(decay, sv.w, acc[k][3]));
                    }
                }
            } else {
                for (int e = tid; e < N * P; e += kThreads) {
                    const int n = e / P, q = e % P;
                    float acc = 0.f;
                    for (int j = 0; j < T; ++j) acc = fmaf(wj[j] * xs[j * P + q], Bs[j * NB + n], acc);
                    S[e] = fmaf(decay, S[e], acc);
                }
            }
            __syncthreads();
        };

        // ---- two passes: the chunk state from a zero state (s_c) and the log of the chunk's decay
        float log_a = 0.f;
        if (two_pass) {
            for (int e = tid; e < N * P; e += kThreads) S[e] = 0.f;
            for (int64_t s0 = c0; s0 < c1; s0 += kSub) {
                const int T = (int)((c1 - s0) < kSub ? (c1 - s0) : kSub);
                load_sub(s0, T, false);
                log_a += cs[kSub - 1];
                advance(T);
            }
        }

        // ---- state entering chunk c
        if (tid == 0)
            s_ok = aborted(hdr, epoch) ? 0
                                       : (c == 0 ? 1 : (int)wait_flag(chk(p.flags, chain * 2 + (c & 1), 1, p.flag_count, hdr, SITE_SIMT_FLAG), chain_tag(epoch, c),
                                                                      epoch, hdr, limit, t, (uint32_t)c));
        __syncthreads();
        if (!s_ok) continue;  // launch aborted: drain the remaining tickets
        const bool publish = !last && c != skip;
        const int64_t slot_in = (chain * 2 + (c & 1)) * (int64_t)(N * P), slot_out = (chain * 2 + ((c + 1) & 1)) * (int64_t)(N * P);
        const float a_c = expf(log_a);  // the chunk's decay (two passes)
        for (int e = tid; e < N * P; e += kThreads) {
            float s_in;
            if (c == 0) {
                const int n = e / P, q = e % P;
                s_in = init ? to_f32(*chk(init, (chain * P + q) * N + n, 1, nstate, hdr, SITE_SIMT_INIT)) : 0.f;
            } else {
                s_in = to_f32(__ldcg(chk(ring, slot_in + e, 1, p.ring_bytes / (int64_t)sizeof(ST), hdr, SITE_SIMT_RING)));
            }
            if (two_pass) {  // the state leaving the chunk, right away
                const float sout = fmaf(a_c, s_in, S[e]);
                if (publish)
                    __stcg(chk(ring, slot_out + e, 1, p.ring_bytes / (int64_t)sizeof(ST), hdr, SITE_SIMT_RING), from_f32<ST>(sout));
                else if (last && fin) {
                    const int n = e / P, q = e % P;
                    *chk(fin, (chain * P + q) * N + n, 1, nstate, hdr, SITE_SIMT_FINAL) = from_f32<ST>(sout);
                }
            }
            S[e] = s_in;
        }
        if (two_pass && publish) {
            __threadfence();
            __syncthreads();
            if (tid == 0)
                st_release_u64(chk(p.flags, chain * 2 + ((c + 1) & 1), 1, p.flag_count, hdr, SITE_SIMT_FLAG),
                               chain_tag(epoch, c + 1));
        }
        __syncthreads();

        // ---- y over the chunk, the running state from S_in
        for (int64_t s0 = c0; s0 < c1; s0 += kSub) {
            const int T = (int)((c1 - s0) < kSub ? (c1 - s0) : kSub);
            load_sub(s0, T, true);
            // step 2 (BMM) with the segsum decay mask: Pm[i][j] = (C_i.B_j) exp(cs_i - cs_j) dt_j, j <= i
            for (int e = tid; e < kSub * kSub; e += kThreads) {
                const int i = e / kSub, j = e % kSub;
                float v = 0.f;
                if (j <= i) {
                    float d = 0.f;
                    for (int n = 0; n < N; ++n) d = fmaf(Cs[i * NB + n], Bs[j * NB + n], d);
                    v = d * expf(cs[i] - cs[j]) * dts[j];
                }
                Pm[e] = v;
            }
            __syncthreads();
            // step 5 (chunk scan): y_i = sum_j Pm_ij x_j + exp(cs_i) C_i . S + D x_i. Where P is a multiple of 4, a
            // thread owns 2 tokens x 4 columns: per step one 16-byte load of x (or S) and two of Pm (or C) feed 8
            // multiply-adds, in the scalar loop's order (row i0's extra term j = i0 + 1 has Pm = 0: exact).
            if ((P & 3) == 0) {
                const int qb_n = P / 4;
                for (int blk = tid; blk < (kSub / 2) * qb_n; blk += kThreads) {
                    const int q0 = 4 * (blk % qb_n), i0 = 2 * (blk / qb_n);
                    if (i0 >= T) continue;
                    float a1[2][4] = {}, a2[2][4] = {};
                    for (int j = 0; j <= i0 + 1; ++j) {
                        const float4 xv = *reinterpret_cast<const float4 *>(xs + j * P + q0);
                        const float p0 = Pm[i0 * kSub + j], p1 = Pm[(i0 + 1) * kSub + j];
                        a1[0][0] = fmaf(p0, xv.x, a1[0][0]); a1[0][1] = fmaf(p0, xv.y, a1[0][1]);
                        a1[0][2] = fmaf(p0, xv.z, a1[0][2]); a1[0][3] = fmaf(p0, xv.w, a1[0][3]);
                        a1[1][0] = fmaf(p1, xv.x, a1[1][0]); a1[1][1] = fmaf(p1, xv.y, a1[1][1]);
                        a1[1][2] = fmaf(p1, xv.z, a1[1][2]); a1[1][3] = fmaf(p1, xv.w, a1[1][3]);
                    }
                    for (int n = 0; n < N; ++n) {
                        const float4 sv = *reinterpret_cast<const float4 *>(S + n * P + q0);
                        const float c0 = Cs[i0 * NB + n], c1 = Cs[(i0 + 1) * NB + n];
                        a2[0][0] = fmaf(c0, sv.x, a2[0][0]); a2[0][1] = fmaf(c0, sv.y, a2[0][1]);
                        a2[0][2] = fmaf(c0, sv.z, a2[0][2]); a2[0][3] = fmaf(c0, sv.w, a2[0][3]);
                        a2[1][0] = fmaf(c1, sv.x, a2[1][0]); a2[1][1] = fmaf(c1, sv.y, a2[1][1]);
                        a2[1][2] = fmaf(c1, sv.z, a2[1][2]); a2[1][3] = fmaf(c1, sv.w, a2[1][3]);
                    }
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int i = i0 + r;
                        if (i >= T) break;
#pragma unroll
                        for (int l = 0; l < 4; ++l) {
                            const float v = a1[r][l] + ecs[i] * a2[r][l] + Dh * xs[i * P + q0 + l];
                            *chk(y, ((s0 + i) * p.H + h) * P + q0 + l, 1, Tt * p.H * P, hdr, SITE_SIMT_Y) = from_f32<IO>(v);
                        }
                    }
                }
            } else {
                for (int e = tid; e < T * P; e += kThreads) {
                    const int i = e / P, q = e % P;
                    float a1 = 0.f, a2 = 0.f;
                    for (int j = 0; j <= i; ++j) a1 = fmaf(Pm[i * kSub + j], xs[j * P + q], a1);
                    for (int n = 0; n < N; ++n) a2 = fmaf(Cs[i * NB + n], S[n * P + q], a2);
                    const float v = a1 + ecs[i] * a2 + Dh * xs[i * P + q];
                    *chk(y, ((s0 + i) * p.H + h) * P + q, 1, Tt * p.H * P, hdr, SITE_SIMT_Y) = from_f32<IO>(v);
                }
            }
            __syncthreads();
            // the state entering the next sub-chunk (two passes: not needed after the last one)
            if (!two_pass || s0 + kSub < c1) advance(T);
        }

        // ---- one pass: publish the state leaving chunk c
        if (!two_pass) {
            if (last) {
                if (fin)
                    for (int e = tid; e < N * P; e += kThreads) {
                        const int q = e / N, n = e % N;
                        *chk(fin, (chain * P + q) * N + n, 1, nstate, hdr, SITE_SIMT_FINAL) = from_f32<ST>(S[n * P + q]);
                    }
            } else if (c != skip) {
                for (int e = tid; e < N * P; e += kThreads)
                    __stcg(chk(ring, slot_out + e, 1, p.ring_bytes / (int64_t)sizeof(ST), hdr, SITE_SIMT_RING), from_f32<ST>(S[e]));
                __threadfence();
                __syncthreads();
                if (tid == 0)
                    st_release_u64(chk(p.flags, chain * 2 + ((c + 1) & 1), 1, p.flag_count, hdr, SITE_SIMT_FLAG),
                                   chain_tag(epoch, c + 1));
            }
        }
        __syncthreads();
    }

    // ---- launch bookkeeping: the last CTA resets the counters and commits the epoch
    __syncthreads();
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

template <typename IO, typename ST>
cudaError_t launch_t(const Params &p, int sms, cudaStream_t stream) {
    const size_t smem = simt_smem_bytes(p.P, p.N);
    auto k = simt_kernel<IO, ST>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t grid = p.ctab ? (int64_t)sms * per_sm : std::min<int64_t>((int64_t)p.total_units, (int64_t)sms * per_sm);
    // two passes where the chains are fewer than the resident CTAs (the hops bound the launch); the
    // simt_two_pass test hook (ssd_debug_knobs) forces one form
    int two_pass = p.nseq * p.H < (int64_t)sms * per_sm;
    const int forced = knobs().simt_two_pass;
    if (forced >= 0) two_pass = forced;
    k<<<(unsigned)grid, kThreads, smem, stream>>>(p, two_pass);
    return cudaGetLastError();
}

}  // namespace

size_t simt_smem_bytes(int64_t P, int64_t N) {
    return sizeof(float) * (size_t)(N * P + kSub * P + 2 * kSub * (N + 1) + kSub * kSub + 4 * kSub);
}

cudaError_t launch_simt(const Params &p, int io_dtype, int state_dtype, int sms, cudaStream_t stream) {
    if (state_dtype == 0) {
        if (io_dtype == 0) return launch_t<float, float>(p, sms, stream);
        if (io_dtype == 1) return launch_t<__nv_bfloat16, float>(p, sms, stream);
        return launch_t<__half, float>(p, sms, stream);
    }
    if (io_dtype == 0) return launch_t<float, __half>(p, sms, stream);
    if (io_dtype == 1) return launch_t<__nv_bfloat16, __half>(p, sms, stream);
    return launch_t<__half, __half>(p, sms, stream);
}

}  // namespace ssd

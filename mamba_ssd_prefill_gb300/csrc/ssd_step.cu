// Single-token step of the SSD recurrence (decode): for every (batch, head)
// chain, with dt = softplus(dt_raw + dt_bias),
//
//   h'[p, n] = exp(dt A) h[p, n] + dt x[p] B[n]
//   y[p]     = sum_n C[n] h'[p, n] + D x[p]
//
// the recurrent form of the state space model ("Mamba-2 state space model
// compiler optimisation", the step function that advances the cached state by
// one token; its state cache is the [batch, heads, headdim, d_state] layout the
// prefill kernels read and write). It is the seqlen = 1 case of the prefill
// problem and reads and writes the same tensors.
//
// Memory-bound: every state element is read once and written once, in fp32
// arithmetic. Warps own state rows p (d_state elements, in 8- or 16-byte
// vectors when the row allows), the C.h' reduction by warp shuffles, a
// grid-stride loop over chains. No workspace and no inter-CTA ordering.
#include <type_traits>

#include "sm100_ptx.cuh"
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// K consecutive elements starting at p (16- or 8-byte vectors when K elements fill one) -> fp32
template <typename T, int K> __device__ __forceinline__ void load_k(const T *p, float (&f)[K]) {
    if constexpr (sizeof(T) * K == 16 || sizeof(T) * K == 8) {
        using V = typename std::conditional<sizeof(T) * K == 16, uint4, uint2>::type;
        const V u = *reinterpret_cast<const V *>(p);
        const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int i = 0; i < K; ++i) f[i] = to_f32(e[i]);
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) f[i] = to_f32(p[i]);
    }
}
template <typename T, int K> __device__ __forceinline__ void store_k(T *p, const float (&f)[K]) {
    if constexpr (sizeof(T) * K == 16 || sizeof(T) * K == 8) {
        using V = typename std::conditional<sizeof(T) * K == 16, uint4, uint2>::type;
        V u;
        T *e = reinterpret_cast<T *>(&u);
#pragma unroll
        for (int i = 0; i < K; ++i) e[i] = from_f32<T>(f[i]);
        *reinterpret_cast<V *>(p) = u;
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) p[i] = from_f32<T>(f[i]);
    }
}

// K state elements per lane per pass (a vector when the row allows, else 1); LPR lanes per state row (32, or 16
// when 16 lanes of K elements cover the row), so a warp holds 32 / LPR rows at a time. Each warp advances two such
// row sets at once, all loads issued before any store (distinct elements, so safe when the state is updated in
// place), which keeps 1 KB per warp in flight.
template <typename IO, typename ST, int K, int LPR>
__global__ void __launch_bounds__(kThreads) step_kernel(Params p) {
    constexpr int SUBS = 32 / LPR, ROWS = 2 * SUBS;  // rows per warp and pass
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPR, l = lane % LPR;
    const IO *x = static_cast<const IO *>(p.x);
    const IO *dtr = static_cast<const IO *>(p.dt_raw);
    const IO *Bm = static_cast<const IO *>(p.B);
    const IO *Cm = static_cast<const IO *>(p.C);
    const ST *hin = static_cast<const ST *>(p.init);
    ST *hout = static_cast<ST *>(p.final_states);
    IO *y = static_cast<IO *>(p.y);
    const int64_t chains = p.batch * p.H;
    // extents of the checked accesses (bounds-checked builds)
    const int64_t nst = chains * p.P * p.N, nbc = p.batch * p.bc_ld, nx = p.batch * p.x_ld;
    (void)nst;
    (void)nbc;
    (void)nx;
    for (int64_t ch = blockIdx.x; ch < chains; ch += gridDim.x) {
        const int64_t b = ch / p.H, h = ch % p.H, g = h / p.heads_per_group;
        const float dt = softplus_f32(to_f32(*chk(dtr, ch, 1, chains, p.hdr, SITE_STEP_IN)) + p.dt_bias[h]);
        const float a = expf(dt * p.A[h]);
        const float Dh = p.D ? p.D[h] : 0.f;
        const IO *Bg = chk(Bm, b * p.bc_ld + g * p.N, p.N, nbc, p.hdr, SITE_STEP_IN);
        const IO *Cg = chk(Cm, b * p.bc_ld + g * p.N, p.N, nbc, p.hdr, SITE_STEP_IN);
        const IO *xh = chk(x, b * p.x_ld + h * p.P, p.P, nx, p.hdr, SITE_STEP_IN);  // this chain's token
        const int64_t base = ch * p.P * p.N;
        const ST *hin_c = hin ? chk(hin, base, p.P * p.N, nst, p.hdr, SITE_STEP_STATE) : nullptr;
        ST *hout_c = hout ? chk(hout, base, p.P * p.N, nst, p.hdr, SITE_STEP_STATE) : nullptr;
        IO *y_c = chk(y, ch * p.P, p.P, chains * p.P, p.hdr, SITE_STEP_Y);
        for (int64_t r0 = (int64_t)warp * ROWS; r0 < p.P; r0 += (int64_t)kWarps * ROWS) {
            const int64_t p0 = r0 + sub, p1 = r0 + SUBS + sub;
            const bool one = p0 < p.P, two = p1 < p.P;
            const float x0 = one ? to_f32(xh[p0]) : 0.f, x1 = two ? to_f32(xh[p1]) : 0.f;
            float acc0 = 0.f, acc1 = 0.f;
            for (int64_t n0 = (int64_t)l * K; n0 < p.N; n0 += LPR * K) {
                float h0[K], h1[K], bv[K], cv[K];
#pragma unroll
                for (int i = 0; i < K; ++i) h0[i] = h1[i] = 0.f;
                if (hin) {
                    if (one) load_k<ST, K>(hin_c + p0 * p.N + n0, h0);
                    if (two) load_k<ST, K>(hin_c + p1 * p.N + n0, h1);
                }
                load_k<IO, K>(Bg + n0, bv);
                load_k<IO, K>(Cg + n0, cv);
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    h0[i] = fmaf(a, h0[i], dt * x0 * bv[i]);
                    h1[i] = fmaf(a, h1[i], dt * x1 * bv[i]);
                    acc0 = fmaf(cv[i], h0[i], acc0);
                    acc1 = fmaf(cv[i], h1[i], acc1);
                }
                if (hout) {
                    if (one) store_k<ST, K>(hout_c + p0 * p.N + n0, h0);
                    if (two) store_k<ST, K>(hout_c + p1 * p.N + n0, h1);
                }
            }
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) {
                acc0 += __shfl_xor_sync(0xffffffffu, acc0, o);
                acc1 += __shfl_xor_sync(0xffffffffu, acc1, o);
            }
            if (l == 0) {
                if (one) y_c[p0] = from_f32<IO>(fmaf(Dh, x0, acc0));
                if (two) y_c[p1] = from_f32<IO>(fmaf(Dh, x1, acc1));
            }
        }
    }
}

// Staged form for rows of 128, 256 or 512 bytes: persistent CTAs (2 per SM with fp32 states, 4 with fp16 ones)
// keep several chains' states in flight in shared memory. Thread 0 loads a chain's state (P x N, contiguous)
// together with its B and C rows and its x by plain bulk copies onto one mbarrier, `stages - 1` chains ahead;
// the warps update the state in place (a lane owns a 16-byte vector of a row, LPR lanes a row), write y, and
// thread 0 sends the state back by one bulk store. The bytes in flight are the stages', not registers', and the
// CTAs of an SM overlap each other's per-chain latencies (measured on GB300: 64 x 80 fp32 states 0.068 -> 0.061
// ms, 256 x 80 fp16 states 0.205 -> 0.121 ms against the register-only form).
constexpr int kBulkThreads = 256;
template <typename ST> constexpr int bulk_ctas() { return sizeof(ST) == 4 ? 2 : 4; }
template <typename ST> constexpr uint32_t bulk_smem() { return 200u * 1024u / bulk_ctas<ST>(); }  // per CTA

__device__ __noinline__ void step_pipe_error(WsHeader *hdr) {
    if (atomicCAS(&hdr->status, 0u, (uint32_t)DEV_PIPE) == 0u) hdr->err_where = WAIT_PIPE;
}

template <typename IO, typename ST, int LPR>
__global__ void __launch_bounds__(kBulkThreads, bulk_ctas<ST>()) step_bulk_kernel(Params p, int stages, uint32_t stride) {
    using namespace sm100;
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int V = 16 / (int)sizeof(ST), RPW = 32 / LPR, kWarpsB = kBulkThreads / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, sub = lane / LPR, l = lane % LPR;
    const IO *x = static_cast<const IO *>(p.x);
    const IO *dtr = static_cast<const IO *>(p.dt_raw);
    const IO *Bm = static_cast<const IO *>(p.B);
    const IO *Cm = static_cast<const IO *>(p.C);
    const ST *hin = static_cast<const ST *>(p.init);
    ST *hout = static_cast<ST *>(p.final_states);
    IO *y = static_cast<IO *>(p.y);
    const uint32_t SB = (uint32_t)(p.P * p.N * sizeof(ST)), BB = (uint32_t)(p.N * sizeof(IO));
    const uint32_t XB = (uint32_t)(p.P * sizeof(IO));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stride);
    const int64_t chains = p.batch * p.H;
    const int64_t mine = blockIdx.x < chains ? (chains - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (tid == 0) {
        for (int i = 0; i < stages; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // thread 0: chain j's state, B and C rows and x into stage j % stages
    auto issue = [&](int64_t j) {
        const int st = (int)(j % stages);
        const int64_t ch = blockIdx.x + j * gridDim.x;
        const int64_t b = ch / p.H, h = ch % p.H, g = h / p.heads_per_group;
        uint8_t *base = smem + (size_t)st * stride;
        mbar_arrive_expect_tx(&full[st], (hin ? SB : 0u) + 2 * BB + XB);
        if (hin) bulk_load(base, chk(hin, ch * p.P * p.N, p.P * p.N, chains * p.P * p.N, p.hdr, SITE_STEP_STATE), SB, &full[st]);
        bulk_load(base + SB, chk(Bm, b * p.bc_ld + g * p.N, p.N, p.batch * p.bc_ld, p.hdr, SITE_STEP_IN), BB, &full[st]);
        bulk_load(base + SB + BB, chk(Cm, b * p.bc_ld + g * p.N, p.N, p.batch * p.bc_ld, p.hdr, SITE_STEP_IN), BB, &full[st]);
        bulk_load(base + SB + 2 * BB, chk(x, b * p.x_ld + h * p.P, p.P, p.batch * p.x_ld, p.hdr, SITE_STEP_IN), XB, &full[st]);
    };
    int64_t issued = 0;
    if (tid == 0)
        for (; issued < stages - 1 && issued < mine; ++issued) issue(issued);
    bool failed = false;
    int64_t j = 0;
    for (; j < mine; ++j) {
        const int st = (int)(j % stages);
        const int64_t ch = blockIdx.x + j * gridDim.x;
        const int64_t h = ch % p.H;
        // bounded wait for the stage (every thread; the outcome is made uniform below)
        if (!mbar_try_wait(&full[st], (uint32_t)((j / stages) & 1))) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(&full[st], (uint32_t)((j / stages) & 1)))
                if (globaltimer() - t0 > kDefaultTimeoutNs) {
                    failed = true;
                    break;
                }
        }
        if (!failed) {
            const float dt = softplus_f32(to_f32(*chk(dtr, ch, 1, chains, p.hdr, SITE_STEP_IN)) + p.dt_bias[h]);
            const float a = expf(dt * p.A[h]);
            const float Dh = p.D ? p.D[h] : 0.f;
            uint8_t *base = smem + (size_t)st * stride;
            IO *y_c = chk(y, ch * p.P, p.P, chains * p.P, p.hdr, SITE_STEP_Y);
            ST *S = reinterpret_cast<ST *>(base);
            const IO *Bs = reinterpret_cast<const IO *>(base + SB);
            const IO *Cs = Bs + p.N;
            const IO *xs = reinterpret_cast<const IO *>(base + SB + 2 * BB);
            float bv[V], cv[V];
#pragma unroll
            for (int i = 0; i < V; ++i) {
                bv[i] = to_f32(Bs[l * V + i]);
                cv[i] = to_f32(Cs[l * V + i]);
            }
            for (int r = warp * RPW + sub; r < p.P; r += kWarpsB * RPW) {
                const float xv = to_f32(xs[r]);
                float hv[V];
                ST *row = S + (int64_t)r * p.N + l * V;
                if (hin) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(row);
                    const ST *e = reinterpret_cast<const ST *>(&u);
#pragma unroll
                    for (int i = 0; i < V; ++i) hv[i] = to_f32(e[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < V; ++i) hv[i] = 0.f;
                }
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    hv[i] = fmaf(a, hv[i], dt * xv * bv[i]);
                    acc = fmaf(cv[i], hv[i], acc);
                }
                if (hout) {
                    uint4 u;
                    ST *e = reinterpret_cast<ST *>(&u);
#pragma unroll
                    for (int i = 0; i < V; ++i) e[i] = from_f32<ST>(hv[i]);
                    *reinterpret_cast<uint4 *>(row) = u;
                }
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (l == 0) y_c[r] = from_f32<IO>(fmaf(Dh, xv, acc));
            }
            if (hout) fence_proxy_async_smem();  // the updated rows, for the bulk store
        }
        if (__syncthreads_or(failed)) {
            failed = true;
            break;
        }
        if (tid == 0) {
            if (hout) {
                bulk_store(chk(hout, ch * p.P * p.N, p.P * p.N, chains * p.P * p.N, p.hdr, SITE_STEP_STATE),
                           smem + (size_t)st * stride, SB);
                bulk_commit();
            }
            // refill the stage of chain j - 1 (its store has been issued one chain ago) with chain j + stages - 1
            if (issued < mine) {
                if (hout) bulk_wait_read1();
                issue(issued);
                ++issued;
            }
        }
    }
    if (tid == 0) {
        if (failed) {  // record it, and let the loads still in flight land before the shared memory is released
            step_pipe_error(p.hdr);
            for (int64_t k = j; k < issued; ++k) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&full[k % stages], (uint32_t)((k / stages) & 1)) &&
                       globaltimer() - t0 < 100000000ull) {
                }
            }
        }
        bulk_wait0();  // every state store has completed
    }
}

template <typename IO, typename ST, int LPR>
cudaError_t launch_bulk(const Params &p, int sms, cudaStream_t stream) {
    const uint32_t SB = (uint32_t)(p.P * p.N * sizeof(ST)), BB = (uint32_t)(p.N * sizeof(IO));
    const uint32_t XB = (uint32_t)(p.P * sizeof(IO));
    const uint32_t stride = (SB + 2 * BB + XB + 127) / 128 * 128;
    const int stages = (int)std::min<uint32_t>(8u, bulk_smem<ST>() / stride);
    const size_t smem = (size_t)stages * stride + 8 * (size_t)stages;
    auto k = step_bulk_kernel<IO, ST, LPR>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(p.batch * p.H, (int64_t)sms * bulk_ctas<ST>());
    k<<<(unsigned)grid, kBulkThreads, smem, stream>>>(p, stages, stride);
    return cudaGetLastError();
}

// The staged kernel takes rows of 128, 256 or 512 bytes whose state, B, C and x rows all start on 16 bytes and
// at least two stages of them fit in a CTA's share of shared memory.
template <typename IO, typename ST>
bool bulk_ok(const Params &p) {
    const int64_t row = p.N * (int64_t)sizeof(ST), es = sizeof(IO);
    const uint64_t stride = ((uint64_t)(p.P * p.N * sizeof(ST) + 2 * p.N * es + p.P * es) + 127) / 128 * 128;
    const bool al = ((reinterpret_cast<uintptr_t>(p.init) | reinterpret_cast<uintptr_t>(p.final_states) |
                      reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.B) |
                      reinterpret_cast<uintptr_t>(p.C)) % 16) == 0;
    return al && (row == 128 || row == 256 || row == 512) && (p.N * es) % 16 == 0 && (p.P * es) % 16 == 0 &&
           (p.bc_ld * es) % 16 == 0 && (p.x_ld * es) % 16 == 0 && 2 * stride <= bulk_smem<ST>() && p.P <= (1 << 20);
}

template <typename IO, typename ST>
cudaError_t launch_t(const Params &p, int sms, cudaStream_t stream) {
    if (bulk_ok<IO, ST>(p)) {
        const int64_t lpr = p.N * (int64_t)sizeof(ST) / 16;
        if (lpr == 32) return launch_bulk<IO, ST, 32>(p, sms, stream);
        if (lpr == 16) return launch_bulk<IO, ST, 16>(p, sms, stream);
        return launch_bulk<IO, ST, 8>(p, sms, stream);
    }
    const int64_t chains = p.batch * p.H;
    const int64_t grid = std::min<int64_t>(chains, (int64_t)sms * 16);
    // 16-byte state vectors (8-byte for short rows) need the row length to be a multiple of the vector and aligned
    // state rows (B and C are 16-byte aligned by the API; where a vector of them is not 8 or 16 bytes they are read
    // element-wise). A row of exactly 16 vectors is split over half-warps.
    constexpr int K16 = 16 / (int)sizeof(ST), K8 = 8 / (int)sizeof(ST);
    const bool aligned = ((reinterpret_cast<uintptr_t>(p.init) | reinterpret_cast<uintptr_t>(p.final_states)) % 16) == 0;
    if (aligned && p.N % K16 == 0 && p.N >= 32 * K16)
        step_kernel<IO, ST, K16, 32><<<(unsigned)grid, kThreads, 0, stream>>>(p);
    else if (aligned && p.N == 16 * K16)
        step_kernel<IO, ST, K16, 16><<<(unsigned)grid, kThreads, 0, stream>>>(p);
    else if (aligned && p.N % K8 == 0)
        step_kernel<IO, ST, K8, 32><<<(unsigned)grid, kThreads, 0, stream>>>(p);
    else
        step_kernel<IO, ST, 1, 32><<<(unsigned)grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_step(const Params &p, int io_dtype, int state_dtype, int sms, cudaStream_t stream) {
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

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
    for (int64_t ch = blockIdx.x; ch < chains; ch += gridDim.x) {
        const int64_t b = ch / p.H, h = ch % p.H, g = h / p.heads_per_group;
        const float dt = softplus_f32(to_f32(dtr[ch]) + p.dt_bias[h]);
        const float a = expf(dt * p.A[h]);
        const float Dh = p.D ? p.D[h] : 0.f;
        const IO *Bg = Bm + b * p.bc_ld + g * p.N;
        const IO *Cg = Cm + b * p.bc_ld + g * p.N;
        const IO *xh = x + b * p.x_ld + h * p.P;  // this chain's token
        const int64_t base = ch * p.P * p.N;
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
                    if (one) load_k<ST, K>(hin + base + p0 * p.N + n0, h0);
                    if (two) load_k<ST, K>(hin + base + p1 * p.N + n0, h1);
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
                    if (one) store_k<ST, K>(hout + base + p0 * p.N + n0, h0);
                    if (two) store_k<ST, K>(hout + base + p1 * p.N + n0, h1);
                }
            }
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) {
                acc0 += __shfl_xor_sync(0xffffffffu, acc0, o);
                acc1 += __shfl_xor_sync(0xffffffffu, acc1, o);
            }
            if (l == 0) {
                if (one) y[ch * p.P + p0] = from_f32<IO>(fmaf(Dh, x0, acc0));
                if (two) y[ch * p.P + p1] = from_f32<IO>(fmaf(Dh, x1, acc1));
            }
        }
    }
}

template <typename IO, typename ST>
cudaError_t launch_t(const Params &p, int sms, cudaStream_t stream) {
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

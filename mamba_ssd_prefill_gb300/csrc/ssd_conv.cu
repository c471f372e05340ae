// Causal depthwise convolution in front of the SSD ("Accelerating Mamba2 with
// Kernel Fusion", Mamba-2 core operations item 3: each channel mixes its most
// recent tokens; "Mamba-2 compiler optimisation" section 2.2: the cache of the
// last k - 1 inputs per channel, [batch, channels, k - 1]):
//
//   out[t, ch] = act(bias[ch] + sum_j w[ch, j] * in[t - (k - 1) + j, ch])
//
// with in[t' < 0] read from the cache (zeros without one) and act the identity
// or SiLU, v * sigmoid(v). The channels are the x | B | C concatenation of the
// SSD inputs, so the SSD reads x, B and C as column slices of the output.
//
// HBM-bound: a thread walks 32 tokens of one 16-byte vector of channels with
// the taps and the last k - 1 inputs in registers, so every input is read once;
// fp32 arithmetic. A second kernel writes the cache for continuing each
// sequence.
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 256;

template <typename IO> __device__ __forceinline__ void load_vec(const IO *p, float (&f)[16 / sizeof(IO)]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const IO *e = reinterpret_cast<const IO *>(&u);
#pragma unroll
    for (int i = 0; i < (int)(16 / sizeof(IO)); ++i) f[i] = to_f32(e[i]);
}

constexpr int kTokens = 32;  // tokens per thread: the taps and the window of the last k - 1 inputs stay in registers

// Inputs before token tt of sequence s for window slot j (token tt - 1 - j): from the rows, else the cache, else 0.
template <typename IO, int V>
__device__ __forceinline__ void load_before(const ConvParams &c, const IO *in, const IO *state, int64_t s, int64_t tt,
                                            int64_t c0, int j, float (&v)[V]) {
    const int64_t tp = tt - 1 - j;
    if (tp >= 0) {
        load_vec<IO>(in + (s * c.L + tp) * c.D + c0, v);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) v[i] = state ? to_f32(state[((s * c.D) + c0 + i) * (c.k - 1) + (c.k - 1 + tp)]) : 0.f;
    }
}

// One thread: a 16-byte vector of channels over kTokens consecutive tokens (a warp covers 512 contiguous bytes of
// each token's row). The window restarts at a sequence start.
template <typename IO, int K>
__global__ void __launch_bounds__(kThreads) conv_kernel(ConvParams c) {
    constexpr int V = 16 / sizeof(IO);
    const IO *in = static_cast<const IO *>(c.in);
    const IO *state = static_cast<const IO *>(c.state);
    IO *out = static_cast<IO *>(c.out);
    const int64_t groups = c.D / V, blocks = (c.T + kTokens - 1) / kTokens, total = blocks * groups;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += (int64_t)gridDim.x * kThreads) {
        const int64_t t0 = (e / groups) * kTokens, c0 = (e % groups) * V;
        float w[K][V], bias[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
            bias[i] = c.bias ? c.bias[c0 + i] : 0.f;
#pragma unroll
            for (int j = 0; j < K; ++j) w[j][i] = c.w[(c0 + i) * K + j];
        }
        float hist[K > 1 ? K - 1 : 1][V];  // hist[j] = input of token t - 1 - j
        int64_t s = t0 / c.L, tt = t0 % c.L;
#pragma unroll
        for (int j = 0; j < K - 1; ++j) load_before<IO, V>(c, in, state, s, tt, c0, j, hist[j]);
        const int64_t t1 = t0 + kTokens < c.T ? t0 + kTokens : c.T;
#pragma unroll 4
        for (int64_t t = t0; t < t1; ++t) {
            if (t != t0 && tt == 0) {  // a new sequence starts: its window comes from its cache
#pragma unroll
                for (int j = 0; j < K - 1; ++j) load_before<IO, V>(c, in, state, s, 0, c0, j, hist[j]);
            }
            float v[V], acc[V];
            load_vec<IO>(in + t * c.D + c0, v);
#pragma unroll
            for (int i = 0; i < V; ++i) {
                acc[i] = fmaf(w[K - 1][i], v[i], bias[i]);
#pragma unroll
                for (int j = 0; j < K - 1; ++j) acc[i] = fmaf(w[K - 2 - j][i], hist[j][i], acc[i]);
            }
            uint4 o;
            IO *oe = reinterpret_cast<IO *>(&o);
#pragma unroll
            for (int i = 0; i < V; ++i) oe[i] = from_f32<IO>(c.silu ? __fdividef(acc[i], 1.f + __expf(-acc[i])) : acc[i]);
            *reinterpret_cast<uint4 *>(out + t * c.D + c0) = o;
#pragma unroll
            for (int j = K - 2; j > 0; --j)
#pragma unroll
                for (int i = 0; i < V; ++i) hist[j][i] = hist[j - 1][i];
            if (K > 1) {
#pragma unroll
                for (int i = 0; i < V; ++i) hist[0][i] = v[i];
            }
            if (++tt == c.L) {
                tt = 0;
                ++s;
            }
        }
    }
}

// The cache for continuing each sequence: its last k - 1 inputs per channel (from the cache given on entry where the
// sequence is shorter). Entries are written in ascending order and each is read before it can be overwritten, so the
// cache may be updated in place.
template <typename IO>
__global__ void __launch_bounds__(kThreads) conv_state_kernel(ConvParams c) {
    const IO *in = static_cast<const IO *>(c.in);
    const IO *state = static_cast<const IO *>(c.state);
    IO *sout = static_cast<IO *>(c.state_out);
    const int64_t total = c.nseq * c.D;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += (int64_t)gridDim.x * kThreads) {
        const int64_t s = e / c.D, ch = e % c.D;
        for (int j = 0; j < c.k - 1; ++j) {
            const int64_t tp = c.L - (c.k - 1) + j;
            IO v = from_f32<IO>(0.f);
            if (tp >= 0)
                v = in[(s * c.L + tp) * c.D + ch];
            else if (state)
                v = state[e * (c.k - 1) + (c.k - 1 + tp)];
            sout[e * (c.k - 1) + j] = v;
        }
    }
}

template <typename IO>
cudaError_t launch_t(const ConvParams &c, int sms, cudaStream_t stream) {
    constexpr int V = 16 / sizeof(IO);
    const int64_t total = (c.T + kTokens - 1) / kTokens * (c.D / V);
    if (total > 0) {
        const int64_t grid = std::min<int64_t>((total + kThreads - 1) / kThreads, (int64_t)sms * 16);
        switch (c.k) {
            case 1: conv_kernel<IO, 1><<<(unsigned)grid, kThreads, 0, stream>>>(c); break;
            case 2: conv_kernel<IO, 2><<<(unsigned)grid, kThreads, 0, stream>>>(c); break;
            case 3: conv_kernel<IO, 3><<<(unsigned)grid, kThreads, 0, stream>>>(c); break;
            case 4: conv_kernel<IO, 4><<<(unsigned)grid, kThreads, 0, stream>>>(c); break;
            case 5: conv_kernel<IO, 5><<<(unsigned)grid, kThreads, 0, stream>>>(c); break;
            case 6: conv_kernel<IO, 6><<<(unsigned)grid, kThreads, 0, stream>>>(c); break;
            case 7: conv_kernel<IO, 7><<<(unsigned)grid, kThreads, 0, stream>>>(c); break;
            case 8: conv_kernel<IO, 8><<<(unsigned)grid, kThreads, 0, stream>>>(c); break;
            default: return cudaErrorInvalidValue;
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (c.state_out && c.k > 1 && c.nseq * c.D > 0) {
        const int64_t grid = std::min<int64_t>((c.nseq * c.D + kThreads - 1) / kThreads, (int64_t)sms * 16);
        conv_state_kernel<IO><<<(unsigned)grid, kThreads, 0, stream>>>(c);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_conv(const ConvParams &c, int io_dtype, int sms, cudaStream_t stream) {
    if (io_dtype == 0) return launch_t<float>(c, sms, stream);
    if (io_dtype == 1) return launch_t<__nv_bfloat16>(c, sms, stream);
    return launch_t<__half>(c, sms, stream);
}

}  // namespace ssd

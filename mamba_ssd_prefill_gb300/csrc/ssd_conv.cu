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
// HBM-bound: tiles of 64 tokens x 512 bytes of channels, with the k - 1 rows before them, go through shared
// memory in a 3-stage pipeline, two CTAs per SM: one TMA box per tile from a 3-D map over [sequence, token,
// channel] (rows outside the sequence and channels past the last read as zeros), or, where the rows are not
// 16-byte multiples, 16-byte asynchronous copies with the same zero fill. A thread walks 32 tokens of one
// 4-byte column of the tile (two 16-bit channels or one fp32 one)
// with the taps and the last k - 1 inputs in registers, fp32 arithmetic (a 16-bit column's two channels in packed
// f32x2 fused multiply-adds), SiLU as h + h tanh(h) with h = v / 2 (one special-function op per channel), and
// stores rows coalesced. A second kernel writes the cache for continuing each sequence.
#include <cuda.h>

#include <stdlib.h>

#include <type_traits>

#include "sm100_ptx.cuh"
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kThreads = 256;
constexpr int kTileT = 64;      // tokens per tile
constexpr int kTileB = 512;     // bytes of channels per tile row
constexpr int kStages = 3;
constexpr int kCols = kTileB / 4;  // 4-byte columns per tile row (one per thread, two token halves)

__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Two fp32 fused multiply-adds in one packed instruction, each rounded like a scalar fmaf.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mov.b64 pc, {%6, %7};\n\tfma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float tanh_approx(float v) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

template <typename IO> struct Col;  // a 4-byte column: two 16-bit channels or one fp32 channel
template <> struct Col<float> {
    static constexpr int C = 1;
    __device__ static void load(const uint8_t *p, float (&v)[1]) { v[0] = *reinterpret_cast<const float *>(p); }
    __device__ static uint32_t pack(const float (&v)[1]) { return __float_as_uint(v[0]); }
};
template <> struct Col<__nv_bfloat16> {
    static constexpr int C = 2;
    __device__ static void load(const uint8_t *p, float (&v)[2]) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
        v[0] = f.x;
        v[1] = f.y;
    }
    __device__ static uint32_t pack(const float (&v)[2]) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[0], v[1]);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};
template <> struct Col<__half> {
    static constexpr int C = 2;
    __device__ static void load(const uint8_t *p, float (&v)[2]) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(p));
        v[0] = f.x;
        v[1] = f.y;
    }
    __device__ static uint32_t pack(const float (&v)[2]) {
        __half2 h = __floats2half2_rn(v[0], v[1]);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

// Item `it` (sequence, token tile, channel tile; channel tiles fastest) from its staged rows: this thread's 4-byte
// column of the output, tokens [tb, tb + 32) of the tile.
template <typename IO, int K>
__device__ __forceinline__ void conv_item(const ConvParams &c, const uint8_t *stage, int64_t it, int64_t ctiles,
                                          int64_t ttiles, int tid) {
    constexpr int NC = Col<IO>::C;
    const int64_t rowb = c.D * (int64_t)sizeof(IO);
    const IO *state = static_cast<const IO *>(c.state);
    uint8_t *out = static_cast<uint8_t *>(c.out);
    const int col = tid % kCols, half = tid / kCols;
    const int64_t cb = it % ctiles, rest = it / ctiles, tt = rest % ttiles, sq = rest / ttiles;
    const int64_t cbyte = cb * kTileB + col * 4;
    if (cbyte >= rowb) return;  // past the last channel
    const int64_t ch0 = cbyte / (int64_t)sizeof(IO);
    const uint8_t *tile = stage + col * 4;
    const int64_t tb = tt * kTileT + half * (kTileT / 2);  // first token of this thread's half
    const int64_t te = tb + kTileT / 2 < c.L ? tb + kTileT / 2 : c.L;
    if (tb >= te) return;
    float w[K][NC], bias[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        bias[i] = c.bias ? c.bias[ch0 + i] : 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j) w[j][i] = c.w[(ch0 + i) * K + j];
    }
    // hist[j] = input of token t - 1 - j: from the tile (rows before the sequence are zeros there), or the cache
    float hist[K > 1 ? K - 1 : 1][NC];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int64_t tp = tb - 1 - j;
        if (tp >= 0 || !state) {
            Col<IO>::load(tile + (int)(tp - (tt * kTileT - (K - 1))) * kTileB, hist[j]);
        } else {
#pragma unroll
            for (int i = 0; i < NC; ++i)
                hist[j][i] = to_f32(*chk(state, ((sq * c.D) + ch0 + i) * (K - 1) + (K - 1 + tp), 1,
                                         c.nseq * c.D * (K - 1), c.hdr, SITE_CONV_STATE));
        }
    }
    int64_t oidx = (sq * c.L + tb) * rowb + cbyte;  // byte index of this thread's output column
    const int64_t nout = c.nseq * c.L * rowb;
    (void)nout;
    const uint8_t *irow = tile + (int)(tb - (tt * kTileT - (K - 1))) * kTileB;
#pragma unroll 4
    for (int64_t t = tb; t < te; ++t) {
        float v[NC], acc[NC];
        Col<IO>::load(irow, v);
        if constexpr (NC == 2) {  // the column's two channels side by side
            float2 a2 = fma2(make_float2(w[K - 1][0], w[K - 1][1]), make_float2(v[0], v[1]),
                             make_float2(bias[0], bias[1]));
#pragma unroll
            for (int j = 0; j < K - 1; ++j)
                a2 = fma2(make_float2(w[K - 2 - j][0], w[K - 2 - j][1]), make_float2(hist[j][0], hist[j][1]), a2);
            acc[0] = a2.x;
            acc[NC - 1] = a2.y;
            if (c.silu) {  // v sigmoid(v) = h + h tanh(h), h = v / 2
                const float2 hv = make_float2(0.5f * a2.x, 0.5f * a2.y);
                const float2 r = fma2(hv, make_float2(tanh_approx(hv.x), tanh_approx(hv.y)), hv);
                acc[0] = r.x;
                acc[NC - 1] = r.y;
            }
        } else {
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                acc[i] = fmaf(w[K - 1][i], v[i], bias[i]);
#pragma unroll
                for (int j = 0; j < K - 1; ++j) acc[i] = fmaf(w[K - 2 - j][i], hist[j][i], acc[i]);
                if (c.silu) {  // v sigmoid(v) = h + h tanh(h), h = v / 2
                    const float hv = 0.5f * acc[i];
                    acc[i] = fmaf(hv, tanh_approx(hv), hv);
                }
            }
        }
        *reinterpret_cast<uint32_t *>(chk(out, oidx, 4, nout, c.hdr, SITE_CONV_OUT)) = Col<IO>::pack(acc);
#pragma unroll
        for (int j = K - 2; j > 0; --j)
#pragma unroll
            for (int i = 0; i < NC; ++i) hist[j][i] = hist[j - 1][i];
        if (K > 1) {
#pragma unroll
            for (int i = 0; i < NC; ++i) hist[0][i] = v[i];
        }
        irow += kTileB;
        oidx += rowb;
    }
    }

template <typename IO, int K>
__global__ void __launch_bounds__(kThreads, 2) conv_kernel(ConvParams c) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int R = kTileT + K - 1;  // rows per stage: the tile and the k - 1 before it
    constexpr int STAGE = R * kTileB;
    const int tid = threadIdx.x;
    const int64_t rowb = c.D * (int64_t)sizeof(IO);  // bytes of one token row
    const int64_t ctiles = (rowb + kTileB - 1) / kTileB, ttiles = (c.L + kTileT - 1) / kTileT;
    const int64_t items = c.nseq * ttiles * ctiles;
    const uint8_t *in = static_cast<const uint8_t *>(c.in);
    // item -> (sequence, token tile, channel tile), channel tiles fastest
    auto load = [&](int64_t it, int st) {
        const int64_t cb = it % ctiles, rest = it / ctiles, tt = rest % ttiles, sq = rest / ttiles;
        const int64_t t0 = tt * kTileT - (K - 1), cbyte = cb * kTileB;
        uint8_t *dst = smem + st * STAGE;
        for (int q = tid; q < R * (kTileB / 16); q += kThreads) {
            const int r = q / (kTileB / 16), off = (q % (kTileB / 16)) * 16;
            const int64_t t = t0 + r;
            const bool valid = t >= 0 && t < c.L && cbyte + off < rowb;
            cp_async16(dst + r * kTileB + off,
                       valid ? chk(in, (sq * c.L + t) * rowb + cbyte + off, 16, c.nseq * c.L * rowb, c.hdr, SITE_CONV_IN)
                             : in,
                       valid ? 16u : 0u);
        }
    };
    const int64_t first = blockIdx.x, step = gridDim.x;
    for (int k = 0; k < kStages - 1; ++k) {
        if (first + k * step < items) load(first + k * step, k);
        cp_async_commit();
    }
    for (int64_t n = 0;; ++n) {
        const int64_t it = first + n * step;
        if (it >= items) break;
        cp_async_wait<kStages - 2>();  // this thread's copies of item n have landed
        __syncthreads();               // everyone's; and stage (n - 1) % kStages has been read by everyone
        {
            const int64_t nx = first + (n + kStages - 1) * step;
            if (nx < items) load(nx, (int)((n + kStages - 1) % kStages));
            cp_async_commit();
        }
        conv_item<IO, K>(c, smem + (int)(n % kStages) * STAGE, it, ctiles, ttiles, tid);
    }
    cp_async_wait<0>();
}

// Bounded wait on a stage's mbarrier phase (the TMA that fills it); false after about 2 s.
__device__ __noinline__ bool stage_wait_slow(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0; i < kMaxSpinIters; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && globaltimer() - t0 > kDefaultTimeoutNs) return false;
    }
    return false;
}
__device__ __forceinline__ bool stage_wait(uint64_t *bar, uint32_t parity) {
    return mbar_try_wait(bar, parity) || stage_wait_slow(bar, parity);
}

// The same pipeline with one TMA box per stage ([1 sequence, R tokens, 512 bytes of channels] of a 3-D map over
// [nseq, L, D]; rows before or past the sequence and channels past D read as zeros), issued by one thread and
// counted on the stage's mbarrier, so no thread spends instructions on addresses. A stage is refilled only after
// the barrier that follows everyone's use of it. A wait that runs out records SSD_ERR_DEVICE and the CTA stops
// (after waiting, bounded, for its copies still in flight).
template <typename IO, int K>
__global__ void __launch_bounds__(kThreads, 2) conv_tma_kernel(ConvParams c, const __grid_constant__ CUtensorMap map) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kStages];
    constexpr int R = kTileT + K - 1;
    constexpr int STAGE = R * kTileB;
    const int tid = threadIdx.x;
    const int64_t rowb = c.D * (int64_t)sizeof(IO);
    const int64_t ctiles = (rowb + kTileB - 1) / kTileB, ttiles = (c.L + kTileT - 1) / kTileT;
    const int64_t items = c.nseq * ttiles * ctiles;
    if (tid == 0) {
        prefetch_tensormap(&map);
        for (int st = 0; st < kStages; ++st) mbar_init(&full[st], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int64_t it, int st) {  // thread 0
        const int64_t cb = it % ctiles, rest = it / ctiles, tt = rest % ttiles, sq = rest / ttiles;
        mbar_arrive_expect_tx(&full[st], (uint32_t)STAGE);
        tma_load_3d(smem + st * STAGE, &map, &full[st], (int)(cb * (kTileB / (int)sizeof(IO))),
                    (int)(tt * kTileT - (K - 1)), (int)sq);
    };
    const int64_t first = blockIdx.x, step = gridDim.x;
    int64_t issued = 0;  // items issued so far (thread 0)
    if (tid == 0)
        for (int k = 0; k < kStages - 1 && first + k * step < items; ++k, ++issued) issue(first + k * step, k);
    int64_t n = 0;
    for (;; ++n) {
        const int64_t it = first + n * step;
        if (it >= items) break;
        const int st = (int)(n % kStages);
        const bool ok = stage_wait(&full[st], (uint32_t)((n / kStages) & 1));
        if (__syncthreads_or(!ok)) {  // also: everyone is done with stage (n - 1) % kStages
            if (!ok && c.hdr && atomicCAS(&c.hdr->status, 0u, (uint32_t)DEV_PIPE) == 0u) c.hdr->err_where = WAIT_PIPE;
            break;
        }
        if (tid == 0) {
            const int64_t nx = first + (n + kStages - 1) * step;
            if (nx < items) {
                issue(nx, (int)((n + kStages - 1) % kStages));
                ++issued;
            }
        }
        conv_item<IO, K>(c, smem + st * STAGE, it, ctiles, ttiles, tid);
    }
    if (tid == 0)  // only after a stop: the copies issued but not waited for land before the CTA exits
        for (int64_t m = n; m < issued; ++m) stage_wait(&full[(int)(m % kStages)], (uint32_t)((m / kStages) & 1));
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
                v = *chk(in, (s * c.L + tp) * c.D + ch, 1, c.nseq * c.L * c.D, c.hdr, SITE_CONV_IN);
            else if (state)
                v = *chk(state, e * (c.k - 1) + (c.k - 1 + tp), 1, total * (c.k - 1), c.hdr, SITE_CONV_STATE);
            *chk(sout, e * (c.k - 1) + j, 1, total * (c.k - 1), c.hdr, SITE_CONV_STATE) = v;
        }
    }
}

// 3-D map over the raw rows [nseq, L, D], box [1, R, 512 bytes of channels], no swizzle, zeros outside. Needs a
// 16-byte aligned base and rows a multiple of 16 bytes (else the cp.async kernel runs).
template <typename IO>
bool conv_map(CUtensorMap *m, const ConvParams &c, int R) {
    const int64_t es = (int64_t)sizeof(IO), rowb = c.D * es;
    if ((reinterpret_cast<uintptr_t>(c.in) & 15) || (rowb & 15) || c.L > INT32_MAX || c.nseq > INT32_MAX) return false;
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)c.D, (cuuint64_t)c.L, (cuuint64_t)c.nseq};
    const cuuint64_t strides[2] = {(cuuint64_t)rowb, (cuuint64_t)(rowb * c.L)};
    const cuuint32_t box[3] = {(cuuint32_t)(kTileB / es), (cuuint32_t)R, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : std::is_same<IO, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return enc(m, dt, 3, const_cast<void *>(c.in), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename IO, int K>
cudaError_t launch_k(const ConvParams &c, int sms, cudaStream_t stream) {
    const size_t smem = (size_t)kStages * (kTileT + K - 1) * kTileB;
    const int64_t rowb = c.D * (int64_t)sizeof(IO);
    const int64_t items = c.nseq * ((c.L + kTileT - 1) / kTileT) * ((rowb + kTileB - 1) / kTileB);
    const int64_t grid = std::min<int64_t>(items, (int64_t)sms * 2);
    CUtensorMap map;
    // conv_tma test hook (ssd_debug_knobs) 0: the cp.async kernel on any rows (it serves rows that are not 16-byte
    // multiples)
    const bool tma_allowed = knobs().conv_tma != 0;
    if (tma_allowed && conv_map<IO>(&map, c, kTileT + K - 1)) {
        auto k = conv_tma_kernel<IO, K>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k<<<(unsigned)grid, kThreads, smem, stream>>>(c, map);
        return cudaGetLastError();
    }
    auto k = conv_kernel<IO, K>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<(unsigned)grid, kThreads, smem, stream>>>(c);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_t(const ConvParams &c, int sms, cudaStream_t stream) {
    if (c.T > 0) {
        cudaError_t e;
        switch (c.k) {
            case 1: e = launch_k<IO, 1>(c, sms, stream); break;
            case 2: e = launch_k<IO, 2>(c, sms, stream); break;
            case 3: e = launch_k<IO, 3>(c, sms, stream); break;
            case 4: e = launch_k<IO, 4>(c, sms, stream); break;
            case 5: e = launch_k<IO, 5>(c, sms, stream); break;
            case 6: e = launch_k<IO, 6>(c, sms, stream); break;
            case 7: e = launch_k<IO, 7>(c, sms, stream); break;
            case 8: e = launch_k<IO, 8>(c, sms, stream); break;
            default: return cudaErrorInvalidValue;
        }
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

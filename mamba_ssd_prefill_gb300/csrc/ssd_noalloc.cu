// ssd_fwd_static_scratch: the SSD prefill forward for callers that cannot
// allocate device memory.
//
// ssd_fwd() needs a caller-provided workspace (a header, the per-chunk
// state-passing flags and the state ring). Some callers have no way to provide
// one: a host application or plugin framework that owns every byte of device
// memory and hands a kernel only its input and output buffers, or a
// latency-critical loop where a cudaMalloc (which can synchronise the whole
// device) is not acceptable. This entry point serves them from a fixed scratch
// array that lives in the library itself.
//
// The scratch is a file-scope __device__ array of kStaticScratchBytes. Every
// GPU that loads this library holds that much memory until the process exits.
// Its device address is looked up once per device (cudaGetSymbolAddress) by
// the first call made with that device current; that first call should come
// before any stream capture. All calls share the one array: calls that overlap
// on the GPU (different streams, or different host threads, without ordering
// between them) race on it and must not be issued. Each call zero-fills the
// part of the array it uses (the part the kernel expects to start at zero) on
// its stream before the launch, so the contents left by the previous call do
// not matter. No call allocates or frees device memory. Where two-level state
// passing (long sequences) would need more than the array, the call runs with
// one state chain per sequence instead.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/ssd.h"
#include "ssd_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// device address of g_static_scratch, per device (null until looked up; host threads that race on a first call
// look it up alike and store the same value)
std::atomic<void *> g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" SSD_API ssd_status_t ssd_fwd_static_scratch(const ssd_problem_t *prob, const void *x, const void *dt_raw,
                                                       const float *dt_bias, const float *A, const void *B,
                                                       const void *C, const float *D, const void *init_states,
                                                       void *y, void *final_states, void *stream) {
    size_t need = 0;
    ssd_status_t st = ssd_fwd_workspace_size(prob, &need);
    if (st != SSD_OK) return st;
    if (need > kStaticScratchBytes) {  // without two-level state passing, if that fits
        st = ssd::workspace_bytes(prob, false, &need);
        if (st != SSD_OK) return st;
        if (need > kStaticScratchBytes) return SSD_ERR_WORKSPACE;  // problem too large for the static scratch
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    void *ws = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!ws) {
        if (cudaGetSymbolAddress(&ws, g_static_scratch) != cudaSuccess || !ws) return SSD_ERR_CUDA;
        g_scratch_addr[dev].store(ws, std::memory_order_release);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (prob->batch > 0 && prob->seqlen > 0 && cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return SSD_ERR_CUDA;
    // the workspace size passed is `need`: ssd_fwd then plans exactly what was sized (and zero-filled) here
    return ssd_fwd(prob, x, dt_raw, dt_bias, A, B, C, D, init_states, y, final_states, ws, need, stream);
}

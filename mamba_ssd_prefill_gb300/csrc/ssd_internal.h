// Host-side interfaces between the C ABI (ssd_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/ssd.h"
#include "ssd_common.cuh"

namespace ssd {

// Workspace bytes of a regular batch with or without two-level state passing (ssd_api.cu).
ssd_status_t workspace_bytes(const ssd_problem_t *prob, bool segments, size_t *bytes);

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry points (ssd_api.cu); null when the
// driver has none
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Launch-configuration overrides set by ssd_debug_knobs (test hooks; -1 = the library's own choice).
struct Knobs {
    int tc_heads_per_unit, tc_late_ticket, simt_two_pass, conv_tma;
    int tc_segment_chunks;  // -1: the library's choice, 0: one state chain per sequence, >= 1: chunks per segment
    int tc_head_flags;      // -1: the library's choice, 0: a release flag per state row, 1: one per head
};
Knobs knobs();

// fp32 SIMT kernel (ssd_simt.cu)
size_t simt_smem_bytes(int64_t P, int64_t N);
cudaError_t launch_simt(const Params &p, int io_dtype, int state_dtype, int sms, cudaStream_t stream);

// variable-length batches (ssd_varlen.cu): chunk table from cu_seqlens, final = initial for empty sequences
cudaError_t launch_varlen_plan(const Params &p, uint32_t *scratch, size_t state_bytes, cudaStream_t stream);

// causal depthwise convolution in front of the SSD (ssd_conv.cu)
cudaError_t launch_conv(const ConvParams &c, int io_dtype, int sms, cudaStream_t stream);

// single-token step (ssd_step.cu)
cudaError_t launch_step(const Params &p, int io_dtype, int state_dtype, int sms, cudaStream_t stream);

// tcgen05 / TMA kernel (ssd_tc.cu)
bool tc_supports(int64_t P, int64_t N, int64_t Q, int io_dtype);
int64_t tc_chunk();  // tokens per state-passing step inside the tensor-core kernel
size_t tc_flag_bytes(int64_t chains);
size_t tc_ring_bytes(int64_t chains, int64_t P, int64_t N, int state_dtype);
uint32_t tc_total_units(int64_t batch, int64_t H, int64_t G, int64_t nc, int heads_per_unit);
int tc_heads_per_unit(int64_t batch, int64_t H, int64_t G, int64_t nc, int sms);
bool tc_late_ticket(int64_t units_per_chunk, int sms);  // ticket order = finishing order (chain-bound problems)
bool tc_head_flags(int64_t chains_per_position, bool late_ticket, int sms);  // fp32 states: one release per head
cudaError_t launch_tc(Params p, int io_dtype, int state_dtype, int heads_per_unit, int sms, cudaStream_t stream);

// two-level state passing (ssd_segstate.cu): segment entering states from block aggregates, before launch_tc
struct SegChoice {
    int64_t nseg, seg_chunks;  // segments per sequence (1: off) and chunks per segment
    int64_t blk, nblk;         // chunks per aggregate block, blocks per sequence with an aggregate
    int hs;                    // heads per block-kernel work unit
};
SegChoice choose_segments(int64_t nseq, int64_t nc, int64_t H, int64_t G, int sms, int64_t forced, bool fp32_states);
struct SegPlan {
    int64_t blk, nblk;
    int hs;
    float *blk_s;  // [nseq][nblk][H][P][N] block aggregates
    float *blk_L;  // [nseq][nblk][H] log2 of the block decays
};
cudaError_t launch_segstate(const Params &p, const SegPlan &sp, int io_dtype, int state_dtype, int sms,
                            cudaStream_t stream);

}  // namespace ssd

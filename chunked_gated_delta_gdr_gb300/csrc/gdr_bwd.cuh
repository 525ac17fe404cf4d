// gdr_bwd.cuh -- the backward of the chunked gated delta rule (gdr_bwd.cu; not installed).
#pragma once

#include "gdr_internal.cuh"

namespace gdr {

// Operands of the backward.  Inputs as the forward's (bf16 q, k, v, beta and dout; fp32
// g); outputs fp32.  dq_h / dk_h are the per-value-head accumulators: the outputs dq / dk
// themselves when every query/key head has one value head, else [T, H, D] scratch that
// the last kernel sums into dq / dk.
struct BwdArgs {
  StageShapes s;
  View q, k, v, g, beta, dout;
  const float *h0, *dht;
  float scale;
  View dq, dk, dv, dg, dbeta;  // outputs (fp32)
  float *dh0;                  // [n_seq, H, D, D] or null
  const SegInfo *seg;
  const int32_t *order;        // segments longest first (launch_seg_order)
  const ChunkInfo *chunks;
  const int32_t *n_chunks;
  void *work;                  // gdr_bwd_work_bytes bytes, 256-byte aligned
};

size_t bwd_work_bytes(int64_t T, int32_t n_seq, int32_t Hk, int32_t H, int32_t D);
cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t stream);

// Tensor-core (tcgen05 / TMA) kernels of the backward (gdr_bwd_tc.cu).  Each returns
// cudaErrorNotSupported, launching nothing, when its operands cannot be loaded by TMA
// (base or strides not 16-byte aligned, head dim other than 64 or 128); the caller then
// runs the warp-tile kernel of the same step.
cudaError_t launch_bwd_dv_intra_tc(const BwdArgs &a, View gcum, View dvp, cudaStream_t stream);
// The S_0 / dS_C products (dq, dk, dW parts and <dS_C, S_0> per 64 key rows) from the bf16
// states h [chunks, H, D, D] and their fp32 gradients dh (same layout); dvp, dh also need
// 16-byte aligned rows (float4 loads).
cudaError_t launch_bwd_sgrad_tc(const BwdArgs &a, const void *h, const float *dh, View gcum,
                               View vnew, View dvp, View dqh, View dkh, View dw, float *sdot,
                               cudaStream_t stream);
cudaError_t read_bwd_tc_status(int32_t *out);

}  // namespace gdr

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

}  // namespace gdr

// gdr_sched.cuh -- dispatch order of the per-segment scans (not installed).
#pragma once

#include "gdr_internal.cuh"

namespace gdr {

// order[0 .. n_seq) = the segments by chunk count, longest first (counting sort on the
// device, one block).  A scan dispatched in this order starts its longest chains first,
// so no long segment is left for the last wave; the order changes no result.
cudaError_t launch_seg_order(const SegInfo *seg, int32_t n_seq, int32_t *order,
                             cudaStream_t stream);

// launch_scan with its blocks dispatched in `order` (null: segment order).
cudaError_t launch_scan_ordered(const StageShapes &s, View k, View w, View u, View gcum,
                                const float *h0, void *h, View v_new, float *ht, Ckpt ck,
                                const SegInfo *seg, const int32_t *order, cudaStream_t stream);

}  // namespace gdr

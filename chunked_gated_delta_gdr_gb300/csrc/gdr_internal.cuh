// gdr_internal.cuh -- shared definitions of the libgdr CUDA sources (not installed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr.h"

namespace gdr {

constexpr int kChunk = 64;  // tokens per chunk

// Per-segment entry of the chunk enumeration: sanitised bounds [start, end),
// id of the segment's first chunk, number of chunks.
struct SegInfo {
  int32_t start, end, chunk_off, n_chunks;
};

// Per-chunk entry: owning segment, first token, token count (1..64).
struct ChunkInfo {
  int32_t seq, start, len, pad;
};

// A [rows, heads, dim] tensor with a contiguous innermost dim, or a [rows, heads]
// tensor (dim stride unused).  Strides are in elements.
struct View {
  void *p;
  int64_t st;  // token (row) stride
  int64_t sh;  // head stride
};

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int64_t chunk_bound(int64_t T, int32_t n_seq) { return ceil_div64(T, kChunk) + n_seq; }

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__device__ __forceinline__ float ldbf(const void *p, int64_t i) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
}

__device__ __forceinline__ void stbf(void *p, int64_t i, float x) {
  reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float ldf(const void *p, int64_t i) {
  return reinterpret_cast<const float *>(p)[i];
}

// ---- host-side launchers implemented in the .cu files ----

// Chunk enumeration (gdr_index.cu).
cudaError_t launch_chunk_index(const int32_t *cu, int32_t n_seq, int64_t T, SegInfo *seg,
                               ChunkInfo *chunks, int64_t chunk_cap, int32_t *n_chunks,
                               cudaStream_t stream);
cudaError_t launch_check_cu(const int32_t *cu, int32_t n_seq, int64_t T, int32_t *out2,
                            cudaStream_t stream);

// Stage kernels (gdr_staged.cu).  All views are validated by the caller.
struct StageShapes {
  int64_t T;
  int32_t n_seq, Hk, H, D;
  int64_t chunk_cap;
};

cudaError_t launch_prep(const StageShapes &s, View k, View v, View g, View beta, View w,
                        View u, View gcum, const SegInfo *seg, const ChunkInfo *chunks,
                        const int32_t *n_chunks, cudaStream_t stream);
// State checkpoints: state after every `every` tokens of each segment (every a positive
// multiple of 64; 0 = none), rows off[n] .. off[n+1]-1 of h [rows, H, D, D] for segment n.
struct Ckpt {
  float *h;
  const int32_t *off;
  int32_t every;
};
cudaError_t launch_scan(const StageShapes &s, View k, View w, View u, View gcum,
                        const float *h0, void *h, View v_new, float *ht, Ckpt ck,
                        const SegInfo *seg, cudaStream_t stream);
// off[n] = sum over segments before n of floor(len / every); off[n_seq] = total
cudaError_t launch_ckpt_offsets(const SegInfo *seg, int32_t n_seq, int32_t every, int32_t *off,
                                cudaStream_t stream);
cudaError_t launch_out(const StageShapes &s, View q, View k, View v_new, const void *h,
                       View gcum, float scale, View o, const SegInfo *seg,
                       const ChunkInfo *chunks, const int32_t *n_chunks, cudaStream_t stream);

// Intra-sequence split (gdr_split.cu): a long segment is cut into pieces of whole
// chunks.  Pass A runs piece 0 from the segment's initial state (outputs and the state
// after it) and every later piece twice: from a zero state (R, the piece's offset) and
// from the identity with v = 0 (M, the piece's transition).  The combine step chains
// S_{p+1} = M_p S_p + R_p; pass B runs pieces 1.. from their initial states S_p.
enum UnitMode : int32_t { kUnitFull = 0, kUnitR = 1, kUnitM = 2, kUnitFinal = 3 };
// state slots (`sin`, `sout`) index [D][D] fp32 blocks of SplitArgs::states;
// sout -1: ht (if requested), -2: no state output; sin -1: h0 or zero (by mode)
struct UnitDesc {
  int32_t seq, head, t0, end, nch, mode, sin, sout;
};
struct SplitArgs {
  const UnitDesc *units;    // null: no split (units are whole segments)
  const int32_t *n_units;   // device count
  float *states;            // [slots][D][D]
  int32_t *counter;         // unit counter, zeroed by the unit builder
  bool empty_states;        // also write ht of empty segments (pass A only)
};
constexpr int kSplitMaxPieces = 8;
constexpr int kSplitMinChunks = 16;  // shortest piece worth splitting off
// pieces per segment for U (segment, head) units on `sms` SMs (1 = do not split), and
// the weight of the first piece against the others (`lead`)
int split_pieces(int64_t units, int sms, int *lead);
struct SplitWs {
  UnitDesc *ua, *ub;
  int32_t *na, *nb, *counters, *seg_pieces;
  float *states;
  size_t bytes;
};
SplitWs carve_split(void *ws, int32_t n_seq, int32_t H, int32_t D, int32_t pieces);
cudaError_t launch_split_units(const SegInfo *seg, int32_t n_seq, int32_t H, int32_t pieces,
                               int32_t lead, const SplitWs &w, cudaStream_t stream);
cudaError_t launch_split_combine(const SplitWs &w, int32_t n_seq, int32_t H, int32_t D,
                                 cudaStream_t stream);

// Fused persistent kernel (gdr_fused.cu).
struct FusedArgs {
  int64_t T;
  int32_t n_seq, Hk, H, D;
  const void *q, *k, *v;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const float *g;
  int64_t g_st, g_sh;
  const void *beta;
  int64_t b_st, b_sh;
  float scale;
  const float *h0;
  void *o;
  int64_t o_st, o_sh;
  float *ht;
  Ckpt ckpt;
  SplitArgs split;
  // The forward recomputed for the backward instead (bwd.h non-null; no o, no ht): the
  // chunk-local cumulative gate G [T][H] fp32, W = Tm diag(beta e^G) K and V' [T][H][D]
  // bf16, the state entering each chunk [chunk][H][D][D] bf16 (chunk ids of `seg`), and
  // Tm = (I + A)^-1 [chunk][H][64][64] fp32 (tmat may be null)
  struct {
    float *gcum;
    void *w, *h, *vnew;
    float *tmat;
  } bwd;
  const SegInfo *seg;
  void *workspace;  // fused-path scratch (work list etc.)
};
bool fused_supported(const FusedArgs &a);
// TMA map of a [T, heads, D] bf16 tensor (element strides st, sh; innermost contiguous):
// boxes of 64 tokens x 1 head x 64 elements, 128-byte swizzle (gdr_fused.cu).  False if the
// driver's encoder rejects it (alignment of base or strides).
bool make_tile_map(CUtensorMap *m, const void *ptr, int64_t D, int64_t heads, int64_t T,
                   int64_t st, int64_t sh);
size_t fused_workspace_bytes(int64_t T, int32_t n_seq, int32_t H);
cudaError_t launch_fused(const FusedArgs &a, cudaStream_t stream);

// Device status word (gdr_fused.cu).
cudaError_t read_device_status(int32_t *out);
cudaError_t launch_wait_selftest(uint32_t limit_us, int32_t code, cudaStream_t stream);
cudaError_t clear_device_status();

}  // namespace gdr

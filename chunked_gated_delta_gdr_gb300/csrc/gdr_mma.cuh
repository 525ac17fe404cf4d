// gdr_mma.cuh -- for the staged and backward kernels: warp-level tensor-core tiles over
// fp32 or bf16 shared-memory operands (tf32 in, fp32 accumulate, mma.sync m16n8k8), and
// tile loads from global memory into shared memory.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gdr_internal.cuh"

namespace gdr {

// Streaming multiprocessors of the current device (cached; 0 if it cannot be queried).
inline int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
  return cache[dev];
}

// Value columns per block of a sequential scan over (segment, head) pairs: 64 (eight
// warps) when that still gives every SM a block, else 32 (four warps, twice the blocks).
inline int scan_cols(int64_t n_seq, int64_t H, int D) {
  return n_seq * H * (D / 64) >= device_sm_count() ? 64 : 32;
}

// Row t, head `head` of a bf16 [rows, heads, dim] view.
__device__ __forceinline__ const __nv_bfloat16 *bf_row(const View &x, int64_t t, int64_t head) {
  return reinterpret_cast<const __nv_bfloat16 *>(x.p) + t * x.st + head * x.sh;
}

// A tf32 operand: the fp32 bits as they are.  The tensor pipe reads the upper 19 bits
// of a tf32 operand, so this truncates the mantissa to 10 bits (relative error below
// 2^-10) and saves a conversion per operand element.
__device__ __forceinline__ uint32_t tf32_rn(float x) { return __float_as_uint(x); }

// A strided view of an fp32 matrix in shared memory: element (r, c) is p[r * rs + c * cs],
// so a transposed operand is the same array with rs and cs swapped.
struct SMat {
  const float *p;
  int rs, cs;
};
// The same for a bf16 matrix (an operand whose values came from a bf16 tensor: it takes
// half the shared memory, and every bf16 value is exactly a tf32 value).
struct SMatH {
  const __nv_bfloat16 *p;
  int rs, cs;
};
// Element i of a view as a tf32 operand.
__device__ __forceinline__ uint32_t tf32_at(const SMat &m, int i) { return tf32_rn(m.p[i]); }
__device__ __forceinline__ uint32_t tf32_at(const SMatH &m, int i) {
  return (uint32_t)reinterpret_cast<const uint16_t *>(m.p)[i] << 16;
}

// One warp: acc[16 x 8] += A[m0 .. m0+16, k0 .. k1) * B[k0 .. k1, n0 .. n0+8), with
// k1 - k0 a multiple of 8.  Accumulator element e (0..3) of lane l holds
// (m0 + l/4 + 8 (e/2), n0 + 2 (l%4) + e%2).
template <class VA, class VB>
__device__ __forceinline__ void mma_16x8(float (&acc)[4], VA A, int m0, VB B, int n0, int k0,
                                         int k1) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int ab = (m0 + g) * A.rs;
  const int bb = (n0 + g) * B.cs;
#pragma unroll 2
  for (int k = k0; k < k1; k += 8) {
    const int ap = ab + (k + t) * A.cs;
    const int bp = bb + (k + t) * B.rs;
    const uint32_t a0 = tf32_at(A, ap), a1 = tf32_at(A, ap + 8 * A.rs);
    const uint32_t a2 = tf32_at(A, ap + 4 * A.cs), a3 = tf32_at(A, ap + 8 * A.rs + 4 * A.cs);
    const uint32_t b0 = tf32_at(B, bp), b1 = tf32_at(B, bp + 4 * B.rs);
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// One warp: NB adjacent tiles, acc[b][16 x 8] += A[m0.., k] B[k, n0 + 8 b ..]; the A
// fragment is loaded once per k step and the NB products are independent, so their
// latencies overlap.
template <int NB, class VA, class VB>
__device__ __forceinline__ void mma_16xN(float (&acc)[NB][4], VA A, int m0, VB B, int n0,
                                         int k0, int k1) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int ab = (m0 + g) * A.rs;
#pragma unroll 2
  for (int k = k0; k < k1; k += 8) {
    const int ap = ab + (k + t) * A.cs;
    const uint32_t a0 = tf32_at(A, ap), a1 = tf32_at(A, ap + 8 * A.rs);
    const uint32_t a2 = tf32_at(A, ap + 4 * A.cs), a3 = tf32_at(A, ap + 8 * A.rs + 4 * A.cs);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int bp = (n0 + 8 * b + g) * B.cs + (k + t) * B.rs;
      const uint32_t b0 = tf32_at(B, bp), b1 = tf32_at(B, bp + 4 * B.rs);
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(acc[b][0]), "+f"(acc[b][1]), "+f"(acc[b][2]), "+f"(acc[b][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
}

// One warp: MB row tiles (m0 + 16 r) sharing one column tile (n0); the B fragment is
// loaded once per k step and the MB products are independent.
template <int MB, class VA, class VB>
__device__ __forceinline__ void mma_Mx8(float (&acc)[MB][4], VA A, int m0, VB B, int n0,
                                        int k0, int k1) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int bb = (n0 + g) * B.cs;
#pragma unroll 2
  for (int k = k0; k < k1; k += 8) {
    const int bp = bb + (k + t) * B.rs;
    const uint32_t b0 = tf32_at(B, bp), b1 = tf32_at(B, bp + 4 * B.rs);
#pragma unroll
    for (int r = 0; r < MB; ++r) {
      const int ap = (m0 + 16 * r + g) * A.rs + (k + t) * A.cs;
      const uint32_t a0 = tf32_at(A, ap), a1 = tf32_at(A, ap + 8 * A.rs);
      const uint32_t a2 = tf32_at(A, ap + 4 * A.cs), a3 = tf32_at(A, ap + 8 * A.rs + 4 * A.cs);
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(acc[r][0]), "+f"(acc[r][1]), "+f"(acc[r][2]), "+f"(acc[r][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
}

// Row and column of accumulator element e of this lane for the tile at (m0, n0).
__device__ __forceinline__ int acc_row(int m0, int e) { return m0 + ((threadIdx.x & 31) >> 2) + 8 * (e >> 1); }
__device__ __forceinline__ int acc_col(int n0, int e) { return n0 + 2 * (threadIdx.x & 3) + (e & 1); }

// Threads of the per-chunk kernels (one block per chunk and head): 16 warps; a 64 x 64
// tile matrix is 32 MMA tiles of 16 x 8, kTPW per warp; in phases where warps own
// row tiles, warp w takes row tile w % 4 and column group w / 4 (of kQ).
constexpr int kChunkThreads = 512, kWarps = kChunkThreads / 32, kTPW = 32 / kWarps,
              kQ = kWarps / 4;

// Row strides of fp32 shared-memory operands.  A warp's fragment read touches rows
// l/4 and columns l%4 (lane l): a stride of 4 mod 32 puts the 32 reads of a row-major
// operand in 32 different banks, a stride of 8 mod 32 those of a transposed one.
__host__ __device__ constexpr int ld_rows(int cols) { return cols + 4; }   // read as rows
__host__ __device__ constexpr int ld_cols(int cols) { return cols + 8; }   // read transposed
// bf16 operands: a word holds two neighbours, so with a stride of 8 mod 64 elements both
// reads map a warp's 32 lanes onto 16 different words (lanes sharing a word get it at once).
__host__ __device__ constexpr int ld_bf16(int cols) { return cols + 8; }
constexpr int kLdY = 24;  // 16 x 16 scratch tiles of the solve (read as the B operand)
constexpr int kSolveScratch = 8 * 16 * kLdY;

// Synchronise the first `nthreads` threads of the block on named barrier `id` (id 0 with
// the whole block is __syncthreads).
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// T = (I + A)^-1 for a strictly lower-triangular 64 x 64 A (row stride lda), written to T
// (row stride ldt), by threads 0 .. nthreads-1 of the block (at least 4 warps, whole
// warps) synchronised on named barrier `bar`: the four 16 x 16 diagonal blocks by
// forward substitution, then the blocks below the diagonal by distance d = 1, 2, 3 as
// T_ij = -T_ii (sum_{k=j}^{i-1} A_ik T_kj), one warp per block pair (tensor tiles).
// `scratch` holds kSolveScratch floats.  Ends with that barrier.
__device__ __forceinline__ void solve_unit_lower64(const float *A, int lda, float *T, int ldt,
                                                   float *scratch, int nthreads, int bar) {
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int idx = tid; idx < 64 * 64; idx += nthreads) {  // blocks above the diagonal are zero
    const int i = idx >> 6, j = idx & 63;
    if ((i >> 4) < (j >> 4)) T[i * ldt + j] = 0.f;
  }
  if (tid < 64) {  // column c of the diagonal block b
    const int b = tid >> 4, c = tid & 15, o = b * 16;
    for (int i = 0; i < 16; ++i) {
      float x = (i == c) ? 1.f : 0.f;
      for (int j = c; j < i; ++j) x -= A[(o + i) * lda + o + j] * T[(o + j) * ldt + o + c];
      T[(o + i) * ldt + o + c] = x;
    }
  }
  bar_sync(bar, nthreads);
  for (int dist = 1; dist < 4; ++dist) {
    if (warp < 4 - dist) {
      const int j = warp, i = warp + dist;
      float *Y = scratch + warp * 16 * kLdY;
      float y0[4] = {0.f, 0.f, 0.f, 0.f}, y1[4] = {0.f, 0.f, 0.f, 0.f};
      // Y = A[i rows, j .. i-1 blocks] T[j .. i-1 blocks, j columns]
      mma_16x8(y0, SMat{A + i * 16 * lda, lda, 1}, 0, SMat{T, ldt, 1}, j * 16, j * 16, i * 16);
      mma_16x8(y1, SMat{A + i * 16 * lda, lda, 1}, 0, SMat{T, ldt, 1}, j * 16 + 8, j * 16,
               i * 16);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        Y[acc_row(0, e) * kLdY + acc_col(0, e)] = y0[e];
        Y[acc_row(0, e) * kLdY + acc_col(8, e)] = y1[e];
      }
      __syncwarp();
      float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
      const float *Tii = T + i * 16 * ldt + i * 16;
      mma_16x8(t0, SMat{Tii, ldt, 1}, 0, SMat{Y, kLdY, 1}, 0, 0, 16);
      mma_16x8(t1, SMat{Tii, ldt, 1}, 0, SMat{Y, kLdY, 1}, 8, 0, 16);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        T[(i * 16 + acc_row(0, e)) * ldt + j * 16 + acc_col(0, e)] = -t0[e];
        T[(i * 16 + acc_row(0, e)) * ldt + j * 16 + acc_col(8, e)] = -t1[e];
      }
      __syncwarp();
    }
    bar_sync(bar, nthreads);
  }
}

// Rows [0, R) x columns [0, C) of a row-major matrix in global memory (row r at
// src + r * rs elements) into fp32 shared memory dst[r * ld + c] (dst 16-byte aligned,
// ld a multiple of 4); rows >= len read as 0.
// With `vec` (src 16-byte aligned, rs a multiple of 16 bytes) every thread issues its
// 16-byte loads, at most eight at a time, before it stores any of them, so a tile costs
// about one memory round trip instead of one per element.  NT threads take part.
template <int R, int C, int NT>
__device__ __forceinline__ void tile_bf16(float *dst, int ld, const __nv_bfloat16 *src, int64_t rs,
                                          int len, bool vec) {
  constexpr int VPR = C / 8, NV = R * VPR;  // 16-byte vectors per row, per tile
  static_assert(C % 8 == 0 && NV % NT == 0, "tile shape");
  constexpr int PER = NV / NT, BATCH = PER < 8 ? PER : 8;
  static_assert(PER % BATCH == 0, "whole batches");
  if (vec) {
#pragma unroll
    for (int b0 = 0; b0 < PER; b0 += BATCH) {
      uint4 x[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int v = threadIdx.x + (b0 + u) * NT, r = v / VPR, c = (v % VPR) * 8;
        x[u] = r < len ? *reinterpret_cast<const uint4 *>(src + r * rs + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int v = threadIdx.x + (b0 + u) * NT, r = v / VPR, c = (v % VPR) * 8;
        const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&x[u]);
        float f[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 y = __bfloat1622float2(p2[q]);
          f[2 * q] = y.x;
          f[2 * q + 1] = y.y;
        }
        float4 *d = reinterpret_cast<float4 *>(dst + r * ld + c);  // ld % 4 == 0
        d[0] = make_float4(f[0], f[1], f[2], f[3]);
        d[1] = make_float4(f[4], f[5], f[6], f[7]);
      }
    }
  } else {
    for (int idx = threadIdx.x; idx < R * C; idx += NT) {
      const int r = idx / C, c = idx % C;
      dst[r * ld + c] = r < len ? __bfloat162float(src[r * rs + c]) : 0.f;
    }
  }
}

// As tile_bf16, into bf16 shared memory as it is (dst 16-byte aligned, ld a multiple of 8).
template <int R, int C, int NT>
__device__ __forceinline__ void tile_bf16_raw(__nv_bfloat16 *dst, int ld, const __nv_bfloat16 *src,
                                              int64_t rs, int len, bool vec) {
  constexpr int VPR = C / 8, NV = R * VPR;
  static_assert(C % 8 == 0 && NV % NT == 0, "tile shape");
  constexpr int PER = NV / NT, BATCH = PER < 8 ? PER : 8;
  static_assert(PER % BATCH == 0, "whole batches");
  if (vec) {
#pragma unroll
    for (int b0 = 0; b0 < PER; b0 += BATCH) {
      uint4 x[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int v = threadIdx.x + (b0 + u) * NT, r = v / VPR, c = (v % VPR) * 8;
        x[u] = r < len ? *reinterpret_cast<const uint4 *>(src + r * rs + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int v = threadIdx.x + (b0 + u) * NT, r = v / VPR, c = (v % VPR) * 8;
        *reinterpret_cast<uint4 *>(dst + r * ld + c) = x[u];
      }
    }
  } else {
    const __nv_bfloat16 zero = __float2bfloat16(0.f);
    for (int idx = threadIdx.x; idx < R * C; idx += NT) {
      const int r = idx / C, c = idx % C;
      dst[r * ld + c] = r < len ? src[r * rs + c] : zero;
    }
  }
}

template <int R, int C, int NT>
__device__ __forceinline__ void tile_f32(float *dst, int ld, const float *src, int64_t rs, int len) {
  constexpr int VPR = C / 4, NV = R * VPR;  // always 16-byte aligned (internal buffers)
  static_assert(C % 4 == 0 && NV % NT == 0, "tile shape");
  constexpr int PER = NV / NT, BATCH = PER < 8 ? PER : 8;
  static_assert(PER % BATCH == 0, "whole batches");
#pragma unroll
  for (int b0 = 0; b0 < PER; b0 += BATCH) {
    float4 x[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int v = threadIdx.x + (b0 + u) * NT, r = v / VPR, c = (v % VPR) * 4;
      x[u] = r < len ? *reinterpret_cast<const float4 *>(src + r * rs + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int v = threadIdx.x + (b0 + u) * NT, r = v / VPR, c = (v % VPR) * 4;
      *reinterpret_cast<float4 *>(dst + r * ld + c) = x[u];  // ld % 4 == 0
    }
  }
}

}  // namespace gdr

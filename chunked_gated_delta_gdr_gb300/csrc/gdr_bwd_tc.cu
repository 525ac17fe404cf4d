// gdr_bwd_tc.cu -- backward kernels of the chunked gated delta rule on the sm_103a tensor
// cores (tcgen05.mma with TMEM accumulators, operand tiles loaded by TMA).
//
// k_bwd_dv_intra_tc: the intra-chunk part of dV' (the gradient of the chunk's V', see
// gdr_bwd.cu), per chunk c of 64 tokens and value head h:
//
//   dV'_intra = scale ((Q K^T) o Gam)^T dO,   Gam_rc = e^{G_r - G_c} for c <= r < len,
//
// with G the chunk-local cumulative gate.  Two MMAs per block, M = 128 on both:
//   X' = [K;Q] Q^T              TMEM lanes 0-63 hold k_c.q_r (lanes 64-127: q.q, unused);
//   P^T[c][r] = Gam_rc X'[c][r]  by the threads of lanes 0-63, bf16, 128-byte swizzled rows;
//   dV'^T = dO^T (P^T)^T          A = dO^T (value dim on lanes, MN-major), B = P^T (K-major).
// The accumulator row of lane dv is stored as fp32 to dV'[t0 + c][h][dv] (each warp writes
// 128 contiguous bytes per token).  Rows of the tiles past the chunk's end (the next
// segment's tokens, or zeros past the tensor's end) only reach masked entries of P^T or
// accumulator columns that are not stored.  The chunk's 64-token grid and the masks are the
// ones the forward uses ("Findings from integrating FlashQLA's Blackwell GDN kernels into
// a JAX trainer", section 1: 64-token chunks over cu_seqlens).
//
// One block of 128 threads per (chunk, value head), 59 KB of shared memory and 128 TMEM
// columns, so three blocks share an SM.  Thread 0 issues the TMA loads and the MMAs.
//
// k_bwd_sgrad_tc: the products with the state entering the chunk (S_0, bf16 as the
// forward recompute stores it) and the gradient of the state leaving it (dS_C, fp32):
//
//   dQ  = scale diag(e^G) dO S_0^T,   dK = diag(e^{G_C - G}) V' dS_C^T,   dW = -dV' S_0^T,
//   sdot = <dS_C, S_0> per 64 key rows,
//
// as three MMAs with the key dim on the TMEM lanes (M = 128) and the chunk's tokens as N:
// A = S_0 or dS_C (rows = key dim, K-major over the value dim), B = dO, V' or dV' (rows =
// tokens).  dS_C and dV' are rounded to bf16 on their way into shared memory (loaded by
// the threads, coalesced, which also form sdot in fp32); S_0, dO and V' hold bf16 values
// already and come by TMA.  113 KB of shared memory and 256 TMEM columns: two blocks per SM.
//
// Every wait is bounded; a wait that runs out makes the block skip the rest of its work
// (its outputs then hold whatever was there before) and records a status word that
// read_bwd_tc_status returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdr_bwd.cuh"
#include "gdr_tc.cuh"

namespace gdr {

__device__ int32_t g_bwd_tc_status = 0;

namespace {

using namespace tc;

constexpr int kTcThreads = 128;
constexpr uint64_t kTcWaitNs = 2000000000ull;
// shared memory (from a 1024-aligned base)
constexpr uint32_t kOffKQ = 0;       // 2 key blocks x [K rows 0-63 | Q rows 64-127] x 128 B
constexpr uint32_t kOffDO = 32768;   // 2 value blocks x 64 token rows x 128 B
constexpr uint32_t kOffPT = 49152;   // P^T bf16 64 x 64
constexpr uint32_t kOffG = 57344;    // G[64] fp32, then barriers
constexpr uint32_t kTcSmem = kOffG + 512 + 1024;
constexpr uint32_t kTcCols = 128;    // X' in columns 0-63, dV'^T in 64-127

struct TcSmall {
  float G[64];
  uint64_t full, mma1, mma2;
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(TcSmall) <= 512, "small area");

template <int D>
__global__ void __launch_bounds__(kTcThreads)
    k_bwd_dv_intra_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mdo, int32_t group, View gcum,
                      float scale, View dvp, const ChunkInfo *__restrict__ chunks,
                      const int32_t *__restrict__ n_chunks) {
  extern __shared__ uint8_t dyn_smem[];
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (cid >= *n_chunks) return;  // (before any TMEM is allocated)
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  TcSmall *sm = reinterpret_cast<TcSmall *>(base + kOffG);
  const uint32_t sbase = smem_u32(base);
  const int warp = tid >> 5;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int t0 = ci.start;
  if (tid == 0) {
    mbar_init(&sm->full, 1);
    mbar_init(&sm->mma1, 1);
    mbar_init(&sm->mma2, 1);
    sm->abort = 0;
    fence_mbar_init();
  }
  if (D != 128) {  // head dim 64: the upper key / value blocks stay zero
    uint32_t *z = reinterpret_cast<uint32_t *>(base + kOffKQ + 16384);
    for (int i = tid; i < 16384 / 4; i += kTcThreads) z[i] = 0;
    z = reinterpret_cast<uint32_t *>(base + kOffDO + 8192);
    for (int i = tid; i < 8192 / 4; i += kTcThreads) z[i] = 0;
    fence_async_smem();
  }
  if (tid < 64)
    sm->G[tid] = tid < len ? ldf(gcum.p, (int64_t)(t0 + tid) * gcum.st + (int64_t)h * gcum.sh) : 0.f;
  if (warp == 0) {
    tmem_alloc(&sm->tmem_base, kTcCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = sm->tmem_base;
  const uint32_t lane_base = (uint32_t)(tid & ~31);
  if (tid == 0) {
    mbar_expect_tx(&sm->full, D == 128 ? 49152u : 24576u);
    uint8_t *kq = base + kOffKQ, *dd = base + kOffDO;
    tma_load_3d(kq, &mk, &sm->full, 0, hk, t0);
    tma_load_3d(kq + 8192, &mq, &sm->full, 0, hk, t0);
    tma_load_3d(dd, &mdo, &sm->full, 0, h, t0);
    if (D == 128) {
      tma_load_3d(kq + 16384, &mk, &sm->full, 64, hk, t0);
      tma_load_3d(kq + 24576, &mq, &sm->full, 64, hk, t0);
      tma_load_3d(dd + 8192, &mdo, &sm->full, 64, h, t0);
    }
  }
  bool bad = !mbar_wait(&sm->full, 0, &sm->abort, kTcWaitNs);
  if (tid == 0 && !bad) {
    // X' = [K;Q] Q^T over the key dim: A = the [K;Q] rows, B = the Q rows (K-major)
    tc_fence_after();
    const uint32_t id = idesc_bf16(128, 64, false, false);
    const uint64_t a = sdesc_sw128(sbase + kOffKQ, 0, 1024);
    const uint64_t b = sdesc_sw128(sbase + kOffKQ + 8192, 0, 1024);
#pragma unroll 1
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
      mma_bf16(tb, a + off, b + off, id, kk > 0);
    }
    mma_commit(&sm->mma1);
  }
  bad = bad || !mbar_wait(&sm->mma1, 0, &sm->abort, kTcWaitNs);
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicCAS(&g_bwd_tc_status, 0, 0x501);
  } else {
    tc_fence_after();
    if (tid < 64) {
      // P^T row c: Gam_rc k_c.q_r for c <= r < len, as bf16 into the K-major B tile
      const int c = tid;
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem_addr(tb, lane_base, 0), r0);
      tmem_ld32(tmem_addr(tb, lane_base, 32), r1);
      tmem_ld_wait();
      const float gc = sm->G[c];
      constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float f[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int r = hh * 32 + u;
          const float x = __uint_as_float(hh ? r1[u] : r0[u]);
          f[u] = (c <= r && r < len) ? ex2((sm->G[r] - gc) * kLog2e) * x : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float *v = f + q * 8;
          const uint32_t addr = sbase + kOffPT + sw128_off(c, hh * 32 + q * 8);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                       "r"(pack_bf16(v[0], v[1])), "r"(pack_bf16(v[2], v[3])),
                       "r"(pack_bf16(v[4], v[5])), "r"(pack_bf16(v[6], v[7])));
        }
      }
      fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      // dV'^T = dO^T (P^T)^T: A = dO^T (value dim on lanes, MN-major over tokens), B = P^T
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, true, false);
      const uint64_t a = sdesc_sw128(sbase + kOffDO, 8192, 1024);
      const uint64_t b = sdesc_sw128(sbase + kOffPT, 0, 1024);
#pragma unroll 1
      for (int kk = 0; kk < 4; ++kk) mma_bf16(tb + 64, a + ((kk * 2048) >> 4), b + ((kk * 32) >> 4), id, kk > 0);
      mma_commit(&sm->mma2);
    }
    bad = !mbar_wait(&sm->mma2, 0, &sm->abort, kTcWaitNs);
    if (__syncthreads_or(bad)) {
      if (tid == 0) atomicCAS(&g_bwd_tc_status, 0, 0x502);
    } else {
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem_addr(tb + 64, lane_base, 0), r0);
      tmem_ld32(tmem_addr(tb + 64, lane_base, 32), r1);
      tmem_ld_wait();
      const int dv = tid;
      if (dv < D) {
        float *out = reinterpret_cast<float *>(dvp.p) + (int64_t)t0 * dvp.st + (int64_t)h * dvp.sh + dv;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          if (u < len) out[(int64_t)u * dvp.st] = scale * __uint_as_float(r0[u]);
          if (32 + u < len) out[(int64_t)(32 + u) * dvp.st] = scale * __uint_as_float(r1[u]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, kTcCols);
  }
}

// ---------------------------------------------------------------- products with S_0, dS_C
constexpr uint32_t kSgOffS0 = 0;       // S_0 bf16: 2 value blocks x 128 key rows x 128 B
constexpr uint32_t kSgOffDO = 32768;   // dO bf16: 2 value blocks x 64 token rows x 128 B
constexpr uint32_t kSgOffVP = 49152;   // V' bf16, same
constexpr uint32_t kSgOffDV = 65536;   // dV' bf16, same
constexpr uint32_t kSgOffSmall = 81920;
constexpr uint32_t kSgSmem = kSgOffSmall + 1024 + 1024;
constexpr uint32_t kSgCols = 256;  // dQ^T 0-63, dK^T 64-127, dW^T 128-191, dS_C (bf16) 192-255

struct SgSmall {
  float EG[64], DEC[64];
  float red[4];
  uint64_t full, mma;
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(SgSmall) <= 1024, "small area");

// Byte offset of element (row, col) of a K-major tile of `rows` rows, 64 bf16 columns per
// 128-byte row and value block (col < 128).
__device__ __forceinline__ uint32_t kmaj_off(uint32_t rows, uint32_t row, uint32_t col) {
  return (col >> 6) * rows * 128u + sw128_off(row, col & 63u);
}

template <int D>
__global__ void __launch_bounds__(kTcThreads)
    k_bwd_sgrad_tc(const __grid_constant__ CUtensorMap mh, const __grid_constant__ CUtensorMap mdo,
                   const __grid_constant__ CUtensorMap mvp, View gcum, float scale, const float *dh,
                   View dvp, View dqh, View dkh, View dw, float *sdot,
                   const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks,
                   int32_t H) {
  extern __shared__ uint8_t dyn_smem[];
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (cid >= *n_chunks) return;  // (before any TMEM is allocated)
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  SgSmall *sm = reinterpret_cast<SgSmall *>(base + kSgOffSmall);
  const uint32_t sbase = smem_u32(base);
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, t0 = ci.start;
  const int64_t sidx = (int64_t)cid * H + h;
  if (tid == 0) {
    mbar_init(&sm->full, 1);
    mbar_init(&sm->mma, 1);
    sm->abort = 0;
    fence_mbar_init();
  }
  if (tid < 64) {
    const float gi =
        tid < len ? ldf(gcum.p, (int64_t)(t0 + tid) * gcum.st + (int64_t)h * gcum.sh) : 0.f;
    const float gl = ldf(gcum.p, (int64_t)(t0 + len - 1) * gcum.st + (int64_t)h * gcum.sh);
    sm->EG[tid] = tid < len ? expf(gi) : 0.f;
    sm->DEC[tid] = tid < len ? expf(gl - gi) : 0.f;
  }
  if (warp == 0) {
    tmem_alloc(&sm->tmem_base, kSgCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = sm->tmem_base;
  const uint32_t lane_base = (uint32_t)(tid & ~31);
  if (tid == 0) {
    // S_0 as the 128 rows from key row 0 of this (chunk, head)'s [D][D] block (rows past D
    // belong to the next block and reach only accumulator lanes that are not stored)
    mbar_expect_tx(&sm->full, D == 128 ? 65536u : 32768u);
    tma_load_2d(base + kSgOffS0, &mh, &sm->full, 0, (int32_t)(sidx * D));
    tma_load_3d(base + kSgOffDO, &mdo, &sm->full, 0, h, t0);
    tma_load_3d(base + kSgOffVP, &mvp, &sm->full, 0, h, t0);
    if (D == 128) {
      tma_load_2d(base + kSgOffS0 + 16384, &mh, &sm->full, 64, (int32_t)(sidx * D));
      tma_load_3d(base + kSgOffDO + 8192, &mdo, &sm->full, 64, h, t0);
      tma_load_3d(base + kSgOffVP + 8192, &mvp, &sm->full, 64, h, t0);
    }
  }
  constexpr int kV4 = D / 4;  // float4 per row
  {
    // dV' -> bf16 B tile: rows past the chunk's end are zero; a warp reads a row's D
    // floats per step (16-byte loads, coalesced)
    const float *dvb =
        reinterpret_cast<const float *>(dvp.p) + (int64_t)t0 * dvp.st + (int64_t)h * dvp.sh;
#pragma unroll 4
    for (int idx = tid; idx < 64 * kV4; idx += kTcThreads) {
      const int r = idx / kV4, c = (idx % kV4) * 4;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < len) x = __ldg(reinterpret_cast<const float4 *>(dvb + (int64_t)r * dvp.st + c));
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(sbase + kSgOffDV + kmaj_off(64, r, c)),
                   "r"(pack_bf16(x.x, x.y)), "r"(pack_bf16(x.z, x.w)));
    }
    fence_async_smem();
  }
  // (warp-uniform: the TMEM stores below are warp-collective)
  bool bad = __any_sync(0xffffffffu, !mbar_wait(&sm->full, 0, &sm->abort, kTcWaitNs));
  float part = 0.f;
  if (!bad && tid < D) {
    // key row r = tid: dS_C row r -> bf16 into TMEM lane r (the A operand of dK^T), and
    // <dS_C, S_0> over the row with S_0 from its tile
    const int r = tid;
    const float *dsr = dh + sidx * D * D + (int64_t)r * D;
#pragma unroll 1
    for (int cb = 0; cb < D / 64; ++cb) {
      uint32_t pk[32];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = cb * 64 + u * 4;
        const float4 x = __ldg(reinterpret_cast<const float4 *>(dsr + c));
        uint32_t s01, s23;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                     : "=r"(s01), "=r"(s23)
                     : "r"(sbase + kSgOffS0 + kmaj_off(128, r, c)));
        part += x.x * __uint_as_float(s01 << 16) + x.y * __uint_as_float(s01 & 0xffff0000u) +
                x.z * __uint_as_float(s23 << 16) + x.w * __uint_as_float(s23 & 0xffff0000u);
        pk[2 * u] = pack_bf16(x.x, x.y);
        pk[2 * u + 1] = pack_bf16(x.z, x.w);
      }
      tmem_st32(tmem_addr(tb + 192, lane_base, cb * 32), pk);
    }
  }
  if (warp < D / 32) tmem_st_wait();
  // fixed-order sums: a shuffle tree in each warp, then two warps per 64 key rows in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) sm->red[warp] = part;
  tc_fence_before();
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicCAS(&g_bwd_tc_status, 0, 0x511);
  } else {
    tc_fence_after();
    if (tid == 0) {
      for (int b = 0; b < D / 64; ++b) sdot[sidx * (D / 64) + b] = sm->red[2 * b] + sm->red[2 * b + 1];
      // over the value dim: dQ^T = S_0 dO^T, dW^T = S_0 dV'^T (A = S_0 tile), dK^T =
      // dS_C V'^T (A = dS_C in TMEM)
      const uint32_t id = idesc_bf16(128, 64, false, false);
      const uint64_t as0 = sdesc_sw128(sbase + kSgOffS0, 0, 1024);
      const uint64_t bdo = sdesc_sw128(sbase + kSgOffDO, 0, 1024);
      const uint64_t bvp = sdesc_sw128(sbase + kSgOffVP, 0, 1024);
      const uint64_t bdv = sdesc_sw128(sbase + kSgOffDV, 0, 1024);
#pragma unroll 1
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t oa = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;  // 128-row A tile
        const uint32_t ob = ((kk / 4) * 8192 + (kk % 4) * 32) >> 4;   // 64-row B tiles
        mma_bf16(tb, as0 + oa, bdo + ob, id, kk > 0);
        mma_bf16(tb + 128, as0 + oa, bdv + ob, id, kk > 0);
        mma_bf16_ts(tb + 64, tb + 192 + kk * 8, bvp + ob, id, kk > 0);
      }
      mma_commit(&sm->mma);
    }
    bad = !mbar_wait(&sm->mma, 0, &sm->abort, kTcWaitNs);
    if (__syncthreads_or(bad)) {
      if (tid == 0) atomicCAS(&g_bwd_tc_status, 0, 0x512);
    } else if (warp < D / 32) {
      tc_fence_after();
      // lane r = key row r; column i = token i of the chunk
      const int r = tid;
      float *qo = reinterpret_cast<float *>(dqh.p) + (int64_t)t0 * dqh.st + (int64_t)h * dqh.sh + r;
      float *ko = reinterpret_cast<float *>(dkh.p) + (int64_t)t0 * dkh.st + (int64_t)h * dkh.sh + r;
      float *wo = reinterpret_cast<float *>(dw.p) + (int64_t)t0 * dw.st + (int64_t)h * dw.sh + r;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t aq[32], ak[32], aw[32];
        tmem_ld32(tmem_addr(tb, lane_base, half * 32), aq);
        tmem_ld32(tmem_addr(tb + 64, lane_base, half * 32), ak);
        tmem_ld32(tmem_addr(tb + 128, lane_base, half * 32), aw);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int i = half * 32 + u;
          if (i < len) {
            qo[(int64_t)i * dqh.st] = scale * sm->EG[i] * __uint_as_float(aq[u]);
            ko[(int64_t)i * dkh.st] = sm->DEC[i] * __uint_as_float(ak[u]);
            wo[(int64_t)i * dw.st] = -__uint_as_float(aw[u]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, kSgCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 2-D map of a [rows, D] bf16 matrix (row-major): boxes of 128 rows x 64 columns, 128-byte
// swizzle (the states S_0 of the forward recompute, one [D][D] block per chunk and head).
bool make_rows_map(CUtensorMap *m, const void *ptr, int64_t D, int64_t rows) {
  auto enc = tc_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(D * 2)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_tc_smem_set[64] = {0};

// Dynamic shared memory limits of the kernels above, once per device.
cudaError_t tc_smem_attrs() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (g_tc_smem_set[dev]) return cudaSuccess;
  const int a = (int)kTcSmem, b = (int)kSgSmem;
  if ((e = cudaFuncSetAttribute(k_bwd_dv_intra_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, a)) ||
      (e = cudaFuncSetAttribute(k_bwd_dv_intra_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, a)) ||
      (e = cudaFuncSetAttribute(k_bwd_sgrad_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, b)) ||
      (e = cudaFuncSetAttribute(k_bwd_sgrad_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, b)))
    return e;
  g_tc_smem_set[dev] = 1;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_dv_intra_tc(const BwdArgs &a, View gcum, View dvp, cudaStream_t stream) {
  const StageShapes &s = a.s;
  if (s.D != 128 && s.D != 64) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mdo;
  if (!make_tile_map(&mq, a.q.p, s.D, s.Hk, s.T, a.q.st, a.q.sh) ||
      !make_tile_map(&mk, a.k.p, s.D, s.Hk, s.T, a.k.st, a.k.sh) ||
      !make_tile_map(&mdo, a.dout.p, s.D, s.H, s.T, a.dout.st, a.dout.sh))
    return cudaErrorNotSupported;
  cudaError_t e = tc_smem_attrs();
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)s.chunk_cap, (unsigned)s.H);
  const int32_t group = s.H / s.Hk;
  if (s.D == 128)
    k_bwd_dv_intra_tc<128><<<grid, kTcThreads, kTcSmem, stream>>>(mq, mk, mdo, group, gcum, a.scale,
                                                                   dvp, a.chunks, a.n_chunks);
  else
    k_bwd_dv_intra_tc<64><<<grid, kTcThreads, kTcSmem, stream>>>(mq, mk, mdo, group, gcum, a.scale,
                                                                  dvp, a.chunks, a.n_chunks);
  return cudaGetLastError();
}

cudaError_t launch_bwd_sgrad_tc(const BwdArgs &a, const void *h, const float *dh, View gcum,
                               View vnew, View dvp, View dqh, View dkh, View dw, float *sdot,
                               cudaStream_t stream) {
  const StageShapes &s = a.s;
  if (s.D != 128 && s.D != 64) return cudaErrorNotSupported;
  auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  // dS_C and dV' rows are read as float4
  if (!al16(dh) || !al16(dvp.p) || (dvp.st % 4) || (dvp.sh % 4)) return cudaErrorNotSupported;
  const int64_t rows = s.chunk_cap * s.H * s.D;  // S_0 rows; the TMA row coordinate is int32
  if (rows >= ((int64_t)1 << 31)) return cudaErrorNotSupported;
  CUtensorMap mh, mdo, mvp;
  if (!make_rows_map(&mh, h, s.D, rows) ||
      !make_tile_map(&mdo, a.dout.p, s.D, s.H, s.T, a.dout.st, a.dout.sh) ||
      !make_tile_map(&mvp, vnew.p, s.D, s.H, s.T, vnew.st, vnew.sh))
    return cudaErrorNotSupported;
  cudaError_t e = tc_smem_attrs();
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)s.chunk_cap, (unsigned)s.H);
  if (s.D == 128)
    k_bwd_sgrad_tc<128><<<grid, kTcThreads, kSgSmem, stream>>>(mh, mdo, mvp, gcum, a.scale, dh, dvp,
                                                               dqh, dkh, dw, sdot, a.chunks,
                                                               a.n_chunks, s.H);
  else
    k_bwd_sgrad_tc<64><<<grid, kTcThreads, kSgSmem, stream>>>(mh, mdo, mvp, gcum, a.scale, dh, dvp,
                                                              dqh, dkh, dw, sdot, a.chunks,
                                                              a.n_chunks, s.H);
  return cudaGetLastError();
}

cudaError_t read_bwd_tc_status(int32_t *out) {
  return cudaMemcpyFromSymbol(out, g_bwd_tc_status, sizeof(int32_t));
}

}  // namespace gdr

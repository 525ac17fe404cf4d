// gdr_staged.cu -- the three stages of the chunked gated delta rule forward as
// separate kernels with their intermediates in HBM (GDR_PATH_STAGED and the
// per-stage entry points).  fp32 arithmetic; every dense product as tf32 tensor-core
// warp tiles over shared-memory operands (bf16 tiles for bf16 values, fp32 otherwise),
// the rest SIMT; bf16 at the same storage points as the fused path (W, U, V', h).
//
// Per chunk of 64 tokens (chunk-local indices i, j) and value head:
//   stage 1  G = cumsum(g);  A_ij = beta_i e^{G_i-G_j} k_i.k_j (j<i);  Tm = (I+A)^-1
//            W = Tm diag(beta e^G) K;  U = Tm diag(beta) V
//   stage 2  h_c = S;  V' = U - W S;  S <- e^{G_last} S + (diag(e^{G_last-G}) K)^T V'
//   stage 3  O = scale [diag(e^G) Q h_c + (M o Q K^T) V'],  M_ij = e^{G_i-G_j} (j<=i)
// These follow from unrolling the gated delta rule recurrence inside a chunk;
// the chunk size is the 64 of FlashQLA's varlen path ("Findings from
// integrating FlashQLA's Blackwell GDN kernels into a JAX trainer", section 1).
#include "gdr_internal.cuh"
#include "gdr_mma.cuh"
#include "gdr_sched.cuh"

namespace gdr {
namespace {

// ---------------------------------------------------------------- stage 1
// K and V stay bf16 in shared memory (half the bytes of fp32 tiles, the same operand
// values): two blocks fit on an SM, so one block's loads overlap another's products.
template <int D>
struct PrepSmem {
  static constexpr int kLd = ld_bf16(D), kLdA = ld_rows(64);
  static constexpr size_t f32 = 3 * 64 * kLdA + 3 * 64 + kSolveScratch;  // floats
  static constexpr size_t bytes = sizeof(float) * f32 + sizeof(__nv_bfloat16) * 2 * 64 * kLd;
};

template <int D>
__global__ void __launch_bounds__(kChunkThreads, 2)
    k_prep(int32_t group, View k, View v, View g, View beta, View w, View u, View gcum,
           const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks, bool vec) {
  extern __shared__ float sm[];
  constexpr int L = PrepSmem<D>::kLd, LA = PrepSmem<D>::kLdA;
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *Am = sm, *Tm = Am + 64 * LA, *TU = Tm + 64 * LA;
  float *G = TU + 64 * LA, *B = G + 64, *BG = B + 64, *scratch = BG + 64;
  __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(sm + PrepSmem<D>::f32), *Vs = Ks + 64 * L;

  tile_bf16_raw<64, D, kChunkThreads>(Ks, L, bf_row(k, t0, hk), k.st, len, vec);
  tile_bf16_raw<64, D, kChunkThreads>(Vs, L, bf_row(v, t0, h), v.st, len, vec);
  if (tid < 64) {
    G[tid] = tid < len ? ldf(g.p, (t0 + tid) * g.st + h * g.sh) : 0.f;
    B[tid] = tid < len ? ldbf(beta.p, (t0 + tid) * beta.st + h * beta.sh) : 0.f;
  }
  __syncthreads();
  if (tid < 32) {  // chunk-local inclusive cumsum of g, two entries per lane
    const float a = G[2 * tid], b = G[2 * tid + 1];
    float s = a + b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, off);
      if (tid >= off) s += y;
    }
    const float excl = s - (a + b);
    G[2 * tid] = excl + a;
    G[2 * tid + 1] = excl + a + b;
  }
  __syncthreads();
  if (tid < 64) BG[tid] = B[tid] * expf(G[tid]);
  const int warp = tid >> 5;
  // A_ij = beta_i e^{G_i - G_j} k_i . k_j (j < i): 32 tiles of the key products
  {
    const int m0 = ((warp * kTPW) >> 3) * 16, nb = ((warp * kTPW) & 7) * 8;
    float accs[kTPW][4] = {};
    mma_16xN<kTPW>(accs, SMatH{Ks, L, 1}, m0, SMatH{Ks, 1, L}, nb, 0, D);
#pragma unroll
    for (int b = 0; b < kTPW; ++b) {
      const int n0 = nb + 8 * b;
      float(&acc)[4] = accs[b];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = acc_row(m0, e), j = acc_col(n0, e);
        Am[i * LA + j] = (j < i && i < len) ? B[i] * expf(G[i] - G[j]) * acc[e] : 0.f;
      }
    }
  }
  __syncthreads();
  solve_unit_lower64(Am, LA, Tm, LA, scratch, blockDim.x, 0);  // Tm = (I + A)^-1
  // Tm diag(beta e^G) into Am's place, Tm diag(beta) into TU
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx >> 6, j = idx & 63;
    Am[i * LA + j] = Tm[i * LA + j] * BG[j];
    TU[i * LA + j] = Tm[i * LA + j] * B[j];
  }
  __syncthreads();
  // W = Tm diag(beta e^G) K, U = Tm diag(beta) V: 64 x D outputs each
  for (int tl = warp; tl < 4 * (D / 8); tl += kWarps) {
    const int m0 = (tl & 3) * 16, n0 = (tl >> 2) * 8;
    float wa[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
    mma_16x8(wa, SMat{Am, LA, 1}, m0, SMatH{Ks, L, 1}, n0, 0, 64);
    mma_16x8(ua, SMat{TU, LA, 1}, m0, SMatH{Vs, L, 1}, n0, 0, 64);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = acc_row(m0, e), d = acc_col(n0, e);
      if (i < len) {
        stbf(w.p, (t0 + i) * w.st + h * w.sh + d, wa[e]);
        stbf(u.p, (t0 + i) * u.st + h * u.sh + d, ua[e]);
      }
    }
  }
  if (tid < len) reinterpret_cast<float *>(gcum.p)[(t0 + tid) * gcum.st + h * gcum.sh] = G[tid];
}

// ---------------------------------------------------------------- stage 2

// W, K and U stay bf16 in shared memory (as stored): two blocks fit on an SM.
template <int D, int kScanCols>
struct ScanSmem {
  static constexpr int kLdW = ld_bf16(D), kLdK = ld_bf16(D), kLdU = ld_bf16(kScanCols),
                       kLdC = ld_cols(kScanCols);
  static constexpr size_t f32 = D * kLdC + 64 * kLdC + 2 * 64;  // floats
  static constexpr size_t bytes =
      sizeof(float) * f32 + sizeof(__nv_bfloat16) * (64 * kLdW + 64 * kLdK + 64 * kLdU);
};

// kScanCols value columns per block, kScanCols / 8 warps
template <int D, int kScanCols>
__global__ void __launch_bounds__(kScanCols * 4, 2)
    k_scan(int32_t H, int32_t group, View k, View w, View u, View gcum, const float *h0,
           __nv_bfloat16 *hbuf, View v_new, float *ht, Ckpt ck,
           const SegInfo *__restrict__ seg, const int32_t *__restrict__ order, bool vec) {
  extern __shared__ float sm[];
  using Sm = ScanSmem<D, kScanCols>;
  constexpr int LW = Sm::kLdW, LK = Sm::kLdK, LU = Sm::kLdU, LC = Sm::kLdC;
  constexpr int NT = kScanCols * 4, NW = kScanCols / 8, CT = kScanCols / 8;  // threads, warps, column tiles
  // one flat grid, head fastest, then column block, then segment rank: the longest
  // segments are dispatched first (a flat x extent allows any segment count)
  const int64_t bid = blockIdx.x, Z = D / kScanCols;
  const int h = (int)(bid % H), rank = (int)(bid / H / Z);
  const int n = order ? order[rank] : rank;
  const int jb = (int)((bid / H) % Z) * kScanCols, tid = threadIdx.x;
  const int hk = h / group;
  const SegInfo si = seg[n];
  float *S = sm, *Vn = S + D * LC, *G = Vn + 64 * LC, *Dec = G + 64;
  __nv_bfloat16 *Ws = reinterpret_cast<__nv_bfloat16 *>(sm + Sm::f32), *Ks = Ws + 64 * LW,
                *Us = Ks + 64 * LK;
  const int64_t sbase = ((int64_t)n * H + h) * D * D;

  for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
    const int d = idx / kScanCols, j = idx % kScanCols;
    S[d * LC + j] = h0 ? h0[sbase + (int64_t)d * D + jb + j] : 0.f;
  }
  // state of this block's columns -> checkpoint row `row` (the state after the
  // segment's first (row - first row + 1) * every tokens)
  auto store_ckpt = [&](int64_t row) {
    float *dst = ck.h + (row * H + h) * D * D;
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      dst[(int64_t)d * D + jb + j] = S[d * LC + j];
    }
  };
  for (int c = 0; c < si.n_chunks; ++c) {
    const int64_t cid = si.chunk_off + c;
    const int64_t t0 = si.start + (int64_t)c * kChunk;
    const int len = min(kChunk, si.end - (int)t0);
    __syncthreads();
    if (ck.h && c > 0 && (c * kChunk) % ck.every == 0)
      store_ckpt(ck.off[n] + (c * kChunk) / ck.every - 1);
    __nv_bfloat16 *hc = hbuf + (cid * H + h) * D * D;
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      hc[(int64_t)d * D + jb + j] = __float2bfloat16_rn(S[d * LC + j]);
    }
    tile_bf16_raw<64, D, NT>(Ws, LW, bf_row(w, t0, h), w.st, len, vec);
    tile_bf16_raw<64, D, NT>(Ks, LK, bf_row(k, t0, hk), k.st, len, vec);
    tile_bf16_raw<64, kScanCols, NT>(Us, LU, bf_row(u, t0, h) + jb, u.st, len, vec);
    if (tid < 64) G[tid] = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    __syncthreads();
    const float glast = G[len - 1];
    if (tid < 64) Dec[tid] = tid < len ? expf(glast - G[tid]) : 0.f;
    __syncthreads();
    const int warp = tid >> 5;
    // V' = U - W S (bf16, as stored), and Vn = diag(e^{G_last - G}) V' for the update:
    // 64 x kScanCols outputs, four 16 x 8 tiles per warp on the tensor pipe
    {
      const int m0 = ((warp * 4) / CT) * 16, nb = ((warp * 4) % CT) * 8;
      float accs[4][4] = {};
      mma_16xN<4>(accs, SMatH{Ws, LW, 1}, m0, SMat{S, LC, 1}, nb, 0, D);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int n0 = nb + 8 * b;
        float(&acc)[4] = accs[b];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = acc_row(m0, e), j = acc_col(n0, e);
          float vn = 0.f;
          if (i < len) {
            const __nv_bfloat16 b = __float2bfloat16_rn(__bfloat162float(Us[i * LU + j]) - acc[e]);
            reinterpret_cast<__nv_bfloat16 *>(v_new.p)[(t0 + i) * v_new.st + h * v_new.sh + jb + j] = b;
            vn = Dec[i] * __bfloat162float(b);
          }
          Vn[i * LC + j] = vn;
        }
      }
    }
    __syncthreads();
    // S <- e^{G_last} S + K^T Vn: D x kScanCols outputs
    const float eg = expf(glast);
    static_assert(NW == CT, "one column tile per warp");
    {
      // warp w: every row tile of column tile w
      constexpr int MB = D / 16;
      const int n0 = warp * 8;
      float acc[MB][4] = {};
      mma_Mx8<MB>(acc, SMatH{Ks, 1, LK}, 0, SMat{Vn, LC, 1}, n0, 0, 64);
#pragma unroll
      for (int r = 0; r < MB; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = acc_row(16 * r, e), j = acc_col(n0, e);
          S[d * LC + j] = eg * S[d * LC + j] + acc[r][e];
        }
    }
  }
  if (ht || ck.h) __syncthreads();
  if (ht) {
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      ht[sbase + (int64_t)d * D + jb + j] = S[d * LC + j];
    }
  }
  const int seg_len = si.end - si.start;
  if (ck.h && seg_len > 0 && seg_len % ck.every == 0) store_ckpt(ck.off[n] + seg_len / ck.every - 1);
}

// ---------------------------------------------------------------- stage 3
constexpr int kOutCols = 64;

// q, k, h and V' stay bf16 in shared memory (as in memory); P is fp32.
template <int D>
struct OutSmem {
  static constexpr int kLd = ld_bf16(D), kLdH = ld_bf16(kOutCols), kLdP = ld_rows(64);
  static constexpr size_t f32 = 64 * kLdP + 2 * 64;  // floats
  static constexpr size_t bytes =
      sizeof(float) * f32 + sizeof(__nv_bfloat16) * (2 * 64 * kLd + D * kLdH + 64 * kLdH);
};

// Block (chunk, head, column block of kOutCols value columns), 8 warps: every product is
// a set of tensor-core tiles, four 16 x 8 tiles per warp.
template <int D>
__global__ void __launch_bounds__(256, 2)
    k_out(int32_t H, int32_t group, View q, View k, View v_new, const __nv_bfloat16 *hbuf,
          View gcum, float scale, View o, const ChunkInfo *__restrict__ chunks,
          const int32_t *__restrict__ n_chunks, bool vec) {
  extern __shared__ float sm[];
  using Sm = OutSmem<D>;
  constexpr int L = Sm::kLd, LH = Sm::kLdH, LP = Sm::kLdP;
  const int cid = blockIdx.x, h = blockIdx.y, cb = blockIdx.z * kOutCols, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *P = sm, *G = P + 64 * LP, *EG = G + 64;
  __nv_bfloat16 *Qs = reinterpret_cast<__nv_bfloat16 *>(sm + Sm::f32), *Ks = Qs + 64 * L,
                *Hs = Ks + 64 * L, *Vn = Hs + D * LH;

  tile_bf16_raw<64, D, 256>(Qs, L, bf_row(q, t0, hk), q.st, len, vec);
  tile_bf16_raw<64, D, 256>(Ks, L, bf_row(k, t0, hk), k.st, len, vec);
  const __nv_bfloat16 *hc = hbuf + ((int64_t)cid * H + h) * D * D;
  tile_bf16_raw<D, kOutCols, 256>(Hs, LH, hc + cb, D, D, vec);
  tile_bf16_raw<64, kOutCols, 256>(Vn, LH, bf_row(v_new, t0, h) + cb, v_new.st, len, vec);
  if (tid < 64) {
    const float gi = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    G[tid] = gi;
    EG[tid] = tid < len ? expf(gi) : 0.f;
  }
  __syncthreads();
  const int warp = tid >> 5;
  const int m0 = ((warp * 4) >> 3) * 16, nb = ((warp * 4) & 7) * 8;  // 16 rows x 32 columns
  // P = tril(Gam) o (Q K^T), Gam_ij = e^{G_i - G_j}
  {
    float accs[4][4] = {};
    mma_16xN<4>(accs, SMatH{Qs, L, 1}, m0, SMatH{Ks, 1, L}, nb, 0, D);
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = acc_row(m0, e), j = acc_col(nb + 8 * b, e);
        P[i * LP + j] = (j <= i && i < len) ? expf(G[i] - G[j]) * accs[b][e] : 0.f;
      }
  }
  __syncthreads();
  // O[:, cb ..] = scale (diag(e^G) Q h + P V')
  {
    float inter[4][4] = {}, intra[4][4] = {};
    mma_16xN<4>(inter, SMatH{Qs, L, 1}, m0, SMatH{Hs, LH, 1}, nb, 0, D);
    mma_16xN<4>(intra, SMat{P, LP, 1}, m0, SMatH{Vn, LH, 1}, nb, 0, 64);
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = acc_row(m0, e), c = acc_col(nb + 8 * b, e);
        if (i < len)
          stbf(o.p, (t0 + i) * o.st + h * o.sh + cb + c,
               scale * (EG[i] * inter[b][e] + intra[b][e]));
      }
  }
}

// 16-byte vector loads of a caller's bf16 tensor when its rows allow it
bool vec_ok(const View &x) {
  return (reinterpret_cast<uintptr_t>(x.p) & 15) == 0 && x.st % 8 == 0 && x.sh % 8 == 0;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_prep(const StageShapes &s, View k, View v, View g, View beta, View w,
                        View u, View gcum, const SegInfo *, const ChunkInfo *chunks,
                        const int32_t *n_chunks, cudaStream_t stream) {
  if (s.chunk_cap <= 0 || s.H <= 0) return cudaSuccess;
  dim3 grid((unsigned)s.chunk_cap, (unsigned)s.H);
  const bool vec = vec_ok(k) && vec_ok(v);
  cudaError_t e;
  if (s.D == 64) {
    if ((e = set_smem(k_prep<64>, PrepSmem<64>::bytes)) != cudaSuccess) return e;
    k_prep<64><<<grid, kChunkThreads, PrepSmem<64>::bytes, stream>>>(s.H / s.Hk, k, v, g, beta, w, u,
                                                           gcum, chunks, n_chunks, vec);
  } else {
    if ((e = set_smem(k_prep<128>, PrepSmem<128>::bytes)) != cudaSuccess) return e;
    k_prep<128><<<grid, kChunkThreads, PrepSmem<128>::bytes, stream>>>(s.H / s.Hk, k, v, g, beta, w, u,
                                                             gcum, chunks, n_chunks, vec);
  }
  return cudaGetLastError();
}

cudaError_t launch_scan(const StageShapes &s, View k, View w, View u, View gcum,
                        const float *h0, void *h, View v_new, float *ht, Ckpt ck,
                        const SegInfo *seg, cudaStream_t stream) {
  return launch_scan_ordered(s, k, w, u, gcum, h0, h, v_new, ht, ck, seg, nullptr, stream);
}

cudaError_t launch_scan_ordered(const StageShapes &s, View k, View w, View u, View gcum,
                                const float *h0, void *h, View v_new, float *ht, Ckpt ck,
                                const SegInfo *seg, const int32_t *order, cudaStream_t stream) {
  if (s.n_seq <= 0 || s.H <= 0) return cudaSuccess;
  auto *hb = reinterpret_cast<__nv_bfloat16 *>(h);
  const bool vec = vec_ok(k) && vec_ok(w) && vec_ok(u);
  auto scan = [&](auto kern, int cols, size_t bytes) -> cudaError_t {
    cudaError_t r = set_smem(kern, bytes);
    if (r != cudaSuccess) return r;
    const int64_t blocks = (int64_t)s.H * (s.D / cols) * s.n_seq;
    kern<<<(unsigned)blocks, cols * 4, bytes, stream>>>(s.H, s.H / s.Hk, k, w, u, gcum, h0, hb,
                                                       v_new, ht, ck, seg, order, vec);
    return cudaGetLastError();
  };
  const bool wide = scan_cols(s.n_seq, s.H, s.D) == 64;
  if (s.D == 64)
    return wide ? scan(k_scan<64, 64>, 64, ScanSmem<64, 64>::bytes)
                : scan(k_scan<64, 32>, 32, ScanSmem<64, 32>::bytes);
  return wide ? scan(k_scan<128, 64>, 64, ScanSmem<128, 64>::bytes)
              : scan(k_scan<128, 32>, 32, ScanSmem<128, 32>::bytes);
}

cudaError_t launch_out(const StageShapes &s, View q, View k, View v_new, const void *h,
                       View gcum, float scale, View o, const SegInfo *, const ChunkInfo *chunks,
                       const int32_t *n_chunks, cudaStream_t stream) {
  if (s.chunk_cap <= 0 || s.H <= 0) return cudaSuccess;
  dim3 grid((unsigned)s.chunk_cap, (unsigned)s.H, (unsigned)(s.D / kOutCols));
  auto *hb = reinterpret_cast<const __nv_bfloat16 *>(h);
  const bool vec = vec_ok(q) && vec_ok(k) && vec_ok(v_new) &&
                   (reinterpret_cast<uintptr_t>(h) & 15) == 0;
  cudaError_t e;
  if (s.D == 64) {
    if ((e = set_smem(k_out<64>, OutSmem<64>::bytes)) != cudaSuccess) return e;
    k_out<64><<<grid, 256, OutSmem<64>::bytes, stream>>>(s.H, s.H / s.Hk, q, k, v_new, hb,
                                                         gcum, scale, o, chunks, n_chunks, vec);
  } else {
    if ((e = set_smem(k_out<128>, OutSmem<128>::bytes)) != cudaSuccess) return e;
    k_out<128><<<grid, 256, OutSmem<128>::bytes, stream>>>(s.H, s.H / s.Hk, q, k, v_new, hb,
                                                           gcum, scale, o, chunks, n_chunks, vec);
  }
  return cudaGetLastError();
}

}  // namespace gdr

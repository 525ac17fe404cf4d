// gdr_bwd.cu -- backward of the chunked gated delta rule: dq, dk, dv, dg, dbeta, dh0 from
// dL/do and dL/dht.  Shared-memory operand tiles in bf16 where their values are bf16
// (inputs and the bf16 intermediates) and fp32 otherwise; the dense products run on the
// tensor pipe as warp tiles (tf32 in, fp32 accumulate, gdr_mma.cuh), the rest in fp32 SIMT.
//
// The pages describe a training backend whose backward is bit-reproducible and
// tolerates length-0 segments ("Findings from integrating FlashQLA's Blackwell GDN
// kernels into a JAX trainer", intro and section 2) and print no backward formula;
// what follows is the gradient of the chunk form the forward evaluates.  Per chunk of
// 64 tokens (chunk-local i, j; G the chunk-local cumulative gate, C the chunk's last
// token, Gam_ij = e^{G_i - G_j} for j <= i, S_0 the state entering the chunk):
//
//   forward   A = strictly-lower(diag(beta) (K K^T) o Gam),  T = (I + A)^-1
//             U = T diag(beta) V,   W = T diag(beta e^G) K,   V' = U - W S_0
//             O = scale [diag(e^G) Q S_0 + ((Q K^T) o Gam) V']
//             S_C = e^{G_C} S_0 + (diag(e^{G_C - G}) K)^T V'
//
//   backward  (dO given; dS_C the gradient of the state leaving the chunk)
//     dV'  = scale ((Q K^T) o Gam)^T dO + diag(e^{G_C - G}) K dS_C
//     dS_0 = e^{G_C} dS_C + scale Q^T diag(e^G) dO - W^T dV'        (the reverse scan)
//     dQ   = scale diag(e^G) dO S_0^T + E K,   E = scale (dO V'^T) o Gam (j <= i)
//     dK  += E^T Q + diag(e^{G_C - G}) V' dS_C^T
//     dW   = -dV' S_0^T;  dU = dV'
//     dV   = diag(beta) T^T dU;          dbeta += rowsum(V o T^T dU)
//     dK  += diag(beta e^G) T^T dW;      dbeta += e^G rowsum(K o T^T dW)
//     dT   = dU (diag(beta) V)^T + dW (diag(beta e^G) K)^T,  dA = -T^T dT T^T (i > j)
//     dK  += B K + B^T K,  B_ij = dA_ij beta_i Gam_ij;  dbeta_i += sum_j dA_ij Gam_ij k_i.k_j
//     dG   collects every e^{G} factor above; dg = reverse cumulative sum of dG in the chunk
//
// Kernels, in launch order (the forward recompute reuses the staged stage 1 and 2):
//   k_bwd_dv_intra  dV' intra-chunk part                      (chunk, head, 64 columns)
//   k_bwd_scan      dS_C per chunk, dV' total, dh0            (segment, head, 32 or 64 columns)
//   k_bwd_sgrad     the S_0 / dS_C products: dQ, dK, dW parts (chunk, head, 64 key rows)
//   k_bwd_intra     E, the intra-chunk parts of dQ, dK, dG    (chunk, head)
//   k_bwd_wy        the WY / solve backward, dv, dbeta, dg    (chunk, head)
//   k_bwd_heads     per-value-head dq, dk summed over grouped heads, in head order
// Every output element is written by one thread per kernel, in a fixed order: the
// result is bit-identical from run to run (no atomics).
#include "gdr_bwd.cuh"
#include "gdr_mma.cuh"
#include "gdr_sched.cuh"

namespace gdr {
namespace {

// ---------------------------------------------------------------- dV' intra part
template <int D>
struct DvIntraSmem {  // q, k, dO stay bf16 (as in memory)
  static constexpr int kLd = ld_bf16(D), kLdD = ld_bf16(64), kLdP = ld_cols(64);
  static constexpr size_t f32 = 64 * kLdP + 64;  // floats
  static constexpr size_t bytes = sizeof(float) * f32 + sizeof(__nv_bfloat16) * (2 * 64 * kLd + 64 * kLdD);
};

template <int D>
__global__ void __launch_bounds__(kChunkThreads)
    k_bwd_dv_intra(int32_t group, View q, View k, View dout, View gcum, float scale, View dvp,
                   const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks,
                   bool vec) {
  extern __shared__ float sm[];
  constexpr int L = DvIntraSmem<D>::kLd, LD = DvIntraSmem<D>::kLdD, LP = DvIntraSmem<D>::kLdP;
  const int cid = blockIdx.x, h = blockIdx.y, cb = blockIdx.z * 64, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *P = sm, *G = P + 64 * LP;
  __nv_bfloat16 *Qs = reinterpret_cast<__nv_bfloat16 *>(sm + DvIntraSmem<D>::f32), *Ks = Qs + 64 * L,
                *Ds = Ks + 64 * L;
  tile_bf16_raw<64, D, kChunkThreads>(Qs, L, bf_row(q, t0, hk), q.st, len, vec);
  tile_bf16_raw<64, D, kChunkThreads>(Ks, L, bf_row(k, t0, hk), k.st, len, vec);
  tile_bf16_raw<64, 64, kChunkThreads>(Ds, LD, bf_row(dout, t0, h) + cb, dout.st, len, vec);
  if (tid < 64) G[tid] = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
  __syncthreads();
  const int warp = tid >> 5;
  // P = (Q K^T) o Gam (j <= i): 32 tiles of 16 x 8, four per warp
  {
    const int m0 = ((warp * kTPW) >> 3) * 16, nb = ((warp * kTPW) & 7) * 8;
    float accs[kTPW][4] = {};
    mma_16xN<kTPW>(accs, SMatH{Qs, L, 1}, m0, SMatH{Ks, 1, L}, nb, 0, D);
#pragma unroll
    for (int b = 0; b < kTPW; ++b) {
      const int n0 = nb + 8 * b;
      float(&acc)[4] = accs[b];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = acc_row(m0, e), c = acc_col(n0, e);
        P[r * LP + c] = (c <= r && r < len) ? expf(G[r] - G[c]) * acc[e] : 0.f;
      }
    }
  }
  __syncthreads();
  // dV'_intra = scale P^T dO (this block's 64 value columns)
  float *out = reinterpret_cast<float *>(dvp.p);
  {
    const int m0 = ((warp * kTPW) >> 3) * 16, nb = ((warp * kTPW) & 7) * 8;
    float accs[kTPW][4] = {};
    mma_16xN<kTPW>(accs, SMat{P, 1, LP}, m0, SMatH{Ds, LD, 1}, nb, 0, 64);
#pragma unroll
    for (int b = 0; b < kTPW; ++b) {
      const int n0 = nb + 8 * b;
      float(&acc)[4] = accs[b];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = acc_row(m0, e), c = acc_col(n0, e);
        if (r < len) out[(t0 + r) * dvp.st + h * dvp.sh + cb + c] = scale * acc[e];
      }
    }
  }
}

// ---------------------------------------------------------------- reverse state scan

template <int D, int kScanCols>
struct BwdScanSmem {  // K, W and Q stay bf16 (as in memory)
  static constexpr int kLdK = ld_bf16(D), kLdQ = ld_bf16(D), kLdC = ld_cols(kScanCols);
  static constexpr size_t f32 = D * kLdC + 2 * 64 * kLdC + 3 * 64;  // floats
  static constexpr size_t bytes =
      sizeof(float) * f32 + sizeof(__nv_bfloat16) * (64 * kLdK + 2 * 64 * kLdQ);
};

// kScanCols value columns per block, kScanCols / 8 warps
template <int D, int kScanCols>
__global__ void __launch_bounds__(kScanCols * 4)
    k_bwd_scan(int32_t H, int32_t group, View q, View k, View w, View dout, View gcum,
               float scale, const float *dht, View dvp, float *dh, float *dh0,
               const SegInfo *__restrict__ seg, const int32_t *__restrict__ order, bool vec) {
  extern __shared__ float sm[];
  using Sm = BwdScanSmem<D, kScanCols>;
  constexpr int LK = Sm::kLdK, LQ = Sm::kLdQ, LC = Sm::kLdC;
  constexpr int NT = kScanCols * 4, NW = kScanCols / 8, CT = kScanCols / 8;  // threads, warps, column tiles
  // one flat grid, head fastest, then column block, then segment rank: the longest
  // segments are dispatched first (a flat x extent allows any segment count)
  const int64_t bid = blockIdx.x, Z = D / kScanCols;
  const int h = (int)(bid % H), n = order[bid / H / Z];
  const int jb = (int)((bid / H) % Z) * kScanCols, tid = threadIdx.x;
  const int hk = h / group;
  const SegInfo si = seg[n];
  float *dS = sm, *Dos = dS + D * LC, *Vd = Dos + 64 * LC, *G = Vd + 64 * LC, *Dec = G + 64,
        *EG = Dec + 64;
  __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(sm + Sm::f32), *Ws = Ks + 64 * LK,
                *Qs = Ws + 64 * LQ;
  const int64_t sbase = ((int64_t)n * H + h) * D * D;
  float *dvt = reinterpret_cast<float *>(dvp.p);
  for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
    const int d = idx / kScanCols, j = idx % kScanCols;
    dS[d * LC + j] = dht ? dht[sbase + (int64_t)d * D + jb + j] : 0.f;
  }
  for (int c = si.n_chunks - 1; c >= 0; --c) {
    const int64_t cid = si.chunk_off + c;
    const int64_t t0 = si.start + (int64_t)c * kChunk;
    const int len = min(kChunk, si.end - (int)t0);
    __syncthreads();
    float *dhc = dh + (cid * H + h) * D * D;
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      dhc[(int64_t)d * D + jb + j] = dS[d * LC + j];
    }
    tile_bf16_raw<64, D, NT>(Ks, LK, bf_row(k, t0, hk), k.st, len, vec);
    tile_bf16_raw<64, D, NT>(Ws, LQ, bf_row(w, t0, h), w.st, len, true);
    tile_bf16_raw<64, D, NT>(Qs, LQ, bf_row(q, t0, hk), q.st, len, vec);
    tile_bf16<64, kScanCols, NT>(Dos, LC, bf_row(dout, t0, h) + jb,
                                  dout.st, len, vec);
    tile_f32<64, kScanCols, NT>(Vd, LC, dvt + t0 * dvp.st + h * dvp.sh + jb, dvp.st, len);
    if (tid < 64) G[tid] = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    __syncthreads();
    const float glast = G[len - 1];
    if (tid < 64) {
      Dec[tid] = tid < len ? expf(glast - G[tid]) : 0.f;
      EG[tid] = tid < len ? expf(G[tid]) : 0.f;
    }
    __syncthreads();
    for (int idx = tid; idx < 64 * kScanCols; idx += blockDim.x)  // dO <- diag(e^G) dO
      Dos[(idx / kScanCols) * LC + idx % kScanCols] *= EG[idx / kScanCols];
    const int warp = tid >> 5;
    // dV' = dV'_intra + diag(e^{G_C - G}) K dS_C: 4 x CT tiles, four per warp
    {
      const int m0 = ((warp * 4) / CT) * 16, nb = ((warp * 4) % CT) * 8;
      float accs[4][4] = {};
      mma_16xN<4>(accs, SMatH{Ks, LK, 1}, m0, SMat{dS, LC, 1}, nb, 0, D);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int n0 = nb + 8 * b;
        float(&acc)[4] = accs[b];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = acc_row(m0, e), j = acc_col(n0, e);
          if (i < len) {
            const float r = Vd[i * LC + j] + Dec[i] * acc[e];
            Vd[i * LC + j] = r;
            dvt[(t0 + i) * dvp.st + h * dvp.sh + jb + j] = r;
          }
        }
      }
    }
    __syncthreads();
    // dS_0 = e^{G_C} dS_C + scale Q^T diag(e^G) dO - W^T dV': D/16 x CT tiles
    const float eg = expf(glast);
    static_assert(NW == CT, "one column tile per warp");
    {
      // warp w: every row tile of column tile w, in two halves (fewer live accumulators)
      const int n0 = warp * 8;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        constexpr int MB = D / 32;
        const int m0 = half * (D / 2);
        float inj[MB][4] = {}, corr[MB][4] = {};
        mma_Mx8<MB>(inj, SMatH{Qs, 1, LQ}, m0, SMat{Dos, LC, 1}, n0, 0, 64);
        mma_Mx8<MB>(corr, SMatH{Ws, 1, LQ}, m0, SMat{Vd, LC, 1}, n0, 0, 64);
#pragma unroll
        for (int r = 0; r < MB; ++r)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = acc_row(m0 + 16 * r, e), j = acc_col(n0, e);
            dS[d * LC + j] = eg * dS[d * LC + j] + scale * inj[r][e] - corr[r][e];
          }
      }
    }
  }
  if (dh0) {
    __syncthreads();
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      dh0[sbase + (int64_t)d * D + jb + j] = dS[d * LC + j];
    }
  }
}

// ---------------------------------------------------------------- products with S_0, dS_C
constexpr int kSRows = 64;  // key rows of S_0 / dS_C per block

// The products reduce over the value dimension, taken 64 columns at a time: per pass
// S_0, dO, V' as bf16 (their values are bf16) and dS_C, dV' as fp32, 63 KB, so two
// blocks fit on an SM.
constexpr int kSCols = 64;
struct SgradSmem {
  static constexpr int kLdB = ld_bf16(kSCols), kLdF = ld_rows(kSCols);
  static constexpr size_t f32 = (kSRows + 64) * kLdF + 2 * 64 + kWarps;  // floats
  static constexpr size_t bytes =
      sizeof(float) * f32 + sizeof(__nv_bfloat16) * (kSRows + 2 * 64) * kLdB;
};

template <int D>
__global__ void __launch_bounds__(kChunkThreads, 2)
    k_bwd_sgrad(View dout, View v_new, View gcum, float scale, const __nv_bfloat16 *hbuf,
                const float *dh, View dvp, View dqh, View dkh, View dw, float *sdot,
                const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks,
                int32_t H, bool vec) {
  extern __shared__ float sm[];
  constexpr int LB = SgradSmem::kLdB, LF = SgradSmem::kLdF;
  const int cid = blockIdx.x, h = blockIdx.y, rb = blockIdx.z * kSRows, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len;
  const int64_t t0 = ci.start;
  float *dS = sm, *dV = dS + kSRows * LF, *Dec = dV + 64 * LF, *EG = Dec + 64, *red = EG + 64;
  __nv_bfloat16 *S0 = reinterpret_cast<__nv_bfloat16 *>(sm + SgradSmem::f32);
  __nv_bfloat16 *Dos = S0 + kSRows * LB, *Vp = Dos + 64 * LB;
  const __nv_bfloat16 *hc = hbuf + ((int64_t)cid * H + h) * D * D + (int64_t)rb * D;
  const float *dhc = dh + ((int64_t)cid * H + h) * D * D + (int64_t)rb * D;
  const float *dvt = reinterpret_cast<const float *>(dvp.p) + t0 * dvp.st + h * dvp.sh;
  if (tid < 64) {
    const float gi = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    const float gl = ldf(gcum.p, (t0 + len - 1) * gcum.st + h * gcum.sh);
    Dec[tid] = tid < len ? expf(gl - gi) : 0.f;
    EG[tid] = tid < len ? expf(gi) : 0.f;
  }
  // 64 x kSRows outputs of each product: 32 tiles, kTPW per warp, accumulated over the
  // passes; <dS_C, S_0> over this block's key rows on the way
  const int warp = tid >> 5;
  const int m0 = ((warp * kTPW) >> 3) * 16, nb = ((warp * kTPW) & 7) * 8;
  float aqs[kTPW][4] = {}, aks[kTPW][4] = {}, aws[kTPW][4] = {};
  float part = 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += kSCols) {
    if (c0 > 0) __syncthreads();  // the previous pass has read its tiles
    tile_bf16_raw<kSRows, kSCols, kChunkThreads>(S0, LB, hc + c0, D, kSRows, true);
    tile_f32<kSRows, kSCols, kChunkThreads>(dS, LF, dhc + c0, D, kSRows);
    tile_bf16_raw<64, kSCols, kChunkThreads>(Dos, LB, bf_row(dout, t0, h) + c0, dout.st, len, vec);
    tile_bf16_raw<64, kSCols, kChunkThreads>(Vp, LB, bf_row(v_new, t0, h) + c0, v_new.st, len, true);
    tile_f32<64, kSCols, kChunkThreads>(dV, LF, dvt + c0, dvp.st, len);
    __syncthreads();
    mma_16xN<kTPW>(aqs, SMatH{Dos, LB, 1}, m0, SMatH{S0, 1, LB}, nb, 0, kSCols);
    mma_16xN<kTPW>(aks, SMatH{Vp, LB, 1}, m0, SMat{dS, 1, LF}, nb, 0, kSCols);
    mma_16xN<kTPW>(aws, SMat{dV, LF, 1}, m0, SMatH{S0, 1, LB}, nb, 0, kSCols);
    for (int idx = tid; idx < kSRows * kSCols; idx += blockDim.x) {
      const int r = idx / kSCols, j = idx % kSCols;
      part += dS[r * LF + j] * __bfloat162float(S0[r * LB + j]);
    }
  }
  float *q_out = reinterpret_cast<float *>(dqh.p), *k_out = reinterpret_cast<float *>(dkh.p);
  float *w_out = reinterpret_cast<float *>(dw.p);
#pragma unroll
  for (int b = 0; b < kTPW; ++b) {
    const int n0 = nb + 8 * b;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = acc_row(m0, e), r = acc_col(n0, e);
      if (i < len) {
        q_out[(t0 + i) * dqh.st + h * dqh.sh + rb + r] = scale * EG[i] * aqs[b][e];
        k_out[(t0 + i) * dkh.st + h * dkh.sh + rb + r] = Dec[i] * aks[b][e];
        w_out[(t0 + i) * dw.st + h * dw.sh + rb + r] = -aws[b][e];
      }
    }
  }
  // the per-thread parts summed in a fixed order: a shuffle tree in each warp, then the
  // warps' sums in warp order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((tid & 31) == 0) red[warp] = part;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += red[w];
    sdot[((int64_t)cid * H + h) * (D / kSRows) + blockIdx.z] = t;
  }
}

// ---------------------------------------------------------------- intra-chunk terms
template <int D>
struct IntraSmem {  // q, k, dO, V' stay bf16 (as in memory): two blocks fit on an SM
  static constexpr int kLd = ld_bf16(D), kLdE = ld_rows(64);
  static constexpr size_t f32 = 2 * 64 * kLdE + (3 + 2 * kQ) * 64;  // floats
  static constexpr size_t bytes = sizeof(float) * f32 + sizeof(__nv_bfloat16) * 4 * 64 * kLd;
};

// Warp w owns rows 16 (w % 4) .. +16 and column group w / 4 (of kQ) of the 64 x D
// products; row sums go through a shuffle inside the tile, then kQ per-warp partials
// added in a fixed order.
template <int D>
__global__ void __launch_bounds__(kChunkThreads, 2)
    k_bwd_intra(int32_t group, View q, View k, View dout, View v_new, View gcum, float scale,
                View dqh, View dkh, float *dga, const ChunkInfo *__restrict__ chunks,
                const int32_t *__restrict__ n_chunks, int32_t H, bool vec) {
  extern __shared__ float sm[];
  constexpr int L = IntraSmem<D>::kLd, LE = IntraSmem<D>::kLdE;
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *E = sm, *R = E + 64 * LE, *G = R + 64 * LE, *rowR = G + 64, *colR = rowR + 64;
  float *aP = colR + 64, *cP = aP + kQ * 64;  // [kQ][64] partial row sums
  __nv_bfloat16 *Qs = reinterpret_cast<__nv_bfloat16 *>(sm + IntraSmem<D>::f32);
  __nv_bfloat16 *Ks = Qs + 64 * L, *Dos = Ks + 64 * L, *Vp = Dos + 64 * L;
  tile_bf16_raw<64, D, kChunkThreads>(Qs, L, bf_row(q, t0, hk), q.st, len, vec);
  tile_bf16_raw<64, D, kChunkThreads>(Ks, L, bf_row(k, t0, hk), k.st, len, vec);
  tile_bf16_raw<64, D, kChunkThreads>(Dos, L, bf_row(dout, t0, h), dout.st, len, vec);
  tile_bf16_raw<64, D, kChunkThreads>(Vp, L, bf_row(v_new, t0, h), v_new.st, len, true);
  if (tid < 64) G[tid] = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
  const int warp = tid >> 5;
  // this thread's elements of the dQ / dK accumulators (written by k_bwd_sgrad), loaded
  // now so that the loads overlap the products below
  float *q_out = reinterpret_cast<float *>(dqh.p), *k_out = reinterpret_cast<float *>(dkh.p);
  const int m0 = (warp & 3) * 16, cg = warp >> 2;
  constexpr int kCT = D / (8 * kQ);  // column tiles per warp
  float qpre[kCT][4], kpre[kCT][4];
#pragma unroll
  for (int c = 0; c < kCT; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = acc_row(m0, e), d = acc_col((cg * kCT + c) * 8, e);
      qpre[c][e] = i < len ? q_out[(t0 + i) * dqh.st + h * dqh.sh + d] : 0.f;
      kpre[c][e] = i < len ? k_out[(t0 + i) * dkh.st + h * dkh.sh + d] : 0.f;
    }
  __syncthreads();
  // E_ij = scale (do_i . v'_j) Gam_ij and R_ij = E_ij (q_i . k_j), j <= i
  {
    const int m0 = ((warp * kTPW) >> 3) * 16, nb = ((warp * kTPW) & 7) * 8;
    float dvs[kTPW][4] = {}, qks[kTPW][4] = {};
    mma_16xN<kTPW>(dvs, SMatH{Dos, L, 1}, m0, SMatH{Vp, 1, L}, nb, 0, D);
    mma_16xN<kTPW>(qks, SMatH{Qs, L, 1}, m0, SMatH{Ks, 1, L}, nb, 0, D);
#pragma unroll
    for (int b = 0; b < kTPW; ++b) {
      const int n0 = nb + 8 * b;
      float(&dv)[4] = dvs[b];
      float(&qk)[4] = qks[b];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = acc_row(m0, e), j = acc_col(n0, e);
        const float ev = (j <= i && i < len) ? scale * dv[e] * expf(G[i] - G[j]) : 0.f;
        E[i * LE + j] = ev;
        R[i * LE + j] = ev * qk[e];
      }
    }
  }
  __syncthreads();
  if (tid < 64) {
    float s = 0.f;
    for (int j = 0; j < 64; ++j) s += R[tid * LE + j];
    rowR[tid] = s;
  } else if (tid < 128) {
    const int j = tid - 64;
    float s = 0.f;
    for (int i = 0; i < 64; ++i) s += R[i * LE + j];
    colR[j] = s;
  }
  // dQ += E K, dK += E^T Q; a_i = q_i . dQ_inter_i and c_i = k_i . dK_state_i on the way
  float ap[2] = {0.f, 0.f}, cp[2] = {0.f, 0.f};
#pragma unroll
  for (int c = 0; c < kCT; ++c) {
    const int n0 = (cg * kCT + c) * 8;
    float dq[4] = {0.f, 0.f, 0.f, 0.f}, dk[4] = {0.f, 0.f, 0.f, 0.f};
    mma_16x8(dq, SMat{E, LE, 1}, m0, SMatH{Ks, L, 1}, n0, 0, 64);
    mma_16x8(dk, SMat{E, 1, LE}, m0, SMatH{Qs, L, 1}, n0, 0, 64);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = acc_row(m0, e), d = acc_col(n0, e);
      if (i < len) {
        ap[e >> 1] += __bfloat162float(Qs[i * L + d]) * qpre[c][e];
        cp[e >> 1] += __bfloat162float(Ks[i * L + d]) * kpre[c][e];
        q_out[(t0 + i) * dqh.st + h * dqh.sh + d] = qpre[c][e] + dq[e];
        k_out[(t0 + i) * dkh.st + h * dkh.sh + d] = kpre[c][e] + dk[e];
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    ap[r] += __shfl_xor_sync(0xffffffffu, ap[r], 1);
    ap[r] += __shfl_xor_sync(0xffffffffu, ap[r], 2);
    cp[r] += __shfl_xor_sync(0xffffffffu, cp[r], 1);
    cp[r] += __shfl_xor_sync(0xffffffffu, cp[r], 2);
  }
  if ((tid & 3) == 0) {
    const int r0 = m0 + ((tid & 31) >> 2);
    aP[cg * 64 + r0] = ap[0];
    aP[cg * 64 + r0 + 8] = ap[1];
    cP[cg * 64 + r0] = cp[0];
    cP[cg * 64 + r0 + 8] = cp[1];
  }
  __syncthreads();
  // dG from the output (e^G on S_0, Gam) and from the state's e^{G_C - G_i} factors;
  // the e^{G_C} S_0 term is added by k_bwd_wy
  if (tid < len) {
    float a_t = 0.f, c_t = 0.f;
    for (int q = 0; q < kQ; ++q) {
      a_t += aP[q * 64 + tid];
      c_t += cP[q * 64 + tid];
    }
    float v = a_t - c_t + rowR[tid] - colR[tid];
    if (tid == len - 1) {
      float sc = 0.f;
      for (int r = 0; r < len; ++r)
        for (int q = 0; q < kQ; ++q) sc += cP[q * 64 + r];
      v += sc;
    }
    dga[(t0 + tid) * H + h] = v;
  }
}

// ---------------------------------------------------------------- WY / solve backward
// The products that reduce over (or produce) the value dimension take it 64 columns at a
// time, from tiles reloaded per pass (K, V bf16 as in memory; dV', dW fp32); the key
// products K K^T stay in registers in the tile layout that dA has later, so the block
// holds only the 64-column tiles and three 64 x 64 fp32 matrices: 111 KB, two blocks on
// an SM.  The solve's scratch reuses the pass tiles.
constexpr int kWyCols = 64;
struct WySmem {
  static constexpr int kLdB = ld_bf16(kWyCols), kLdF = ld_rows(kWyCols), kLdT = ld_cols(64);
  static constexpr size_t pass_bytes =
      sizeof(__nv_bfloat16) * 2 * 64 * kLdB + sizeof(float) * 2 * 64 * kLdF;
  static constexpr size_t f32 = 3 * 64 * kLdT + 5 * 64 + 4 * kQ * 64;  // floats after the pass tiles
  static constexpr size_t bytes = pass_bytes + sizeof(float) * f32;
  static_assert(pass_bytes % 16 == 0 && pass_bytes >= sizeof(float) * kSolveScratch, "layout");
};

template <int D>
__global__ void __launch_bounds__(kChunkThreads, 2)
    k_bwd_wy(int32_t group, View k, View v, View beta, View gcum, View dvp, View dw, View dkh,
             const float *dga, const float *sdot, const float *tg, View dv_out, View dbeta_out,
             View dg_out, const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks,
             int32_t H, bool vec) {
  extern __shared__ float sm[];
  constexpr int LB = WySmem::kLdB, LF = WySmem::kLdF, LT = WySmem::kLdT;
  static_assert(kQ == 4 && kTPW == 2, "tile mapping below");
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  uint8_t *base = reinterpret_cast<uint8_t *>(sm);
  __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(base), *Vs = Ks + 64 * LB;
  float *dVs = reinterpret_cast<float *>(base + sizeof(__nv_bfloat16) * 2 * 64 * LB);
  float *dWs = dVs + 64 * LF;
  float *scratch = reinterpret_cast<float *>(base);  // during the solve only
  float *Tm = reinterpret_cast<float *>(base + WySmem::pass_bytes), *dT = Tm + 64 * LT,
        *X = dT + 64 * LT;
  float *G = X + 64 * LT, *B = G + 64, *BG = B + 64, *EGv = BG + 64, *dGt = EGv + 64;
  float *baP = dGt + 64, *bbP = baP + kQ * 64;    // [kQ][64] partial row sums (dbeta)
  float *rowP = bbP + kQ * 64, *colP = rowP + kQ * 64;  // [4][64] partial sums of P
  const float *dvt = reinterpret_cast<const float *>(dvp.p) + t0 * dvp.st + h * dvp.sh;
  const float *dwt = reinterpret_cast<const float *>(dw.p) + t0 * dw.st + h * dw.sh;
  auto load_pass = [&](int c0) {
    tile_bf16_raw<64, kWyCols, kChunkThreads>(Ks, LB, bf_row(k, t0, hk) + c0, k.st, len, vec);
    tile_bf16_raw<64, kWyCols, kChunkThreads>(Vs, LB, bf_row(v, t0, h) + c0, v.st, len, vec);
    tile_f32<64, kWyCols, kChunkThreads>(dVs, LF, dvt + c0, dvp.st, len);
    tile_f32<64, kWyCols, kChunkThreads>(dWs, LF, dwt + c0, dw.st, len);
  };
  if (tid < 64) {
    const bool in = tid < len;
    const float gi = in ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    const float bi = in ? ldbf(beta.p, (t0 + tid) * beta.st + h * beta.sh) : 0.f;
    const float ei = in ? expf(gi) : 0.f;
    G[tid] = gi;
    B[tid] = bi;
    EGv[tid] = ei;
    BG[tid] = bi * ei;
  }
  const int warp = tid >> 5;
  // 64 x 64 products: warp w owns tiles (m0, nb) and (m0, nb + 8)
  const int tm0 = ((warp * kTPW) >> 3) * 16, tnb = ((warp * kTPW) & 7) * 8;
  // raw key products k_i . k_j, dU_i . v_j and dW_i . k_j over the value passes
  float kk[kTPW][4] = {}, du[kTPW][4] = {}, dwk[kTPW][4] = {};
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += kWyCols) {
    if (c0 > 0) __syncthreads();
    load_pass(c0);
    __syncthreads();
    mma_16xN<kTPW>(kk, SMatH{Ks, LB, 1}, tm0, SMatH{Ks, 1, LB}, tnb, 0, kWyCols);
    mma_16xN<kTPW>(du, SMat{dVs, LF, 1}, tm0, SMatH{Vs, 1, LB}, tnb, 0, kWyCols);
    mma_16xN<kTPW>(dwk, SMat{dWs, LF, 1}, tm0, SMatH{Ks, 1, LB}, tnb, 0, kWyCols);
  }
  // A_ij = beta_i Gam_ij k_i . k_j into X (the solve's input) and dT_ij = beta_j (dU_i . v_j)
  // + beta_j e^{G_j} (dW_i . k_j), i > j (the only part dA needs)
#pragma unroll
  for (int b = 0; b < kTPW; ++b)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = acc_row(tm0, e), j = acc_col(tnb + 8 * b, e);
      const bool lo = j < i && i < len;
      kk[b][e] = lo ? kk[b][e] : 0.f;
      X[i * LT + j] = lo ? B[i] * expf(G[i] - G[j]) * kk[b][e] : 0.f;
      dT[i * LT + j] = lo ? B[j] * du[b][e] + BG[j] * dwk[b][e] : 0.f;
    }
  __syncthreads();  // also: every warp is done with the pass tiles (the solve's scratch)
  if (tg) {  // T = (I + A)^-1 as the fused recompute formed it
    const float *tc = tg + ((int64_t)cid * H + h) * 4096;
    for (int idx = tid; idx < 64 * 16; idx += kChunkThreads) {
      const int i = idx >> 4, j = (idx & 15) * 4;
      const float4 x = *reinterpret_cast<const float4 *>(tc + i * 64 + j);
      Tm[i * LT + j] = x.x;
      Tm[i * LT + j + 1] = x.y;
      Tm[i * LT + j + 2] = x.z;
      Tm[i * LT + j + 3] = x.w;
    }
    __syncthreads();
  } else {
    solve_unit_lower64(X, LT, Tm, LT, scratch, kChunkThreads, 0);  // T = (I + A)^-1
  }
  // X = dT T^T
  {
    float accs[kTPW][4] = {};
    mma_16xN<kTPW>(accs, SMat{dT, LT, 1}, tm0, SMat{Tm, 1, LT}, tnb, 0, 64);
#pragma unroll
    for (int b = 0; b < kTPW; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) X[acc_row(tm0, e) * LT + acc_col(tnb + 8 * b, e)] = accs[b][e];
  }
  __syncthreads();
  // dA = -T^T X (i > j), in registers; P_ij = dA_ij Gam_ij (k_i . k_j) gives the dbeta term
  // (row sums), and with B_ij = dA_ij beta_i Gam_ij the dG terms sum_j B_ij k_i.k_j =
  // beta_i (row sum of P) and sum_i B_ij k_i.k_j (column sums of beta_i P_ij).  X then
  // holds B + B^T (B is strictly lower: the owner of (i, j), i > j, writes both halves,
  // the diagonal is zero), which is symmetric, so (B + B^T) K is one product.
  float dA[kTPW][4] = {};
  mma_16xN<kTPW>(dA, SMat{Tm, 1, LT}, tm0, SMat{X, LT, 1}, tnb, 0, 64);
  __syncthreads();  // every warp has read X
  {
    float rs[2] = {0.f, 0.f}, cs[kTPW][2] = {};
#pragma unroll
    for (int b = 0; b < kTPW; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = acc_row(tm0, e), j = acc_col(tnb + 8 * b, e);
        const bool lo = j < i && i < len;
        // the decay only where it is a ratio e^{G_i - G_j}, j < i (at most 1 for g <= 0):
        // elsewhere e^{G_i - G_j} can overflow and 0 * inf would be NaN
        const float gam = lo ? expf(G[i] - G[j]) : 0.f;
        const float a = lo ? -dA[b][e] : 0.f;
        const float pij = a * gam * kk[b][e];
        if (j < i) {
          const float bij = a * B[i] * gam;
          X[i * LT + j] = bij;
          X[j * LT + i] = bij;
        } else if (j == i) {
          X[i * LT + j] = 0.f;
        }
        rs[e >> 1] += pij;
        cs[b][e & 1] += B[i] * pij;
      }
    // rows: the four lanes of a row (lane % 4); columns: the eight row groups (lane / 4)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
      rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
    }
#pragma unroll
    for (int b = 0; b < kTPW; ++b)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        cs[b][c] += __shfl_xor_sync(0xffffffffu, cs[b][c], 4);
        cs[b][c] += __shfl_xor_sync(0xffffffffu, cs[b][c], 8);
        cs[b][c] += __shfl_xor_sync(0xffffffffu, cs[b][c], 16);
      }
    const int lane = tid & 31;
    if ((lane & 3) == 0) {
      const int r0 = tm0 + (lane >> 2);
      rowP[(warp & 3) * 64 + r0] = rs[0];
      rowP[(warp & 3) * 64 + r0 + 8] = rs[1];
    }
    if (lane < 4) {
#pragma unroll
      for (int b = 0; b < kTPW; ++b)
#pragma unroll
        for (int c = 0; c < 2; ++c) colP[(warp >> 2) * 64 + tnb + 8 * b + 2 * lane + c] = cs[b][c];
    }
  }
  // per row j, for each value pass: T^T dU, T^T dW, (B + B^T) K; warp w owns rows
  // 16 (w % 4) .. +16 and column group w / 4 of the pass
  float *dvo = reinterpret_cast<float *>(dv_out.p), *dko = reinterpret_cast<float *>(dkh.p);
  const int m0 = (warp & 3) * 16, cg = warp >> 2;
  constexpr int kCT = kWyCols / (8 * kQ);
  float ba[2] = {0.f, 0.f}, bb[2] = {0.f, 0.f};
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += kWyCols) {
    __syncthreads();  // X written (first pass) / the previous pass's tiles read
    // this thread's dK accumulator elements (written by earlier kernels), loaded with the
    // pass's tiles so that the loads overlap
    float kpre[kCT][4];
#pragma unroll
    for (int c = 0; c < kCT; ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = acc_row(m0, e), d = acc_col((cg * kCT + c) * 8, e);
        kpre[c][e] = j < len ? dko[(t0 + j) * dkh.st + h * dkh.sh + c0 + d] : 0.f;
      }
    load_pass(c0);
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kCT; ++c) {
      const int n0 = (cg * kCT + c) * 8;
      float tdu[4] = {0.f, 0.f, 0.f, 0.f}, tdw[4] = {0.f, 0.f, 0.f, 0.f}, kc[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16x8(tdu, SMat{Tm, 1, LT}, m0, SMat{dVs, LF, 1}, n0, 0, 64);
      mma_16x8(tdw, SMat{Tm, 1, LT}, m0, SMat{dWs, LF, 1}, n0, 0, 64);
      mma_16x8(kc, SMat{X, 1, LT}, m0, SMatH{Ks, LB, 1}, n0, 0, 64);  // (B + B^T) K
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = acc_row(m0, e), d = acc_col(n0, e);
        if (j < len) {
          dvo[(t0 + j) * dv_out.st + h * dv_out.sh + c0 + d] = B[j] * tdu[e];
          ba[e >> 1] += __bfloat162float(Vs[j * LB + d]) * tdu[e];
          bb[e >> 1] += __bfloat162float(Ks[j * LB + d]) * tdw[e];
          dko[(t0 + j) * dkh.st + h * dkh.sh + c0 + d] = kpre[c][e] + BG[j] * tdw[e] + kc[e];
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    ba[r] += __shfl_xor_sync(0xffffffffu, ba[r], 1);
    ba[r] += __shfl_xor_sync(0xffffffffu, ba[r], 2);
    bb[r] += __shfl_xor_sync(0xffffffffu, bb[r], 1);
    bb[r] += __shfl_xor_sync(0xffffffffu, bb[r], 2);
  }
  if ((tid & 3) == 0) {
    const int r0 = m0 + ((tid & 31) >> 2);
    baP[cg * 64 + r0] = ba[0];
    baP[cg * 64 + r0 + 8] = ba[1];
    bbP[cg * 64 + r0] = bb[0];
    bbP[cg * 64 + r0 + 8] = bb[1];
  }
  __syncthreads();
  if (tid < len) {
    const int r = tid;
    float dba = 0.f, dbb = 0.f, dbc = 0.f, colq = 0.f;
    for (int q = 0; q < kQ; ++q) {
      dba += baP[q * 64 + r];
      dbb += bbP[q * 64 + r];
    }
    for (int q = 0; q < 4; ++q) {
      dbc += rowP[q * 64 + r];
      colq += colP[q * 64 + r];
    }
    float *dbo = reinterpret_cast<float *>(dbeta_out.p);
    dbo[(t0 + r) * dbeta_out.st + h * dbeta_out.sh] = dba + EGv[r] * dbb + dbc;
    float gt = dga[(t0 + r) * H + h] + BG[r] * dbb + B[r] * dbc - colq;
    if (r == len - 1) {
      float sd = 0.f;
      for (int b = 0; b < D / kSRows; ++b) sd += sdot[((int64_t)cid * H + h) * (D / kSRows) + b];
      gt += EGv[r] * sd;
    }
    dGt[r] = gt;
  }
  __syncthreads();
  if (tid < len) {  // dg = reverse cumulative sum of dG inside the chunk
    float acc = 0.f;
    for (int r = len - 1; r >= tid; --r) acc += dGt[r];
    reinterpret_cast<float *>(dg_out.p)[(t0 + tid) * dg_out.st + h * dg_out.sh] = acc;
  }
}

// ---------------------------------------------------------------- grouped heads
// dq[t, hk] = sum over the value heads of hk (in head order) of dq_h[t, h]; same for dk.
__global__ void k_bwd_heads(int32_t group, int32_t D, View dqh, View dkh, View dq, View dk,
                            const ChunkInfo *__restrict__ chunks,
                            const int32_t *__restrict__ n_chunks) {
  const int cid = blockIdx.x, hk = blockIdx.y;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const float *qh = reinterpret_cast<const float *>(dqh.p), *kh = reinterpret_cast<const float *>(dkh.p);
  float *qo = reinterpret_cast<float *>(dq.p), *ko = reinterpret_cast<float *>(dk.p);
  for (int idx = threadIdx.x; idx < ci.len * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    const int64_t t = ci.start + i;
    float a = 0.f, b = 0.f;
    for (int r = 0; r < group; ++r) {
      const int h = hk * group + r;
      a += qh[t * dqh.st + h * dqh.sh + d];
      b += kh[t * dkh.st + h * dkh.sh + d];
    }
    qo[t * dq.st + hk * dq.sh + d] = a;
    ko[t * dk.st + hk * dk.sh + d] = b;
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Workspace of the backward after the chunk tables (all 256-byte aligned).
struct BwdWs {
  float *gcum;
  void *w, *u, *vnew;
  void *h;
  float *dvp, *dh, *dqh, *dkh, *dw, *dga, *sdot;
  void *fws;    // the fused recompute's scratch (work list)
  float *tmat;  // Tm per chunk and head from the fused recompute [chunk][H][64][64]
  size_t bytes;
};

BwdWs carve_bwd(void *ws, int64_t T, int32_t n_seq, int32_t Hk, int32_t H, int32_t D) {
  BwdWs r{};
  char *p = reinterpret_cast<char *>(ws);
  size_t off = 0;
  auto take = [&](size_t b) {
    char *q = p + off;
    off += align256(b);
    return q;
  };
  const size_t tok = (size_t)T * H, cap = (size_t)chunk_bound(T, n_seq);
  r.gcum = reinterpret_cast<float *>(take(tok * sizeof(float)));
  r.w = take(tok * D * 2);
  r.u = take(tok * D * 2);
  r.vnew = take(tok * D * 2);
  r.h = take(cap * H * D * D * 2);
  r.dvp = reinterpret_cast<float *>(take(tok * D * sizeof(float)));
  r.dh = reinterpret_cast<float *>(take(cap * H * D * D * sizeof(float)));
  if (H != Hk) {
    r.dqh = reinterpret_cast<float *>(take(tok * D * sizeof(float)));
    r.dkh = reinterpret_cast<float *>(take(tok * D * sizeof(float)));
  }
  r.dw = reinterpret_cast<float *>(take(tok * D * sizeof(float)));
  r.dga = reinterpret_cast<float *>(take(tok * sizeof(float)));
  r.sdot = reinterpret_cast<float *>(take(cap * H * (D / kSRows) * sizeof(float)));
  r.fws = take(fused_workspace_bytes(T, n_seq, H));
  r.tmat = reinterpret_cast<float *>(take(cap * H * 64 * 64 * sizeof(float)));
  r.bytes = off;
  return r;
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs &a, const BwdWs &w, cudaStream_t stream) {
  const StageShapes &s = a.s;
  const int32_t group = s.H / s.Hk;
  const int64_t HD = (int64_t)s.H * D;
  const View vw{w.w, HD, D}, vu{w.u, HD, D}, vn{w.vnew, HD, D}, vg{w.gcum, s.H, 1};
  const View vdvp{w.dvp, HD, D}, vdw{w.dw, HD, D};
  const View vdqh = group > 1 ? View{w.dqh, HD, D} : a.dq;
  const View vdkh = group > 1 ? View{w.dkh, HD, D} : a.dk;
  // 16-byte vector loads of the caller's bf16 tensors when their rows allow it
  auto al = [](const View &x) {
    return (reinterpret_cast<uintptr_t>(x.p) & 15) == 0 && x.st % 8 == 0 && x.sh % 8 == 0;
  };
  const bool vec = al(a.q) && al(a.k) && al(a.v) && al(a.dout);
  cudaError_t e;
  // forward recompute: G, W, the chunk states h and V', by the fused forward kernel's
  // backward variant when TMA can load q, k and v; else by the staged stage 1 (G, W, U)
  // and stage 2 (h, V')
  FusedArgs fa{};
  fa.T = s.T;
  fa.n_seq = s.n_seq;
  fa.Hk = s.Hk;
  fa.H = s.H;
  fa.D = D;
  fa.q = a.q.p;
  fa.k = a.k.p;
  fa.v = a.v.p;
  fa.q_st = a.q.st;
  fa.q_sh = a.q.sh;
  fa.k_st = a.k.st;
  fa.k_sh = a.k.sh;
  fa.v_st = a.v.st;
  fa.v_sh = a.v.sh;
  fa.g = reinterpret_cast<const float *>(a.g.p);
  fa.g_st = a.g.st;
  fa.g_sh = a.g.sh;
  fa.beta = a.beta.p;
  fa.b_st = a.beta.st;
  fa.b_sh = a.beta.sh;
  fa.scale = a.scale;
  fa.h0 = a.h0;
  fa.ckpt = Ckpt{nullptr, nullptr, 0};
  fa.bwd.gcum = w.gcum;
  fa.bwd.w = w.w;
  fa.bwd.h = w.h;
  fa.bwd.vnew = w.vnew;
  fa.bwd.tmat = w.tmat;
  fa.seg = a.seg;
  fa.workspace = w.fws;
  bool fused = fused_supported(fa);
  if (fused) {
    e = launch_fused(fa, stream);
    if (e == cudaErrorInvalidValue) {  // a TMA map was refused: the staged recompute
      (void)cudaGetLastError();
      fused = false;
    } else if (e != cudaSuccess) {
      return e;
    }
  }
  if (!fused) {
    if ((e = launch_prep(s, a.k, a.v, a.g, a.beta, vw, vu, vg, a.seg, a.chunks, a.n_chunks,
                         stream)) != cudaSuccess)
      return e;
    if ((e = launch_scan_ordered(s, a.k, vw, vu, vg, a.h0, w.h, vn, nullptr,
                                 Ckpt{nullptr, nullptr, 0}, a.seg, a.order, stream)) != cudaSuccess)
      return e;
  }
  const dim3 gc((unsigned)s.chunk_cap, (unsigned)s.H);
  // dV' intra-chunk part on the tensor cores when TMA can load q, k and dout; the
  // warp-tile kernel otherwise
  e = launch_bwd_dv_intra_tc(a, vg, vdvp, stream);
  if (e == cudaErrorNotSupported) {
    (void)cudaGetLastError();
    if ((e = set_smem(k_bwd_dv_intra<D>, DvIntraSmem<D>::bytes)) != cudaSuccess) return e;
    k_bwd_dv_intra<D><<<dim3(gc.x, gc.y, D / 64), kChunkThreads, DvIntraSmem<D>::bytes, stream>>>(
        group, a.q, a.k, a.dout, vg, a.scale, vdvp, a.chunks, a.n_chunks, vec);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  auto scan = [&](auto kern, int cols, size_t bytes) -> cudaError_t {
    cudaError_t r = set_smem(kern, bytes);
    if (r != cudaSuccess) return r;
    const int64_t blocks = (int64_t)s.H * (D / cols) * s.n_seq;
    kern<<<(unsigned)blocks, cols * 4, bytes, stream>>>(s.H, group, a.q, a.k, vw, a.dout, vg,
                                                       a.scale, a.dht, vdvp, w.dh, a.dh0, a.seg,
                                                       a.order, vec);
    return cudaGetLastError();
  };
  // at d = 128 the 32-column blocks (bf16 operand tiles, 94 KB) fit two to an SM and ran
  // faster than 64-column blocks at one per SM
  const int bcols = D == 128 ? 32 : scan_cols(s.n_seq, s.H, D);
  e = bcols == 64 ? scan(k_bwd_scan<D, 64>, 64, BwdScanSmem<D, 64>::bytes)
                  : scan(k_bwd_scan<D, 32>, 32, BwdScanSmem<D, 32>::bytes);
  if (e != cudaSuccess) return e;
  // the S_0 / dS_C products on the tensor cores when TMA can load dout; the warp-tile
  // kernel otherwise
  e = launch_bwd_sgrad_tc(a, w.h, w.dh, vg, vn, vdvp, vdqh, vdkh, vdw, w.sdot, stream);
  if (e == cudaErrorNotSupported) {
    (void)cudaGetLastError();
    if ((e = set_smem(k_bwd_sgrad<D>, SgradSmem::bytes)) != cudaSuccess) return e;
    k_bwd_sgrad<D><<<dim3(gc.x, gc.y, D / kSRows), kChunkThreads, SgradSmem::bytes, stream>>>(
        a.dout, vn, vg, a.scale, reinterpret_cast<const __nv_bfloat16 *>(w.h), w.dh, vdvp, vdqh,
        vdkh, vdw, w.sdot, a.chunks, a.n_chunks, s.H, vec);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  if ((e = set_smem(k_bwd_intra<D>, IntraSmem<D>::bytes)) != cudaSuccess) return e;
  k_bwd_intra<D><<<gc, kChunkThreads, IntraSmem<D>::bytes, stream>>>(group, a.q, a.k, a.dout, vn, vg,
                                                            a.scale, vdqh, vdkh, w.dga,
                                                            a.chunks, a.n_chunks, s.H, vec);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = set_smem(k_bwd_wy<D>, WySmem::bytes)) != cudaSuccess) return e;
  k_bwd_wy<D><<<gc, kChunkThreads, WySmem::bytes, stream>>>(group, a.k, a.v, a.beta, vg, vdvp, vdw,
                                                      vdkh, w.dga, w.sdot, fused ? w.tmat : nullptr,
                                                      a.dv, a.dbeta, a.dg,
                                                      a.chunks, a.n_chunks, s.H, vec);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (group > 1) {
    k_bwd_heads<<<dim3((unsigned)s.chunk_cap, (unsigned)s.Hk), 256, 0, stream>>>(
        group, D, vdqh, vdkh, a.dq, a.dk, a.chunks, a.n_chunks);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t bwd_work_bytes(int64_t T, int32_t n_seq, int32_t Hk, int32_t H, int32_t D) {
  return carve_bwd(nullptr, T, n_seq, Hk, H, D).bytes;
}

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t stream) {
  const StageShapes &s = a.s;
  if (s.n_seq <= 0) return cudaSuccess;
  const BwdWs w = carve_bwd(a.work, s.T, s.n_seq, s.Hk, s.H, s.D);
  if (s.T == 0 || s.chunk_cap <= 0) {
    // only empty segments: dh0 = dht
    if (a.dh0) {
      const size_t b = sizeof(float) * (size_t)s.n_seq * s.H * s.D * s.D;
      return a.dht ? cudaMemcpyAsync(a.dh0, a.dht, b, cudaMemcpyDeviceToDevice, stream)
                   : cudaMemsetAsync(a.dh0, 0, b, stream);
    }
    return cudaSuccess;
  }
  return s.D == 64 ? launch_bwd_d<64>(a, w, stream) : launch_bwd_d<128>(a, w, stream);
}

}  // namespace gdr

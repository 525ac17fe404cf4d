// gdr_bwd.cu -- backward of the chunked gated delta rule: dq, dk, dv, dg, dbeta, dh0 from
// dL/do and dL/dht.  Plain fp32 SIMT arithmetic over shared-memory tiles.
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
//   k_bwd_scan      dS_C per chunk, dV' total, dh0            (segment, head, 32 columns)
//   k_bwd_sgrad     the S_0 / dS_C products: dQ, dK, dW parts (chunk, head, 32 key rows)
//   k_bwd_intra     E, the intra-chunk parts of dQ, dK, dG    (chunk, head)
//   k_bwd_wy        the WY / solve backward, dv, dbeta, dg    (chunk, head)
//   k_bwd_heads     per-value-head dq, dk summed over grouped heads, in head order
// Every output element is written by one thread per kernel, in a fixed order: the
// result is bit-identical from run to run (no atomics).
#include "gdr_bwd.cuh"

namespace gdr {
namespace {

// ---------------------------------------------------------------- dV' intra part
template <int D>
struct DvIntraSmem {
  static constexpr int kLd = D + 1;
  static constexpr size_t bytes = sizeof(float) * (2 * 64 * kLd + 2 * 64 * 65 + 64);
};

template <int D>
__global__ void __launch_bounds__(256)
    k_bwd_dv_intra(int32_t group, View q, View k, View dout, View gcum, float scale, View dvp,
                   const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks) {
  extern __shared__ float sm[];
  constexpr int L = DvIntraSmem<D>::kLd;
  const int cid = blockIdx.x, h = blockIdx.y, cb = blockIdx.z * 64, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *Qs = sm, *Ks = Qs + 64 * L, *Ds = Ks + 64 * L, *P = Ds + 64 * 65, *G = P + 64 * 65;
  for (int idx = tid; idx < 64 * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    float qv = 0.f, kv = 0.f;
    if (i < len) {
      qv = ldbf(q.p, (t0 + i) * q.st + hk * q.sh + d);
      kv = ldbf(k.p, (t0 + i) * k.st + hk * k.sh + d);
    }
    Qs[i * L + d] = qv;
    Ks[i * L + d] = kv;
  }
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx / 64, c = idx % 64;
    Ds[i * 65 + c] = i < len ? ldbf(dout.p, (t0 + i) * dout.st + h * dout.sh + cb + c) : 0.f;
  }
  if (tid < 64) G[tid] = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
  __syncthreads();
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx / 64, j = idx % 64;
    float pv = 0.f;
    if (j <= i && i < len) {
      float dot = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) dot += Qs[i * L + d] * Ks[j * L + d];
      pv = expf(G[i] - G[j]) * dot;
    }
    P[i * 65 + j] = pv;
  }
  __syncthreads();
  float *out = reinterpret_cast<float *>(dvp.p);
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int j = idx / 64, c = idx % 64;
    if (j >= len) continue;
    float acc = 0.f;
    for (int i = j; i < len; ++i) acc += P[i * 65 + j] * Ds[i * 65 + c];
    out[(t0 + j) * dvp.st + h * dvp.sh + cb + c] = scale * acc;
  }
}

// ---------------------------------------------------------------- reverse state scan
constexpr int kScanCols = 32;

template <int D>
struct BwdScanSmem {
  static constexpr int kLd = D + 1;
  static constexpr size_t bytes =
      sizeof(float) * (D * 33 + 3 * 64 * kLd + 2 * 64 * 33 + 3 * 64);
};

template <int D>
__global__ void __launch_bounds__(128)
    k_bwd_scan(int32_t H, int32_t group, View q, View k, View w, View dout, View gcum,
               float scale, const float *dht, View dvp, float *dh, float *dh0,
               const SegInfo *__restrict__ seg) {
  extern __shared__ float sm[];
  constexpr int L = BwdScanSmem<D>::kLd;
  const int n = blockIdx.x, h = blockIdx.y, jb = blockIdx.z * kScanCols, tid = threadIdx.x;
  const int hk = h / group;
  const SegInfo si = seg[n];
  float *dS = sm, *Ks = dS + D * 33, *Ws = Ks + 64 * L, *Qs = Ws + 64 * L, *Dos = Qs + 64 * L;
  float *Vd = Dos + 64 * 33, *G = Vd + 64 * 33, *Dec = G + 64, *EG = Dec + 64;
  const int64_t sbase = ((int64_t)n * H + h) * D * D;
  float *dvt = reinterpret_cast<float *>(dvp.p);
  for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
    const int d = idx / kScanCols, j = idx % kScanCols;
    dS[d * 33 + j] = dht ? dht[sbase + (int64_t)d * D + jb + j] : 0.f;
  }
  for (int c = si.n_chunks - 1; c >= 0; --c) {
    const int64_t cid = si.chunk_off + c;
    const int64_t t0 = si.start + (int64_t)c * kChunk;
    const int len = min(kChunk, si.end - (int)t0);
    __syncthreads();
    float *dhc = dh + (cid * H + h) * D * D;
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      dhc[(int64_t)d * D + jb + j] = dS[d * 33 + j];
    }
    for (int idx = tid; idx < 64 * D; idx += blockDim.x) {
      const int i = idx / D, d = idx % D;
      float kv = 0.f, wv = 0.f, qv = 0.f;
      if (i < len) {
        kv = ldbf(k.p, (t0 + i) * k.st + hk * k.sh + d);
        wv = ldbf(w.p, (t0 + i) * w.st + h * w.sh + d);
        qv = ldbf(q.p, (t0 + i) * q.st + hk * q.sh + d);
      }
      Ks[i * L + d] = kv;
      Ws[i * L + d] = wv;
      Qs[i * L + d] = qv;
    }
    for (int idx = tid; idx < 64 * kScanCols; idx += blockDim.x) {
      const int i = idx / kScanCols, j = idx % kScanCols;
      float dov = 0.f, vd = 0.f;
      if (i < len) {
        dov = ldbf(dout.p, (t0 + i) * dout.st + h * dout.sh + jb + j);
        vd = dvt[(t0 + i) * dvp.st + h * dvp.sh + jb + j];
      }
      Dos[i * 33 + j] = dov;
      Vd[i * 33 + j] = vd;
    }
    if (tid < 64) G[tid] = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    __syncthreads();
    const float glast = G[len - 1];
    if (tid < 64) {
      Dec[tid] = tid < len ? expf(glast - G[tid]) : 0.f;
      EG[tid] = tid < len ? expf(G[tid]) : 0.f;
    }
    __syncthreads();
    // dV' = dV'_intra + diag(e^{G_C - G}) K dS_C
    for (int idx = tid; idx < 64 * kScanCols; idx += blockDim.x) {
      const int i = idx / kScanCols, j = idx % kScanCols;
      if (i >= len) continue;
      float acc = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) acc += Ks[i * L + d] * dS[d * 33 + j];
      const float r = Vd[i * 33 + j] + Dec[i] * acc;
      Vd[i * 33 + j] = r;
      dvt[(t0 + i) * dvp.st + h * dvp.sh + jb + j] = r;
    }
    __syncthreads();
    // dS_0 = e^{G_C} dS_C + scale Q^T diag(e^G) dO - W^T dV'
    const float eg = expf(glast);
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      float inj = 0.f, corr = 0.f;
      for (int i = 0; i < len; ++i) {
        inj += Qs[i * L + d] * EG[i] * Dos[i * 33 + j];
        corr += Ws[i * L + d] * Vd[i * 33 + j];
      }
      dS[d * 33 + j] = eg * dS[d * 33 + j] + scale * inj - corr;
    }
  }
  if (dh0) {
    __syncthreads();
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      dh0[sbase + (int64_t)d * D + jb + j] = dS[d * 33 + j];
    }
  }
}

// ---------------------------------------------------------------- products with S_0, dS_C
constexpr int kSRows = 32;  // key rows of S_0 / dS_C per block

template <int D>
struct SgradSmem {
  static constexpr int kLd = D + 1;
  static constexpr size_t bytes =
      sizeof(float) * (2 * kSRows * kLd + 3 * 64 * kLd + 2 * 64 + 256);
};

template <int D>
__global__ void __launch_bounds__(256)
    k_bwd_sgrad(View dout, View v_new, View gcum, float scale, const __nv_bfloat16 *hbuf,
                const float *dh, View dvp, View dqh, View dkh, View dw, float *sdot,
                const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks,
                int32_t H) {
  extern __shared__ float sm[];
  constexpr int L = SgradSmem<D>::kLd;
  const int cid = blockIdx.x, h = blockIdx.y, rb = blockIdx.z * kSRows, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len;
  const int64_t t0 = ci.start;
  float *S0 = sm, *dS = S0 + kSRows * L, *Dos = dS + kSRows * L, *Vp = Dos + 64 * L;
  float *dV = Vp + 64 * L, *Dec = dV + 64 * L, *EG = Dec + 64, *red = EG + 64;
  const __nv_bfloat16 *hc = hbuf + ((int64_t)cid * H + h) * D * D;
  const float *dhc = dh + ((int64_t)cid * H + h) * D * D;
  for (int idx = tid; idx < kSRows * D; idx += blockDim.x) {
    const int r = idx / D, j = idx % D;
    S0[r * L + j] = __bfloat162float(hc[(int64_t)(rb + r) * D + j]);
    dS[r * L + j] = dhc[(int64_t)(rb + r) * D + j];
  }
  const float *dvt = reinterpret_cast<const float *>(dvp.p);
  for (int idx = tid; idx < 64 * D; idx += blockDim.x) {
    const int i = idx / D, j = idx % D;
    float a = 0.f, b = 0.f, c = 0.f;
    if (i < len) {
      a = ldbf(dout.p, (t0 + i) * dout.st + h * dout.sh + j);
      b = ldbf(v_new.p, (t0 + i) * v_new.st + h * v_new.sh + j);
      c = dvt[(t0 + i) * dvp.st + h * dvp.sh + j];
    }
    Dos[i * L + j] = a;
    Vp[i * L + j] = b;
    dV[i * L + j] = c;
  }
  if (tid < 64) {
    const float gi = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    const float gl = ldf(gcum.p, (t0 + len - 1) * gcum.st + h * gcum.sh);
    Dec[tid] = tid < len ? expf(gl - gi) : 0.f;
    EG[tid] = tid < len ? expf(gi) : 0.f;
  }
  __syncthreads();
  float *q_out = reinterpret_cast<float *>(dqh.p), *k_out = reinterpret_cast<float *>(dkh.p);
  float *w_out = reinterpret_cast<float *>(dw.p);
  for (int idx = tid; idx < 64 * kSRows; idx += blockDim.x) {
    const int i = idx / kSRows, r = idx % kSRows;
    if (i >= len) continue;
    float aq = 0.f, ak = 0.f, aw = 0.f;
#pragma unroll 4
    for (int j = 0; j < D; ++j) {
      aq += Dos[i * L + j] * S0[r * L + j];
      ak += Vp[i * L + j] * dS[r * L + j];
      aw += dV[i * L + j] * S0[r * L + j];
    }
    q_out[(t0 + i) * dqh.st + h * dqh.sh + rb + r] = scale * EG[i] * aq;
    k_out[(t0 + i) * dkh.st + h * dkh.sh + rb + r] = Dec[i] * ak;
    w_out[(t0 + i) * dw.st + h * dw.sh + rb + r] = -aw;
  }
  // <dS_C, S_0> over this block's key rows (fixed-order tree reduction)
  float part = 0.f;
  for (int idx = tid; idx < kSRows * D; idx += blockDim.x) {
    const int r = idx / D, j = idx % D;
    part += dS[r * L + j] * S0[r * L + j];
  }
  red[tid] = part;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (tid < s) red[tid] += red[tid + s];
    __syncthreads();
  }
  if (tid == 0) sdot[((int64_t)cid * H + h) * (D / kSRows) + blockIdx.z] = red[0];
}

// ---------------------------------------------------------------- intra-chunk terms
template <int D>
struct IntraSmem {
  static constexpr int kLd = D + 1;
  static constexpr size_t bytes = sizeof(float) * (4 * 64 * kLd + 2 * 64 * 65 + 5 * 64);
};

// Threads cover a 64 x D tile as (row i = tid / 4, columns tid % 4 + 4 m): the four
// threads of a row are neighbouring lanes, so row sums are two shuffles.
template <int D>
__global__ void __launch_bounds__(256)
    k_bwd_intra(int32_t group, View q, View k, View dout, View v_new, View gcum, float scale,
                View dqh, View dkh, float *dga, const ChunkInfo *__restrict__ chunks,
                const int32_t *__restrict__ n_chunks, int32_t H) {
  extern __shared__ float sm[];
  constexpr int L = IntraSmem<D>::kLd;
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *Qs = sm, *Ks = Qs + 64 * L, *Dos = Ks + 64 * L, *Vp = Dos + 64 * L;
  float *E = Vp + 64 * L, *R = E + 64 * 65, *G = R + 64 * 65, *rowR = G + 64, *colR = rowR + 64;
  float *aS = colR + 64, *cS = aS + 64;
  for (int idx = tid; idx < 64 * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    float a = 0.f, b = 0.f, c = 0.f, e = 0.f;
    if (i < len) {
      a = ldbf(q.p, (t0 + i) * q.st + hk * q.sh + d);
      b = ldbf(k.p, (t0 + i) * k.st + hk * k.sh + d);
      c = ldbf(dout.p, (t0 + i) * dout.st + h * dout.sh + d);
      e = ldbf(v_new.p, (t0 + i) * v_new.st + h * v_new.sh + d);
    }
    Qs[i * L + d] = a;
    Ks[i * L + d] = b;
    Dos[i * L + d] = c;
    Vp[i * L + d] = e;
  }
  if (tid < 64) G[tid] = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
  __syncthreads();
  // E_ij = scale (do_i . v'_j) Gam_ij and R_ij = E_ij (q_i . k_j), j <= i
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx / 64, j = idx % 64;
    float e = 0.f, r = 0.f;
    if (j <= i && i < len) {
      float dv = 0.f, qk = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) {
        dv += Dos[i * L + d] * Vp[j * L + d];
        qk += Qs[i * L + d] * Ks[j * L + d];
      }
      e = scale * dv * expf(G[i] - G[j]);
      r = e * qk;
    }
    E[i * 65 + j] = e;
    R[i * 65 + j] = r;
  }
  __syncthreads();
  if (tid < 64) {
    float s = 0.f;
    for (int j = 0; j < 64; ++j) s += R[tid * 65 + j];
    rowR[tid] = s;
  } else if (tid < 128) {
    const int j = tid - 64;
    float s = 0.f;
    for (int i = 0; i < 64; ++i) s += R[i * 65 + j];
    colR[j] = s;
  }
  const int i = tid >> 2, sub = tid & 3;
  float apart = 0.f, cpart = 0.f;
  float *q_out = reinterpret_cast<float *>(dqh.p), *k_out = reinterpret_cast<float *>(dkh.p);
  if (i < len) {
    for (int d = sub; d < D; d += 4) {
      float dq = 0.f, dk = 0.f;
      for (int j = 0; j <= i; ++j) dq += E[i * 65 + j] * Ks[j * L + d];
      for (int a = i; a < len; ++a) dk += E[a * 65 + i] * Qs[a * L + d];
      const int64_t oq = (t0 + i) * dqh.st + h * dqh.sh + d;
      const int64_t ok = (t0 + i) * dkh.st + h * dkh.sh + d;
      const float q_inter = q_out[oq], k_state = k_out[ok];
      apart += Qs[i * L + d] * q_inter;
      cpart += Ks[i * L + d] * k_state;
      q_out[oq] = q_inter + dq;
      k_out[ok] = k_state + dk;
    }
  }
  apart += __shfl_xor_sync(0xffffffffu, apart, 1);
  apart += __shfl_xor_sync(0xffffffffu, apart, 2);
  cpart += __shfl_xor_sync(0xffffffffu, cpart, 1);
  cpart += __shfl_xor_sync(0xffffffffu, cpart, 2);
  if (sub == 0) {
    aS[i] = apart;
    cS[i] = cpart;
  }
  __syncthreads();
  // dG from the output (e^G on S_0, Gam) and from the state's e^{G_C - G_i} factors;
  // the e^{G_C} S_0 term is added by k_bwd_wy
  if (tid < len) {
    float v = aS[tid] - cS[tid] + rowR[tid] - colR[tid];
    if (tid == len - 1) {
      float sc = 0.f;
      for (int r = 0; r < len; ++r) sc += cS[r];
      v += sc;
    }
    dga[(t0 + tid) * H + h] = v;
  }
}

// ---------------------------------------------------------------- WY / solve backward
template <int D>
struct WySmem {
  static constexpr int kLd = D + 1;
  static constexpr size_t bytes = sizeof(float) * (4 * 64 * kLd + 4 * 64 * 65 + 8 * 64);
};

template <int D>
__global__ void __launch_bounds__(256)
    k_bwd_wy(int32_t group, View k, View v, View beta, View gcum, View dvp, View dw, View dkh,
             const float *dga, const float *sdot, View dv_out, View dbeta_out, View dg_out,
             const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks,
             int32_t H) {
  extern __shared__ float sm[];
  constexpr int L = WySmem<D>::kLd;
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *Ks = sm, *Vs = Ks + 64 * L, *dVs = Vs + 64 * L, *dWs = dVs + 64 * L;
  float *KK = dWs + 64 * L, *Tm = KK + 64 * 65, *dT = Tm + 64 * 65, *X = dT + 64 * 65;
  float *G = X + 64 * 65, *B = G + 64, *BG = B + 64, *EGv = BG + 64, *dGt = EGv + 64;
  float *dbS = dGt + 64, *dgbS = dbS + 64;
  const float *dvt = reinterpret_cast<const float *>(dvp.p), *dwt = reinterpret_cast<const float *>(dw.p);
  for (int idx = tid; idx < 64 * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    float a = 0.f, b = 0.f, c = 0.f, e = 0.f;
    if (i < len) {
      a = ldbf(k.p, (t0 + i) * k.st + hk * k.sh + d);
      b = ldbf(v.p, (t0 + i) * v.st + h * v.sh + d);
      c = dvt[(t0 + i) * dvp.st + h * dvp.sh + d];
      e = dwt[(t0 + i) * dw.st + h * dw.sh + d];
    }
    Ks[i * L + d] = a;
    Vs[i * L + d] = b;
    dVs[i * L + d] = c;
    dWs[i * L + d] = e;
  }
  if (tid < 64) {
    const bool in = tid < len;
    G[tid] = in ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    B[tid] = in ? ldbf(beta.p, (t0 + tid) * beta.st + h * beta.sh) : 0.f;
  }
  __syncthreads();
  if (tid < 64) {
    EGv[tid] = tid < len ? expf(G[tid]) : 0.f;
    BG[tid] = B[tid] * EGv[tid];
  }
  // raw key products k_i . k_j, j < i
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx / 64, j = idx % 64;
    float dot = 0.f;
    if (j < i && i < len) {
#pragma unroll 8
      for (int d = 0; d < D; ++d) dot += Ks[i * L + d] * Ks[j * L + d];
    }
    KK[i * 65 + j] = dot;
    X[i * 65 + j] = (j < i && i < len) ? B[i] * expf(G[i] - G[j]) * dot : 0.f;  // A_ij
  }
  __syncthreads();
  if (tid < 64) {  // column c of T = (I + A)^-1, A_ij = beta_i Gam_ij k_i.k_j
    const int c = tid;
    for (int i = 0; i < 64; ++i) {
      float x = (i == c) ? 1.f : 0.f;
      for (int j = c; j < i; ++j) x -= X[i * 65 + j] * Tm[j * 65 + c];
      Tm[i * 65 + c] = x;
    }
  }
  // dT_ij = dU_i . (beta_j v_j) + dW_i . (beta_j e^{G_j} k_j), i > j (the only part dA needs)
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx / 64, j = idx % 64;
    float acc = 0.f;
    if (j < i && i < len) {
      float du = 0.f, dwk = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) {
        du += dVs[i * L + d] * Vs[j * L + d];
        dwk += dWs[i * L + d] * Ks[j * L + d];
      }
      acc = B[j] * du + BG[j] * dwk;
    }
    dT[i * 65 + j] = acc;
  }
  __syncthreads();
  // X = dT T^T:  X_ab = sum_{c} dT_ac T_bc  (c < a, c <= b)
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int a = idx / 64, b = idx % 64;
    float acc = 0.f;
    const int cmax = min(a, b + 1);
    for (int c = 0; c < cmax; ++c) acc += dT[a * 65 + c] * Tm[b * 65 + c];
    X[a * 65 + b] = acc;
  }
  __syncthreads();
  // dA = -T^T X, i > j:  dA_ij = -sum_{a >= i} T_ai X_aj; then Q_ij = dA_ij A_ij into X's
  // place is not needed: dA goes to dT (dT is dead once X is formed)
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx / 64, j = idx % 64;
    float acc = 0.f;
    if (j < i && i < len) {
      for (int a = i; a < len; ++a) acc += Tm[a * 65 + i] * X[a * 65 + j];
      acc = -acc;
    }
    dT[i * 65 + j] = acc;
  }
  __syncthreads();
  // X <- B_ij = dA_ij beta_i Gam_ij (i > j); dbeta_c and dG_c from dA o A
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx / 64, j = idx % 64;
    X[i * 65 + j] = (j < i && i < len) ? dT[i * 65 + j] * B[i] * expf(G[i] - G[j]) : 0.f;
  }
  __syncthreads();
  // per row j (tid / 4), columns tid % 4 + 4 m
  const int j = tid >> 2, sub = tid & 3;
  float dba = 0.f, dbb = 0.f;
  float *dvo = reinterpret_cast<float *>(dv_out.p), *dko = reinterpret_cast<float *>(dkh.p);
  if (j < len) {
    for (int d = sub; d < D; d += 4) {
      float tdu = 0.f, tdw = 0.f;
      for (int i = j; i < len; ++i) {
        tdu += Tm[i * 65 + j] * dVs[i * L + d];
        tdw += Tm[i * 65 + j] * dWs[i * L + d];
      }
      dvo[(t0 + j) * dv_out.st + h * dv_out.sh + d] = B[j] * tdu;
      dba += Vs[j * L + d] * tdu;
      dbb += Ks[j * L + d] * tdw;
      float kc = 0.f;
      for (int x = 0; x < j; ++x) kc += X[j * 65 + x] * Ks[x * L + d];
      for (int a = j + 1; a < len; ++a) kc += X[a * 65 + j] * Ks[a * L + d];
      const int64_t ok = (t0 + j) * dkh.st + h * dkh.sh + d;
      dko[ok] = dko[ok] + BG[j] * tdw + kc;
    }
  }
  dba += __shfl_xor_sync(0xffffffffu, dba, 1);
  dba += __shfl_xor_sync(0xffffffffu, dba, 2);
  dbb += __shfl_xor_sync(0xffffffffu, dbb, 1);
  dbb += __shfl_xor_sync(0xffffffffu, dbb, 2);
  if (sub == 0) {
    dbS[j] = dba;
    dgbS[j] = dbb;
  }
  __syncthreads();
  if (tid < 64) {
    const int r = tid;
    float dbc = 0.f, rowq = 0.f, colq = 0.f;
    if (r < len) {
      for (int x = 0; x < r; ++x) {
        const float gam = expf(G[r] - G[x]);
        dbc += dT[r * 65 + x] * gam * KK[r * 65 + x];
        rowq += X[r * 65 + x] * KK[r * 65 + x];
      }
      for (int a = r + 1; a < len; ++a) colq += X[a * 65 + r] * KK[a * 65 + r];
      float* dbo = reinterpret_cast<float *>(dbeta_out.p);
      dbo[(t0 + r) * dbeta_out.st + h * dbeta_out.sh] = dbS[r] + EGv[r] * dgbS[r] + dbc;
      float gt = dga[(t0 + r) * H + h] + BG[r] * dgbS[r] + rowq - colq;
      if (r == len - 1) {
        float sd = 0.f;
        for (int b = 0; b < D / kSRows; ++b) sd += sdot[((int64_t)cid * H + h) * (D / kSRows) + b];
        gt += EGv[r] * sd;
      }
      dGt[r] = gt;
    }
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
  cudaError_t e;
  // forward recompute: G, W, U (stage 1), chunk states h and V' (stage 2)
  if ((e = launch_prep(s, a.k, a.v, a.g, a.beta, vw, vu, vg, a.seg, a.chunks, a.n_chunks,
                       stream)) != cudaSuccess)
    return e;
  if ((e = launch_scan(s, a.k, vw, vu, vg, a.h0, w.h, vn, nullptr, Ckpt{nullptr, nullptr, 0},
                       a.seg, stream)) != cudaSuccess)
    return e;
  const dim3 gc((unsigned)s.chunk_cap, (unsigned)s.H);
  if ((e = set_smem(k_bwd_dv_intra<D>, DvIntraSmem<D>::bytes)) != cudaSuccess) return e;
  k_bwd_dv_intra<D><<<dim3(gc.x, gc.y, D / 64), 256, DvIntraSmem<D>::bytes, stream>>>(
      group, a.q, a.k, a.dout, vg, a.scale, vdvp, a.chunks, a.n_chunks);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = set_smem(k_bwd_scan<D>, BwdScanSmem<D>::bytes)) != cudaSuccess) return e;
  k_bwd_scan<D><<<dim3((unsigned)s.n_seq, (unsigned)s.H, D / kScanCols), 128,
                  BwdScanSmem<D>::bytes, stream>>>(s.H, group, a.q, a.k, vw, a.dout, vg,
                                                   a.scale, a.dht, vdvp, w.dh, a.dh0, a.seg);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = set_smem(k_bwd_sgrad<D>, SgradSmem<D>::bytes)) != cudaSuccess) return e;
  k_bwd_sgrad<D><<<dim3(gc.x, gc.y, D / kSRows), 256, SgradSmem<D>::bytes, stream>>>(
      a.dout, vn, vg, a.scale, reinterpret_cast<const __nv_bfloat16 *>(w.h), w.dh, vdvp, vdqh,
      vdkh, vdw, w.sdot, a.chunks, a.n_chunks, s.H);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = set_smem(k_bwd_intra<D>, IntraSmem<D>::bytes)) != cudaSuccess) return e;
  k_bwd_intra<D><<<gc, 256, IntraSmem<D>::bytes, stream>>>(group, a.q, a.k, a.dout, vn, vg,
                                                            a.scale, vdqh, vdkh, w.dga,
                                                            a.chunks, a.n_chunks, s.H);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = set_smem(k_bwd_wy<D>, WySmem<D>::bytes)) != cudaSuccess) return e;
  k_bwd_wy<D><<<gc, 256, WySmem<D>::bytes, stream>>>(group, a.k, a.v, a.beta, vg, vdvp, vdw,
                                                      vdkh, w.dga, w.sdot, a.dv, a.dbeta, a.dg,
                                                      a.chunks, a.n_chunks, s.H);
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

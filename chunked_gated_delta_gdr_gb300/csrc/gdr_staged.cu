// gdr_staged.cu -- the three stages of the chunked gated delta rule forward as
// separate kernels with their intermediates in HBM (GDR_PATH_STAGED and the
// per-stage entry points).  Plain fp32 SIMT arithmetic over shared-memory
// tiles; bf16 at the same storage points as the fused path (W, U, V', h).
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

namespace gdr {
namespace {

// ---------------------------------------------------------------- stage 1
template <int D>
struct PrepSmem {
  static constexpr int kLd = D + 1;
  static constexpr size_t bytes =
      sizeof(float) * (2 * 64 * kLd + 2 * 64 * 65 + 3 * 64);
};

template <int D>
__global__ void __launch_bounds__(256)
    k_prep(int32_t group, View k, View v, View g, View beta, View w, View u, View gcum,
           const ChunkInfo *__restrict__ chunks, const int32_t *__restrict__ n_chunks) {
  extern __shared__ float sm[];
  constexpr int L = PrepSmem<D>::kLd;
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *Ks = sm, *Vs = Ks + 64 * L, *Am = Vs + 64 * L, *Tm = Am + 64 * 65;
  float *G = Tm + 64 * 65, *B = G + 64, *BG = B + 64;

  for (int idx = tid; idx < 64 * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    float kv = 0.f, vv = 0.f;
    if (i < len) {
      kv = ldbf(k.p, (t0 + i) * k.st + hk * k.sh + d);
      vv = ldbf(v.p, (t0 + i) * v.st + h * v.sh + d);
    }
    Ks[i * L + d] = kv;
    Vs[i * L + d] = vv;
  }
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
  for (int idx = tid; idx < 64 * 64; idx += blockDim.x) {
    const int i = idx / 64, j = idx % 64;
    float a = 0.f;
    if (j < i && i < len) {
      float dot = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) dot += Ks[i * L + d] * Ks[j * L + d];
      a = B[i] * expf(G[i] - G[j]) * dot;
    }
    Am[i * 65 + j] = a;
  }
  __syncthreads();
  if (tid < 64) {  // column c of (I + A)^-1 by forward substitution
    const int c = tid;
    for (int i = 0; i < 64; ++i) {
      float x = (i == c) ? 1.f : 0.f;
      for (int j = c; j < i; ++j) x -= Am[i * 65 + j] * Tm[j * 65 + c];
      Tm[i * 65 + c] = x;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < 64 * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    if (i >= len) continue;
    float wa = 0.f, ua = 0.f;
    for (int j = 0; j <= i; ++j) {
      const float t = Tm[i * 65 + j];
      wa += t * BG[j] * Ks[j * L + d];
      ua += t * B[j] * Vs[j * L + d];
    }
    stbf(w.p, (t0 + i) * w.st + h * w.sh + d, wa);
    stbf(u.p, (t0 + i) * u.st + h * u.sh + d, ua);
  }
  if (tid < len) reinterpret_cast<float *>(gcum.p)[(t0 + tid) * gcum.st + h * gcum.sh] = G[tid];
}

// ---------------------------------------------------------------- stage 2
constexpr int kScanCols = 32;  // value columns of S per block

template <int D>
struct ScanSmem {
  static constexpr int kLd = D + 1;
  static constexpr size_t bytes =
      sizeof(float) * (D * 33 + 2 * 64 * kLd + 2 * 64 * 33 + 2 * 64);
};

template <int D>
__global__ void __launch_bounds__(128)
    k_scan(int32_t H, int32_t group, View k, View w, View u, View gcum, const float *h0,
           __nv_bfloat16 *hbuf, View v_new, float *ht, Ckpt ck,
           const SegInfo *__restrict__ seg) {
  extern __shared__ float sm[];
  constexpr int L = ScanSmem<D>::kLd;
  const int n = blockIdx.x, h = blockIdx.y, jb = blockIdx.z * kScanCols, tid = threadIdx.x;
  const int hk = h / group;
  const SegInfo si = seg[n];
  float *S = sm, *Ws = S + D * 33, *Ks = Ws + 64 * L, *Us = Ks + 64 * L, *Vn = Us + 64 * 33;
  float *G = Vn + 64 * 33, *Dec = G + 64;
  const int64_t sbase = ((int64_t)n * H + h) * D * D;

  for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
    const int d = idx / kScanCols, j = idx % kScanCols;
    S[d * 33 + j] = h0 ? h0[sbase + (int64_t)d * D + jb + j] : 0.f;
  }
  // state of this block's columns -> checkpoint row `row` (the state after the
  // segment's first (row - first row + 1) * every tokens)
  auto store_ckpt = [&](int64_t row) {
    float *dst = ck.h + (row * H + h) * D * D;
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      dst[(int64_t)d * D + jb + j] = S[d * 33 + j];
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
      hc[(int64_t)d * D + jb + j] = __float2bfloat16_rn(S[d * 33 + j]);
    }
    for (int idx = tid; idx < 64 * D; idx += blockDim.x) {
      const int i = idx / D, d = idx % D;
      float wv = 0.f, kv = 0.f;
      if (i < len) {
        wv = ldbf(w.p, (t0 + i) * w.st + h * w.sh + d);
        kv = ldbf(k.p, (t0 + i) * k.st + hk * k.sh + d);
      }
      Ws[i * L + d] = wv;
      Ks[i * L + d] = kv;
    }
    for (int idx = tid; idx < 64 * kScanCols; idx += blockDim.x) {
      const int i = idx / kScanCols, j = idx % kScanCols;
      Us[i * 33 + j] = i < len ? ldbf(u.p, (t0 + i) * u.st + h * u.sh + jb + j) : 0.f;
    }
    if (tid < 64) G[tid] = tid < len ? ldf(gcum.p, (t0 + tid) * gcum.st + h * gcum.sh) : 0.f;
    __syncthreads();
    const float glast = G[len - 1];
    if (tid < 64) Dec[tid] = tid < len ? expf(glast - G[tid]) : 0.f;
    for (int idx = tid; idx < 64 * kScanCols; idx += blockDim.x) {
      const int i = idx / kScanCols, j = idx % kScanCols;
      float vn = 0.f;
      if (i < len) {
        float acc = Us[i * 33 + j];
#pragma unroll 8
        for (int d = 0; d < D; ++d) acc -= Ws[i * L + d] * S[d * 33 + j];
        const __nv_bfloat16 b = __float2bfloat16_rn(acc);
        reinterpret_cast<__nv_bfloat16 *>(v_new.p)[(t0 + i) * v_new.st + h * v_new.sh + jb + j] = b;
        vn = __bfloat162float(b);
      }
      Vn[i * 33 + j] = vn;
    }
    __syncthreads();
    const float eg = expf(glast);
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      float acc = eg * S[d * 33 + j];
      for (int i = 0; i < len; ++i) acc += Dec[i] * Ks[i * L + d] * Vn[i * 33 + j];
      S[d * 33 + j] = acc;
    }
  }
  if (ht || ck.h) __syncthreads();
  if (ht) {
    for (int idx = tid; idx < D * kScanCols; idx += blockDim.x) {
      const int d = idx / kScanCols, j = idx % kScanCols;
      ht[sbase + (int64_t)d * D + jb + j] = S[d * 33 + j];
    }
  }
  const int seg_len = si.end - si.start;
  if (ck.h && seg_len > 0 && seg_len % ck.every == 0) store_ckpt(ck.off[n] + seg_len / ck.every - 1);
}

// ---------------------------------------------------------------- stage 3
constexpr int kOutCols = 64;

template <int D>
struct OutSmem {
  static constexpr int kLd = D + 1;
  static constexpr size_t bytes =
      sizeof(float) * (2 * 64 * kLd + D * 65 + 2 * 64 * 65 + 64);
};

template <int D>
__global__ void __launch_bounds__(256)
    k_out(int32_t H, int32_t group, View q, View k, View v_new, const __nv_bfloat16 *hbuf,
          View gcum, float scale, View o, const ChunkInfo *__restrict__ chunks,
          const int32_t *__restrict__ n_chunks) {
  extern __shared__ float sm[];
  constexpr int L = OutSmem<D>::kLd;
  const int cid = blockIdx.x, h = blockIdx.y, cb = blockIdx.z * kOutCols, tid = threadIdx.x;
  if (cid >= *n_chunks) return;
  const ChunkInfo ci = chunks[cid];
  const int len = ci.len, hk = h / group;
  const int64_t t0 = ci.start;
  float *Qs = sm, *Ks = Qs + 64 * L, *Hs = Ks + 64 * L, *Vn = Hs + D * 65, *P = Vn + 64 * 65;
  float *G = P + 64 * 65;

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
  const __nv_bfloat16 *hc = hbuf + ((int64_t)cid * H + h) * D * D;
  for (int idx = tid; idx < D * kOutCols; idx += blockDim.x) {
    const int d = idx / kOutCols, c = idx % kOutCols;
    Hs[d * 65 + c] = __bfloat162float(hc[(int64_t)d * D + cb + c]);
  }
  for (int idx = tid; idx < 64 * kOutCols; idx += blockDim.x) {
    const int i = idx / kOutCols, c = idx % kOutCols;
    Vn[i * 65 + c] = i < len ? ldbf(v_new.p, (t0 + i) * v_new.st + h * v_new.sh + cb + c) : 0.f;
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
  for (int idx = tid; idx < 64 * kOutCols; idx += blockDim.x) {
    const int i = idx / kOutCols, c = idx % kOutCols;
    if (i >= len) continue;
    float inter = 0.f, intra = 0.f;
#pragma unroll 8
    for (int d = 0; d < D; ++d) inter += Qs[i * L + d] * Hs[d * 65 + c];
    for (int j = 0; j <= i; ++j) intra += P[i * 65 + j] * Vn[j * 65 + c];
    const float r = scale * (expf(G[i]) * inter + intra);
    stbf(o.p, (t0 + i) * o.st + h * o.sh + cb + c, r);
  }
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
  cudaError_t e;
  if (s.D == 64) {
    if ((e = set_smem(k_prep<64>, PrepSmem<64>::bytes)) != cudaSuccess) return e;
    k_prep<64><<<grid, 256, PrepSmem<64>::bytes, stream>>>(s.H / s.Hk, k, v, g, beta, w, u,
                                                           gcum, chunks, n_chunks);
  } else {
    if ((e = set_smem(k_prep<128>, PrepSmem<128>::bytes)) != cudaSuccess) return e;
    k_prep<128><<<grid, 256, PrepSmem<128>::bytes, stream>>>(s.H / s.Hk, k, v, g, beta, w, u,
                                                             gcum, chunks, n_chunks);
  }
  return cudaGetLastError();
}

cudaError_t launch_scan(const StageShapes &s, View k, View w, View u, View gcum,
                        const float *h0, void *h, View v_new, float *ht, Ckpt ck,
                        const SegInfo *seg, cudaStream_t stream) {
  if (s.n_seq <= 0 || s.H <= 0) return cudaSuccess;
  dim3 grid((unsigned)s.n_seq, (unsigned)s.H, (unsigned)(s.D / kScanCols));
  auto *hb = reinterpret_cast<__nv_bfloat16 *>(h);
  cudaError_t e;
  if (s.D == 64) {
    if ((e = set_smem(k_scan<64>, ScanSmem<64>::bytes)) != cudaSuccess) return e;
    k_scan<64><<<grid, 128, ScanSmem<64>::bytes, stream>>>(s.H, s.H / s.Hk, k, w, u, gcum, h0,
                                                           hb, v_new, ht, ck, seg);
  } else {
    if ((e = set_smem(k_scan<128>, ScanSmem<128>::bytes)) != cudaSuccess) return e;
    k_scan<128><<<grid, 128, ScanSmem<128>::bytes, stream>>>(s.H, s.H / s.Hk, k, w, u, gcum,
                                                             h0, hb, v_new, ht, ck, seg);
  }
  return cudaGetLastError();
}

cudaError_t launch_out(const StageShapes &s, View q, View k, View v_new, const void *h,
                       View gcum, float scale, View o, const SegInfo *, const ChunkInfo *chunks,
                       const int32_t *n_chunks, cudaStream_t stream) {
  if (s.chunk_cap <= 0 || s.H <= 0) return cudaSuccess;
  dim3 grid((unsigned)s.chunk_cap, (unsigned)s.H, (unsigned)(s.D / kOutCols));
  auto *hb = reinterpret_cast<const __nv_bfloat16 *>(h);
  cudaError_t e;
  if (s.D == 64) {
    if ((e = set_smem(k_out<64>, OutSmem<64>::bytes)) != cudaSuccess) return e;
    k_out<64><<<grid, 256, OutSmem<64>::bytes, stream>>>(s.H, s.H / s.Hk, q, k, v_new, hb,
                                                         gcum, scale, o, chunks, n_chunks);
  } else {
    if ((e = set_smem(k_out<128>, OutSmem<128>::bytes)) != cudaSuccess) return e;
    k_out<128><<<grid, 256, OutSmem<128>::bytes, stream>>>(s.H, s.H / s.Hk, q, k, v_new, hb,
                                                           gcum, scale, o, chunks, n_chunks);
  }
  return cudaGetLastError();
}

}  // namespace gdr

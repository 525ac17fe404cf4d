// gdr_index.cu -- chunk enumeration from cu_seqlens, entirely on the device.
//
// FlashQLA derives its chunk grid on the host through a cache keyed by the
// Python id() of cu_seqlens, which served stale grids for recycled addresses
// ("Findings from integrating FlashQLA's Blackwell GDN kernels into a JAX
// trainer", section 1).  Here the grid is rebuilt from the array's contents
// on every call, on the stream, with no host read-back.
//
// Reading of cu_seqlens: offsets are clamped to [0, T] and made
// non-decreasing by a running maximum; segment n is [c[n], c[n+1]).
// Length-0 segments ("Findings ...", section 2) get zero chunks.
#include "gdr_internal.cuh"
#include "gdr_sched.cuh"

namespace gdr {
namespace {

constexpr int kScanThreads = 1024;

template <bool kMax>
__device__ int block_inclusive_scan(int x, int *warp_buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x = kMax ? max(x, y) : x + y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_buf[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w = kMax ? max(w, y) : w + y;
    }
    warp_buf[lane] = w;
  }
  __syncthreads();
  if (warp > 0) {
    int y = warp_buf[warp - 1];
    x = kMax ? max(x, y) : x + y;
  }
  __syncthreads();
  return x;
}

// One block: sanitised bounds, per-segment chunk counts, exclusive prefix.
__global__ void __launch_bounds__(kScanThreads)
    k_seg_index(const int32_t *__restrict__ cu, int32_t n_seq, int64_t T, SegInfo *seg,
                int32_t *n_chunks) {
  __shared__ int warp_buf[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int Tc = (int)(T < 0x7fffffff ? T : 0x7fffffff);
  for (int base = 0; base <= n_seq; base += kScanThreads) {
    const int i = base + (int)threadIdx.x;
    int x = 0;
    if (i <= n_seq) x = min(max(cu[i], 0), Tc);
    x = block_inclusive_scan<true>(x, warp_buf);
    x = max(x, carry);
    if (i <= n_seq) {
      if (i < n_seq) seg[i].start = x;
      if (i > 0) seg[i - 1].end = x;
    }
    __syncthreads();
    if (threadIdx.x == kScanThreads - 1) carry = x;
    __syncthreads();
  }
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n_seq; base += kScanThreads) {
    const int i = base + (int)threadIdx.x;
    int nc = 0;
    if (i < n_seq) nc = (seg[i].end - seg[i].start + kChunk - 1) / kChunk;
    const int incl = block_inclusive_scan<false>(nc, warp_buf);
    if (i < n_seq) {
      seg[i].chunk_off = carry + incl - nc;
      seg[i].n_chunks = nc;
    }
    __syncthreads();
    if (threadIdx.x == kScanThreads - 1) carry += incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_chunks = carry;
}

// Chunk table: chunk id -> (segment, first token, length), by binary search
// over the non-decreasing chunk offsets.
__global__ void k_chunk_table(const SegInfo *__restrict__ seg, int32_t n_seq,
                              const int32_t *__restrict__ n_chunks, ChunkInfo *chunks,
                              int64_t cap) {
  const int total = *n_chunks;
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < cap;
       c += (int64_t)gridDim.x * blockDim.x) {
    ChunkInfo ci{-1, 0, 0, 0};
    if (c < total) {
      int lo = 0, hi = n_seq - 1;  // last n with chunk_off[n] <= c
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg[mid].chunk_off <= c) lo = mid; else hi = mid - 1;
      }
      const SegInfo s = seg[lo];
      const int local = (int)c - s.chunk_off;
      ci.seq = lo;
      ci.start = s.start + local * kChunk;
      ci.len = min(kChunk, s.end - ci.start);
    }
    chunks[c] = ci;
  }
}

// Checkpoint offsets: exclusive prefix of floor(len / every) over the segments.
__global__ void __launch_bounds__(kScanThreads)
    k_ckpt_offsets(const SegInfo *__restrict__ seg, int32_t n_seq, int32_t every,
                   int32_t *off) {
  __shared__ int warp_buf[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n_seq; base += kScanThreads) {
    const int i = base + (int)threadIdx.x;
    const int nc = i < n_seq ? (seg[i].end - seg[i].start) / every : 0;
    const int incl = block_inclusive_scan<false>(nc, warp_buf);
    if (i < n_seq) off[i] = carry + incl - nc;
    __syncthreads();
    if (threadIdx.x == kScanThreads - 1) carry += incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) off[n_seq] = carry;
}

// Segments by chunk count, longest first: counting sort over kScanThreads buckets
// (counts beyond the last bucket share it); positions within a bucket are arbitrary.
__global__ void __launch_bounds__(kScanThreads)
    k_seg_order(const SegInfo *__restrict__ seg, int32_t n_seq, int32_t *order) {
  __shared__ int warp_buf[32];
  __shared__ int pos[kScanThreads];
  const int b0 = threadIdx.x;
  pos[b0] = 0;
  __syncthreads();
  auto bucket = [](int nc) { return kScanThreads - 1 - min(nc, kScanThreads - 1); };
  for (int n = threadIdx.x; n < n_seq; n += kScanThreads) atomicAdd(&pos[bucket(seg[n].n_chunks)], 1);
  __syncthreads();
  const int x = pos[b0];
  const int incl = block_inclusive_scan<false>(x, warp_buf);
  pos[b0] = incl - x;
  __syncthreads();
  for (int n = threadIdx.x; n < n_seq; n += kScanThreads)
    order[atomicAdd(&pos[bucket(seg[n].n_chunks)], 1)] = n;
}

__global__ void k_check_cu(const int32_t *__restrict__ cu, int32_t n_seq, int64_t T,
                           int32_t *out2) {
  // out2[0]: count of bad offsets, out2[1]: first bad index (or -1); single block
  __shared__ int cnt, first;
  if (threadIdx.x == 0) { cnt = 0; first = 0x7fffffff; }
  __syncthreads();
  for (int i = threadIdx.x; i <= n_seq; i += blockDim.x) {
    const int c = cu[i];
    const bool bad = c < 0 || (int64_t)c > T || (i > 0 && c < cu[i - 1]);
    if (bad) { atomicAdd(&cnt, 1); atomicMin(&first, i); }
  }
  __syncthreads();
  if (threadIdx.x == 0) { out2[0] = cnt; out2[1] = cnt ? first : -1; }
}

}  // namespace

cudaError_t launch_ckpt_offsets(const SegInfo *seg, int32_t n_seq, int32_t every, int32_t *off,
                                cudaStream_t stream) {
  if (every <= 0) return cudaErrorInvalidValue;
  k_ckpt_offsets<<<1, kScanThreads, 0, stream>>>(seg, n_seq, every, off);
  return cudaGetLastError();
}

cudaError_t launch_chunk_index(const int32_t *cu, int32_t n_seq, int64_t T, SegInfo *seg,
                               ChunkInfo *chunks, int64_t chunk_cap, int32_t *n_chunks,
                               cudaStream_t stream) {
  k_seg_index<<<1, kScanThreads, 0, stream>>>(cu, n_seq, T, seg, n_chunks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || chunks == nullptr || chunk_cap <= 0) return e;
  const int threads = 256;
  int64_t blocks = ceil_div64(chunk_cap, threads);
  if (blocks > 4096) blocks = 4096;
  k_chunk_table<<<(unsigned)blocks, threads, 0, stream>>>(seg, n_seq, n_chunks, chunks, chunk_cap);
  return cudaGetLastError();
}

cudaError_t launch_seg_order(const SegInfo *seg, int32_t n_seq, int32_t *order,
                             cudaStream_t stream) {
  if (n_seq <= 0) return cudaSuccess;
  k_seg_order<<<1, kScanThreads, 0, stream>>>(seg, n_seq, order);
  return cudaGetLastError();
}

cudaError_t launch_check_cu(const int32_t *cu, int32_t n_seq, int64_t T, int32_t *out2,
                            cudaStream_t stream) {
  k_check_cu<<<1, 1024, 0, stream>>>(cu, n_seq, T, out2);
  return cudaGetLastError();
}

}  // namespace gdr

// gdr_split.cu -- intra-sequence split of long segments (few (segment, head) units).
//
// The state after a span of tokens is affine in the state before it,
// S_out = M S_in + R (M: the span's dk x dk transition, R: its zero-start state), which
// is how a sequence is carried across ranks in context-parallel delta-rule kernels
// (the final_correction of "feat(cake_kda): add paired recurrent training for SM100a and
// SM103a").  Here the pieces of one segment run on different SMs: pass A gives R and M of
// every piece after the first, the combine step below chains the initial states, pass B
// produces the outputs of the later pieces.  Everything is decided on the device from
// cu_seqlens; the host only picks the number of pieces from the unit count.
#include "gdr_internal.cuh"

namespace gdr {

int split_pieces(int64_t units, int sms, int *lead) {
  *lead = 1;
  if (units <= 0 || sms <= 0 || units * 3 > sms) return 1;
  // A segment is cut into the first piece (weight `a`) and P - 1 pieces of weight 1;
  // per (segment, head) pass A runs the first piece and R and M of the P - 2 middle
  // ones, pass B the P - 1 later pieces, each pass on `sms` SMs that take units in
  // table order as they come free (first pieces first).  Pick the P and `a` with the
  // shortest pass A + pass B in units of the whole segment; ties go to fewer pieces.
  int best = 1, best_a = 1;
  double best_cost = 1.0;
  for (int P = 3; P <= kSplitMaxPieces; ++P)
    for (int a = 1; a <= 3; ++a) {
      const int64_t rm = units * 2 * (P - 2);  // R and M units, length 1
      // pass A: the first pieces occupy `units` SMs for time a; the smallest integer
      // time t >= a by which the other SMs (from 0) and those (from a) fit all of rm
      int64_t t = a;
      while ((sms - units) * t + units * (t - a) < rm) ++t;
      const int64_t tb = (units * (P - 1) + sms - 1) / sms;
      const double cost = (double)(t + tb) / (a + P - 1);
      if (cost < best_cost - 1e-9) { best_cost = cost; best = P; best_a = a; }
    }
  *lead = best_a;
  return best;
}

namespace {
inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

SplitWs carve_split(void *ws, int32_t n_seq, int32_t H, int32_t D, int32_t pieces) {
  SplitWs w{};
  char *p = reinterpret_cast<char *>(ws);
  size_t off = 0;
  const size_t nu = (size_t)(n_seq > 0 ? n_seq : 1) * H;
  const size_t P = (size_t)(pieces < 1 ? 1 : pieces);
  const size_t na = nu * (2 * P - 1), nb = nu * P;
  w.ua = reinterpret_cast<UnitDesc *>(p + off); off += al256(na * sizeof(UnitDesc));
  w.ub = reinterpret_cast<UnitDesc *>(p + off); off += al256(nb * sizeof(UnitDesc));
  w.na = reinterpret_cast<int32_t *>(p + off);
  w.nb = w.na + 1;
  w.counters = w.na + 2;  // [0] pass A, [1] pass B
  off += 256;
  w.seg_pieces = reinterpret_cast<int32_t *>(p + off);  // (first piece id, piece count)
  off += al256((size_t)(n_seq > 0 ? n_seq : 1) * 2 * sizeof(int32_t));
  w.states = reinterpret_cast<float *>(p + off);
  off += al256(nu * P * 3 * (size_t)D * D * sizeof(float));
  w.bytes = off;
  return w;
}

namespace {

// One block: piece layout per segment and the unit tables of both passes.
__global__ void k_split_units(const SegInfo *__restrict__ seg, int32_t n_seq, int32_t H,
                              int32_t P, int32_t lead, UnitDesc *ua, int32_t *na, UnitDesc *ub,
                              int32_t *nb, int32_t *counters, int32_t *seg_pieces) {
  __shared__ int32_t s_off_a, s_off_b, s_pid;
  if (threadIdx.x == 0) { s_off_a = 0; s_off_b = 0; s_pid = 0; }
  __syncthreads();
  // segments one at a time (few by construction); threads fill that segment's units
  for (int n = 0; n < n_seq; ++n) {
    const SegInfo si = seg[n];
    const int nc = si.n_chunks;
    // pieces: the first of weight `lead`, the others of weight 1, none shorter than
    // about kSplitMinChunks; fewer than 3 pieces gain nothing (two run one after the
    // other), so such a segment stays whole
    int pn = nc / kSplitMinChunks - (lead - 1);
    pn = nc <= 0 ? 0 : (pn < 3 ? 1 : (pn > P ? P : pn));
    const int a = pn > 1 ? lead : 1, wsum = a + pn - 1;
    // first chunk of piece p (p = pn: the end)
    auto cstart = [&](int p) { return p == 0 ? 0 : (p >= pn ? nc : (int)(((int64_t)(a + p - 1) * nc) / wsum)); };
    const int pid0 = s_pid, base_a = s_off_a, base_b = s_off_b;
    // slot of (piece id, head, which): which 0 = R, 1 = M, 2 = initial state
    auto slot = [&](int pid, int h, int which) { return (pid * H + h) * 3 + which; };
    // pass A: the first piece, and R and M of pieces 1 .. pn-2 (the last piece's are
    // never needed); pass B: pieces 1 .. pn-1 from their initial states
    const int units_a = pn > 0 ? H * (pn > 1 ? 2 * pn - 3 : 1) : 0;
    const int units_b = pn > 1 ? H * (pn - 1) : 0;
    for (int u = threadIdx.x; u < units_a; u += blockDim.x) {
      // u < H: piece 0; then (piece p in 1 .. pn-2, R/M, head)
      int p, h, mode;
      if (u < H) { p = 0; h = u; mode = kUnitFull; }
      else {
        const int v = u - H;
        p = 1 + v / (2 * H);
        mode = ((v / H) & 1) ? kUnitM : kUnitR;
        h = v % H;
      }
      const int c0 = cstart(p), c1 = cstart(p + 1);
      UnitDesc d;
      d.seq = n;
      d.head = h;
      d.t0 = si.start + c0 * kChunk;
      d.end = min(si.end, si.start + c1 * kChunk);
      d.nch = c1 - c0;
      d.mode = mode;
      d.sin = -1;
      if (mode == kUnitFull) d.sout = pn > 1 ? slot(pid0 + 1, h, 2) : -1;
      else d.sout = slot(pid0 + p, h, mode == kUnitR ? 0 : 1);
      ua[base_a + u] = d;
    }
    for (int u = threadIdx.x; u < units_b; u += blockDim.x) {
      const int p = 1 + u / H, h = u % H;
      const int c0 = cstart(p), c1 = cstart(p + 1);
      UnitDesc d;
      d.seq = n;
      d.head = h;
      d.t0 = si.start + c0 * kChunk;
      d.end = min(si.end, si.start + c1 * kChunk);
      d.nch = c1 - c0;
      d.mode = kUnitFinal;
      d.sin = slot(pid0 + p, h, 2);
      d.sout = p == pn - 1 ? -1 : -2;
      ub[base_b + u] = d;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      seg_pieces[2 * n] = pid0;
      seg_pieces[2 * n + 1] = pn;
      s_pid = pid0 + pn;
      s_off_a = base_a + units_a;
      s_off_b = base_b + units_b;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *na = s_off_a;
    *nb = s_off_b;
    counters[0] = 0;
    counters[1] = 0;
  }
}

// Initial states of pieces 2.. of every split segment: S_{p+1} = M_p S_p + R_p, fp32.
// Block (segment, head, 32 value columns); S_1 comes from pass A (piece 0's final
// state).  M_p is staged in shared memory with rows padded to kLdM floats, so that the
// four rows a warp reads at one key index fall in different banks; each thread keeps a
// (D / 32) x 4 tile of the product in registers.
constexpr int kCombCols = 32;
constexpr int kLdM = 129;
__global__ void __launch_bounds__(256)
    k_split_combine(const int32_t *__restrict__ seg_pieces, int32_t H, int32_t D,
                    float *states) {
  extern __shared__ float smem[];
  float *sM = smem;              // [D][kLdM]
  float *sS = smem + D * kLdM;   // [D][kCombCols]
  const int n = blockIdx.x, h = blockIdx.y, cb = blockIdx.z * kCombCols;
  const int pid0 = seg_pieces[2 * n], pn = seg_pieces[2 * n + 1];
  if (pn < 3) return;  // S_1 is all pass B needs for two pieces
  const int64_t DD = (int64_t)D * D;
  auto blk = [&](int pid, int which) { return states + ((int64_t)(pid * H + h) * 3 + which) * DD; };
  const int tx = threadIdx.x % 8, ty = threadIdx.x / 8;  // 4 columns, D / 32 rows
  const int rpt = D / 32, c = tx * 4;
  // all loads of a block are issued before the first is used (unrolled, 16 bytes each),
  // so that one step waits for about one memory round trip, not one per element
  const float *S1 = blk(pid0 + 1, 2);
  {
    float4 x[4];  // D x 32 floats: at most 1024 float4 over 256 threads
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = threadIdx.x + u * 256, j = f / 8, c4 = (f % 8) * 4;
      if (j < D) x[u] = *reinterpret_cast<const float4 *>(S1 + (int64_t)j * D + cb + c4);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = threadIdx.x + u * 256, j = f / 8, c4 = (f % 8) * 4;
      if (j < D) *reinterpret_cast<float4 *>(sS + j * kCombCols + c4) = x[u];
    }
  }
  for (int p = 1; p + 1 < pn; ++p) {
    const float *M = blk(pid0 + p, 1), *R = blk(pid0 + p, 0);
    float *out = blk(pid0 + p + 1, 2);
    {
      float4 x[16];  // D x D floats: at most 4096 float4 over 256 threads
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int f = threadIdx.x + u * 256;
        if (f * 4 < D * D) x[u] = *reinterpret_cast<const float4 *>(M + (int64_t)f * 4);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int f = threadIdx.x + u * 256;
        if (f * 4 < D * D) {
          float *d = sM + ((f * 4) / D) * kLdM + (f * 4) % D;  // rows padded: scalar stores
          d[0] = x[u].x; d[1] = x[u].y; d[2] = x[u].z; d[3] = x[u].w;
        }
      }
    }
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (r < rpt) {
        const float4 x = *reinterpret_cast<const float4 *>(R + (int64_t)(ty * rpt + r) * D + cb + c);
        acc[r][0] = x.x; acc[r][1] = x.y; acc[r][2] = x.z; acc[r][3] = x.w;
      }
    }
#pragma unroll 4
    for (int j = 0; j < D; ++j) {
      const float4 sv = *reinterpret_cast<const float4 *>(sS + j * kCombCols + c);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        if (r < rpt) {
          const float m = sM[(ty * rpt + r) * kLdM + j];
          acc[r][0] = fmaf(m, sv.x, acc[r][0]);
          acc[r][1] = fmaf(m, sv.y, acc[r][1]);
          acc[r][2] = fmaf(m, sv.z, acc[r][2]);
          acc[r][3] = fmaf(m, sv.w, acc[r][3]);
        }
      }
    }
    __syncthreads();  // every read of sS and sM is done
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (r < rpt) {
        const int i = ty * rpt + r;
        const float4 x = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        *reinterpret_cast<float4 *>(sS + i * kCombCols + c) = x;
        *reinterpret_cast<float4 *>(out + (int64_t)i * D + cb + c) = x;
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_split_units(const SegInfo *seg, int32_t n_seq, int32_t H, int32_t pieces,
                               int32_t lead, const SplitWs &w, cudaStream_t stream) {
  k_split_units<<<1, 1024, 0, stream>>>(seg, n_seq, H, pieces, lead, w.ua, w.na, w.ub, w.nb,
                                        w.counters, w.seg_pieces);
  return cudaGetLastError();
}

cudaError_t launch_split_combine(const SplitWs &w, int32_t n_seq, int32_t H, int32_t D,
                                 cudaStream_t stream) {
  if (n_seq <= 0) return cudaSuccess;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const size_t smem = sizeof(float) * D * (kLdM + kCombCols);
  if (!attr_set[dev]) {
    const int most = (int)(sizeof(float) * 128 * (kLdM + kCombCols));
    if ((e = cudaFuncSetAttribute(k_split_combine, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  most)) != cudaSuccess)
      return e;
    attr_set[dev] = true;
  }
  dim3 grid((unsigned)n_seq, (unsigned)H, (unsigned)(D / kCombCols));
  k_split_combine<<<grid, 256, smem, stream>>>(w.seg_pieces, H, D, w.states);
  return cudaGetLastError();
}

}  // namespace gdr

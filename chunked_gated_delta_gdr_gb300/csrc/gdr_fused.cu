// gdr_fused.cu -- fused persistent forward of the chunked gated delta rule on
// sm_103a (GB300), plus the device status word.
//
// One CTA per SM walks a work list of (segment, value head) units, longest
// segments first.  For each 64-token chunk of a unit it runs the chunkwise (WY)
// form with every intermediate on chip:
//
//   prep   G = cumsum(g); X1 = [K;Q] K^T (KK^T and QK^T);  A, P masks;
//          Tm = (I + A)^-1;  Tm diag(beta) and Tm diag(beta e^G) as bf16 operands
//   scan   Y = S^T K^T;  U^T = V^T (Tm diag(beta))^T;  V'^T = U^T - Y (Tm diag(beta e^G))^T
//          (so V' = U - W S with W = Tm diag(beta e^G) K, never formed);
//          S^T <- e^{G_last} S^T + V''^T K,  V'' = diag(e^{G_last-G}) V'
//   out    O^T = e^G-scaled S^T Q^T + V'^T P^T,  P_ij = e^{G_i-G_j} q_i.k_j (j <= i)
//
// The state is kept transposed (S^T: value dim on TMEM lanes, key dim on
// columns) so that every tcgen05.mma has M = 128: the head dimension is the M
// side and the chunk's 64 tokens are N or K.  Operands that come from the state
// side (S^T, Y, V'^T, V''^T) stay in TMEM as bf16 A operands; the rest are bf16
// in 128-byte swizzled shared memory; accumulators are fp32 in TMEM.  The chunk
// size (64) is the one FlashQLA's varlen path uses ("Findings from integrating
// FlashQLA's Blackwell GDN kernels into a JAX trainer", section 1); a unit with no
// chunks (a length-0 segment, section 2 of the same page) is never scheduled, so
// it can store no output.
//
// Warp roles (352 threads):
//   warp 0      TMA producer: K, Q, V tiles and g, beta of each chunk into a 3-stage ring
//   warp 1      MMA issuer P (one thread: X1, U, O1, O2) and TMEM owner
//   warp 2      MMA issuer C (one thread: Y, V', S update)
//   warps 3-6   prep warpgroup (one TMEM lane quadrant per warp)
//   warps 7-10  state warpgroup: bf16 conversions on the state chain, output epilogue
// Every wait is bounded in time; a wait that runs out sets the device status
// word and a CTA-wide abort flag, each role drains what it has in flight and
// the CTA releases its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdr_internal.cuh"
#include "gdr_tc.cuh"

namespace gdr {

// Nonzero once a bounded wait in a fused kernel ran out; read by gdr_device_status.
__device__ int32_t g_device_status = 0;

namespace {

using namespace tc;

constexpr int kThreads = 352;
constexpr int kStages = 3;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kUnitRing = 4;

// ---- shared memory map (bytes from a 1024-aligned base) ----
constexpr uint32_t kKQBytes = 32768;  // 2 key blocks x [K rows 0-63 | Q rows 64-127] x 128 B
constexpr uint32_t kVBytes = 16384;   // 2 value blocks x 64 rows x 128 B
constexpr uint32_t kStageBytes = kKQBytes + kVBytes;
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_P = OFF_STAGE + kStages * kStageBytes;  // P bf16, 2 buffers of 64 x 64
constexpr uint32_t OFF_TB = OFF_P + 16384;     // Tm diag(beta) bf16 64 x 64
constexpr uint32_t OFF_TBG = OFF_TB + 8192;    // -Tm diag(beta e^G) bf16 64 x 64
constexpr uint32_t OFF_STG = OFF_TBG + 8192;   // output staging [64 tokens][128 dv] bf16
constexpr uint32_t OFF_A = OFF_STG + 16384;    // solve scratch fp32 64 x kLdA
constexpr uint32_t OFF_Y = OFF_A + 17408;      // solve scratch fp32 32 x kLdY
constexpr uint32_t OFF_SMALL = OFF_Y + 5120;
constexpr uint32_t kSmallBytes = 9216;
constexpr uint32_t kSmemBytes = OFF_SMALL + kSmallBytes + 1024;  // + alignment slack
constexpr int kLdA = 68, kLdY = 40, kLdX = 24;  // padded leading dims of the fp32 scratch
static_assert(kSmemBytes <= 232448, "shared memory over the per-block limit");

// ---- TMEM columns ----
constexpr uint32_t TM_S = 0;     // S^T fp32, 128 columns (key dim)
constexpr uint32_t TM_SB = 128;  // S^T bf16 pairs (A operand), 64 columns
constexpr uint32_t TM_U = 192;   // two buffers of 64 columns, by chunk parity: X1, then U^T ->
                                 // V'^T fp32, then bf16 V'^T (cols 0-31) and V''^T (32-63)
constexpr uint32_t TM_Y = 320;   // Y = S^T K^T fp32, then bf16 pairs in cols 0-31
constexpr uint32_t TM_O = 384;   // S^T Q^T (inter-chunk part of O^T), 64 columns
constexpr uint32_t TM_O2 = 448;  // V'^T P^T (intra-chunk part of O^T), 64 columns
constexpr uint32_t kTmemCols = 512;

struct UnitInfo {
  int32_t seq, head, t0, end, nch, mode, sin, sout;  // the last three: split units only
};

// kernel variants: the plain forward, with state checkpoints, split-segment pieces, and the
// forward recomputed for the backward (no output; the chunk quantities the backward reads)
constexpr int kVarPlain = 0, kVarCkpt = 1, kVarSplit = 2, kVarBwd = 3;

// Per-chunk vectors, computed by the producer warp from g and beta.  Five slots
// (by chunk index): the producer refills chunk c's slot for chunk c+5 only after
// chunk c+2's stage is released, which follows chunk c's output epilogue.
constexpr int kInfo = 5;
struct ChunkVec {
  alignas(16) float G[64];     // chunk-local inclusive cumsum of g, times log2(e)
  alignas(16) float eG[64];    // exp(G_j)
  alignas(16) float eGs[64];   // scale * exp(G_j)
  alignas(16) float bfac[64];  // 2^(Gref - G_j) (valid when fac != 0)
  alignas(16) float dec[64];   // exp(G_last - G_j)
  alignas(16) float beta[64];  // beta (0 past the chunk's end)
  float eL;                    // exp(G_last)
  float Gref;                  // max_j G_j
  int32_t fac;                 // 1: max G - min G is small enough to factor 2^(G_i - G_j)
  int32_t ckrow;               // checkpoint row of the state entering this chunk, or -1
};
// 2^(G_i - G_j) = 2^(G_i - Gref) 2^(Gref - G_j) with both factors normal fp32 numbers
// as long as the chunk's range of G (log2 units) stays below this bound.
constexpr float kFacRange = 100.f;

struct Small {
  uint64_t full[kStages], empty[kStages];
  uint64_t x1_full, x1_free, t_ready, uw_full, s_ready, y_full, y_ready, vp_full, vp_ready,
      s_full, o1_full, o_full, o_free, drain;
  uint64_t unit_full[kUnitRing], unit_empty[kUnitRing];
  UnitInfo unit[kUnitRing];
  ChunkVec cv[kInfo];
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Small) <= kSmallBytes, "small area too large");

struct Params {
  int32_t T, n_seq, Hk, H, D, has_h0;
  int32_t n_units;  // filled on the device (work list)
  const float *g;
  int64_t g_st, g_sh;
  const __nv_bfloat16 *beta;
  int64_t b_st, b_sh;
  float scale;
  const float *h0;
  __nv_bfloat16 *o;
  int64_t o_st, o_sh;
  float *ht;
  Ckpt ckpt;                // state checkpoints (ckpt.h null: none)
  // backward recompute (kVarBwd): G [T][H] fp32 (natural log), W and V' [T][H][D] bf16,
  // the state entering each chunk [chunk][H][D dk][D dv] bf16
  float *bw_gcum;
  __nv_bfloat16 *bw_w, *bw_h, *bw_vn;
  float *bw_t;  // Tm = (I + A)^-1 per chunk [chunk][H][64][64] fp32 (null: not stored)
  SplitArgs split;          // split-segment pieces (split.units null: none)
  const SegInfo *seg;
  const int32_t *order;     // non-empty segments, longest first
  const int32_t *n_active;  // number of non-empty segments
  int32_t *counter;         // unit counter (zeroed by the work-list kernel)
};

// ------------------------------------------------------------------ helpers
__device__ __noinline__ void fail(Small *sm, int code) {
  sm->abort = 1;
  atomicCAS(&g_device_status, 0, code);
}

// Named barrier over `n` threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Bounded waits whose outcome is the same for every thread of the caller's group,
// so that no thread leaves a loop that contains barriers or warp-aligned
// tcgen05 instructions while another stays in it.
__device__ __forceinline__ bool wait1(Small *sm, uint64_t &bar, uint32_t parity, int code) {
  if (mbar_wait(&bar, parity, &sm->abort, kWaitLimitNs)) return true;
  fail(sm, code);
  return false;
}
__device__ __forceinline__ bool wait_warp(Small *sm, uint64_t &bar, uint32_t parity, int code) {
  const bool bad = !mbar_wait(&bar, parity, &sm->abort, kWaitLimitNs);
  if (__any_sync(0xffffffffu, bad)) {
    fail(sm, code);
    return false;
  }
  return true;
}
__device__ __forceinline__ bool wait_wg(Small *sm, uint64_t &bar, uint32_t parity, int code,
                                        uint32_t bar_id) {
  const bool bad = !mbar_wait(&bar, parity, &sm->abort, kWaitLimitNs);
  if (named_bar_or(bar_id, 128, bad)) {
    fail(sm, code);
    return false;
  }
  return true;
}
constexpr uint32_t kBarPrep = 1, kBarState = 2;


__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d));
}

// Two fp32 products, or two fused multiply-adds, in one packed instruction (sm_100 and
// later).  Each lane rounds exactly as the scalar operation does (round to nearest, no
// flush to zero), so the results are those of the scalar code with half the instructions.
// a, b: fp32 bit patterns (TMEM loads), times x, y.
__device__ __forceinline__ void mul_x2(uint32_t &a, uint32_t &b, float x, float y) {
  asm("{\n\t.reg .b64 s, t;\n\tmov.b64 s, {%0, %1};\n\tmov.b64 t, {%2, %3};\n\t"
      "mul.rn.f32x2 s, s, t;\n\tmov.b64 {%0, %1}, s;\n\t}"
      : "+r"(a), "+r"(b)
      : "f"(x), "f"(y));
}
__device__ __forceinline__ void mul_x2(float &a, float &b, float x, float y) {
  asm("{\n\t.reg .b64 s, t;\n\tmov.b64 s, {%0, %1};\n\tmov.b64 t, {%2, %3};\n\t"
      "mul.rn.f32x2 s, s, t;\n\tmov.b64 {%0, %1}, s;\n\t}"
      : "+f"(a), "+f"(b)
      : "f"(x), "f"(y));
}
// (a, b) = (x a + u, y b + v)
__device__ __forceinline__ void fma_x2(float &a, float &b, float x, float y, float u, float v) {
  asm("{\n\t.reg .b64 s, t, c;\n\tmov.b64 s, {%0, %1};\n\tmov.b64 t, {%2, %3};\n\t"
      "mov.b64 c, {%4, %5};\n\tfma.rn.f32x2 s, s, t, c;\n\tmov.b64 {%0, %1}, s;\n\t}"
      : "+f"(a), "+f"(b)
      : "f"(x), "f"(y), "f"(u), "f"(v));
}

__device__ __forceinline__ void zero_row(uint32_t tile, int row) {
#pragma unroll
  for (int q = 0; q < 8; ++q) st_shared_v4(tile + row * 128 + q * 16, 0u, 0u, 0u, 0u);
}

// Fetch the next unit (segment, head) for this CTA into ring slot `slot`.
__device__ void fetch_unit(const Params &p, Small *sm, int slot) {
  const int32_t active = *p.n_active;
  const int32_t n_units = active * p.H;
  const int32_t u = atomicAdd(p.counter, 1);
  UnitInfo ui{-1, 0, 0, 0, 0, 0, 0, 0};
  if (u < n_units) {
    const int32_t s = p.order[u / p.H];
    const SegInfo si = p.seg[s];
    ui.seq = s;
    ui.head = u % p.H;
    ui.t0 = si.start;
    ui.end = si.end;
    ui.nch = si.n_chunks;
  }
  sm->unit[slot] = ui;
  mbar_arrive(&sm->unit_full[slot]);
}
// the same from a split unit table
__device__ void fetch_unit_split(const Params &p, Small *sm, int slot) {
  const int32_t u = atomicAdd(p.counter, 1);
  UnitInfo ui{-1, 0, 0, 0, 0, 0, 0, 0};
  if (u < *p.split.n_units) {
    const UnitDesc d = p.split.units[u];
    ui = UnitInfo{d.seq, d.head, d.t0, d.end, d.nch, d.mode, d.sin, d.sout};
  }
  sm->unit[slot] = ui;
  mbar_arrive(&sm->unit_full[slot]);
}

// ------------------------------------------------------------------ roles
template <int kVar>
__device__ void role_producer(const Params &p, Small *sm, uint8_t *base,
                              const CUtensorMap *mq, const CUtensorMap *mk,
                              const CUtensorMap *mv) {
  const int lane = threadIdx.x & 31;
  const uint32_t tx = p.D == 128 ? kStageBytes : kStageBytes / 2;
  uint32_t g = 0;  // chunk counter
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    const int slot = k % kUnitRing;
    if (k >= (uint32_t)kUnitRing &&
        !wait_warp(sm, sm->unit_empty[slot], ((k / kUnitRing) - 1) & 1, 0x101)) {
      ok = false;
      break;
    }
    if (lane == 0) {
      if constexpr (kVar == kVarSplit) fetch_unit_split(p, sm, slot);
      else fetch_unit(p, sm, slot);
    }
    __syncwarp();
    if (!wait_warp(sm, sm->unit_full[slot], (k / kUnitRing) & 1, 0x102)) {
      ok = false;
      break;
    }
    const UnitInfo ui = sm->unit[slot];
    if (ui.seq < 0) break;
    const int hk = ui.head / (p.H / p.Hk);
    for (int c = 0; c < ui.nch; ++c, ++g) {
      const int s = g % kStages;
      const int t = ui.t0 + c * kChunk;
      const int len = min(kChunk, ui.end - t);
      // g and beta of tokens 2*lane and 2*lane+1 (issued before waiting for the stage)
      const int j0 = 2 * lane, j1 = 2 * lane + 1;
      const int64_t r0 = (int64_t)(t + j0), r1 = (int64_t)(t + j1);
      const float g0 = j0 < len ? p.g[r0 * p.g_st + (int64_t)ui.head * p.g_sh] : 0.f;
      const float g1 = j1 < len ? p.g[r1 * p.g_st + (int64_t)ui.head * p.g_sh] : 0.f;
      const float b0 =
          j0 < len ? __bfloat162float(p.beta[r0 * p.b_st + (int64_t)ui.head * p.b_sh]) : 0.f;
      const float b1 =
          j1 < len ? __bfloat162float(p.beta[r1 * p.b_st + (int64_t)ui.head * p.b_sh]) : 0.f;
      if (g >= (uint32_t)kStages &&
          !wait_warp(sm, sm->empty[s], ((g / kStages) - 1) & 1, 0x103)) {
        ok = false;
        break;
      }
      uint8_t *kq = base + OFF_STAGE + s * kStageBytes;
      uint8_t *vv = kq + kKQBytes;
      if (lane == 0) {
        mbar_expect_tx(&sm->full[s], tx);
        tma_load_3d(kq, mk, &sm->full[s], 0, hk, t);
        tma_load_3d(kq + 8192, mq, &sm->full[s], 0, hk, t);
        tma_load_3d(vv, mv, &sm->full[s], 0, ui.head, t);
        if (p.D == 128) {
          tma_load_3d(kq + 16384, mk, &sm->full[s], 64, hk, t);
          tma_load_3d(kq + 24576, mq, &sm->full[s], 64, hk, t);
          tma_load_3d(vv + 8192, mv, &sm->full[s], 64, ui.head, t);
        }
      }
      {
        // chunk-local cumsum of g and the decay vectors (the slot's previous chunk is
        // done: see kInfo)
        ChunkVec &cv = sm->cv[g % kInfo];
        float sum = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, sum, off);
          if (lane >= off) sum += y;
        }
        // decay factors e^x are evaluated as 2^(x log2 e) on the special-function unit
        constexpr float kLog2e = 1.4426950408889634f;
        const float G0 = (sum - g1) * kLog2e, G1 = sum * kLog2e;
        const float GL = __shfl_sync(0xffffffffu, G1, 31);
        float gmax = fmaxf(G0, G1), gmin = fminf(G0, G1);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
          gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, off));
          gmin = fminf(gmin, __shfl_xor_sync(0xffffffffu, gmin, off));
        }
        const bool fac = gmax - gmin <= kFacRange;
        cv.G[j0] = G0;
        cv.G[j1] = G1;
        const float e0 = ex2(G0), e1 = ex2(G1);
        cv.eG[j0] = e0;
        cv.eG[j1] = e1;
        cv.eGs[j0] = p.scale * e0;
        cv.eGs[j1] = p.scale * e1;
        cv.bfac[j0] = fac ? ex2(gmax - G0) : 0.f;
        cv.bfac[j1] = fac ? ex2(gmax - G1) : 0.f;
        cv.dec[j0] = ex2(GL - G0);
        cv.dec[j1] = ex2(GL - G1);
        cv.beta[j0] = b0;
        cv.beta[j1] = b1;
        if constexpr (kVar == kVarBwd) {
          float *gc = p.bw_gcum + (int64_t)t * p.H + ui.head;
          if (j0 < len) gc[(int64_t)j0 * p.H] = sum - g1;
          if (j1 < len) gc[(int64_t)j1 * p.H] = sum;
        }
        if (lane == 0) {
          cv.eL = ex2(GL);
          cv.Gref = gmax;
          cv.fac = fac ? 1 : 0;
          if constexpr (kVar == kVarCkpt)
            cv.ckrow = (c > 0 && (c * kChunk) % p.ckpt.every == 0)
                           ? p.ckpt.off[ui.seq] + (c * kChunk) / p.ckpt.every - 1
                           : -1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->full[s]);
    }
  }
  // drain: make sure no TMA write of ours is still in flight
  for (uint32_t i = 0; i < (uint32_t)kStages && i < g; ++i) {
    const uint32_t gi = g - 1 - i;
    mbar_wait(&sm->full[gi % kStages], (gi / kStages) & 1, nullptr, kWaitLimitNs);
  }
}

// MMA issue is split over two threads in different warps, because one thread
// issues a tcgen05.mma only every ~100 cycles whatever its size.  Issuer P
// runs the MMAs off the state chain (X1, U, O1, O2); issuer C runs the chain
// (Y, V', S update).  A stage is released once both have committed.
__device__ void issuer_drain(Small *sm) {
  mma_commit(&sm->drain);
  mbar_wait(&sm->drain, 0, nullptr, kWaitLimitNs);
}

// A shared-memory descriptor moved by `bytes` (a multiple of 16; the address field
// does not overflow inside the 227 KB window).
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

template <int kVar>
__device__ void role_issue_p(const Params &p, Small *sm, uint8_t *base) {
  const uint32_t tb = sm->tmem_base;
  const uint32_t sbase = smem_u32(base);
  const uint32_t id_x1 = idesc_bf16(128, 64, false, false);
  const uint32_t id_uw = idesc_bf16(128, 64, true, false);  // A = V^T (MN-major)
  const uint32_t id_n64 = idesc_bf16(128, 64, false, false);
  // descriptors of stage 0 / buffer 0; stages are kStageBytes apart
  const uint64_t d_kq = sdesc_sw128(sbase + OFF_STAGE, 0, 1024);          // K rows (K-major)
  const uint64_t d_q = sdesc_sw128(sbase + OFF_STAGE + 8192, 0, 1024);    // Q rows (K-major)
  const uint64_t d_v = sdesc_sw128(sbase + OFF_STAGE + kKQBytes, 8192, 1024);  // V (MN-major)
  const uint64_t d_tb = sdesc_sw128(sbase + OFF_TB, 0, 1024);
  const uint64_t d_p = sdesc_sw128(sbase + OFF_P, 0, 1024);
  const uint64_t d_kmn = sdesc_sw128(sbase + OFF_STAGE, 16384, 1024);  // K (MN-major)
  const uint64_t d_tbg = sdesc_sw128(sbase + OFF_TBG, 0, 1024);
  uint32_t g = 0;
  bool ok = true;
  // X1 of chunk gg into its U buffer (by parity).  It needs its stage, prep done
  // reading X1 of chunk gg-1 (one x1_full phase at a time), and chunk gg-2's
  // MMAs (the last readers of that U buffer and of the P buffer) complete, i.e.
  // chunk gg-2's stage released.
  auto x1_wait = [&](uint32_t gg, int code) {
    if (!wait1(sm, sm->full[gg % kStages], (gg / kStages) & 1, code)) return false;
    if (gg >= 1 && !wait1(sm, sm->x1_free, (gg - 1) & 1, code + 1)) return false;
    if (gg >= 2 && !wait1(sm, sm->empty[(gg - 2) % kStages], ((gg - 2) / kStages) & 1, code + 2))
      return false;
    tc_fence_after();
    return true;
  };
  auto issue_x1 = [&](uint32_t gg) {
    const uint64_t a = dadd(d_kq, (gg % kStages) * kStageBytes);
    const uint32_t d = tb + TM_U + (gg & 1) * 64;
#pragma unroll 1
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t ak = dadd(a, (kk / 4) * 16384 + (kk % 4) * 32);
      mma_bf16(d, ak, ak, id_x1, kk > 0);
    }
    mma_commit(&sm->x1_full);
  };
  for (uint32_t k = 0; ok; ++k) {
    const int slot = k % kUnitRing;
    if (!wait1(sm, sm->unit_full[slot], (k / kUnitRing) & 1, 0x201)) { ok = false; break; }
    const UnitInfo ui = sm->unit[slot];
    mbar_arrive(&sm->unit_empty[slot]);
    if (ui.seq < 0) break;
    for (int c = 0; c < ui.nch; ++c, ++g) {
      const uint32_t s = g % kStages;
      const uint32_t tu = tb + TM_U + (g & 1) * 64;
      if (c == 0) {
        if (!x1_wait(g, 0x202)) { ok = false; break; }
        issue_x1(g);
      }
      // next chunk's X1 first: prep of c+1 starts as soon as prep of c ends
      if (c + 1 < ui.nch) {
        if (!x1_wait(g + 1, 0x205)) { ok = false; break; }
        issue_x1(g + 1);
      }
      // U^T = V^T (Tm diag beta)^T
      if (!wait1(sm, sm->t_ready, g & 1, 0x208)) { ok = false; break; }
      tc_fence_after();
      if (kVar != kVarSplit || ui.mode != kUnitM) {  // a transition unit has v = 0: U = 0
        const uint64_t dv = dadd(d_v, s * kStageBytes);
#pragma unroll 1
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tu, dadd(dv, kk * 2048), dadd(d_tb, kk * 32), id_uw, kk > 0);
      }
      mma_commit(&sm->uw_full);
      if constexpr (kVar == kVarBwd) {
        // no output: -W^T = K^T (-Tm diag(beta e^G))^T into the O accumulator instead, once
        // the state warpgroup has read the previous chunk's and has started this chunk (its
        // s_ready arrival follows its o1_full wait for the previous chunk: without it, at a
        // unit boundary, this thread could commit o1_full twice ahead of that wait)
        if (!wait1(sm, sm->s_ready, g & 1, 0x209)) { ok = false; break; }
        if (g >= 1 && !wait1(sm, sm->o_free, (g - 1) & 1, 0x20a)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dk = dadd(d_kmn, s * kStageBytes);
#pragma unroll 1
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tb + TM_O, dadd(dk, kk * 2048), dadd(d_tbg, kk * 32), id_uw, kk > 0);
        mma_commit(&sm->o1_full);
        mma_commit(&sm->o_full);
        mma_commit(&sm->empty[s]);
        continue;
      }
      // O^T (inter-chunk part) = S^T Q^T, once the epilogue has read the previous chunk's
      if (!wait1(sm, sm->s_ready, g & 1, 0x209)) { ok = false; break; }
      if (g >= 1 && !wait1(sm, sm->o_free, (g - 1) & 1, 0x20a)) { ok = false; break; }
      tc_fence_after();
      {
        const uint64_t dq = dadd(d_q, s * kStageBytes);
#pragma unroll 1
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tb + TM_O, tb + TM_SB + kk * 8, dadd(dq, (kk / 4) * 16384 + (kk % 4) * 32),
                      id_n64, kk > 0);
      }
      mma_commit(&sm->o1_full);  // the bf16 copy of S^T is free as far as O1 goes
      // O2^T = V'^T P^T
      if (!wait1(sm, sm->vp_ready, g & 1, 0x20b)) { ok = false; break; }
      tc_fence_after();
      {
        const uint64_t dp = dadd(d_p, (g & 1) * 8192);
#pragma unroll 1
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ts(tb + TM_O2, tu + kk * 8, dadd(dp, kk * 32), id_n64, kk > 0);
      }
      mma_commit(&sm->o_full);
      mma_commit(&sm->empty[s]);
    }
  }
  issuer_drain(sm);
}

template <int kVar>
__device__ void role_issue_c(const Params &p, Small *sm, uint8_t *base) {
  const uint32_t tb = sm->tmem_base;
  const uint32_t sbase = smem_u32(base);
  const uint32_t id_n64 = idesc_bf16(128, 64, false, false);
  const uint32_t id_su = idesc_bf16(128, 128, false, true);  // B = K (MN-major)
  const uint64_t d_k = sdesc_sw128(sbase + OFF_STAGE, 0, 1024);        // K rows (K-major)
  const uint64_t d_kmn = sdesc_sw128(sbase + OFF_STAGE, 16384, 1024);  // K (MN-major)
  const uint64_t d_tbg = sdesc_sw128(sbase + OFF_TBG, 0, 1024);
  uint32_t g = 0;
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    const int slot = k % kUnitRing;
    if (!wait1(sm, sm->unit_full[slot], (k / kUnitRing) & 1, 0x211)) { ok = false; break; }
    const UnitInfo ui = sm->unit[slot];
    mbar_arrive(&sm->unit_empty[slot]);
    if (ui.seq < 0) break;
    for (int c = 0; c < ui.nch; ++c, ++g) {
      const uint32_t s = g % kStages;
      const uint32_t tu = tb + TM_U + (g & 1) * 64;
      const uint64_t dk = dadd(d_k, s * kStageBytes), dkmn = dadd(d_kmn, s * kStageBytes);
      // Y = S^T K^T  (S before this chunk, bf16 in TMEM)
      if (!wait1(sm, sm->s_ready, g & 1, 0x212)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16_ts(tb + TM_Y, tb + TM_SB + kk * 8, dadd(dk, (kk / 4) * 16384 + (kk % 4) * 32),
                    id_n64, kk > 0);
      mma_commit(&sm->y_full);
      // V'^T = U^T + Y (-Tm diag(beta e^G))^T
      if (!wait1(sm, sm->y_ready, g & 1, 0x213)) { ok = false; break; }
      if (!wait1(sm, sm->uw_full, g & 1, 0x214)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int kk = 0; kk < 4; ++kk)  // (a transition unit has no U to add to)
        mma_bf16_ts(tu, tb + TM_Y + kk * 8, dadd(d_tbg, kk * 32), id_n64,
                    (kVar != kVarSplit || ui.mode != kUnitM || kk > 0) ? 1u : 0u);
      mma_commit(&sm->vp_full);
      // S^T += V''^T K
      if (!wait1(sm, sm->vp_ready, g & 1, 0x215)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16_ts(tb + TM_S, tu + 32 + kk * 8, dadd(dkmn, kk * 2048), id_su, 1);
      mma_commit(&sm->s_full);
      mma_commit(&sm->empty[s]);
    }
  }
  issuer_drain(sm);
}

__device__ __forceinline__ void store_chunk8(uint32_t tile, int row, int col, const float *v) {
  st_shared_v4(tile + sw128_off(row, col), pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
               pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}

__device__ __forceinline__ void ld_f4(const float *p, float *v) {
  const float4 x = *reinterpret_cast<const float4 *>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void st_f4(float *p, const float *v) {
  *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

// One warp: c[16 x 16] += A[16 x K] * B[K x 16] on the tensor pipe (tf32 in, fp32
// accumulate, mma.sync m16n8k8); A and B are fp32 row-major in shared memory.  The fp32
// bit patterns go to the tensor core as they are: it reads the sign, exponent and top 10
// mantissa bits of each tf32 operand, i.e. the operands are truncated to tf32 (relative
// error below 2^-10) instead of rounded by a conversion instruction per element.
__device__ __forceinline__ void warp_mm16(const float *A, int lda, const float *B, int ldb,
                                          int K, float (&c)[2][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  for (int k = 0; k < K; k += 8) {
    const uint32_t a0 = __float_as_uint(A[g * lda + k + t]);
    const uint32_t a1 = __float_as_uint(A[(g + 8) * lda + k + t]);
    const uint32_t a2 = __float_as_uint(A[g * lda + k + t + 4]);
    const uint32_t a3 = __float_as_uint(A[(g + 8) * lda + k + t + 4]);
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const uint32_t b0 = __float_as_uint(B[(k + t) * ldb + n * 8 + g]);
      const uint32_t b1 = __float_as_uint(B[(k + t + 4) * ldb + n * 8 + g]);
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[n][0]), "+f"(c[n][1]), "+f"(c[n][2]), "+f"(c[n][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
}

__device__ __forceinline__ void warp_store16(float *C, int ldc, const float (&c)[2][4], float s) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    C[g * ldc + n * 8 + 2 * t] = s * c[n][0];
    C[g * ldc + n * 8 + 2 * t + 1] = s * c[n][1];
    C[(g + 8) * ldc + n * 8 + 2 * t] = s * c[n][2];
    C[(g + 8) * ldc + n * 8 + 2 * t + 1] = s * c[n][3];
  }
}

// The prep warpgroup.  `row` is this thread's TMEM lane (0..127).
template <bool kVarW>
__device__ void role_prep(const Params &p, Small *sm, uint8_t *base, int row) {
  const uint32_t tb = sm->tmem_base;
  const uint32_t sbase = smem_u32(base);
  const uint32_t lane_base = (uint32_t)(row & ~31);
  float *AS = reinterpret_cast<float *>(base + OFF_A);  // 64 x kLdA fp32
  float *YS = reinterpret_cast<float *>(base + OFF_Y);  // 32 x kLdY fp32 (also 2 x 16 x kLdX)
  const int pid = row;           // 0..127, unique in the warpgroup
  const int wq = pid >> 5;       // warp index by lane quadrant
  // the operand tiles Tm diag(beta) and -Tm diag(beta e^G) are zero above the diagonal's
  // 8-column groups: cleared once here, only the lower groups are rewritten per chunk
  for (int i = pid; i < 16384 / 16; i += 128) st_shared_v4(sbase + OFF_TB + i * 16, 0u, 0u, 0u, 0u);
  fence_async_smem();
  uint32_t g = 0;
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    const int slot = k % kUnitRing;
    if (!wait_wg(sm, sm->unit_full[slot], (k / kUnitRing) & 1, 0x301, kBarPrep)) break;
    const UnitInfo ui = sm->unit[slot];
    mbar_arrive(&sm->unit_empty[slot]);
    if (ui.seq < 0) break;
    for (int c = 0; c < ui.nch; ++c, ++g) {
      const uint32_t s = g % kStages;
      const int t = ui.t0 + c * kChunk;
      const int len = min(kChunk, ui.end - t);
      const uint32_t kq_a = sbase + OFF_STAGE + s * kStageBytes;
      const int cb2 = g & 1;
      // the chunk's stage and X1 (one barrier for both waits)
      {
        const bool bad = !mbar_wait(&sm->full[s], (g / kStages) & 1, &sm->abort, kWaitLimitNs) ||
                         !mbar_wait(&sm->x1_full, g & 1, &sm->abort, kWaitLimitNs);
        if (named_bar_or(kBarPrep, 128, bad)) {
          fail(sm, 0x302);
          ok = false;
          break;
        }
      }
      tc_fence_after();
      // zero the rows past the chunk's end (they hold the next segment's tokens); the
      // MMAs that read them before this (X1, Y, O1) only feed masked or unstored values
      if (len < kChunk) {
        for (int idx = pid; idx < (kChunk - len) * 6; idx += 128) {
          const int r = len + idx / 6, which = idx % 6;
          // which: 0,1 = K in key blocks 0,1; 2,3 = Q in key blocks 0,1; 4,5 = V blocks 0,1
          uint32_t tile;
          int rr = r;
          if (which < 2) tile = kq_a + which * 16384;
          else if (which < 4) { tile = kq_a + (which - 2) * 16384; rr = r + 64; }
          else tile = kq_a + kKQBytes + (which - 4) * 8192;
          zero_row(tile, rr);
        }
        fence_async_smem();
      }
      const ChunkVec &cv = sm->cv[g % kInfo];
      // X1 rows: lanes 0-63 = K K^T (rows of A), lanes 64-127 = Q K^T (rows of P)
      {
        // A_ij = beta_i e^{G_i-G_j} k_i.k_j (j < i);  P_ij = scale e^{G_i-G_j} q_i.k_j (j <= i).
        // Only what the solve and the O2 MMA read is masked: A's entries on and above the
        // diagonal are never read except the two 16 x 16 blocks inside the 32 x 32
        // diagonal blocks (rows 0-15 / 32-47, the next 16 columns), which must be zero;
        // P is an MMA operand, so all its entries above the diagonal must be zero.  Rows
        // past the chunk's end are zero (ci = 0).  Per 32-column half, the warp's rows
        // (one lane quadrant) lie either below, on or above the half's diagonal block.
        const int i = row & 63;
        const bool is_a = row < 64;
        const bool upper = i < 32;  // same for the whole warp
        const float scl = is_a ? cv.beta[i] : p.scale;
        const bool fac = cv.fac != 0;  // same for the whole chunk
        const float gi = cv.G[i];
        const float ci = i < len ? (fac ? scl * ex2(gi - cv.Gref) : scl) : 0.f;
        const uint32_t tx1 = tb + TM_U + (g & 1) * 64;
        const uint32_t ptile = sbase + OFF_P + cb2 * 8192;
        // kept columns u (within the diagonal half) satisfy u <= keep
        const int keep = is_a ? (((i & 31) < 16) ? 15 : 31) : (i & 31);
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {  // 32 columns at a time
          if (hh == 1 && upper) {  // above the diagonal: A is never read there, P is zero
            if (!is_a) {
              const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int q = 0; q < 4; ++q) store_chunk8(ptile, i, 32 + q * 8, z);
            }
            continue;
          }
          const int lim = (hh == 0) == upper ? keep : 31;  // diagonal half or fully below
          uint32_t r[32];
          tmem_ld32(tmem_addr(tx1, lane_base, hh * 32), r);
          float f[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) ld_f4((fac ? cv.bfac : cv.G) + hh * 32 + q * 4, f + q * 4);
          if (!fac) {
#pragma unroll
            for (int u = 0; u < 32; ++u) f[u] = ex2(gi - f[u]);
          }
          tmem_ld_wait();
          if ((hh == 0) != upper) {  // the whole half is below the diagonal: nothing to mask
#pragma unroll
            for (int u = 0; u < 32; u += 2) {
              mul_x2(f[u], f[u + 1], ci, ci);
              mul_x2(f[u], f[u + 1], __uint_as_float(r[u]), __uint_as_float(r[u + 1]));
            }
          } else {
#pragma unroll
            for (int u = 0; u < 32; u += 2) {
              float p0 = f[u], p1 = f[u + 1];
              mul_x2(p0, p1, ci, ci);
              mul_x2(p0, p1, __uint_as_float(r[u]), __uint_as_float(r[u + 1]));
              f[u] = u <= lim ? p0 : 0.f;
              f[u + 1] = u + 1 <= lim ? p1 : 0.f;
            }
          }
          if (is_a) {
#pragma unroll
            for (int q = 0; q < 8; ++q) st_f4(AS + i * kLdA + hh * 32 + q * 4, f + q * 4);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) store_chunk8(ptile, i, hh * 32 + q * 8, f + q * 8);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm->x1_free);
      named_bar(kBarPrep, 128);
      // ---- Tm = (I + A)^-1, 64 x 64 unit lower triangular, fp32 ----
      // phase 1: the four 16 x 16 diagonal blocks by forward substitution, one
      // column per thread (threads 0..63; a block's 16 threads share a warp); the next
      // row's entries are loaded while the current row is solved
      if (pid < 64) {
        const int b = (pid >> 4) & 3, cc = pid & 15;
        float *blk = AS + 16 * b * kLdA + 16 * b;
        float x[16];
        float an[16];  // entries m < r of the next row r
#pragma unroll
        for (int m = 0; m < 16; ++m) an[m] = 0.f;
        an[0] = blk[1 * kLdA];
        x[0] = (cc == 0) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
          float a[16];
#pragma unroll
          for (int m = 0; m < 16; ++m) a[m] = an[m];
          if (r + 1 < 16) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (q * 4 < r + 1) ld_f4(blk + (r + 1) * kLdA + q * 4, an + q * 4);
          }
          float s0 = (r == cc) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
          for (int m = 0; m < r; ++m) {
            if (m & 1) s1 -= a[m] * x[m]; else s0 -= a[m] * x[m];
          }
          x[r] = s0 + s1;
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 16; ++r) blk[r * kLdA + cc] = x[r];
      }
      named_bar(kBarPrep, 128);
      // phase 2: T_{b+1,b} = -D_{b+1} A_{b+1,b} D_b for b = 0, 2 (warps 0 and 1)
      {
        float *X = YS + wq * 16 * kLdX;
        const int ob = 32 * wq, oa = ob + 16;
        if (wq < 2) {
          float acc[2][4] = {};
          warp_mm16(AS + oa * kLdA + ob, kLdA, AS + ob * kLdA + ob, kLdA, 16, acc);
          warp_store16(X, kLdX, acc, 1.f);
          __syncwarp();  // X is this warp's own scratch
          float acc2[2][4] = {};
          warp_mm16(AS + oa * kLdA + oa, kLdA, X, kLdX, 16, acc2);
          warp_store16(AS + oa * kLdA + ob, kLdA, acc2, -1.f);
        }
      }
      named_bar(kBarPrep, 128);
      // phase 3: Tm[32:64, 0:32] = -T2 (A[32:64, 0:32] T1), one 16 x 16 tile per warp
      {
        const int mt = wq >> 1, nt = wq & 1;
        float acc[2][4] = {};
        warp_mm16(AS + (32 + 16 * mt) * kLdA, kLdA, AS + 16 * nt, kLdA, 32, acc);
        warp_store16(YS + 16 * mt * kLdY + 16 * nt, kLdY, acc, 1.f);
        named_bar(kBarPrep, 128);
        float acc2[2][4] = {};
        warp_mm16(AS + (32 + 16 * mt) * kLdA + 32, kLdA, YS + 16 * nt, kLdY, 32, acc2);
        // the result overwrites A[32:64, 0:32], which every warp finished reading before
        // the barrier above
        warp_store16(AS + (32 + 16 * mt) * kLdA + 16 * nt, kLdA, acc2, -1.f);
      }
      named_bar(kBarPrep, 128);
      if (kVarW && p.bw_t) {
        // Tm itself for the backward (fp32), half a row per thread; the scratch holds only
        // its lower triangle and diagonal
        const int ri = pid & 63, hc = (pid >> 6) * 32;
        const int64_t cid = p.seg[ui.seq].chunk_off + c;
        float *tg = p.bw_t + ((cid * p.H + ui.head) * 64 + ri) * 64 + hc;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float v4[4];
          ld_f4(AS + ri * kLdA + hc + q * 4, v4);
#pragma unroll
          for (int u = 0; u < 4; ++u) v4[u] = hc + q * 4 + u <= ri ? v4[u] : 0.f;
          st_f4(tg + q * 4, v4);
        }
      }
      // Tm diag(beta) and -Tm diag(beta e^G) as bf16 operands, once the previous chunk's
      // MMAs that read them are done
      {
        if (g >= 1 && !wait_wg(sm, sm->vp_full, (g - 1) & 1, 0x305, kBarPrep)) { ok = false; break; }
        // (the backward recompute's W MMA reads Tm diag(beta e^G) too)
        if (kVarW && g >= 1 && !wait_wg(sm, sm->o_full, (g - 1) & 1, 0x306, kBarPrep)) {
          ok = false;
          break;
        }
        // 8 columns at a time, lower-triangle groups only: row r holds r/8 + 1 of them, so
        // rows q and 63 - q together hold 9, which the pair's four threads share (at most
        // three each).  A rolled loop keeps this block small in the instruction cache,
        // which the SMs of a GPC share at full occupancy.
        const int q = pid >> 2, nq = (q >> 3) + 1;
#pragma unroll 1
        for (int gi = pid & 3; gi < 9; gi += 4) {
          const int ri = gi < nq ? q : 63 - q;
          const int c0 = 8 * (gi < nq ? gi : gi - nq);
          const int lim = ri - c0;  // column c0 + u is on or below the diagonal for u <= lim
          float t8[8], b8[8], e8[8], v[8];
          ld_f4(AS + ri * kLdA + c0, t8);
          ld_f4(AS + ri * kLdA + c0 + 4, t8 + 4);
          ld_f4(cv.beta + c0, b8);
          ld_f4(cv.beta + c0 + 4, b8 + 4);
          ld_f4(cv.eG + c0, e8);
          ld_f4(cv.eG + c0 + 4, e8 + 4);
#pragma unroll
          for (int u = 0; u < 8; u += 2) {
            mul_x2(t8[u], t8[u + 1], b8[u], b8[u + 1]);
            v[u] = (u <= lim) ? t8[u] : 0.f;
            v[u + 1] = (u + 1 <= lim) ? t8[u + 1] : 0.f;
          }
          store_chunk8(sbase + OFF_TB, ri, c0, v);
#pragma unroll
          for (int u = 0; u < 8; u += 2) mul_x2(v[u], v[u + 1], -e8[u], -e8[u + 1]);
          store_chunk8(sbase + OFF_TBG, ri, c0, v);
        }
      }
      fence_async_smem();
      mbar_arrive(&sm->t_ready);
    }
  }
}

// Pack 64 fp32 values (two TMEM loads of 32 columns) into 32 bf16 pairs.
__device__ __forceinline__ void pack64(const uint32_t (&a)[32], const uint32_t (&b)[32],
                                       uint32_t (&o)[32]) {
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    o[u] = pack_bf16(__uint_as_float(a[2 * u]), __uint_as_float(a[2 * u + 1]));
    o[16 + u] = pack_bf16(__uint_as_float(b[2 * u]), __uint_as_float(b[2 * u + 1]));
  }
}

// Row dv of the unit's initial state (S^T row = column dv of h0, zero without h0)
// into TMEM; once per unit, so kept out of line.
__device__ __noinline__ void state_from_h0(const Params &p, uint32_t taddr, int64_t sidx, int dv) {
  const int D = p.D;
  const bool from_h0 = p.has_h0 && dv < D;
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    uint32_t r[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int j = cb * 32 + u;
      r[u] = __float_as_uint((from_h0 && j < D) ? p.h0[sidx + (int64_t)j * D + dv] : 0.f);
    }
    tmem_st32(taddr + cb * 32, r);
  }
  tmem_st_wait();
}

// Row dv of S^T (TMEM, fp32) -> column dv of a [dk][dv] fp32 state at `dst` (state
// checkpoints), kept out of line.
__device__ __noinline__ void store_state(uint32_t taddr, float *dst, int D, int dv) {
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    uint32_t r[32];
    tmem_ld32(taddr + cb * 32, r);
    tmem_ld_wait();
    if (dv < D) {
#pragma unroll
      for (int u = 0; u < 32; ++u)
        if (cb * 32 + u < D) dst[(int64_t)(cb * 32 + u) * D + dv] = __uint_as_float(r[u]);
    }
  }
}

// Initial state of a split unit (row dv of S^T): zero (piece offset), the identity (piece
// transition), or a [dk][dv] state from the split buffer; kept out of line.
__device__ __noinline__ void state_from_split(const Params &p, uint32_t taddr, const UnitInfo &ui,
                                              int dv) {
  const int D = p.D;
  const float *src = ui.mode == kUnitFinal ? p.split.states + (int64_t)ui.sin * D * D : nullptr;
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    uint32_t r[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int j = cb * 32 + u;
      float x = 0.f;
      if (j < D && dv < D) {
        if (src) x = src[(int64_t)j * D + dv];
        else if (ui.mode == kUnitM) x = j == dv ? 1.f : 0.f;
      }
      r[u] = __float_as_uint(x);
    }
    tmem_st32(taddr + cb * 32, r);
  }
  tmem_st_wait();
}

// The state warpgroup.  `row` is this thread's TMEM lane = value dimension dv.  The
// checkpoint and split variants are separate instantiations, so that the plain
// forward's code is untouched.
// Per chunk: S^T -> bf16 (A operand of Y and O1) and e^{G_last} S^T; Y -> bf16;
// V'^T -> bf16 V'^T and V''^T; and the previous chunk's output.
template <int kVar>
__device__ void role_state(const Params &p, Small *sm, uint8_t *base, int row) {
  const uint32_t tb = sm->tmem_base;
  const uint32_t lane_base = (uint32_t)(row & ~31);
  const int dv = row;
  const int D = p.D;
  uint8_t *stage_o = base + OFF_STG;  // output staging [64 tokens][128 dv] bf16
  uint32_t g = 0;
  bool ok = true;
  int prev_t = 0, prev_len = 0, prev_head = 0;
  // output of chunk gg, part 1: O = scale e^{G_i} (S^T Q^T)_i + (V'^T P^T)_i (P carries
  // the scale) from TMEM into the staging tile (frees the accumulators early)
  auto epi_read = [&](uint32_t gg) -> bool {
    if (!wait_wg(sm, sm->o_full, gg & 1, 0x401, kBarState)) return false;
    tc_fence_after();
    const float *eG = sm->cv[gg % kInfo].eGs;
    __nv_bfloat16 *st = reinterpret_cast<__nv_bfloat16 *>(stage_o) + dv;
#pragma unroll 1
    for (int hb = 0; hb < 2; ++hb) {
      uint32_t r1[32], r2[32];
      tmem_ld32(tmem_addr(tb + TM_O, lane_base, hb * 32), r1);
      tmem_ld32(tmem_addr(tb + TM_O2, lane_base, hb * 32), r2);
      float e[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) ld_f4(eG + hb * 32 + q * 4, e + q * 4);
      tmem_ld_wait();
      if (hb == 1) {
        tc_fence_before();
        mbar_arrive(&sm->o_free);
      }
#pragma unroll
      for (int u = 0; u < 32; u += 2) {
        float o0 = __uint_as_float(r1[u]), o1 = __uint_as_float(r1[u + 1]);
        fma_x2(o0, o1, e[u], e[u + 1], __uint_as_float(r2[u]), __uint_as_float(r2[u + 1]));
        st[(hb * 32 + u) * 128] = __float2bfloat16_rn(o0);
        st[(hb * 32 + u + 1) * 128] = __float2bfloat16_rn(o1);
      }
    }
    return true;
  };
  // backward recompute: W of chunk gg (-W^T, key dim on the lanes, in the O accumulator)
  // to W[t][head][dk] bf16 for the chunk's tokens
  auto w_out = [&](uint32_t gg) -> bool {
    if (!wait_wg(sm, sm->o_full, gg & 1, 0x401, kBarState)) return false;
    tc_fence_after();
    uint32_t r0[32], r1[32];
    tmem_ld32(tmem_addr(tb + TM_O, lane_base, 0), r0);
    tmem_ld32(tmem_addr(tb + TM_O, lane_base, 32), r1);
    tmem_ld_wait();
    tc_fence_before();
    mbar_arrive(&sm->o_free);
    if (dv < D) {
      const int64_t st = (int64_t)p.H * D;
      __nv_bfloat16 *wp = p.bw_w + (int64_t)prev_t * st + (int64_t)prev_head * D + dv;
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        if (u < prev_len) wp[u * st] = __float2bfloat16_rn(-__uint_as_float(r0[u]));
        if (32 + u < prev_len) wp[(32 + u) * st] = __float2bfloat16_rn(-__uint_as_float(r1[u]));
      }
    }
    return true;
  };
  // part 2: the staging tile to global memory, 16 bytes per store
  auto epi_store = [&]() {
    named_bar(kBarState, 128);
    const int chunks_per_row = D / 8;
#pragma unroll 2
    for (int idx = row; idx < prev_len * 16; idx += 128) {
      const int i = idx >> 4, ch = idx & 15;
      if (ch < chunks_per_row) {
        const uint4 val = *reinterpret_cast<const uint4 *>(stage_o + i * 256 + ch * 16);
        *reinterpret_cast<uint4 *>(p.o + (int64_t)(prev_t + i) * p.o_st +
                                   (int64_t)prev_head * p.o_sh + ch * 8) = val;
      }
    }
  };
  for (uint32_t k = 0; ok; ++k) {
    const int slot = k % kUnitRing;
    if (!wait_wg(sm, sm->unit_full[slot], (k / kUnitRing) & 1, 0x402, kBarState)) break;
    const UnitInfo ui = sm->unit[slot];
    mbar_arrive(&sm->unit_empty[slot]);
    if (ui.seq < 0) break;
    const int64_t sidx = ((int64_t)ui.seq * p.H + ui.head) * D * D;
    // row dv of S^T, key columns [c0, c0 + 64)
    auto load_s = [&](int c0, uint32_t (&r0)[32], uint32_t (&r1)[32]) {
      tmem_ld32(tmem_addr(tb + TM_S, lane_base, c0), r0);
      tmem_ld32(tmem_addr(tb + TM_S, lane_base, c0 + 32), r1);
      tmem_ld_wait();
    };
    for (int c = 0; c < ui.nch; ++c, ++g) {
      const int t = ui.t0 + c * kChunk;
      const int len = min(kChunk, ui.end - t);
      // the chunk's vectors are written before its stage is marked full
      if (!wait_wg(sm, sm->full[g % kStages], (g / kStages) & 1, 0x403, kBarState)) { ok = false; break; }
      const ChunkVec &cv = sm->cv[g % kInfo];
      if (c >= 1 && !wait_wg(sm, sm->s_full, (g - 1) & 1, 0x404, kBarState)) { ok = false; break; }
      // the bf16 copy of S^T is rewritten once the previous chunk's O1 has read it
      if (g >= 1 && !wait_wg(sm, sm->o1_full, (g - 1) & 1, 0x408, kBarState)) { ok = false; break; }
      tc_fence_after();
      if (c == 0) {
        if constexpr (kVar == kVarSplit) {
          if (ui.mode == kUnitFull) state_from_h0(p, tmem_addr(tb + TM_S, lane_base, 0), sidx, dv);
          else state_from_split(p, tmem_addr(tb + TM_S, lane_base, 0), ui, dv);
        } else if (p.has_h0) {
          state_from_h0(p, tmem_addr(tb + TM_S, lane_base, 0), sidx, dv);
        } else {  // zero state, inline (the out-of-line call cost ~6000 cycles per unit)
          uint32_t z[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) z[u] = 0u;
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) tmem_st32(tmem_addr(tb + TM_S, lane_base, cb * 32), z);
        }
      }
      if constexpr (kVar == kVarCkpt) {
        // the state entering this chunk, after c * 64 of the segment's tokens (row chosen
        // by the producer)
        if (cv.ckrow >= 0)
          store_state(tmem_addr(tb + TM_S, lane_base, 0),
                      p.ckpt.h + ((int64_t)cv.ckrow * p.H + ui.head) * D * D, D, dv);
      }
      // S^T -> bf16 pairs (A operand of Y and O1), and e^{G_last} S^T (the base of this
      // chunk's S^T += V''^T K) back in place
      const float eL = cv.eL;
#pragma unroll 1
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t r0[32], r1[32], pk[32];
        load_s(hb * 64, r0, r1);
        pack64(r0, r1, pk);
        tmem_st32(tmem_addr(tb + TM_SB, lane_base, hb * 32), pk);
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          mul_x2(r0[u], r0[u + 1], eL, eL);
          mul_x2(r1[u], r1[u + 1], eL, eL);
        }
        tmem_st32(tmem_addr(tb + TM_S, lane_base, hb * 64), r0);
        tmem_st32(tmem_addr(tb + TM_S, lane_base, hb * 64 + 32), r1);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm->s_ready);
      if constexpr (kVar == kVarBwd) {
        // the state entering this chunk as the products use it (bf16) to h[chunk][dk][dv]:
        // column m of the bf16 copy holds key dims 2m, 2m + 1 (rewritten only by this
        // warpgroup's next state conversion)
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem_addr(tb + TM_SB, lane_base, 0), r0);
        tmem_ld32(tmem_addr(tb + TM_SB, lane_base, 32), r1);
        tmem_ld_wait();
        if (dv < D) {
          const int64_t cid = p.seg[ui.seq].chunk_off + c;
          uint16_t *hp = reinterpret_cast<uint16_t *>(p.bw_h) + (cid * p.H + ui.head) * D * D + dv;
#pragma unroll
          for (int m = 0; m < 32; ++m) {
            hp[(2 * m) * D] = (uint16_t)(r0[m] & 0xffffu);
            hp[(2 * m + 1) * D] = (uint16_t)(r0[m] >> 16);
          }
          if (D == 128) {
#pragma unroll
            for (int m = 0; m < 32; ++m) {
              hp[(64 + 2 * m) * D] = (uint16_t)(r1[m] & 0xffffu);
              hp[(64 + 2 * m + 1) * D] = (uint16_t)(r1[m] >> 16);
            }
          }
        }
        if (c >= 1 && !w_out(g - 1)) { ok = false; break; }
      }
      // previous chunk's output accumulators (same unit) -> staging, while Y is computed
      if (kVar != kVarBwd && c >= 1 && !epi_read(g - 1)) { ok = false; break; }
      // Y -> bf16 pairs in place; token columns past the chunk's end are zeroed so that
      // whatever the stage holds there cannot reach V'
      if (!wait_wg(sm, sm->y_full, g & 1, 0x405, kBarState)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t r0[32], r1[32], pk[32];
        tmem_ld32(tmem_addr(tb + TM_Y, lane_base, 0), r0);
        tmem_ld32(tmem_addr(tb + TM_Y, lane_base, 32), r1);
        tmem_ld_wait();
        if (len < kChunk) {
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            if (u >= len) r0[u] = 0u;
            if (32 + u >= len) r1[u] = 0u;
          }
        }
        pack64(r0, r1, pk);
        tmem_st32(tmem_addr(tb + TM_Y, lane_base, 0), pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm->y_ready);
      if (kVar != kVarBwd && c >= 1) epi_store();
      // V'^T -> bf16 V'^T (columns 0-31) and V''^T = V'^T diag(e^{G_last - G}) (32-63)
      if (!wait_wg(sm, sm->vp_full, g & 1, 0x406, kBarState)) { ok = false; break; }
      tc_fence_after();
      {
        const uint32_t tu = tb + TM_U + (g & 1) * 64;
        uint32_t r0[32], r1[32], pk[32];
        tmem_ld32(tmem_addr(tu, lane_base, 0), r0);
        tmem_ld32(tmem_addr(tu, lane_base, 32), r1);
        tmem_ld_wait();
        pack64(r0, r1, pk);
        tmem_st32(tmem_addr(tu, lane_base, 0), pk);
        if constexpr (kVar == kVarBwd) {
          // V' (bf16, as the products use it) to V'[t][head][dv]; pk[m] holds tokens 2m, 2m + 1
          if (dv < D) {
            const int64_t st = (int64_t)p.H * D;
            uint16_t *vp = reinterpret_cast<uint16_t *>(p.bw_vn) + (int64_t)t * st +
                           (int64_t)ui.head * D + dv;
#pragma unroll
            for (int m = 0; m < 32; ++m) {
              if (2 * m < len) vp[(2 * m) * st] = (uint16_t)(pk[m] & 0xffffu);
              if (2 * m + 1 < len) vp[(2 * m + 1) * st] = (uint16_t)(pk[m] >> 16);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float d[4];
          ld_f4(cv.dec + q * 4, d);
#pragma unroll
          for (int u = 0; u < 4; u += 2) mul_x2(r0[q * 4 + u], r0[q * 4 + u + 1], d[u], d[u + 1]);
          ld_f4(cv.dec + 32 + q * 4, d);
#pragma unroll
          for (int u = 0; u < 4; u += 2) mul_x2(r1[q * 4 + u], r1[q * 4 + u + 1], d[u], d[u + 1]);
        }
        pack64(r0, r1, pk);
        tmem_st32(tmem_addr(tu, lane_base, 32), pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm->vp_ready);
      prev_t = t;
      // offset and transition units of a split segment store no output
      prev_len = (kVar == kVarSplit && (ui.mode == kUnitR || ui.mode == kUnitM)) ? 0 : len;
      prev_head = ui.head;
    }
    if (!ok) break;
    // end of the unit: final state, then the last chunk's output
    if (!wait_wg(sm, sm->s_full, (g - 1) & 1, 0x407, kBarState)) break;
    tc_fence_after();
    if constexpr (kVar == kVarSplit) {
      float *dst = ui.sout >= 0 ? p.split.states + (int64_t)ui.sout * D * D
                                : (ui.sout == -1 && p.ht ? p.ht + sidx : nullptr);
      if (dst) store_state(tmem_addr(tb + TM_S, lane_base, 0), dst, D, dv);
    } else {
      if (p.ht) {
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tb + TM_S, lane_base, cb * 32), r);
          tmem_ld_wait();
          if (dv < D) {
#pragma unroll
            for (int u = 0; u < 32; ++u)
              if (cb * 32 + u < D) p.ht[sidx + (int64_t)(cb * 32 + u) * D + dv] = __uint_as_float(r[u]);
          }
        }
      }
    }
    if constexpr (kVar == kVarCkpt) {
      const int seg_len = ui.end - ui.t0;
      if (seg_len % p.ckpt.every == 0) {
        const int64_t r = p.ckpt.off[ui.seq] + seg_len / p.ckpt.every - 1;
        store_state(tmem_addr(tb + TM_S, lane_base, 0), p.ckpt.h + (r * p.H + ui.head) * D * D,
                    D, dv);
      }
    }
    if constexpr (kVar == kVarBwd) {
      if (!w_out(g - 1)) break;
    } else {
      if (!epi_read(g - 1)) break;
      epi_store();
    }
  }
}

// kVar: the plain forward, the variant that also writes state checkpoints, or the one
// that runs split-segment pieces (separate kernels, so the plain forward's code is not
// touched by the others)
template <int kVar>
__global__ void __launch_bounds__(kThreads, 1)
    k_fused(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
            const __grid_constant__ CUtensorMap mv, const Params p) {
  extern __shared__ uint8_t dyn_smem[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  Small *sm = reinterpret_cast<Small *>(base + OFF_SMALL);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm->full[s], 2);
      mbar_init(&sm->empty[s], 2);  // one commit from each MMA issuer
    }
    mbar_init(&sm->x1_full, 1);
    mbar_init(&sm->x1_free, 128);
    mbar_init(&sm->t_ready, 128);
    mbar_init(&sm->uw_full, 1);
    mbar_init(&sm->o1_full, 1);
    mbar_init(&sm->s_ready, 128);
    mbar_init(&sm->y_full, 1);
    mbar_init(&sm->y_ready, 128);
    mbar_init(&sm->vp_full, 1);
    mbar_init(&sm->vp_ready, 128);
    mbar_init(&sm->s_full, 1);
    mbar_init(&sm->o_full, 1);
    mbar_init(&sm->o_free, 128);
    mbar_init(&sm->drain, 2);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&sm->unit_full[i], 1);
      mbar_init(&sm->unit_empty[i], 2 + 128 + 128);
    }
    sm->abort = 0;
    fence_mbar_init();
  }
  if (p.D != 128) {  // head dim 64: the upper key/value blocks stay zero
    for (int s = 0; s < kStages; ++s) {
      uint32_t *z = reinterpret_cast<uint32_t *>(base + OFF_STAGE + s * kStageBytes + 16384);
      for (int i = threadIdx.x; i < 16384 / 4; i += kThreads) z[i] = 0;
      z = reinterpret_cast<uint32_t *>(base + OFF_STAGE + s * kStageBytes + kKQBytes + 8192);
      for (int i = threadIdx.x; i < 8192 / 4; i += kThreads) z[i] = 0;
    }
    fence_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&mq);
    tma_prefetch_map(&mk);
    tma_prefetch_map(&mv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    role_producer<kVar>(p, sm, base, &mq, &mk, &mv);
  } else if (warp == 1) {
    if (lane == 0) role_issue_p<kVar>(p, sm, base);
  } else if (warp == 2) {
    if (lane == 0) role_issue_c<kVar>(p, sm, base);
  } else if (warp < 7) {
    role_prep<kVar == kVarBwd>(p, sm, base, 32 * (warp & 3) + lane);
  } else {
    role_state<kVar>(p, sm, base, 32 * (warp & 3) + lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(sm->tmem_base, kTmemCols);
  }
}

// Work list: non-empty segments ordered longest first by a counting sort on the
// chunk count (exact below 4096 chunks; longer segments share the top bucket).
// The order among equal counts only affects scheduling, never results.
constexpr int kSortBuckets = 4096;
__global__ void __launch_bounds__(1024)
    k_worklist(const SegInfo *__restrict__ seg, int32_t n_seq, int32_t *order,
               int32_t *n_active, int32_t *counter) {
  __shared__ int cnt[kSortBuckets];
  __shared__ int warp_sum[32];
  for (int b = threadIdx.x; b < kSortBuckets; b += blockDim.x) cnt[b] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n_seq; i += blockDim.x) {
    const int nc = seg[i].n_chunks;
    if (nc > 0) atomicAdd(&cnt[min(nc, kSortBuckets - 1)], 1);
  }
  __syncthreads();
  // exclusive scan from the largest bucket down: 4 buckets per thread
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  int v[4], tot = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    v[u] = cnt[kSortBuckets - 1 - (4 * t + u)];
    tot += v[u];
  }
  int incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    warp_sum[lane] = w;
  }
  __syncthreads();
  int run = incl - tot + (warp > 0 ? warp_sum[warp - 1] : 0);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    cnt[kSortBuckets - 1 - (4 * t + u)] = run;
    run += v[u];
  }
  if (t == 0) {
    *n_active = warp_sum[31];
    *counter = 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n_seq; i += blockDim.x) {
    const int nc = seg[i].n_chunks;
    if (nc > 0) order[atomicAdd(&cnt[min(nc, kSortBuckets - 1)], 1)] = i;
  }
}

// Final states of empty segments: ht[n] = h0[n] (or zero).
__global__ void k_empty_states(const SegInfo *__restrict__ seg, int32_t H, int32_t D,
                               const float *h0, float *ht) {
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  if (seg[n].n_chunks > 0) return;
  const int64_t b = ((int64_t)n * H + h) * D * D;
  for (int i = threadIdx.x; i < D * D; i += blockDim.x) ht[b + i] = h0 ? h0[b + i] : 0.f;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

bool make_map(CUtensorMap *m, const void *ptr, int64_t D, int64_t heads, int64_t T, int64_t st,
              int64_t sh) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)(sh * 2), (cuuint64_t)(st * 2)};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_num_sms[64] = {0};

}  // namespace

bool make_tile_map(CUtensorMap *m, const void *ptr, int64_t D, int64_t heads, int64_t T,
                   int64_t st, int64_t sh) {
  return make_map(m, ptr, D, heads, T, st, sh);
}

bool fused_supported(const FusedArgs &a) {
  if (a.D != 128 && a.D != 64) return false;
  auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (a.T > 0) {
    if (!al16(a.q) || !al16(a.k) || !al16(a.v)) return false;
    if ((a.q_st % 8) || (a.q_sh % 8) || (a.k_st % 8) || (a.k_sh % 8) || (a.v_st % 8) ||
        (a.v_sh % 8))
      return false;
    if (!al16(a.o) || (a.o_st % 8) || (a.o_sh % 8)) return false;
  }
  return true;
}

size_t fused_workspace_bytes(int64_t, int32_t n_seq, int32_t) {
  return align256(sizeof(int32_t) * (size_t)(n_seq > 0 ? n_seq : 1)) + 256;
}

cudaError_t launch_fused(const FusedArgs &a, cudaStream_t stream) {
  char *w = reinterpret_cast<char *>(a.workspace);
  int32_t *counters = reinterpret_cast<int32_t *>(w);  // [0] = unit counter, [1] = n_active
  int32_t *order = reinterpret_cast<int32_t *>(w + 256);
  const bool split = a.split.units != nullptr;
  cudaError_t e = cudaSuccess;
  if (!split) {
    k_worklist<<<1, 1024, 0, stream>>>(a.seg, a.n_seq, order, counters + 1, counters);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.ht && a.n_seq > 0 && (!split || a.split.empty_states)) {
    k_empty_states<<<a.n_seq * a.H, 256, 0, stream>>>(a.seg, a.H, a.D, a.h0, a.ht);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.T == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.D, a.Hk, a.T, a.q_st, a.q_sh) ||
      !make_map(&mk, a.k, a.D, a.Hk, a.T, a.k_st, a.k_sh) ||
      !make_map(&mv, a.v, a.D, a.H, a.T, a.v_st, a.v_sh))
    return cudaErrorInvalidValue;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (g_num_sms[dev] == 0) {
    int n = 0;
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(k_fused<kVarPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBytes)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(k_fused<kVarCkpt>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBytes)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(k_fused<kVarSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBytes)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(k_fused<kVarBwd>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBytes)) != cudaSuccess)
      return e;
    g_num_sms[dev] = n;
  }
  Params p{};
  p.T = (int32_t)a.T;
  p.n_seq = a.n_seq;
  p.Hk = a.Hk;
  p.H = a.H;
  p.D = a.D;
  p.has_h0 = a.h0 != nullptr;
  p.g = a.g;
  p.g_st = a.g_st;
  p.g_sh = a.g_sh;
  p.beta = reinterpret_cast<const __nv_bfloat16 *>(a.beta);
  p.b_st = a.b_st;
  p.b_sh = a.b_sh;
  p.scale = a.scale;
  p.h0 = a.h0;
  p.o = reinterpret_cast<__nv_bfloat16 *>(a.o);
  p.o_st = a.o_st;
  p.o_sh = a.o_sh;
  p.ht = a.ht;
  p.ckpt = a.ckpt;
  p.bw_gcum = a.bwd.gcum;
  p.bw_w = reinterpret_cast<__nv_bfloat16 *>(a.bwd.w);
  p.bw_h = reinterpret_cast<__nv_bfloat16 *>(a.bwd.h);
  p.bw_vn = reinterpret_cast<__nv_bfloat16 *>(a.bwd.vnew);
  p.bw_t = a.bwd.tmat;
  p.split = a.split;
  p.seg = a.seg;
  p.order = order;
  p.n_active = counters + 1;
  p.counter = split ? a.split.counter : counters;
  // one CTA per SM, never more than the number of units that can exist
  int64_t units_max = (int64_t)a.H * a.n_seq;
  const int64_t by_tokens = (int64_t)a.H * ceil_div64(a.T, kChunk);
  if (by_tokens < units_max) units_max = by_tokens;
  int grid = g_num_sms[dev];
  if (!split && units_max < grid) grid = (int)units_max;
  if (grid <= 0) return cudaSuccess;
  if (split)
    k_fused<kVarSplit><<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  else if (p.bw_h)
    k_fused<kVarBwd><<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  else if (p.ckpt.h)
    k_fused<kVarCkpt><<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  else
    k_fused<kVarPlain><<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

namespace {
// A bounded wait on an mbarrier that nothing ever arrives on: it must run out
// after `limit_ns`, record `code` in the status word and return.
__global__ void k_wait_selftest(uint64_t limit_ns, int32_t code) {
  __shared__ uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const bool done = mbar_wait(&bar, 0, &abort_flag, limit_ns);
  if (!done && threadIdx.x == 0) atomicCAS(&g_device_status, 0, code);
}
}  // namespace

cudaError_t launch_wait_selftest(uint32_t limit_us, int32_t code, cudaStream_t stream) {
  k_wait_selftest<<<1, 32, 0, stream>>>((uint64_t)limit_us * 1000ull, code);
  return cudaGetLastError();
}

cudaError_t read_device_status(int32_t *out) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  return cudaMemcpyFromSymbol(out, g_device_status, sizeof(int32_t));
}

cudaError_t clear_device_status() {
  const int32_t zero = 0;
  return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int32_t));
}

}  // namespace gdr

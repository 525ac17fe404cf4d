// gdr_fused.cu -- fused persistent forward of the chunked gated delta rule on
// sm_103a (GB300), plus the device status word.
//
// One CTA per SM walks a work list of (segment, value head) units, longest
// segments first.  For each 64-token chunk of a unit it runs the three stages
// of the chunkwise (WY) form with every intermediate on chip:
//
//   prep   G = cumsum(g); X1 = [K;Q] K^T (KK^T and QK^T);  A, P masks;
//          Tm = (I + A)^-1;  U^T = V^T (Tm diag(beta))^T;  W^T = K^T (Tm diag(beta e^G))^T
//   scan   V'^T = U^T - S^T W^T;  S^T <- e^{G_last} S^T + V''^T K,  V'' = diag(e^{G_last-G}) V'
//   out    O^T = S^T (diag(e^G) Q)^T + V'^T P^T,  P_ij = e^{G_i-G_j} q_i.k_j (j <= i)
//
// The state is kept transposed (S^T: value dim on TMEM lanes, key dim on
// columns) so that every tcgen05.mma has M = 128: the head dimension is the M
// side and the chunk's 64 tokens are N or K.  Operands are bf16 in 128-byte
// swizzled shared memory, accumulators fp32 in TMEM.  The chunk size (64) is
// the one FlashQLA's varlen path uses ("Findings from integrating FlashQLA's
// Blackwell GDN kernels into a JAX trainer", section 1); a unit with no chunks
// (a length-0 segment, section 2 of the same page) is never scheduled, so it
// can store no output.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: K, Q, V tiles and g, beta of each chunk into a 2-stage ring
//   warp 1      MMA issuer (one thread) and TMEM owner
//   warps 2-5   prep warpgroup (one TMEM lane quadrant per warp)
//   warps 6-9   state warpgroup
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

constexpr int kThreads = 320;
constexpr int kStages = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kUnitRing = 4;

// ---- shared memory map (bytes from a 1024-aligned base) ----
constexpr uint32_t kKQBytes = 32768;  // 2 key blocks x [K rows 0-63 | Q rows 64-127] x 128 B
constexpr uint32_t kVBytes = 16384;   // 2 value blocks x 64 rows x 128 B
constexpr uint32_t kStageBytes = kKQBytes + kVBytes;
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_ST = OFF_STAGE + kStages * kStageBytes;  // S^T bf16, 2 key blocks x 128 rows
constexpr uint32_t OFF_WT = OFF_ST + 32768;                     // W^T bf16, 128 rows (dk) x 64 tok
constexpr uint32_t OFF_TB = OFF_WT + 16384;                     // Tm diag(beta) bf16, 64 x 64
constexpr uint32_t OFF_TBG = OFF_TB + 8192;                     // Tm diag(beta e^G) bf16
constexpr uint32_t OFF_P = OFF_TBG + 8192;                      // P bf16, 64 x 64
constexpr uint32_t OFF_VT = OFF_P + 8192;                       // V'^T bf16, 128 rows (dv) x 64 tok
constexpr uint32_t OFF_VS = OFF_VT + 16384;                     // V''^T bf16
constexpr uint32_t OFF_A = OFF_VS + 16384;                      // solve scratch fp32 64 x 64
constexpr uint32_t OFF_Y = OFF_A + 16384;                       // solve scratch fp32 32 x 32
constexpr uint32_t OFF_SMALL = OFF_Y + 4096;
constexpr uint32_t kSmemBytes = OFF_SMALL + 2048 + 1024;  // + small arrays + alignment slack

// ---- TMEM columns ----
constexpr uint32_t TM_S = 0;     // S^T fp32, 128 columns (key dim)
constexpr uint32_t TM_X1 = 128;  // [KK^T ; QK^T], 64 columns
constexpr uint32_t TM_U0 = 192;  // U^T / V'^T, two buffers of 64 columns
constexpr uint32_t TM_W = 320;   // W^T, 64 columns
constexpr uint32_t TM_O = 384;   // O^T, 64 columns
constexpr uint32_t kTmemCols = 512;

struct UnitInfo {
  int32_t seq, head, t0, end, nch, pad0, pad1, pad2;
};

struct Small {
  uint64_t full[kStages], empty[kStages];
  uint64_t x1_full, x1_free, t_ready, uw_full, wt_ready, s_ready, vp_full, vp_ready, s_full,
      o_full, o_free, drain;
  uint64_t unit_full[kUnitRing], unit_empty[kUnitRing];
  UnitInfo unit[kUnitRing];
  float gsm[kStages][64];  // g of the chunk (0 past its end)
  float bsm[kStages][64];  // beta of the chunk (0 past its end)
  float G[2][64];          // chunk-local inclusive cumsum of g
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Small) <= 2048, "small area too large");

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
  const SegInfo *seg;
  const int32_t *order;     // non-empty segments, longest first
  const int32_t *n_active;  // number of non-empty segments
  int32_t *counter;         // unit counter (zeroed by the work-list kernel)
};

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ void fail(Small *sm, int code) {
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

// swizzled index of fp32 element (r, c) in a 64-wide scratch matrix
__device__ __forceinline__ int aix(int r, int c) { return r * 64 + (c ^ (r & 31)); }
__device__ __forceinline__ int yix(int r, int c) { return r * 32 + (c ^ (r & 31)); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t &a, uint32_t &b,
                                             uint32_t &c, uint32_t &d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr)
               : "memory");
}

// Write 64 fp32 values (as bf16) into row `row` of a 128-byte-swizzled tile whose
// rows are 64 bf16 wide (one 8 KB / 16 KB block).
__device__ __forceinline__ void store_row64(uint32_t tile, int row, const float *v) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    st_shared_v4(tile + sw128_off(row, q * 8), pack_bf16(v[q * 8 + 0], v[q * 8 + 1]),
                 pack_bf16(v[q * 8 + 2], v[q * 8 + 3]), pack_bf16(v[q * 8 + 4], v[q * 8 + 5]),
                 pack_bf16(v[q * 8 + 6], v[q * 8 + 7]));
  }
}

__device__ __forceinline__ void zero_row(uint32_t tile, int row) {
#pragma unroll
  for (int q = 0; q < 8; ++q) st_shared_v4(tile + row * 128 + q * 16, 0u, 0u, 0u, 0u);
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

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

// ------------------------------------------------------------------ roles
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
    if (lane == 0) fetch_unit(p, sm, slot);
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
      if (g >= (uint32_t)kStages &&
          !wait_warp(sm, sm->empty[s], ((g / kStages) - 1) & 1, 0x103)) {
        ok = false;
        break;
      }
      const int t = ui.t0 + c * kChunk;
      const int len = min(kChunk, ui.end - t);
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
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = lane + 32 * r;
        float gv = 0.f, bv = 0.f;
        if (j < len) {
          gv = p.g[(int64_t)(t + j) * p.g_st + (int64_t)ui.head * p.g_sh];
          bv = __bfloat162float(p.beta[(int64_t)(t + j) * p.b_st + (int64_t)ui.head * p.b_sh]);
        }
        sm->gsm[s][j] = gv;
        sm->bsm[s][j] = bv;
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

__device__ void role_mma(const Params &p, Small *sm, uint8_t *base) {
  const uint32_t tb = sm->tmem_base;
  const uint32_t sbase = smem_u32(base);
  const uint32_t id_x1 = idesc_bf16(128, 64, false, false);
  const uint32_t id_uw = idesc_bf16(128, 64, true, false);
  const uint32_t id_vp = idesc_bf16(128, 64, false, true, true);
  const uint32_t id_o1 = idesc_bf16(128, 64, false, false);
  const uint32_t id_su = idesc_bf16(128, 128, false, true);
  const uint32_t id_o2 = idesc_bf16(128, 64, false, false);
  uint32_t g = 0;
  bool ok = true;
  auto issue_x1 = [&](uint32_t gg) {
    const uint32_t kq = sbase + OFF_STAGE + (gg % kStages) * kStageBytes;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t a = kq + (kk / 4) * 16384 + (kk % 4) * 32;
      mma_bf16(tb + TM_X1, sdesc_sw128(a, 0, 1024), sdesc_sw128(a, 0, 1024), id_x1, kk > 0);
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
      const uint32_t kq = sbase + OFF_STAGE + s * kStageBytes;
      const uint32_t vv = kq + kKQBytes;
      if (c == 0) {
        if (!wait1(sm, sm->full[s], (g / kStages) & 1, 0x202)) { ok = false; break; }
        if (g >= 1 && !wait1(sm, sm->x1_free, (g - 1) & 1, 0x203)) { ok = false; break; }
        tc_fence_after();
        issue_x1(g);
      }
      // U^T = V^T (Tm diag beta)^T ; W^T = K^T (Tm diag(beta e^G))^T
      if (!wait1(sm, sm->t_ready, g & 1, 0x204)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tu = tb + TM_U0 + (g & 1) * 64;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tu, sdesc_sw128(vv + kk * 2048, 8192, 1024),
                 sdesc_sw128(sbase + OFF_TB + kk * 32, 0, 1024), id_uw, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tb + TM_W, sdesc_sw128(kq + kk * 2048, 16384, 1024),
                 sdesc_sw128(sbase + OFF_TBG + kk * 32, 0, 1024), id_uw, kk > 0);
      }
      mma_commit(&sm->uw_full);
      // next chunk's X1 (prep of c+1 overlaps this chunk's scan)
      if (c + 1 < ui.nch) {
        if (!wait1(sm, sm->full[(g + 1) % kStages], ((g + 1) / kStages) & 1, 0x205)) { ok = false; break; }
        if (!wait1(sm, sm->x1_free, g & 1, 0x206)) { ok = false; break; }
        tc_fence_after();
        issue_x1(g + 1);
      }
      // V'^T = U^T - S^T W^T
      if (!wait1(sm, sm->s_ready, g & 1, 0x207)) { ok = false; break; }
      if (!wait1(sm, sm->wt_ready, g & 1, 0x208)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        mma_bf16(tu, sdesc_sw128(sbase + OFF_ST + (kk / 4) * 16384 + (kk % 4) * 32, 0, 1024),
                 sdesc_sw128(sbase + OFF_WT + kk * 2048, 16384, 1024), id_vp, 1);
      }
      mma_commit(&sm->vp_full);
      // O^T = S^T Q~^T
      if (g >= 1 && !wait1(sm, sm->o_free, (g - 1) & 1, 0x209)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        mma_bf16(tb + TM_O,
                 sdesc_sw128(sbase + OFF_ST + (kk / 4) * 16384 + (kk % 4) * 32, 0, 1024),
                 sdesc_sw128(kq + (kk / 4) * 16384 + 8192 + (kk % 4) * 32, 0, 1024), id_o1,
                 kk > 0);
      }
      // S^T += V''^T K ;  O^T += V'^T P^T
      if (!wait1(sm, sm->vp_ready, g & 1, 0x20a)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tb + TM_S, sdesc_sw128(sbase + OFF_VS + kk * 32, 0, 1024),
                 sdesc_sw128(kq + kk * 2048, 16384, 1024), id_su, 1);
      }
      mma_commit(&sm->s_full);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tb + TM_O, sdesc_sw128(sbase + OFF_VT + kk * 32, 0, 1024),
                 sdesc_sw128(sbase + OFF_P + kk * 32, 0, 1024), id_o2, 1);
      }
      mma_commit(&sm->o_full);
      mma_commit(&sm->empty[s]);
    }
  }
  // drain: every MMA issued so far must finish before TMEM is released
  mma_commit(&sm->drain);
  mbar_wait(&sm->drain, 0, nullptr, kWaitLimitNs);
}

// The prep warpgroup.  `row` is this thread's TMEM lane (0..127).
__device__ void role_prep(const Params &p, Small *sm, uint8_t *base, int row) {
  const uint32_t tb = sm->tmem_base;
  const uint32_t sbase = smem_u32(base);
  const uint32_t lane_base = (uint32_t)(row & ~31);
  float *Asc = reinterpret_cast<float *>(base + OFF_A);
  float *Ysc = reinterpret_cast<float *>(base + OFF_Y);
  const int pid = row;  // 0..127, unique in the warpgroup
  uint32_t g = 0;
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    const int slot = k % kUnitRing;
    if (!wait_wg(sm, sm->unit_full[slot], (k / kUnitRing) & 1, 0x301, kBarPrep)) { ok = false; break; }
    const UnitInfo ui = sm->unit[slot];
    mbar_arrive(&sm->unit_empty[slot]);
    if (ui.seq < 0) break;
    for (int c = 0; c < ui.nch; ++c, ++g) {
      const uint32_t s = g % kStages;
      const int t = ui.t0 + c * kChunk;
      const int len = min(kChunk, ui.end - t);
      uint8_t *kq = base + OFF_STAGE + s * kStageBytes;
      const uint32_t kq_a = smem_u32(kq);
      if (!wait_wg(sm, sm->full[s], (g / kStages) & 1, 0x302, kBarPrep)) { ok = false; break; }
      // zero the rows past the chunk's end (they hold the next segment's tokens)
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
      float *Gc = sm->G[g & 1];
      if (pid < 32) {  // chunk-local inclusive cumsum, two tokens per lane
        const float a = sm->gsm[s][2 * pid], b = sm->gsm[s][2 * pid + 1];
        float sum = a + b;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, sum, off);
          if (pid >= off) sum += y;
        }
        const float ex = sum - (a + b);
        Gc[2 * pid] = ex + a;
        Gc[2 * pid + 1] = ex + a + b;
      }
      named_bar(1, 128);
      // X1 rows: lanes 0-63 = K K^T (rows of A), lanes 64-127 = Q K^T (rows of P)
      if (!wait_wg(sm, sm->x1_full, g & 1, 0x303, kBarPrep)) { ok = false; break; }
      tc_fence_after();
      float xr[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem_addr(tb + TM_X1, lane_base, 0), r0);
        tmem_ld32(tmem_addr(tb + TM_X1, lane_base, 32), r1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          xr[j] = __uint_as_float(r0[j]);
          xr[j + 32] = __uint_as_float(r1[j]);
        }
      }
      tc_fence_before();
      mbar_arrive(&sm->x1_free);
      uint32_t pk[32];  // packed P row (bf16x2), rows 64..127 only
      if (row < 64) {
        const int i = row;
        const float bi = sm->bsm[s][i], gi = Gc[i];
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float a = (j < i && i < len) ? bi * __expf(gi - Gc[j]) * xr[j] : 0.f;
          Asc[aix(i, j)] = a;
        }
      } else {
        const int i = row - 64;
        const float gi = Gc[i];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int j0 = 2 * j, j1 = 2 * j + 1;
          const float p0 = (j0 <= i && i < len) ? __expf(gi - Gc[j0]) * xr[j0] : 0.f;
          const float p1 = (j1 <= i && i < len) ? __expf(gi - Gc[j1]) * xr[j1] : 0.f;
          pk[j] = pack_bf16(p0, p1);
        }
        // Q~ row i = e^{G_i} q_i (in place in the stage; rows past len are zero)
        if (i < len) {
          const float e = __expf(gi);
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t addr = kq_a + kb * 16384 + sw128_off(64 + i, q * 8);
              uint32_t w0, w1, w2, w3;
              ld_shared_v4(addr, w0, w1, w2, w3);
              st_shared_v4(addr, pack_bf16(bf_lo(w0) * e, bf_hi(w0) * e),
                           pack_bf16(bf_lo(w1) * e, bf_hi(w1) * e),
                           pack_bf16(bf_lo(w2) * e, bf_hi(w2) * e),
                           pack_bf16(bf_lo(w3) * e, bf_hi(w3) * e));
            }
          }
        }
      }
      named_bar(1, 128);
      // ---- Tm = (I + A)^-1, 64 x 64 unit lower triangular, fp32 ----
      // phase 1: the four 16 x 16 diagonal blocks, one column per thread
      float x[16];
      if (pid < 64) {
        const int b = pid >> 4, cc = pid & 15, o = 16 * b;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float v = (r == cc) ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < r; ++m) v -= Asc[aix(o + r, o + m)] * x[m];
          x[r] = v;
        }
      }
      named_bar(1, 128);
      if (pid < 64) {
        const int b = pid >> 4, cc = pid & 15, o = 16 * b;
#pragma unroll
        for (int r = 0; r < 16; ++r) Asc[aix(o + r, o + cc)] = x[r];
      }
      named_bar(1, 128);
      // phase 2: T_{b+1,b} = -D_{b+1} A_{b+1,b} D_b for b = 0, 2
      {
        const int blk = pid >> 6, q = pid & 63, r = q >> 2, c0 = (q & 3) * 4;
        const int ob = 32 * blk, oa = ob + 16;  // D_b at ob, the block below at oa
        float xv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float a = Asc[aix(oa + r, ob + m)];
#pragma unroll
          for (int u = 0; u < 4; ++u) xv[u] += a * Asc[aix(ob + m, ob + c0 + u)];
        }
        named_bar(1, 128);
        float *Xs = Ysc + blk * 256;
#pragma unroll
        for (int u = 0; u < 4; ++u) Xs[r * 16 + ((c0 + u) ^ r)] = xv[u];
        named_bar(1, 128);
        float tv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float d = Asc[aix(oa + r, oa + m)];
#pragma unroll
          for (int u = 0; u < 4; ++u) tv[u] -= d * Xs[m * 16 + ((c0 + u) ^ m)];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) Asc[aix(oa + r, ob + c0 + u)] = tv[u];
      }
      named_bar(1, 128);
      // phase 3: Tm[32:64, 0:32] = -T2 (A[32:64, 0:32] T1)
      {
        const int r = pid >> 2, c0 = (pid & 3) * 8;
        float yv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) yv[u] = 0.f;
        for (int m = c0; m < 32; ++m) {
          const float a = Asc[aix(32 + r, m)];
#pragma unroll
          for (int u = 0; u < 8; ++u) yv[u] += a * Asc[aix(m, c0 + u)];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) Ysc[yix(r, c0 + u)] = yv[u];
        named_bar(1, 128);
        float tv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) tv[u] = 0.f;
        for (int m = 0; m <= r; ++m) {
          const float d = Asc[aix(32 + r, 32 + m)];
#pragma unroll
          for (int u = 0; u < 8; ++u) tv[u] -= d * Ysc[yix(m, c0 + u)];
        }
        named_bar(1, 128);
#pragma unroll
        for (int u = 0; u < 8; ++u) Asc[aix(32 + r, c0 + u)] = tv[u];
      }
      named_bar(1, 128);
      // Tm diag(beta) and Tm diag(beta e^G) as bf16 MMA operands (row i = thread i)
      if (row < 64) {
        const int i = row;
        float v[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = (j <= i) ? Asc[aix(i, j)] * sm->bsm[s][j] : 0.f;
        store_row64(sbase + OFF_TB, i, v);
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] *= __expf(Gc[j]);
        store_row64(sbase + OFF_TBG, i, v);
      }
      // P waits until the previous chunk's output MMA has read the buffer
      if (g >= 1 && !wait_wg(sm, sm->o_full, (g - 1) & 1, 0x304, kBarPrep)) { ok = false; break; }
      if (row >= 64) {
        {
          const int i = row - 64;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(sbase + OFF_P + sw128_off(i, q * 8), pk[4 * q], pk[4 * q + 1],
                         pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      fence_async_smem();
      mbar_arrive(&sm->t_ready);
      // W^T (lane = key dim) -> bf16 operand; waits until the previous V'^T MMA read it
      if (!wait_wg(sm, sm->uw_full, g & 1, 0x305, kBarPrep)) { ok = false; break; }
      if (g >= 1 && !wait_wg(sm, sm->vp_full, (g - 1) & 1, 0x306, kBarPrep)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem_addr(tb + TM_W, lane_base, 0), r0);
        tmem_ld32(tmem_addr(tb + TM_W, lane_base, 32), r1);
        tmem_ld_wait();
        float v[64];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] = __uint_as_float(r0[j]);
          v[j + 32] = __uint_as_float(r1[j]);
        }
        store_row64(sbase + OFF_WT, row, v);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&sm->wt_ready);
    }
  }
}

// The state warpgroup.  `row` is this thread's TMEM lane = value dimension dv.
__device__ void role_state(const Params &p, Small *sm, uint8_t *base, int row) {
  const uint32_t tb = sm->tmem_base;
  const uint32_t sbase = smem_u32(base);
  const uint32_t lane_base = (uint32_t)(row & ~31);
  const int dv = row;
  const int D = p.D;
  uint32_t g = 0;
  bool ok = true;
  int prev_t = 0, prev_len = 0, prev_head = 0;
  auto epilogue = [&](uint32_t gg) -> bool {
    if (!wait_wg(sm, sm->o_full, gg & 1, 0x401, kBarState)) return false;
    tc_fence_after();
    uint32_t r0[32], r1[32];
    tmem_ld32(tmem_addr(tb + TM_O, lane_base, 0), r0);
    tmem_ld32(tmem_addr(tb + TM_O, lane_base, 32), r1);
    tmem_ld_wait();
    tc_fence_before();
    mbar_arrive(&sm->o_free);
    if (dv < D) {
      __nv_bfloat16 *op = p.o + (int64_t)prev_head * p.o_sh + dv;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < prev_len)
          op[(int64_t)(prev_t + i) * p.o_st] = __float2bfloat16_rn(p.scale * __uint_as_float(r0[i]));
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i + 32 < prev_len)
          op[(int64_t)(prev_t + 32 + i) * p.o_st] =
              __float2bfloat16_rn(p.scale * __uint_as_float(r1[i]));
    }
    return true;
  };
  for (uint32_t k = 0; ok; ++k) {
    const int slot = k % kUnitRing;
    if (!wait_wg(sm, sm->unit_full[slot], (k / kUnitRing) & 1, 0x402, kBarState)) { ok = false; break; }
    const UnitInfo ui = sm->unit[slot];
    mbar_arrive(&sm->unit_empty[slot]);
    if (ui.seq < 0) break;
    const int64_t sbase_idx = ((int64_t)ui.seq * p.H + ui.head) * D * D;
    for (int c = 0; c < ui.nch; ++c, ++g) {
      const int t = ui.t0 + c * kChunk;
      const int len = min(kChunk, ui.end - t);
      if (!wait_wg(sm, sm->t_ready, g & 1, 0x403, kBarState)) { ok = false; break; }
      const float *Gc = sm->G[g & 1];
      const float GL = Gc[len - 1];
      const float eL = __expf(GL);
      // current state row dv of S^T: from h0 at a unit's first chunk, else from TMEM
      float sr[128];
      if (c == 0) {
#pragma unroll
        for (int j = 0; j < 128; ++j)
          sr[j] = (p.has_h0 && dv < D && j < D) ? p.h0[sbase_idx + (int64_t)j * D + dv] : 0.f;
      } else {
        if (!wait_wg(sm, sm->s_full, (g - 1) & 1, 0x404, kBarState)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tb + TM_S, lane_base, cb * 32), r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) sr[cb * 32 + j] = __uint_as_float(r[j]);
        }
      }
      store_row64(sbase + OFF_ST, row, sr);
      store_row64(sbase + OFF_ST + 16384, row, sr + 64);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(sr[cb * 32 + j] * eL);
        tmem_st32(tmem_addr(tb + TM_S, lane_base, cb * 32), r);
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&sm->s_ready);
      // previous chunk's output (same unit) while this chunk's V'^T is computed
      if (c >= 1) {
        if (!epilogue(g - 1)) { ok = false; break; }
      }
      if (!wait_wg(sm, sm->vp_full, g & 1, 0x405, kBarState)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem_addr(tb + TM_U0 + (g & 1) * 64, lane_base, 0), r0);
        tmem_ld32(tmem_addr(tb + TM_U0 + (g & 1) * 64, lane_base, 32), r1);
        tmem_ld_wait();
        float v[64];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] = __uint_as_float(r0[j]);
          v[j + 32] = __uint_as_float(r1[j]);
        }
        store_row64(sbase + OFF_VT, row, v);
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] *= __expf(GL - Gc[j]);
        store_row64(sbase + OFF_VS, row, v);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&sm->vp_ready);
      prev_t = t;
      prev_len = len;
      prev_head = ui.head;
    }
    if (!ok) break;
    // end of the unit: final state, then the last chunk's output
    if (ui.nch > 0) {
      if (!wait_wg(sm, sm->s_full, (g - 1) & 1, 0x406, kBarState)) { ok = false; break; }
      tc_fence_after();
      if (p.ht) {
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tb + TM_S, lane_base, cb * 32), r);
          tmem_ld_wait();
          if (dv < D) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (cb * 32 + j < D)
                p.ht[sbase_idx + (int64_t)(cb * 32 + j) * D + dv] = __uint_as_float(r[j]);
          }
        }
      }
      if (!epilogue(g - 1)) { ok = false; break; }
    }
  }
}

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
      mbar_init(&sm->empty[s], 1);
    }
    mbar_init(&sm->x1_full, 1);
    mbar_init(&sm->x1_free, 128);
    mbar_init(&sm->t_ready, 128);
    mbar_init(&sm->uw_full, 1);
    mbar_init(&sm->wt_ready, 128);
    mbar_init(&sm->s_ready, 128);
    mbar_init(&sm->vp_full, 1);
    mbar_init(&sm->vp_ready, 128);
    mbar_init(&sm->s_full, 1);
    mbar_init(&sm->o_full, 1);
    mbar_init(&sm->o_free, 128);
    mbar_init(&sm->drain, 1);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&sm->unit_full[i], 1);
      mbar_init(&sm->unit_empty[i], 1 + 128 + 128);
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
    role_producer(p, sm, base, &mq, &mk, &mv);
  } else if (warp == 1) {
    if (lane == 0) role_mma(p, sm, base);
  } else if (warp < 6) {
    role_prep(p, sm, base, 32 * (warp & 3) + lane);
  } else {
    role_state(p, sm, base, 32 * (warp & 3) + lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(sm->tmem_base, kTmemCols);
  }
}

// Work list: non-empty segments ordered longest first (bucketed by log2 of the
// chunk count; the order inside a bucket only affects scheduling, never results).
__global__ void __launch_bounds__(1024)
    k_worklist(const SegInfo *__restrict__ seg, int32_t n_seq, int32_t *order,
               int32_t *n_active, int32_t *counter) {
  __shared__ int cnt[33], cur[33];
  if (threadIdx.x < 33) cnt[threadIdx.x] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n_seq; i += blockDim.x) {
    const int nc = seg[i].n_chunks;
    if (nc > 0) atomicAdd(&cnt[31 - __clz(nc)], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 31; b >= 0; --b) {
      cur[b] = acc;
      acc += cnt[b];
    }
    *n_active = acc;
    *counter = 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n_seq; i += blockDim.x) {
    const int nc = seg[i].n_chunks;
    if (nc > 0) order[atomicAdd(&cur[31 - __clz(nc)], 1)] = i;
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

bool fused_supported(const FusedArgs &a) {
  if (a.D != 128 && a.D != 64) return false;
  auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (a.T > 0) {
    if (!al16(a.q) || !al16(a.k) || !al16(a.v)) return false;
    if ((a.q_st % 8) || (a.q_sh % 8) || (a.k_st % 8) || (a.k_sh % 8) || (a.v_st % 8) ||
        (a.v_sh % 8))
      return false;
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
  k_worklist<<<1, 1024, 0, stream>>>(a.seg, a.n_seq, order, counters + 1, counters);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.ht && a.n_seq > 0) {
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
    if ((e = cudaFuncSetAttribute(k_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  p.seg = a.seg;
  p.order = order;
  p.n_active = counters + 1;
  p.counter = counters;
  // one CTA per SM, never more than the number of units that can exist
  int64_t units_max = (int64_t)a.H * a.n_seq;
  const int64_t by_tokens = (int64_t)a.H * ceil_div64(a.T, kChunk);
  if (by_tokens < units_max) units_max = by_tokens;
  int grid = g_num_sms[dev];
  if (units_max < grid) grid = (int)units_max;
  if (grid <= 0) return cudaSuccess;
  k_fused<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
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

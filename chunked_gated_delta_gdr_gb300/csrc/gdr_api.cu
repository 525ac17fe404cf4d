// gdr_api.cu -- the extern "C" boundary of libgdr: descriptor validation,
// workspace carving and stream-ordered launches.  No host synchronisation
// except in gdr_debug_check_cu_seqlens and gdr_device_status.
#include <mutex>
#include <string.h>

#include "gdr_bwd.cuh"
#include "gdr_internal.cuh"
#include "gdr_sched.cuh"

using namespace gdr;

namespace {

struct Desc {
  void *p;
  int ndim;
  int64_t shape[4];
  int64_t stride[4];
};

int read_desc(const gdr_tensor_t *t, int dtype, int ndim, Desc *d) {
  if (!t) return GDR_ERR_NULL;
  if (t->dtype != dtype) return GDR_ERR_DTYPE;
  if (t->ndim != ndim) return GDR_ERR_SHAPE;
  int64_t numel = 1;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return GDR_ERR_SHAPE;
    d->shape[i] = t->shape[i];
    numel *= t->shape[i];
  }
  if (!t->data && numel > 0) return GDR_ERR_NULL;
  d->p = t->data;
  d->ndim = ndim;
  if (t->strides) {
    for (int i = 0; i < ndim; ++i) {
      if (t->strides[i] < 0) return GDR_ERR_STRIDE;
      d->stride[i] = t->strides[i];
    }
    if (d->shape[ndim - 1] > 1 && d->stride[ndim - 1] != 1) return GDR_ERR_STRIDE;
    d->stride[ndim - 1] = 1;
  } else {
    int64_t s = 1;
    for (int i = ndim - 1; i >= 0; --i) {
      d->stride[i] = s;
      s *= d->shape[i];
    }
  }
  return GDR_OK;
}

bool compact(const Desc &d) {
  int64_t s = 1;
  for (int i = d.ndim - 1; i >= 0; --i) {
    if (d.shape[i] > 1 && d.stride[i] != s) return false;
    s *= d.shape[i];
  }
  return true;
}

View view_of(const Desc &d) { return View{d.p, d.stride[0], d.ndim > 1 ? d.stride[1] : 0}; }

int device_ok() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDR_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return GDR_ERR_CUDA;
  return (major == 10 && minor == 3) ? GDR_OK : GDR_ERR_DEVICE;
}

// Validated problem: extents and views of every operand of the forward.
struct Problem {
  int64_t T;
  int32_t n_seq, Hk, H, D;
  Desc q, k, v, g, beta, o, h0, ht;
  bool has_h0, has_ht;
  Ckpt ck{};  // state checkpoints (ck.h null: none)
};

int validate_fwd(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                 const gdr_tensor_t *g, const gdr_tensor_t *beta, const gdr_tensor_t *h0,
                 const int32_t *cu, int32_t n_seq, const gdr_tensor_t *o,
                 const gdr_tensor_t *ht, Problem *P) {
  int r;
  if ((r = read_desc(q, GDR_BF16, 3, &P->q))) return r;
  if ((r = read_desc(k, GDR_BF16, 3, &P->k))) return r;
  if ((r = read_desc(v, GDR_BF16, 3, &P->v))) return r;
  if ((r = read_desc(g, GDR_F32, 2, &P->g))) return r;
  if ((r = read_desc(beta, GDR_BF16, 2, &P->beta))) return r;
  if ((r = read_desc(o, GDR_BF16, 3, &P->o))) return r;
  P->T = P->q.shape[0];
  P->Hk = (int32_t)P->q.shape[1];
  P->D = (int32_t)P->q.shape[2];
  P->H = (int32_t)P->v.shape[1];
  for (int i = 0; i < 3; ++i)
    if (P->k.shape[i] != P->q.shape[i]) return GDR_ERR_SHAPE;
  if (P->v.shape[0] != P->T || P->o.shape[0] != P->T || P->g.shape[0] != P->T ||
      P->beta.shape[0] != P->T)
    return GDR_ERR_SHAPE;
  if (P->o.shape[1] != P->H || P->g.shape[1] != P->H || P->beta.shape[1] != P->H)
    return GDR_ERR_SHAPE;
  if (P->v.shape[2] != P->o.shape[2]) return GDR_ERR_SHAPE;
  if (P->v.shape[2] != P->D) return GDR_ERR_DIM;
  if (P->D != 64 && P->D != 128) return GDR_ERR_DIM;
  if (P->Hk <= 0 || P->H <= 0) return GDR_ERR_SHAPE;
  if (P->H % P->Hk != 0) return GDR_ERR_HEADS;
  if (P->T > 0x7fffffffLL) return GDR_ERR_SHAPE;
  if (n_seq < 0) return GDR_ERR_NSEQ;
  if (n_seq > 0 && !cu) return GDR_ERR_NULL;
  P->n_seq = n_seq;
  P->has_h0 = h0 != nullptr;
  P->has_ht = ht != nullptr;
  const int64_t sshape[4] = {n_seq, P->H, P->D, P->D};
  if (P->has_h0) {
    if ((r = read_desc(h0, GDR_F32, 4, &P->h0))) return r;
    if (P->h0.shape[0] != n_seq) return GDR_ERR_NSEQ;
    for (int i = 1; i < 4; ++i)
      if (P->h0.shape[i] != sshape[i]) return GDR_ERR_SHAPE;
    if (!compact(P->h0)) return GDR_ERR_STRIDE;
  }
  if (P->has_ht) {
    if ((r = read_desc(ht, GDR_F32, 4, &P->ht))) return r;
    if (P->ht.shape[0] != n_seq) return GDR_ERR_NSEQ;
    for (int i = 1; i < 4; ++i)
      if (P->ht.shape[i] != sshape[i]) return GDR_ERR_SHAPE;
    if (!compact(P->ht)) return GDR_ERR_STRIDE;
  }
  return GDR_OK;
}

// Workspace carving: the chunk tables come first (both paths), then path-specific.
struct IndexWs {
  SegInfo *seg;
  ChunkInfo *chunks;
  int32_t *n_chunks;
  int32_t *order;  // segments longest first, for the per-segment scans
  size_t bytes;
};

IndexWs carve_index(void *ws, int64_t T, int32_t n_seq) {
  IndexWs r{};
  char *p = reinterpret_cast<char *>(ws);
  size_t off = 0;
  r.n_chunks = reinterpret_cast<int32_t *>(p + off);
  off += 256;
  r.seg = reinterpret_cast<SegInfo *>(p + off);
  off += align256(sizeof(SegInfo) * (size_t)(n_seq > 0 ? n_seq : 1));
  r.chunks = reinterpret_cast<ChunkInfo *>(p + off);
  off += align256(sizeof(ChunkInfo) * (size_t)chunk_bound(T, n_seq));
  r.order = reinterpret_cast<int32_t *>(p + off);
  off += align256(sizeof(int32_t) * (size_t)(n_seq > 0 ? n_seq : 1));
  r.bytes = off;
  return r;
}

size_t staged_bytes(int64_t T, int32_t n_seq, int32_t H, int32_t D) {
  const size_t tok = (size_t)T * H;
  size_t b = carve_index(nullptr, T, n_seq).bytes;
  b += align256(tok * sizeof(float));            // gcum
  b += 3 * align256(tok * D * 2);                // W, U, V'
  b += align256((size_t)chunk_bound(T, n_seq) * H * D * D * 2);  // h
  return b;
}

FusedArgs fused_args(const Problem &P, float scale, void *work) {
  FusedArgs a{};
  a.T = P.T;
  a.n_seq = P.n_seq;
  a.Hk = P.Hk;
  a.H = P.H;
  a.D = P.D;
  a.q = P.q.p; a.q_st = P.q.stride[0]; a.q_sh = P.q.stride[1];
  a.k = P.k.p; a.k_st = P.k.stride[0]; a.k_sh = P.k.stride[1];
  a.v = P.v.p; a.v_st = P.v.stride[0]; a.v_sh = P.v.stride[1];
  a.g = reinterpret_cast<const float *>(P.g.p); a.g_st = P.g.stride[0]; a.g_sh = P.g.stride[1];
  a.beta = P.beta.p; a.b_st = P.beta.stride[0]; a.b_sh = P.beta.stride[1];
  a.scale = scale;
  a.h0 = P.has_h0 ? reinterpret_cast<const float *>(P.h0.p) : nullptr;
  a.o = P.o.p; a.o_st = P.o.stride[0]; a.o_sh = P.o.stride[1];
  a.ht = P.has_ht ? reinterpret_cast<float *>(P.ht.p) : nullptr;
  a.ckpt = P.ck;
  a.workspace = work;
  return a;
}

// Pieces per segment of the fused path's sequence split on the current device (1: none).
int split_plan(int64_t T, int32_t n_seq, int32_t H, bool ckpt, int *lead = nullptr) {
  static int sms[64] = {0};
  int lead_dummy = 1;
  if (!lead) lead = &lead_dummy;
  *lead = 1;
  // no segment can be cut when none reaches three of the shortest pieces
  if (ckpt || n_seq <= 0 || T <= (int64_t)(3 * kSplitMinChunks - 1) * kChunk) return 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 1;
  }
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    sms[dev] = n;
  }
  return split_pieces((int64_t)n_seq * H, sms[dev], lead);
}

int run_fwd(const Problem &P, float scale, const int32_t *cu, int32_t path, void *ws,
            size_t ws_bytes, cudaStream_t stream) {
  if (P.n_seq == 0) return GDR_OK;
  const IndexWs ix = carve_index(ws, P.T, P.n_seq);
  char *rest = reinterpret_cast<char *>(ws) + ix.bytes;
  const int64_t cap = chunk_bound(P.T, P.n_seq);
  cudaError_t e;
  if (path == GDR_PATH_FUSED || path == GDR_PATH_FUSED_WHOLE) {
    FusedArgs a = fused_args(P, scale, rest);
    a.seg = ix.seg;
    e = launch_chunk_index(cu, P.n_seq, P.T, ix.seg, nullptr, 0, ix.n_chunks, stream);
    if (e != cudaSuccess) return GDR_ERR_CUDA;
    if (P.ck.h && (e = launch_ckpt_offsets(ix.seg, P.n_seq, P.ck.every,
                                           const_cast<int32_t *>(P.ck.off), stream)) != cudaSuccess)
      return GDR_ERR_CUDA;
    int lead = 1;
    const int pieces =
        path == GDR_PATH_FUSED ? split_plan(P.T, P.n_seq, P.H, P.ck.h != nullptr, &lead) : 1;
    if (pieces <= 1) {
      e = launch_fused(a, stream);
      return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    }
    // sequence split: pass A (first pieces, R and M of the middle ones), the chain of
    // initial states, pass B (the later pieces)
    const SplitWs sw = carve_split(rest + fused_workspace_bytes(P.T, P.n_seq, P.H), P.n_seq,
                                   P.H, P.D, pieces);
    if ((e = launch_split_units(ix.seg, P.n_seq, P.H, pieces, lead, sw, stream)) != cudaSuccess)
      return GDR_ERR_CUDA;
    a.split = SplitArgs{sw.ua, sw.na, sw.states, sw.counters, true};
    if ((e = launch_fused(a, stream)) != cudaSuccess) return GDR_ERR_CUDA;
    if ((e = launch_split_combine(sw, P.n_seq, P.H, P.D, stream)) != cudaSuccess)
      return GDR_ERR_CUDA;
    a.split = SplitArgs{sw.ub, sw.nb, sw.states, sw.counters + 1, false};
    e = launch_fused(a, stream);
    return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
  }
  // staged
  const size_t tok = (size_t)P.T * P.H;
  char *p = rest;
  float *gcum = reinterpret_cast<float *>(p);
  p += align256(tok * sizeof(float));
  void *w = p;
  p += align256(tok * P.D * 2);
  void *u = p;
  p += align256(tok * P.D * 2);
  void *vn = p;
  p += align256(tok * P.D * 2);
  void *h = p;
  (void)ws_bytes;
  const int64_t D = P.D;
  const View vg{gcum, P.H, 1}, vw{w, P.H * D, D}, vu{u, P.H * D, D}, vv{vn, P.H * D, D};
  const StageShapes s{P.T, P.n_seq, P.Hk, P.H, P.D, cap};
  e = launch_chunk_index(cu, P.n_seq, P.T, ix.seg, ix.chunks, cap, ix.n_chunks, stream);
  if (e != cudaSuccess) return GDR_ERR_CUDA;
  if (P.ck.h && (e = launch_ckpt_offsets(ix.seg, P.n_seq, P.ck.every,
                                         const_cast<int32_t *>(P.ck.off), stream)) != cudaSuccess)
    return GDR_ERR_CUDA;
  e = launch_prep(s, view_of(P.k), view_of(P.v), view_of(P.g), view_of(P.beta), vw, vu, vg,
                  ix.seg, ix.chunks, ix.n_chunks, stream);
  if (e != cudaSuccess) return GDR_ERR_CUDA;
  if ((e = launch_seg_order(ix.seg, P.n_seq, ix.order, stream)) != cudaSuccess)
    return GDR_ERR_CUDA;
  e = launch_scan_ordered(s, view_of(P.k), vw, vu, vg,
                          P.has_h0 ? reinterpret_cast<const float *>(P.h0.p) : nullptr, h, vv,
                          P.has_ht ? reinterpret_cast<float *>(P.ht.p) : nullptr, P.ck, ix.seg,
                          ix.order, stream);
  if (e != cudaSuccess) return GDR_ERR_CUDA;
  e = launch_out(s, view_of(P.q), view_of(P.k), vv, h, vg, scale, view_of(P.o), ix.seg,
                 ix.chunks, ix.n_chunks, stream);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

size_t ws_bytes_for(int64_t T, int32_t n_seq, int32_t H, int32_t D, int32_t path) {
  const size_t ix = carve_index(nullptr, T, n_seq).bytes;
  const size_t st = staged_bytes(T, n_seq, H, D);
  const size_t fw = ix + fused_workspace_bytes(T, n_seq, H);
  const int pieces = split_plan(T, n_seq, H, false);
  const size_t fu = fw + (pieces > 1 ? carve_split(nullptr, n_seq, H, D, pieces).bytes : 0);
  if (path == GDR_PATH_STAGED) return st;
  if (path == GDR_PATH_FUSED_WHOLE) return fw;
  if (path == GDR_PATH_FUSED) return fu;
  return st > fu ? st : fu;
}

int choose_path(const Problem &P, float scale, int32_t path) {
  if (path == GDR_PATH_STAGED) return GDR_PATH_STAGED;
  const bool fused_ok = fused_supported(fused_args(P, scale, nullptr));
  if (path == GDR_PATH_FUSED || path == GDR_PATH_FUSED_WHOLE)
    return fused_ok ? path : GDR_ERR_PATH;
  if (path == GDR_PATH_AUTO) return fused_ok ? GDR_PATH_FUSED : GDR_PATH_STAGED;
  return GDR_ERR_PATH;
}

}  // namespace

extern "C" {

int gdr_version(void) { return 100; }

const char *gdr_status_string(int status) {
  switch (status) {
    case GDR_OK: return "ok";
    case GDR_ERR_NULL: return "a required pointer or descriptor is NULL";
    case GDR_ERR_DTYPE: return "wrong element type";
    case GDR_ERR_SHAPE: return "wrong rank or inconsistent extents";
    case GDR_ERR_STRIDE: return "unsupported strides (innermost must be 1, states compact)";
    case GDR_ERR_DIM: return "unsupported head dimension (dk == dv in {64, 128})";
    case GDR_ERR_HEADS: return "value heads must be a multiple of query/key heads";
    case GDR_ERR_NSEQ: return "n_seq negative or inconsistent with h0/ht";
    case GDR_ERR_WORKSPACE: return "workspace NULL, too small or not 256-byte aligned";
    case GDR_ERR_PATH: return "unknown path, or the fused path does not support these inputs";
    case GDR_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case GDR_ERR_ALIGN: return "a base pointer or row stride is not 16-byte aligned";
    case GDR_ERR_DEVICE: return "the current device is not sm_103 (GB300)";
    case GDR_ERR_SCRATCH_LIMIT:
      return "problem too large for the 4 MiB static scratch of gdr_chunk_out_noalloc";
    case GDR_ERR_CKPT:
      return "checkpoint interval not a positive multiple of 64, or checkpoint buffers wrong";
    default: return "unknown status";
  }
}

int64_t gdr_chunk_count_bound(int64_t T, int32_t n_seq) {
  if (T < 0 || n_seq < 0) return 0;
  return chunk_bound(T, n_seq);
}

size_t gdr_stage_workspace_bytes(int64_t T, int32_t n_seq) {
  if (T < 0 || n_seq < 0) return 0;
  return carve_index(nullptr, T, n_seq).bytes;
}

size_t gdr_chunk_fwd_workspace_bytes(int64_t T, int32_t n_seq, int32_t H, int32_t dk,
                                     int32_t dv, int32_t path) {
  if (T < 0 || n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0) return 0;
  const int32_t D = dk > dv ? dk : dv;
  return ws_bytes_for(T, n_seq, H, D, path);
}

int gdr_chunk_fwd_ws(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                     const gdr_tensor_t *g, const gdr_tensor_t *beta, float scale,
                     const gdr_tensor_t *h0, const int32_t *cu_seqlens, int32_t n_seq,
                     gdr_tensor_t *o, gdr_tensor_t *ht, int32_t path, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  Problem P;
  int r = validate_fwd(q, k, v, g, beta, h0, cu_seqlens, n_seq, o, ht, &P);
  if (r) return r;
  if ((r = device_ok())) return r;
  const int chosen = choose_path(P, scale, path);
  if (chosen < 0) return chosen;
  if (P.n_seq == 0) return GDR_OK;
  const size_t need = ws_bytes_for(P.T, P.n_seq, P.H, P.D, chosen);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return GDR_ERR_WORKSPACE;
  return run_fwd(P, scale, cu_seqlens, chosen, workspace, workspace_bytes, stream);
}

int32_t gdr_fused_split_pieces(int64_t T, int32_t n_seq, int32_t H) {
  if (T < 0 || n_seq <= 0 || H <= 0) return 1;
  return split_plan(T, n_seq, H, false);
}

int32_t gdr_split_plan(int64_t units, int32_t sms, int32_t *lead) {
  int l = 1;
  const int p = split_pieces(units, sms, &l);
  if (lead) *lead = l;
  return p;
}

int64_t gdr_ckpt_count_bound(int64_t T, int32_t ckpt_every) {
  if (T < 0 || ckpt_every <= 0) return 0;
  return T / ckpt_every;
}

int gdr_chunk_fwd_ckpt(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                       const gdr_tensor_t *g, const gdr_tensor_t *beta, float scale,
                       const gdr_tensor_t *h0, const int32_t *cu_seqlens, int32_t n_seq,
                       gdr_tensor_t *o, gdr_tensor_t *ht, gdr_tensor_t *state_checkpoints,
                       int32_t *checkpoint_cu_starts, int32_t checkpoint_every_n_tokens,
                       int32_t path, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
  Problem P;
  int r = validate_fwd(q, k, v, g, beta, h0, cu_seqlens, n_seq, o, ht, &P);
  if (r) return r;
  const int32_t every = checkpoint_every_n_tokens;
  if (every <= 0 || every % kChunk != 0) return GDR_ERR_CKPT;
  if (!state_checkpoints || !checkpoint_cu_starts) return GDR_ERR_NULL;
  Desc C;
  if ((r = read_desc(state_checkpoints, GDR_F32, 4, &C))) return r;
  if (C.shape[0] < P.T / every || C.shape[1] != P.H || C.shape[2] != P.D || C.shape[3] != P.D)
    return GDR_ERR_CKPT;
  if (!compact(C)) return GDR_ERR_STRIDE;
  P.ck.h = reinterpret_cast<float *>(C.p);
  P.ck.off = checkpoint_cu_starts;
  P.ck.every = every;
  if ((r = device_ok())) return r;
  const int chosen = choose_path(P, scale, path);
  if (chosen < 0) return chosen;
  if (P.n_seq == 0) {
    return cudaMemsetAsync(checkpoint_cu_starts, 0, sizeof(int32_t), stream) == cudaSuccess
               ? GDR_OK
               : GDR_ERR_CUDA;
  }
  const size_t need = ws_bytes_for(P.T, P.n_seq, P.H, P.D, chosen);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return GDR_ERR_WORKSPACE;
  return run_fwd(P, scale, cu_seqlens, chosen, workspace, workspace_bytes, stream);
}

int gdr_chunk_fwd(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                  const gdr_tensor_t *g, const gdr_tensor_t *beta, float scale,
                  const gdr_tensor_t *h0, const int32_t *cu_seqlens, int32_t n_seq,
                  gdr_tensor_t *o, gdr_tensor_t *ht, cudaStream_t stream) {
  Problem P;
  int r = validate_fwd(q, k, v, g, beta, h0, cu_seqlens, n_seq, o, ht, &P);
  if (r) return r;
  if ((r = device_ok())) return r;
  const int chosen = choose_path(P, scale, GDR_PATH_AUTO);
  if (chosen < 0) return chosen;
  if (P.n_seq == 0) return GDR_OK;
  const size_t need = ws_bytes_for(P.T, P.n_seq, P.H, P.D, chosen);
  void *ws = nullptr;
  if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) return GDR_ERR_CUDA;
  r = run_fwd(P, scale, cu_seqlens, chosen, ws, need, stream);
  if (cudaFreeAsync(ws, stream) != cudaSuccess && r == GDR_OK) r = GDR_ERR_CUDA;
  return r;
}

size_t gdr_chunk_bwd_workspace_bytes(int64_t T, int32_t n_seq, int32_t Hk, int32_t H,
                                     int32_t dk, int32_t dv) {
  if (T < 0 || n_seq < 0 || Hk <= 0 || H <= 0 || dk <= 0 || dv <= 0 || H % Hk) return 0;
  const int32_t D = dk > dv ? dk : dv;
  return carve_index(nullptr, T, n_seq).bytes + bwd_work_bytes(T, n_seq, Hk, H, D);
}

int gdr_chunk_bwd(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                  const gdr_tensor_t *g, const gdr_tensor_t *beta, float scale,
                  const gdr_tensor_t *h0, const int32_t *cu_seqlens, int32_t n_seq,
                  const gdr_tensor_t *dout, const gdr_tensor_t *dht, gdr_tensor_t *dq,
                  gdr_tensor_t *dk, gdr_tensor_t *dv, gdr_tensor_t *dg, gdr_tensor_t *dbeta,
                  gdr_tensor_t *dh0, void *workspace, size_t workspace_bytes,
                  cudaStream_t stream) {
  Problem P;
  // dout is checked as the forward's o, dht as its ht
  int r = validate_fwd(q, k, v, g, beta, h0, cu_seqlens, n_seq, dout, dht, &P);
  if (r) return r;
  Desc Dq, Dk, Dv, Dg, Db, Dh;
  const int64_t qs[3] = {P.T, P.Hk, P.D}, vs[3] = {P.T, P.H, P.D}, gs[2] = {P.T, P.H};
  if ((r = read_desc(dq, GDR_F32, 3, &Dq)) || (r = read_desc(dk, GDR_F32, 3, &Dk)) ||
      (r = read_desc(dv, GDR_F32, 3, &Dv)) || (r = read_desc(dg, GDR_F32, 2, &Dg)) ||
      (r = read_desc(dbeta, GDR_F32, 2, &Db)))
    return r;
  for (int i = 0; i < 3; ++i)
    if (Dq.shape[i] != qs[i] || Dk.shape[i] != qs[i] || Dv.shape[i] != vs[i]) return GDR_ERR_SHAPE;
  for (int i = 0; i < 2; ++i)
    if (Dg.shape[i] != gs[i] || Db.shape[i] != gs[i]) return GDR_ERR_SHAPE;
  if (!compact(Dq) || !compact(Dk) || !compact(Dv) || !compact(Dg) || !compact(Db))
    return GDR_ERR_STRIDE;
  if (dh0) {
    if ((r = read_desc(dh0, GDR_F32, 4, &Dh))) return r;
    if (Dh.shape[0] != n_seq) return GDR_ERR_NSEQ;
    if (Dh.shape[1] != P.H || Dh.shape[2] != P.D || Dh.shape[3] != P.D) return GDR_ERR_SHAPE;
    if (!compact(Dh)) return GDR_ERR_STRIDE;
  }
  if ((r = device_ok())) return r;
  if (P.n_seq == 0) return GDR_OK;
  const size_t need = gdr_chunk_bwd_workspace_bytes(P.T, P.n_seq, P.Hk, P.H, P.D, P.D);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return GDR_ERR_WORKSPACE;
  // tokens outside every segment keep zero gradients
  const size_t tq = sizeof(float) * (size_t)P.T * P.Hk * P.D;
  const size_t tv = sizeof(float) * (size_t)P.T * P.H * P.D, tg = sizeof(float) * (size_t)P.T * P.H;
  if (cudaMemsetAsync(Dq.p, 0, tq, stream) != cudaSuccess ||
      cudaMemsetAsync(Dk.p, 0, tq, stream) != cudaSuccess ||
      cudaMemsetAsync(Dv.p, 0, tv, stream) != cudaSuccess ||
      cudaMemsetAsync(Dg.p, 0, tg, stream) != cudaSuccess ||
      cudaMemsetAsync(Db.p, 0, tg, stream) != cudaSuccess)
    return GDR_ERR_CUDA;
  const IndexWs ix = carve_index(workspace, P.T, P.n_seq);
  const int64_t cap = chunk_bound(P.T, P.n_seq);
  if (launch_chunk_index(cu_seqlens, P.n_seq, P.T, ix.seg, ix.chunks, cap, ix.n_chunks,
                         stream) != cudaSuccess ||
      launch_seg_order(ix.seg, P.n_seq, ix.order, stream) != cudaSuccess)
    return GDR_ERR_CUDA;
  BwdArgs a{};
  a.s = StageShapes{P.T, P.n_seq, P.Hk, P.H, P.D, cap};
  a.q = view_of(P.q);
  a.k = view_of(P.k);
  a.v = view_of(P.v);
  a.g = view_of(P.g);
  a.beta = view_of(P.beta);
  a.dout = view_of(P.o);
  a.h0 = P.has_h0 ? reinterpret_cast<const float *>(P.h0.p) : nullptr;
  a.dht = P.has_ht ? reinterpret_cast<const float *>(P.ht.p) : nullptr;
  a.scale = scale;
  a.dq = view_of(Dq);
  a.dk = view_of(Dk);
  a.dv = view_of(Dv);
  a.dg = view_of(Dg);
  a.dbeta = view_of(Db);
  a.dh0 = dh0 ? reinterpret_cast<float *>(Dh.p) : nullptr;
  a.seg = ix.seg;
  a.order = ix.order;
  a.chunks = ix.chunks;
  a.n_chunks = ix.n_chunks;
  a.work = reinterpret_cast<char *>(workspace) + ix.bytes;
  return launch_bwd(a, stream) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

int gdr_chunk_index(const int32_t *cu_seqlens, int32_t n_seq, int64_t T, int32_t *seg_table,
                    int32_t *chunk_table, int32_t *n_chunks, cudaStream_t stream) {
  if (n_seq < 0) return GDR_ERR_NSEQ;
  if (T < 0 || T > 0x7fffffffLL) return GDR_ERR_SHAPE;
  if (!n_chunks) return GDR_ERR_NULL;
  if (n_seq > 0 && (!cu_seqlens || !seg_table || !chunk_table)) return GDR_ERR_NULL;
  int r;
  if ((r = device_ok())) return r;
  if (n_seq == 0) {
    return cudaMemsetAsync(n_chunks, 0, sizeof(int32_t), stream) == cudaSuccess ? GDR_OK
                                                                                 : GDR_ERR_CUDA;
  }
  const cudaError_t e = launch_chunk_index(
      cu_seqlens, n_seq, T, reinterpret_cast<SegInfo *>(seg_table),
      reinterpret_cast<ChunkInfo *>(chunk_table), chunk_bound(T, n_seq), n_chunks, stream);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

static int check_stage_ws(void *ws, size_t bytes, int64_t T, int32_t n_seq) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) ||
      bytes < carve_index(nullptr, T, n_seq).bytes)
    return GDR_ERR_WORKSPACE;
  return GDR_OK;
}

int gdr_chunk_prep(const gdr_tensor_t *k, const gdr_tensor_t *v, const gdr_tensor_t *g,
                   const gdr_tensor_t *beta, const int32_t *cu_seqlens, int32_t n_seq,
                   gdr_tensor_t *w, gdr_tensor_t *u, gdr_tensor_t *gcum, void *workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  Desc K, V, Gd, B, Wd, Ud, Gc;
  int r;
  if ((r = read_desc(k, GDR_BF16, 3, &K)) || (r = read_desc(v, GDR_BF16, 3, &V)) ||
      (r = read_desc(g, GDR_F32, 2, &Gd)) || (r = read_desc(beta, GDR_BF16, 2, &B)) ||
      (r = read_desc(w, GDR_BF16, 3, &Wd)) || (r = read_desc(u, GDR_BF16, 3, &Ud)) ||
      (r = read_desc(gcum, GDR_F32, 2, &Gc)))
    return r;
  const int64_t T = K.shape[0], Hk = K.shape[1], D = K.shape[2], H = V.shape[1];
  if (V.shape[0] != T || Gd.shape[0] != T || B.shape[0] != T || Wd.shape[0] != T ||
      Ud.shape[0] != T || Gc.shape[0] != T)
    return GDR_ERR_SHAPE;
  if (Gd.shape[1] != H || B.shape[1] != H || Wd.shape[1] != H || Ud.shape[1] != H ||
      Gc.shape[1] != H || Wd.shape[2] != D || Ud.shape[2] != D)
    return GDR_ERR_SHAPE;
  if (V.shape[2] != D || (D != 64 && D != 128)) return GDR_ERR_DIM;
  if (Hk <= 0 || H <= 0) return GDR_ERR_SHAPE;
  if (H % Hk) return GDR_ERR_HEADS;
  if (T > 0x7fffffffLL) return GDR_ERR_SHAPE;
  if (n_seq < 0) return GDR_ERR_NSEQ;
  if (n_seq > 0 && !cu_seqlens) return GDR_ERR_NULL;
  if ((r = device_ok())) return r;
  if (n_seq == 0) return GDR_OK;
  if ((r = check_stage_ws(workspace, workspace_bytes, T, n_seq))) return r;
  const IndexWs ix = carve_index(workspace, T, n_seq);
  const StageShapes s{T, n_seq, (int32_t)Hk, (int32_t)H, (int32_t)D, chunk_bound(T, n_seq)};
  cudaError_t e = launch_chunk_index(cu_seqlens, n_seq, T, ix.seg, ix.chunks, s.chunk_cap,
                                     ix.n_chunks, stream);
  if (e == cudaSuccess)
    e = launch_prep(s, view_of(K), view_of(V), view_of(Gd), view_of(B), view_of(Wd),
                    view_of(Ud), view_of(Gc), ix.seg, ix.chunks, ix.n_chunks, stream);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

int gdr_state_scan(const gdr_tensor_t *k, const gdr_tensor_t *w, const gdr_tensor_t *u,
                   const gdr_tensor_t *gcum, const gdr_tensor_t *h0,
                   const int32_t *cu_seqlens, int32_t n_seq, gdr_tensor_t *h,
                   gdr_tensor_t *v_new, gdr_tensor_t *ht, void *workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  Desc K, Wd, Ud, Gc, Hd, Vn, H0, HT;
  int r;
  if ((r = read_desc(k, GDR_BF16, 3, &K)) || (r = read_desc(w, GDR_BF16, 3, &Wd)) ||
      (r = read_desc(u, GDR_BF16, 3, &Ud)) || (r = read_desc(gcum, GDR_F32, 2, &Gc)) ||
      (r = read_desc(h, GDR_BF16, 4, &Hd)) || (r = read_desc(v_new, GDR_BF16, 3, &Vn)))
    return r;
  const int64_t T = K.shape[0], Hk = K.shape[1], D = K.shape[2], H = Wd.shape[1];
  if (Wd.shape[0] != T || Ud.shape[0] != T || Gc.shape[0] != T || Vn.shape[0] != T)
    return GDR_ERR_SHAPE;
  if (Ud.shape[1] != H || Gc.shape[1] != H || Vn.shape[1] != H || Wd.shape[2] != D ||
      Ud.shape[2] != D || Vn.shape[2] != D)
    return GDR_ERR_SHAPE;
  if (D != 64 && D != 128) return GDR_ERR_DIM;
  if (Hk <= 0 || H <= 0) return GDR_ERR_SHAPE;
  if (H % Hk) return GDR_ERR_HEADS;
  if (T > 0x7fffffffLL) return GDR_ERR_SHAPE;
  if (n_seq < 0) return GDR_ERR_NSEQ;
  if (n_seq > 0 && !cu_seqlens) return GDR_ERR_NULL;
  const int64_t cap = chunk_bound(T, n_seq);
  if (Hd.shape[0] < cap || Hd.shape[1] != H || Hd.shape[2] != D || Hd.shape[3] != D)
    return GDR_ERR_SHAPE;
  if (!compact(Hd)) return GDR_ERR_STRIDE;
  const int64_t sshape[4] = {n_seq, H, D, D};
  if (h0) {
    if ((r = read_desc(h0, GDR_F32, 4, &H0))) return r;
    for (int i = 0; i < 4; ++i)
      if (H0.shape[i] != sshape[i]) return i ? GDR_ERR_SHAPE : GDR_ERR_NSEQ;
    if (!compact(H0)) return GDR_ERR_STRIDE;
  }
  if (ht) {
    if ((r = read_desc(ht, GDR_F32, 4, &HT))) return r;
    for (int i = 0; i < 4; ++i)
      if (HT.shape[i] != sshape[i]) return i ? GDR_ERR_SHAPE : GDR_ERR_NSEQ;
    if (!compact(HT)) return GDR_ERR_STRIDE;
  }
  if ((r = device_ok())) return r;
  if (n_seq == 0) return GDR_OK;
  if ((r = check_stage_ws(workspace, workspace_bytes, T, n_seq))) return r;
  const IndexWs ix = carve_index(workspace, T, n_seq);
  const StageShapes s{T, n_seq, (int32_t)Hk, (int32_t)H, (int32_t)D, cap};
  cudaError_t e = launch_chunk_index(cu_seqlens, n_seq, T, ix.seg, ix.chunks, cap,
                                     ix.n_chunks, stream);
  if (e == cudaSuccess) e = launch_seg_order(ix.seg, n_seq, ix.order, stream);
  if (e == cudaSuccess)
    e = launch_scan_ordered(s, view_of(K), view_of(Wd), view_of(Ud), view_of(Gc),
                            h0 ? reinterpret_cast<const float *>(H0.p) : nullptr, Hd.p,
                            view_of(Vn), ht ? reinterpret_cast<float *>(HT.p) : nullptr, Ckpt{},
                            ix.seg, ix.order, stream);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

int gdr_chunk_out(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v_new,
                  const gdr_tensor_t *h, const gdr_tensor_t *gcum, float scale,
                  const int32_t *cu_seqlens, int32_t n_seq, gdr_tensor_t *o, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
  Desc Q, K, Vn, Hd, Gc, O;
  int r;
  if ((r = read_desc(q, GDR_BF16, 3, &Q)) || (r = read_desc(k, GDR_BF16, 3, &K)) ||
      (r = read_desc(v_new, GDR_BF16, 3, &Vn)) || (r = read_desc(h, GDR_BF16, 4, &Hd)) ||
      (r = read_desc(gcum, GDR_F32, 2, &Gc)) || (r = read_desc(o, GDR_BF16, 3, &O)))
    return r;
  const int64_t T = Q.shape[0], Hk = Q.shape[1], D = Q.shape[2], H = Vn.shape[1];
  for (int i = 0; i < 3; ++i)
    if (K.shape[i] != Q.shape[i]) return GDR_ERR_SHAPE;
  if (Vn.shape[0] != T || Gc.shape[0] != T || O.shape[0] != T) return GDR_ERR_SHAPE;
  if (Gc.shape[1] != H || O.shape[1] != H || Vn.shape[2] != D || O.shape[2] != D)
    return GDR_ERR_SHAPE;
  if (D != 64 && D != 128) return GDR_ERR_DIM;
  if (Hk <= 0 || H <= 0) return GDR_ERR_SHAPE;
  if (H % Hk) return GDR_ERR_HEADS;
  if (T > 0x7fffffffLL) return GDR_ERR_SHAPE;
  if (n_seq < 0) return GDR_ERR_NSEQ;
  if (n_seq > 0 && !cu_seqlens) return GDR_ERR_NULL;
  const int64_t cap = chunk_bound(T, n_seq);
  if (Hd.shape[0] < cap || Hd.shape[1] != H || Hd.shape[2] != D || Hd.shape[3] != D)
    return GDR_ERR_SHAPE;
  if (!compact(Hd)) return GDR_ERR_STRIDE;
  if ((r = device_ok())) return r;
  if (n_seq == 0) return GDR_OK;
  if ((r = check_stage_ws(workspace, workspace_bytes, T, n_seq))) return r;
  const IndexWs ix = carve_index(workspace, T, n_seq);
  const StageShapes s{T, n_seq, (int32_t)Hk, (int32_t)H, (int32_t)D, cap};
  cudaError_t e = launch_chunk_index(cu_seqlens, n_seq, T, ix.seg, ix.chunks, cap,
                                     ix.n_chunks, stream);
  if (e == cudaSuccess)
    e = launch_out(s, view_of(Q), view_of(K), view_of(Vn), Hd.p, view_of(Gc), scale,
                   view_of(O), ix.seg, ix.chunks, ix.n_chunks, stream);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

int gdr_debug_check_cu_seqlens(const int32_t *cu_seqlens, int32_t n_seq, int64_t T,
                               int32_t *n_bad, int32_t *first_bad, cudaStream_t stream) {
  if (!cu_seqlens || !n_bad || !first_bad) return GDR_ERR_NULL;
  if (n_seq < 0) return GDR_ERR_NSEQ;
  int r;
  if ((r = device_ok())) return r;
  int32_t *d = nullptr;
  if (cudaMallocAsync(&d, 2 * sizeof(int32_t), stream) != cudaSuccess) return GDR_ERR_CUDA;
  int32_t hbuf[2] = {0, -1};
  cudaError_t e = launch_check_cu(cu_seqlens, n_seq, T, d, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(hbuf, d, sizeof hbuf, cudaMemcpyDeviceToHost, stream);
  const cudaError_t f = cudaFreeAsync(d, stream);
  if (e == cudaSuccess) e = f;
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return GDR_ERR_CUDA;
  *n_bad = hbuf[0];
  *first_bad = hbuf[1];
  return GDR_OK;
}

int gdr_device_status(int32_t *status_out) {
  if (!status_out) return GDR_ERR_NULL;
  return read_device_status(status_out) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

int gdr_debug_wait_selftest(uint32_t limit_us, cudaStream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return GDR_ERR_SHAPE;
  int r;
  if ((r = device_ok())) return r;
  return launch_wait_selftest(limit_us, GDR_STATUS_WAIT_SELFTEST, stream) == cudaSuccess
             ? GDR_OK
             : GDR_ERR_CUDA;
}

int gdr_clear_device_status(void) {
  return clear_device_status() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gdr_chunk_out_noalloc: stage 3 with its chunk tables in a static device array,
// for callers that cannot allocate device memory.  Host code may not pass the
// array's name to a kernel (in host code it names a host-side shadow); the
// device address is looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = GDR_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up on first use).
int noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDR_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return GDR_OK;
}

}  // namespace

extern "C" int gdr_chunk_out_noalloc(const gdr_tensor_t *q, const gdr_tensor_t *k,
                                     const gdr_tensor_t *v_new, const gdr_tensor_t *h,
                                     const gdr_tensor_t *gcum, float scale,
                                     const int32_t *cu_seqlens, int32_t n_seq, gdr_tensor_t *o,
                                     cudaStream_t stream) {
  Desc Q, K, Vn, Hd, Gc, O;
  int r;
  if ((r = read_desc(q, GDR_BF16, 3, &Q)) || (r = read_desc(k, GDR_BF16, 3, &K)) ||
      (r = read_desc(v_new, GDR_BF16, 3, &Vn)) || (r = read_desc(h, GDR_BF16, 4, &Hd)) ||
      (r = read_desc(gcum, GDR_F32, 2, &Gc)) || (r = read_desc(o, GDR_BF16, 3, &O)))
    return r;
  const int64_t T = Q.shape[0], Hk = Q.shape[1], D = Q.shape[2], H = Vn.shape[1];
  for (int i = 0; i < 3; ++i)
    if (K.shape[i] != Q.shape[i]) return GDR_ERR_SHAPE;
  if (Vn.shape[0] != T || Gc.shape[0] != T || O.shape[0] != T) return GDR_ERR_SHAPE;
  if (Gc.shape[1] != H || O.shape[1] != H || Vn.shape[2] != D || O.shape[2] != D)
    return GDR_ERR_SHAPE;
  if (D != 64 && D != 128) return GDR_ERR_DIM;
  if (Hk <= 0 || H <= 0) return GDR_ERR_SHAPE;
  if (H % Hk) return GDR_ERR_HEADS;
  if (T > 0x7fffffffLL) return GDR_ERR_SHAPE;
  if (n_seq < 0) return GDR_ERR_NSEQ;
  if (n_seq > 0 && !cu_seqlens) return GDR_ERR_NULL;
  const int64_t cap = chunk_bound(T, n_seq);
  if (Hd.shape[0] < cap || Hd.shape[1] != H || Hd.shape[2] != D || Hd.shape[3] != D)
    return GDR_ERR_SHAPE;
  if (!compact(Hd)) return GDR_ERR_STRIDE;
  if ((r = device_ok())) return r;
  if (n_seq == 0) return GDR_OK;
  if (carve_index(nullptr, T, n_seq).bytes > kNoAllocScratchBytes) return GDR_ERR_SCRATCH_LIMIT;
  void *scratch = nullptr;
  if ((r = noalloc_scratch(&scratch))) return r;
  const IndexWs ix = carve_index(scratch, T, n_seq);
  const StageShapes s{T, n_seq, (int32_t)Hk, (int32_t)H, (int32_t)D, cap};
  cudaError_t e = launch_chunk_index(cu_seqlens, n_seq, T, ix.seg, ix.chunks, cap,
                                     ix.n_chunks, stream);
  if (e == cudaSuccess)
    e = launch_out(s, view_of(Q), view_of(K), view_of(Vn), Hd.p, view_of(Gc), scale,
                   view_of(O), ix.seg, ix.chunks, ix.n_chunks, stream);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

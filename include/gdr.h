/*
 * gdr.h -- C ABI of libgdr: the chunked gated delta rule forward on GB300 (sm_103a).
 *
 * The operation (per packed segment n and value head h, state S of dk x dv):
 *
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   S_{start-1} = h0[n,h] or 0
 *     o_t = scale * S_t^T q_t,                                          ht[n,h] = S_last
 *
 * evaluated chunkwise with chunks of 64 tokens, the chunk size of FlashQLA's
 * chunk_gated_delta_rule varlen path ("Findings from integrating FlashQLA's
 * Blackwell GDN kernels into a JAX trainer", section 1: prepare_chunk_indices(cu, 64);
 * "FlashQLA GDN backend produces different tokens from FLA Triton on
 * correctness-test prompts", Setup: chunk_size=64, varlen API).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every data pointer is a DEVICE pointer on the current CUDA device, except
 *   the gdr_tensor_t structs themselves and their `strides` arrays, which live
 *   in host memory and are only read during the call.  The caller owns every
 *   buffer; the library keeps no pointer after a call returns and has no
 *   cache keyed on addresses (the stale-cache failure in "Findings ...",
 *   section 1, cannot occur).
 * - Layouts (row-major by default):
 *       q, k   [T, Hk, dk]  bf16          v, o   [T, H, dv]  bf16
 *       g      [T, H]       f32 (natural-log decay, exp(g) multiplies the state)
 *       beta   [T, H]       bf16          h0, ht [N, H, dk, dv] f32 (row = key dim)
 *   H % Hk == 0 and value head h reads query/key head h / (H / Hk).
 *   dk == dv, with dk in {64, 128}.
 * - `strides == NULL` means compact row-major, as DLPack defines it ("Findings
 *   ...", section 3: stubs that rejected NULL strides).  Explicit strides are
 *   in elements; the innermost stride must be 1.  h0/ht must be compact.
 * - cu_seqlens: DEVICE int32 array of n_seq + 1 offsets into the token axis.
 *   It is never read on the host.  Offsets are clamped to [0, T] and made
 *   non-decreasing by a running maximum, so a malformed array cannot cause an
 *   out-of-bounds access.  Repeated offsets are length-0 ("ghost") segments
 *   ("Findings ...", section 2): they write no o and, when ht is requested,
 *   ht[n] = h0[n] (or zeros).  Tokens outside every segment are not written.
 * - Return value: GDR_OK (0) or a negative gdr_status code.  Nothing is
 *   thrown across the ABI.  Kernels are enqueued on `stream` and the call does
 *   not synchronise; asynchronous device errors surface on the stream.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of gdr_tensor_t::dtype. */
enum gdr_dtype { GDR_BF16 = 1, GDR_F32 = 2, GDR_I32 = 3 };

/* Status codes. */
enum gdr_status {
  GDR_OK = 0,
  GDR_ERR_NULL = -1,      /* a required pointer or descriptor is NULL          */
  GDR_ERR_DTYPE = -2,     /* wrong element type                                 */
  GDR_ERR_SHAPE = -3,     /* wrong rank or inconsistent extents                 */
  GDR_ERR_STRIDE = -4,    /* innermost stride != 1, negative stride, non-compact state */
  GDR_ERR_DIM = -5,       /* head dimension not supported (dk == dv in {64,128}) */
  GDR_ERR_HEADS = -6,     /* H % Hk != 0                                        */
  GDR_ERR_NSEQ = -7,      /* n_seq < 0 or n_seq inconsistent with h0/ht         */
  GDR_ERR_WORKSPACE = -8, /* workspace NULL, too small or not 256-byte aligned   */
  GDR_ERR_PATH = -9,      /* unknown path, or FUSED requested but unsupported    */
  GDR_ERR_CUDA = -10,     /* a CUDA runtime call or kernel launch failed         */
  GDR_ERR_ALIGN = -11,    /* a base pointer or row stride is not 16-byte aligned */
  GDR_ERR_DEVICE = -12,   /* the current device is not sm_103 (GB300)            */
  GDR_ERR_SCRATCH_LIMIT = -13, /* problem too large for gdr_chunk_out_noalloc's static scratch */
  GDR_ERR_CKPT = -14           /* checkpoint interval not a positive multiple of 64, or
                                  checkpoint buffer of the wrong type, shape or size  */
};

/* Execution paths of the forward. */
enum gdr_path {
  GDR_PATH_AUTO = 0,   /* fused when its alignment preconditions hold, else staged */
  GDR_PATH_FUSED = 1,  /* one persistent kernel per call; intermediates stay on chip.
                          When the (segment, head) pairs are too few to fill the GPU
                          (3 x n_seq x H <= its SM count) and no checkpoints are asked
                          for, segments of 48 chunks or more are cut into 3 to 8
                          pieces that run on different SMs, joined through the affine
                          state map S_out = M S_in + R of each piece (FlashQLA's
                          sequence split, `seq_split_idx`, "Findings ...", section 2) */
  GDR_PATH_STAGED = 2, /* the three stages as separate kernels with HBM intermediates */
  GDR_PATH_FUSED_WHOLE = 3 /* the fused kernel with every (segment, head) in one piece */
};

typedef struct gdr_tensor {
  void *data;             /* device pointer to element [0,...,0]           */
  int32_t dtype;          /* enum gdr_dtype                                  */
  int32_t ndim;           /* 1..4                                            */
  int64_t shape[4];       /* extents, outermost first                        */
  const int64_t *strides; /* host array of ndim strides in elements, or NULL */
} gdr_tensor_t;

/*
 * gdr_chunk_fwd -- the whole forward: q, k, v, g, beta (+ optional h0) -> o (+ optional ht).
 *
 *   q, k    [T, Hk, dk] bf16; v [T, H, dv] bf16; g [T, H] f32; beta [T, H] bf16
 *   scale   multiplies the output (o = scale * S^T q)
 *   h0      [n_seq, H, dk, dv] f32 initial states, or NULL for zero states
 *   cu_seqlens, n_seq   see the conventions above
 *   o       [T, H, dv] bf16 output (round-to-nearest-even); covered tokens only
 *   ht      [n_seq, H, dk, dv] f32 final states, or NULL to skip them
 *           (FlashQLA drops dead h0/ht parameters in this case: "Findings ...", section 4)
 *
 * Runs GDR_PATH_AUTO.  Scratch memory is taken with cudaMallocAsync on `stream`
 * and released with cudaFreeAsync on the same stream.  Errors: any gdr_status.
 */
int gdr_chunk_fwd(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                  const gdr_tensor_t *g, const gdr_tensor_t *beta, float scale,
                  const gdr_tensor_t *h0, const int32_t *cu_seqlens, int32_t n_seq,
                  gdr_tensor_t *o, gdr_tensor_t *ht, cudaStream_t stream);

/* Bytes of device scratch gdr_chunk_fwd_ws needs for these extents and path
 * (GDR_PATH_AUTO sizes for the larger of the two) on the current device: the
 * fused path's sequence split depends on its SM count, and takes up to
 * 24 x n_seq x H x dv x dv x 4 bytes for the pieces' states.  Never fails;
 * returns 0 for negative arguments. */
size_t gdr_chunk_fwd_workspace_bytes(int64_t T, int32_t n_seq, int32_t H, int32_t dk,
                                     int32_t dv, int32_t path);

/*
 * gdr_chunk_fwd_ws -- gdr_chunk_fwd with a caller-owned workspace and an explicit path.
 *   workspace   device pointer, 256-byte aligned, at least
 *               gdr_chunk_fwd_workspace_bytes(T, n_seq, H, dk, dv, path) bytes.
 *               Stream-ordered: it may be reused once the call's work on `stream` is done.
 * Errors: as gdr_chunk_fwd, plus GDR_ERR_WORKSPACE and GDR_ERR_PATH.
 */
int gdr_chunk_fwd_ws(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                     const gdr_tensor_t *g, const gdr_tensor_t *beta, float scale,
                     const gdr_tensor_t *h0, const int32_t *cu_seqlens, int32_t n_seq,
                     gdr_tensor_t *o, gdr_tensor_t *ht, int32_t path, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream);

/*
 * gdr_chunk_fwd_ckpt -- gdr_chunk_fwd_ws that also writes state checkpoints every
 * checkpoint_every_n_tokens tokens of each segment, for prefix caching.  The FlashInfer
 * KDA prefill keeps this surface (state_checkpoints / checkpoint_cu_starts /
 * checkpoint_every_n_tokens kwargs, "feat(cake_kda): add paired recurrent training for
 * SM100a and SM103a", the released inference surface kept by the cherry-picked commit);
 * the pages describe no layout, so the one below is this library's.
 *   checkpoint_every_n_tokens  positive multiple of 64 (the chunk size).
 *   state_checkpoints   [rows, H, dk, dv] fp32 out, compact; rows >=
 *                       gdr_ckpt_count_bound(T, checkpoint_every_n_tokens).  Checkpoint m
 *                       (m = 1 .. floor(len_n / every)) of segment n is the state S
 *                       ([dk][dv], as ht) after the segment's first m * every tokens, in row
 *                       checkpoint_cu_starts[n] + m - 1.  Other rows are not written.
 *   checkpoint_cu_starts  device int32 [n_seq + 1] out: the running sum of
 *                       floor(len_n / every) (lengths after the cu_seqlens reading); the last
 *                       entry is the number of checkpoints written.
 * Workspace as gdr_chunk_fwd_ws.  Errors: as gdr_chunk_fwd_ws, plus GDR_ERR_CKPT.
 */
int gdr_chunk_fwd_ckpt(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                       const gdr_tensor_t *g, const gdr_tensor_t *beta, float scale,
                       const gdr_tensor_t *h0, const int32_t *cu_seqlens, int32_t n_seq,
                       gdr_tensor_t *o, gdr_tensor_t *ht, gdr_tensor_t *state_checkpoints,
                       int32_t *checkpoint_cu_starts, int32_t checkpoint_every_n_tokens,
                       int32_t path, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Rows gdr_chunk_fwd_ckpt may write: floor(T / checkpoint_every_n_tokens) (0 for bad
 * arguments). */
int64_t gdr_ckpt_count_bound(int64_t T, int32_t checkpoint_every_n_tokens);

/* Pieces per segment that GDR_PATH_FUSED cuts long segments into on the current
 * device for T tokens in n_seq segments of H value heads (1: no split; else 3..8).
 * The first piece may weigh 2 or 3 of the others (it runs while the others' state
 * maps are formed); a segment of c chunks gets at most floor(c / 16) - (weight - 1)
 * pieces, and stays whole when that is under 3.  Returns 1 when no device can be
 * queried. */
int32_t gdr_fused_split_pieces(int64_t T, int32_t n_seq, int32_t H);

/* The split planner behind gdr_fused_split_pieces, for any machine size: for `units`
 * (segment, value head) pairs on `sms` SMs, the pieces per long segment (1: no split;
 * else 3..8) and, in *lead (may be NULL), the first piece's weight (1..3).  The plan
 * minimises pass A + pass B of the split in units of the whole segment: pass A runs the
 * first pieces (weight `lead`) and, for every middle piece, its state map's offset R and
 * transition M (weight 1 each); pass B the P - 1 later pieces; each pass on `sms` SMs
 * taking units in that order as they come free; ties go to fewer pieces, and no split
 * unless 3 * units <= sms.  Pure host arithmetic; non-positive arguments give 1 and
 * lead 1. */
int32_t gdr_split_plan(int64_t units, int32_t sms, int32_t *lead);

/*
 * gdr_chunk_bwd -- the backward: gradients of gdr_chunk_fwd's outputs with respect to
 * all its inputs.  FlashQLA's GDN kernels serve as a training backend whose backward
 * is bit-reproducible and tolerates length-0 segments ("Findings ...", intro and
 * section 2); the pages print no backward formula, so this is the gradient of the
 * forward defined above (its chunk form is written out in gdr_bwd.cu).
 *
 *   q, k, v, g, beta, scale, h0, cu_seqlens, n_seq
 *           the forward's inputs, as gdr_chunk_fwd takes them (the forward is
 *           recomputed from them; nothing of a previous forward call is kept)
 *   dout    [T, H, dv] bf16, dL/do (read for covered tokens only)
 *   dht     [n_seq, H, dk, dv] f32 compact, dL/dht, or NULL for zero
 *   dq, dk  [T, Hk, dk] f32 compact out (grouped heads: summed over the value heads
 *           that share a query/key head, in head order)
 *   dv      [T, H, dv] f32 compact out
 *   dg, dbeta  [T, H] f32 compact out
 *   dh0     [n_seq, H, dk, dv] f32 compact out, or NULL to skip: the gradient for the
 *           initial state (h0 or the zero state); an empty segment's dh0 is its dht
 *   workspace   device, 256-byte aligned, >= gdr_chunk_bwd_workspace_bytes(...) bytes
 *
 * Tokens outside every segment get zero gradients.  Deterministic: every output
 * element is written by one thread per kernel in a fixed order (no atomics), so
 * results are bit-identical from run to run.  Stream-ordered, no host synchronisation.
 * Errors: as gdr_chunk_fwd_ws (dout is checked like o, dht like ht), GDR_ERR_STRIDE
 * for non-compact outputs, GDR_ERR_WORKSPACE.
 */
int gdr_chunk_bwd(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v,
                  const gdr_tensor_t *g, const gdr_tensor_t *beta, float scale,
                  const gdr_tensor_t *h0, const int32_t *cu_seqlens, int32_t n_seq,
                  const gdr_tensor_t *dout, const gdr_tensor_t *dht, gdr_tensor_t *dq,
                  gdr_tensor_t *dk, gdr_tensor_t *dv, gdr_tensor_t *dg, gdr_tensor_t *dbeta,
                  gdr_tensor_t *dh0, void *workspace, size_t workspace_bytes,
                  cudaStream_t stream);

/* Bytes of device scratch gdr_chunk_bwd needs (0 for bad arguments). */
size_t gdr_chunk_bwd_workspace_bytes(int64_t T, int32_t n_seq, int32_t Hk, int32_t H,
                                     int32_t dk, int32_t dv);

/* Upper bound on the number of 64-token chunks: ceil(T / 64) + n_seq. */
int64_t gdr_chunk_count_bound(int64_t T, int32_t n_seq);

/* Bytes of device scratch each stage entry point below needs (chunk tables). */
size_t gdr_stage_workspace_bytes(int64_t T, int32_t n_seq);

/*
 * Chunk enumeration from cu_seqlens, on the device.
 *   seg_table   [n_seq, 4] int32 out: (start, end, first chunk id, chunk count) per segment
 *   chunk_table [gdr_chunk_count_bound(T, n_seq), 4] int32 out: (segment, first token,
 *               length 1..64, 0) per chunk id; ids are assigned segment by segment.
 *   n_chunks    device int32 out: the number of chunks.
 * Errors: GDR_ERR_NULL, GDR_ERR_NSEQ, GDR_ERR_SHAPE (T < 0), GDR_ERR_CUDA.
 */
int gdr_chunk_index(const int32_t *cu_seqlens, int32_t n_seq, int64_t T, int32_t *seg_table,
                    int32_t *chunk_table, int32_t *n_chunks, cudaStream_t stream);

/*
 * Stage 1, gdr_chunk_prep: per (chunk, value head) with chunk-local index i, j:
 *   G_i  = sum_{t<=i} g_t (chunk-local inclusive cumsum)
 *   A_ij = beta_i exp(G_i - G_j) k_i.k_j (j < i), Tm = (I + A)^-1
 *   W = Tm diag(beta exp(G)) K,  U = Tm diag(beta) V
 * Outputs (compact, covered tokens only): w [T, H, dk] bf16, u [T, H, dv] bf16,
 * gcum [T, H] f32.  workspace: gdr_stage_workspace_bytes(T, n_seq) bytes.
 */
int gdr_chunk_prep(const gdr_tensor_t *k, const gdr_tensor_t *v, const gdr_tensor_t *g,
                   const gdr_tensor_t *beta, const int32_t *cu_seqlens, int32_t n_seq,
                   gdr_tensor_t *w, gdr_tensor_t *u, gdr_tensor_t *gcum, void *workspace,
                   size_t workspace_bytes, cudaStream_t stream);

/*
 * Stage 2, gdr_state_scan: per (segment, value head), sequential over chunks, fp32 state:
 *   h[c] = S (bf16);  V' = U - W S;  S <- exp(G_last) S + (diag(exp(G_last - G)) K)^T V'
 * Inputs: k [T, Hk, dk] bf16, w/u/gcum from stage 1, h0 (or NULL).
 * Outputs: h [gdr_chunk_count_bound, H, dk, dv] bf16 indexed by chunk id,
 * v_new [T, H, dv] bf16 (V'), ht (or NULL).  workspace as for stage 1.
 */
int gdr_state_scan(const gdr_tensor_t *k, const gdr_tensor_t *w, const gdr_tensor_t *u,
                   const gdr_tensor_t *gcum, const gdr_tensor_t *h0,
                   const int32_t *cu_seqlens, int32_t n_seq, gdr_tensor_t *h,
                   gdr_tensor_t *v_new, gdr_tensor_t *ht, void *workspace,
                   size_t workspace_bytes, cudaStream_t stream);

/*
 * Stage 3, gdr_chunk_out: per (chunk, value head):
 *   O = scale [ diag(exp(G)) Q h[c] + (M o Q K^T) V' ],  M_ij = exp(G_i - G_j) for j <= i, else 0
 * Inputs: q, k [T, Hk, dk] bf16, v_new [T, H, dv] bf16, h and gcum as above.
 * Output: o [T, H, dv] bf16, covered tokens only.  workspace as for stage 1.
 */
int gdr_chunk_out(const gdr_tensor_t *q, const gdr_tensor_t *k, const gdr_tensor_t *v_new,
                  const gdr_tensor_t *h, const gdr_tensor_t *gcum, float scale,
                  const int32_t *cu_seqlens, int32_t n_seq, gdr_tensor_t *o, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream);

/*
 * Debug check of cu_seqlens (synchronises `stream`): *n_bad receives the number of
 * offsets that are negative, above T, or below their predecessor, and *first_bad the
 * index of the first such offset (-1 if none).  Errors: GDR_ERR_NULL, GDR_ERR_NSEQ, GDR_ERR_CUDA.
 */
int gdr_debug_check_cu_seqlens(const int32_t *cu_seqlens, int32_t n_seq, int64_t T,
                               int32_t *n_bad, int32_t *first_bad, cudaStream_t stream);

/*
 * Device status word of the fused kernel.  Every bounded wait inside the fused
 * kernel that runs out (after 2 s) sets a nonzero code here: 0x1xx producer,
 * 0x2xx MMA issuer, 0x3xx prep warps, 0x4xx state warps; the CTA then drains its
 * copies and MMAs in flight, releases its Tensor Memory and returns instead of
 * hanging.  gdr_device_status synchronises the current device and
 * reads the word; gdr_clear_device_status resets it.  0 means no wait ran out.
 */
int gdr_device_status(int32_t *status_out);
int gdr_clear_device_status(void);

/*
 * Self-test of the bounded waits: launches one block that waits on an mbarrier
 * nothing ever arrives on.  The wait gives up after `limit_us` microseconds
 * (1..1000000), records GDR_STATUS_WAIT_SELFTEST in the device status word (if it
 * was 0) and the kernel returns normally; the context stays usable.  Read the word
 * with gdr_device_status.  Errors: GDR_ERR_SHAPE for a limit out of range,
 * GDR_ERR_DEVICE, GDR_ERR_CUDA.
 */
#define GDR_STATUS_WAIT_SELFTEST 0x7001
int gdr_debug_wait_selftest(uint32_t limit_us, cudaStream_t stream);

/*
 * gdr_chunk_out_noalloc -- gdr_chunk_out for callers that cannot allocate device memory.
 *
 * The papers behind this library have no counterpart of this entry point; it exists for
 * embedders that may not call cudaMalloc or hand out a workspace: engines with a fixed,
 * pre-planned memory budget, custom-call hosts that own every buffer, or code that must
 * not touch the allocator while it runs.  It computes exactly what gdr_chunk_out computes,
 * with the same arguments minus the workspace, and calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *
 * Scratch: the chunk tables (segment table, chunk table, chunk count) live in one static
 * device array of GDR_NOALLOC_SCRATCH_BYTES (4 MiB) inside libgdr; every GPU that loads
 * the library holds that array until the process exits.  A problem needs
 * 256 + 16 * max(n_seq, 1) + 16 * gdr_chunk_count_bound(T, n_seq) + 4 * max(n_seq, 1)
 * bytes, each term rounded up to 256 (the chunk count, the segment table, the chunk
 * table and the segment order); larger problems return GDR_ERR_SCRATCH_LIMIT (roughly
 * 260k chunks).
 * The tables are rewritten completely by every call, so nothing needs clearing between
 * calls.  Every call on a device shares the same array: calls whose work overlaps on the
 * GPU (different streams without ordering between them) race and may produce wrong
 * output; order them on one stream or with events.
 *
 * Set-up: the first call on each device (with that device current) looks up the array's
 * device address with cudaGetSymbolAddress and caches it; make that first call before
 * any stream capture on that device.
 *
 * Errors: as gdr_chunk_out (without GDR_ERR_WORKSPACE), plus GDR_ERR_SCRATCH_LIMIT, and
 * GDR_ERR_CUDA if the address lookup fails.
 */
#define GDR_NOALLOC_SCRATCH_BYTES (4u << 20)
int gdr_chunk_out_noalloc(const gdr_tensor_t *q, const gdr_tensor_t *k,
                          const gdr_tensor_t *v_new, const gdr_tensor_t *h,
                          const gdr_tensor_t *gcum, float scale, const int32_t *cu_seqlens,
                          int32_t n_seq, gdr_tensor_t *o, cudaStream_t stream);

/* Human-readable text for a gdr_status code (static storage). */
const char *gdr_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int gdr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H_ */

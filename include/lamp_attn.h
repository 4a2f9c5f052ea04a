/*
 * lamp_attn.h -- C ABI of the GB300 (sm_103a) LampAttention forward pass.
 *
 * Operation: the forward pass of look-ahead mixed-precision FlashAttention
 * described in "LampAttention: Look-Ahead Mixed-Precision FlashAttention for
 * Dedicated Accelerators" (arXiv 2609.39361), abstract: the key-query
 * products are accumulated, and their exponentials evaluated, in 8-bit
 * formats; sensitive sub-blocks are identified adaptively and recomputed in
 * 16-bit formats; the thresholds delta (first stage, default 2^-8, can be
 * disabled) and tau (recompute threshold, default 2^-1) and the per-tile
 * count of 16-bit sub-blocks (0 / 1 / 2+) follow Table 1's caption and
 * header and the captions of Figures 1-8.
 *
 * The paper gives no formulas; this library implements these readings:
 *   - 8-bit format FP8 E4M3 (OCP "fn": max 448, RNE, saturating);
 *   - S8 = fl8(sigma * sum_t fl8(q_t) fl8(k_t)), the sum taken exactly;
 *   - running max m_j of S8 over 64-key tiles in ascending key order;
 *   - x8 = fl8(S8 - m_j), P8 = fl8(exp(x8));
 *   - tiles of 64 queries x 64 keys, sub-blocks of 16 queries x 64 keys;
 *   - stage 1 of a sub-block: some visible entry has P8 >= delta;
 *     flagged: some visible entry has P8 >= delta and half-ulp8(S8) >= tau;
 *   - flagged rows: S16 = sigma * sum bf16(q) bf16(k) (FP32 accumulation),
 *     P16 = fp16(exp(S16 - m_j)); other rows use P8;
 *   - P.V in FP16 operands (V16 = fp16(v), saturating) with FP32
 *     accumulation; out = O / l, LSE = m + ln l.
 * The mask bytes and the histogram are bit-identical to a CPU statement of
 * these readings; out and LSE agree with it to 2e-3 / 1e-3 (plus the final
 * rounding of out to its dtype).
 *
 * All tensor pointers are DEVICE pointers owned by the caller; the library
 * keeps no reference after the call returns.  Work is enqueued on
 * `shapes->stream` and the call returns without synchronising.
 */
#ifndef LAMP_ATTN_H
#define LAMP_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LAMP_OK = 0,
  LAMP_ERR_INVALID_ARG = 1,  /* bad pointer, shape, stride, dtype or threshold */
  LAMP_ERR_UNSUPPORTED = 2,  /* head_dim not in {64,128,256}, or not an sm_103 device */
  LAMP_ERR_CUDA = 3,         /* a CUDA runtime / driver call failed */
  LAMP_ERR_TIMEOUT = 4,      /* a device-side wait hit its time limit (status word) */
  LAMP_ERR_WORKSPACE = 5,    /* caller workspace smaller than lamp_attn_workspace_bytes() */
  LAMP_ERR_TOO_LARGE = 6     /* lamp_attn_fwd_noalloc: the shapes need more scratch than
                                LAMP_NOALLOC_SCRATCH_BYTES */
} lamp_status;

/* Size of the fixed device array behind lamp_attn_fwd_noalloc (32 MiB). */
#define LAMP_NOALLOC_SCRATCH_BYTES (32u << 20)

typedef enum {
  LAMP_MASK_NONE = 0,    /* every key visible to every query */
  LAMP_MASK_CAUSAL = 1,  /* key c visible to query r iff c <= r */
  LAMP_MASK_SLIDING = 2  /* key c visible to query r iff r - window < c <= r */
} lamp_mask_kind;

typedef enum { LAMP_DT_BF16 = 0, LAMP_DT_FP32 = 1 } lamp_dtype;

typedef enum {
  LAMP_FORCE_OFF = 0,    /* the detector decides which sub-blocks run in 16 bits */
  LAMP_FORCE_ALL16 = 1,  /* every visible sub-block is recomputed in 16 bits */
  LAMP_FORCE_ALL8 = 2    /* no sub-block is recomputed (plain 8-bit path) */
} lamp_force;

/* Precision of P.V.  The paper ("LampAttention: Look-Ahead Mixed-Precision
 * FlashAttention for Dedicated Accelerators", abstract) puts the key-query
 * products and their exponentials in 8 bits and does not say how P.V is
 * computed. */
typedef enum {
  LAMP_PV_FP16 = 0,  /* P and V as FP16 for every row (P8 is exact in FP16) */
  LAMP_PV_FP8 = 1    /* rows of unflagged sub-blocks: P8 . fl8(v) on the FP8
                        tensor path (V rounded once, RNE, saturating); rows of
                        flagged sub-blocks keep P16 . fp16(v).  head_dim 64 or
                        128 (LAMP_ERR_UNSUPPORTED for 256) */
} lamp_pv_mode;

/* How the 8-bit key-query products accumulate into an 8-bit logit (the
 * abstract of the same paper: "accumulated ... in 8-bit formats"). */
typedef enum {
  LAMP_QK_EXACT = 0,   /* exact sum of the products, one E4M3 rounding:
                          S8 = fl8(sigma * sum_i fl8(q_i) fl8(k_i)) */
  LAMP_QK_CHUNK32 = 1  /* the running logit rounded to E4M3 after every
                          32-element chunk of d, in ascending order:
                          a_c = fl8(a_{c-1} + sigma * A_c) (product and sum in
                          double), S8 = the last a_c.  head_dim 64 or 128
                          (LAMP_ERR_UNSUPPORTED for 256); not together with
                          LAMP_PV_FP8 (LAMP_ERR_UNSUPPORTED) */
} lamp_qk_accum;

/* Counter slots of lamp_stats.counters (uint64 each). */
enum {
  LAMP_CNT_TILES = 0,       /* visited 64x64 tiles (>= 1 visible entry) */
  LAMP_CNT_HIST0 = 1,       /* visited tiles with 0 flagged sub-blocks */
  LAMP_CNT_HIST1 = 2,       /*                    1 flagged sub-block */
  LAMP_CNT_HIST2 = 3,       /*                    2 or more           */
  LAMP_CNT_STRIPS = 4,      /* visited sub-blocks (>= 1 visible entry) */
  LAMP_CNT_STAGE1 = 5,      /* sub-blocks passing the first stage */
  LAMP_CNT_FLAGGED = 6,     /* sub-blocks recomputed in 16 bits */
  LAMP_CNT_SAT = 7,         /* visible logits with |S8| = 448 */
  LAMP_CNT_FIXUPS = 8,      /* logits re-derived exactly (near an 8-bit rounding boundary,
                               where the two candidate codes could differ in a result) */
  LAMP_CNT_STATUS = 9,      /* device-side status (lamp_status), 0 = ok */
  LAMP_CNT_RECOMP_STEPS = 10, /* 128-query x 64-key kernel steps with a flagged
                                 sub-block: their 16-bit products are computed and used */
  LAMP_CNT_SPEC_WASTE = 11, /* steps whose 16-bit products were computed ahead of the
                               decision (the first step of a 128-query tile, or the
                               step before had a flagged sub-block) but not needed;
                               16-bit QK work issued = RECOMP_STEPS + this */
  LAMP_CNT_RECOMP_LATE = 12, /* steps with a flagged sub-block whose 16-bit products were
                                computed only after the decision (the step before had
                                none) */
  LAMP_CNT_GUARD_RESOLVED = 13, /* logits near an 8-bit rounding boundary whose two
                                   candidate codes give the same P8, flag and
                                   saturation results (no exact re-derivation needed) */
  LAMP_CNT_FIXUPS_MAX = 14, /* of LAMP_CNT_FIXUPS: logits re-derived because they could
                               be their row's maximum in the tile */
  LAMP_NUM_COUNTERS = 16
};

typedef struct {
  int32_t batch, seqlen, heads_q, heads_kv, head_dim;
  /* strides in ELEMENTS for the (batch, sequence, head) dimensions of the
   * BSHD tensors; the head_dim dimension is contiguous.  q/out are
   * [B, N, Hq, d], k/v are [B, N, Hkv, d].  Byte strides must be multiples
   * of 16 and the base pointers 16-byte aligned. */
  int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3];
  int32_t window;        /* LAMP_MASK_SLIDING: window length W >= 1 */
  float softmax_scale;   /* sigma; 0 -> 1/sqrt(head_dim) (rounded once from double) */
  int32_t in_dtype;      /* lamp_dtype of q, k, v */
  int32_t out_dtype;     /* lamp_dtype of out */
  int32_t force;         /* lamp_force */
  void* workspace;       /* device scratch, >= lamp_attn_workspace_bytes(); NULL ->
                            the call allocates and frees it stream-ordered */
  size_t workspace_bytes;
  void* stream;          /* cudaStream_t; NULL = legacy default stream */
  void* stage_events[3]; /* optional cudaEvent_t, recorded on `stream` before the
                            pre-pass, between it and the fused kernel, and after
                            the fused kernel (per-stage timing); NULL = none */
  int32_t pv_mode;       /* lamp_pv_mode; 0 = LAMP_PV_FP16 (zero-initialised
                            shapes keep the FP16 path) */
  int32_t qk_accum;      /* lamp_qk_accum; 0 = LAMP_QK_EXACT */
  int32_t kv_prepared;   /* 1: `workspace` already holds this k / v's 8-bit and
                            16-bit copies and key-tile norms, written by
                            lamp_kv_prepare with the same shapes (the forward
                            call then skips that work); 0: the call writes them */
  int32_t q_prepared;    /* 1: `workspace` already holds this q's E4M3 copy and
                            row / chunk norms, written by lamp_qkv_project with
                            the same shapes (bf16 q only; the forward call then
                            neither runs the query part of the pre-pass nor
                            rounds Q in its CTAs); 0: the call derives them */
} lamp_shapes;

typedef struct {
  uint8_t* mask;  /* DEVICE [B][Hq][T][T], T = ceil(seqlen/64), or NULL.
                     Byte (b,h,i,j): bit s (0..3) = sub-block s of tile (i,j)
                     flagged; bit 4+s = it passed stage 1; 0 for tiles that are
                     not visited.  Written in full by every call. */
  uint64_t* counters; /* DEVICE [LAMP_NUM_COUNTERS] or NULL; zeroed, then
                         accumulated, by every call (stream-ordered). */
} lamp_stats;

/*
 * lamp_attn_fwd: out = LampAttention(q, k, v) and lse (natural log,
 * [B, Hq, N] fp32, contiguous; may be NULL).
 *   q, k, v   DEVICE, BSHD with the strides above, dtype shapes->in_dtype.
 *   out       DEVICE, BSHD [B, N, Hq, d] with o_stride, dtype shapes->out_dtype.
 *   mask_kind lamp_mask_kind; causal and sliding use the same N for queries
 *             and keys.
 *   delta     first-stage threshold (>= 0; 0 disables the first stage).
 *   tau       recompute threshold (<= 0 flags every stage-1 sub-block).
 *   stats     may be NULL.
 * Returns LAMP_OK or an error code.  Argument errors are detected before
 * any launch and nothing is enqueued.  A device-side failure (a wait that
 * exceeded its time limit, 2 s by default, LAMP_WAIT_TIMEOUT_NS in the
 * environment overrides it) ends the kernel early: it is written to
 * counters[LAMP_CNT_STATUS] when counters are given and is visible after the
 * stream is synchronised; out / lse / mask are then incomplete.
 * head_dim must be 64, 128 or 256; seqlen >= 1 (any value, not only
 * multiples of 64); heads_q a multiple of heads_kv.
 */
int lamp_attn_fwd(const void* q, const void* k, const void* v, void* out,
                  float* lse, const lamp_shapes* shapes, int mask_kind,
                  float delta, float tau, lamp_stats* stats);

/*
 * lamp_kv_prepare: the key/value half of lamp_attn_fwd's pre-pass on its
 * own: writes into shapes->workspace the E4M3 copy of k, the fp16 copy of v
 * (and, for fp32 inputs, the bf16 copy of k; for LAMP_PV_FP8 the
 * transposed E4M3 copy of v) and the per-key-tile norms that size the
 * exactness guard.  A K/V cache in the attention's own formats: any number
 * of lamp_attn_fwd calls with shapes->kv_prepared = 1, the same workspace,
 * the same k and v (unchanged since) and the same batch, seqlen, heads_kv,
 * head_dim, in_dtype, k / v strides and modes then skip that work and give
 * bit-identical results; their heads_q (any multiple of heads_kv), q, out
 * and strides may differ (the keys' and values' place in the workspace does
 * not depend on them).
 *   k, v      DEVICE, as for lamp_attn_fwd.
 *   shapes    workspace must be given (>= lamp_attn_workspace_bytes() of
 *             these shapes; the later calls check their own size);
 *             kv_prepared and q_prepared are ignored; q_stride /
 *             o_stride are not used.
 * Asynchronous on shapes->stream; LAMP_ERR_INVALID_ARG for a missing
 * workspace, otherwise errors as lamp_attn_fwd.  Not for
 * lamp_attn_fwd_host / lamp_attn_fwd_noalloc (their scratch is their own:
 * they return LAMP_ERR_INVALID_ARG for kv_prepared = 1 or q_prepared = 1).
 */
int lamp_kv_prepare(const void* k, const void* v, const lamp_shapes* shapes);

/*
 * lamp_qkv_project: the QKV projection upstream of the attention, with the
 * attention's key/value cache written by its epilogue.  y = x W^T (BF16
 * operands, FP32 tensor-core accumulation, one rounding to BF16), its
 * columns split into q, k and v; for the key and value columns it also
 * writes what lamp_kv_prepare writes (the E4M3 copy of k, the fp16 copy of
 * v and the key-tile norms) into shapes->workspace, and for the query
 * columns the E4M3 copy of q and its row and chunk norms, so that
 * lamp_attn_fwd on these q, k, v with shapes->kv_prepared = 1,
 * shapes->q_prepared = 1 and the same workspace runs without a pre-pass
 * and without rounding Q in its CTAs (the E4M3 copies of q and k are the
 * projection's outputs rounded once more, as the pre-pass would round
 * them).
 *   x        DEVICE bf16 [batch * seqlen, hidden], row-major (token-major).
 *   w        DEVICE bf16 [(heads_q + 2 heads_kv) * head_dim, hidden],
 *            row-major: the query heads' rows, then the key heads', then
 *            the value heads' (the layout of a linear layer's weight).
 *   hidden   a multiple of 64.
 *   q, k, v  DEVICE bf16 outputs, dense BSHD: q [B, N, Hq, d], k and v
 *            [B, N, Hkv, d].
 *   shapes   batch, seqlen, heads_q, heads_kv, head_dim; in_dtype bf16;
 *            q/k/v strides, if non-zero, must be the dense ones; workspace
 *            given (>= lamp_attn_workspace_bytes()); pv_mode FP16 or FP8
 *            (FP8: the transposed E4M3 copy of v is written too).
 *   stats    optional: counters[LAMP_CNT_STATUS] receives the device status.
 * Asynchronous on shapes->stream.  Errors as lamp_attn_fwd
 * (LAMP_ERR_INVALID_ARG for a missing workspace, an fp32 in_dtype, a hidden
 * size that is not a positive multiple of 64, or non-dense strides).
 */
int lamp_qkv_project(const void* x, const void* w, int hidden, void* q, void* k, void* v,
                     const lamp_shapes* shapes, lamp_stats* stats);

/* Bytes of device workspace lamp_attn_fwd needs for these shapes (E4M3
 * copies of q and k, an fp16 copy of v, bf16 copies of fp32 inputs,
 * per-row norms and, for LAMP_PV_FP8, an E4M3 copy of v).  0 on invalid
 * shapes. */
size_t lamp_attn_workspace_bytes(const lamp_shapes* shapes);

/*
 * lamp_attn_fwd_noalloc: the same forward pass as lamp_attn_fwd, for callers
 * that must not allocate device memory during the call -- e.g. a plug-in of
 * a host framework that owns all device memory through its own pooling
 * allocator (raw cudaMalloc/cudaFree would bypass it, and cudaFree
 * synchronises the device), or a latency-bound serving loop that must stay
 * free of implicit synchronisation.  The paper has no counterpart: this is
 * a memory-management variant only.
 *
 * Arguments, layouts and results are those of lamp_attn_fwd; the caller
 * still passes inputs, outputs and (optionally) stats.  shapes->workspace
 * and workspace_bytes are ignored: the scratch is a file-scope device array
 * of LAMP_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds
 * until process exit.  Shapes whose lamp_attn_workspace_bytes() exceeds it
 * are rejected with LAMP_ERR_TOO_LARGE before anything is enqueued.  No
 * cudaMalloc, cudaFree or other allocating call is made.
 *
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress), so a cudaDeviceReset between calls is harmless;
 * make the first call on each device before any stream capture (that
 * lookup may load the module).  Status codes as lamp_attn_fwd
 * (LAMP_ERR_UNSUPPORTED for a head_dim other than 64, 128, 256).  All calls share the array and it keeps the
 * last call's contents (each call clears what must start at zero); calls
 * whose work overlaps on the GPU race on it and must be serialised.
 */
int lamp_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out,
                          float* lse, const lamp_shapes* shapes, int mask_kind,
                          float delta, float tau, lamp_stats* stats);

/*
 * lamp_attn_fwd_host: lamp_attn_fwd on HOST q, k, v, out and lse, for
 * callers whose tensors live in host memory (page-locked memory lets the
 * copies run asynchronously and at full link speed).  The paper has no
 * counterpart: this is a data-movement variant only, and the results are
 * bit-identical to lamp_attn_fwd on the same inputs.
 *
 * The batch -- and, while batch * groups < 16, the kv-head groups -- is cut
 * into chunks; per chunk the inputs are copied to the device, the forward
 * pass runs and the outputs are copied back, on two internal copy streams,
 * so the copies of one chunk overlap the computation of its neighbours.
 * Each chunk has its own device slot while the slots fit 1 GiB (else at
 * least two slots are reused in turn; the environment variable
 * LAMP_HOST_MAX_SLOTS, >= 2, lowers the count).  Chunks compute in turn on
 * shapes->stream and three internal streams (joined back into
 * shapes->stream before the call returns), so one chunk's kernels start on
 * the SMs the previous chunks' tails leave idle.
 *   q, k, v, out  HOST, BSHD with the strides of `shapes` (elements); the
 *                 head and head_dim dimensions must be dense
 *                 (stride[2] == head_dim).
 *   lse           HOST [B, Hq, N] fp32 or NULL.
 *   stats         DEVICE buffers as for lamp_attn_fwd (mask written per
 *                 chunk; counters summed over the chunks), or NULL.
 *   dev_buffer    DEVICE scratch of lamp_attn_host_buffer_bytes() bytes,
 *                 256-byte aligned, or NULL (allocated and freed
 *                 stream-ordered on shapes->stream); shapes->workspace is
 *                 not used.
 * Synchronous: returns after out and lse hold the results (the status of
 * the device side is in counters[LAMP_CNT_STATUS] when counters are given).
 * The internal streams and events are created once per device (anew after
 * the device's context changes, e.g. a cudaDeviceReset); calls on one
 * device from several host threads run one after the other.
 * Errors as lamp_attn_fwd; LAMP_ERR_WORKSPACE if dev_buffer is too small or
 * misaligned.
 */
int lamp_attn_fwd_host(const void* q, const void* k, const void* v, void* out,
                       float* lse, const lamp_shapes* shapes, int mask_kind,
                       float delta, float tau, lamp_stats* stats,
                       void* dev_buffer, size_t dev_buffer_bytes);

/* Device scratch lamp_attn_fwd_host needs for these shapes; 0 on invalid
 * shapes. */
size_t lamp_attn_host_buffer_bytes(const lamp_shapes* shapes);

/*
 * lamp_attn_tau_sweep: the histograms of 16-bit sub-blocks per tile (the
 * 0 / 1 / 2+ buckets of Tables 1-6) for up to 8 values of tau at once,
 * from one pass -- the tau sweeps of Figures 1-3 and 8.  The running max,
 * the 8-bit exponentials and the first stage do not depend on tau, and a
 * sub-block is flagged at tau iff one of its stage-1 entries has
 * half-ulp8(S8) >= tau, so the pass records per sub-block the largest such
 * half-ulp; no 16-bit recompute, no P.V and no output are computed.  The
 * histograms equal the counters LAMP_CNT_TILES / HIST0 / HIST1 / HIST2 of
 * lamp_attn_fwd at each tau (force off).
 *   q, k      DEVICE, as for lamp_attn_fwd (shapes: v_stride, o_stride and
 *             out_dtype are not used).
 *   taus      HOST float[ntau], 0 <= ntau <= 8.
 *   records   DEVICE uint32 [B][Hq][T][T], T = ceil(seqlen/64), written in
 *             full: bits 0-3 visible sub-blocks, 4-7 stage-1 sub-blocks,
 *             8+4s..11+4s the code of sub-block s = log2(largest stage-1
 *             half-ulp8) + 11 (1..15), 0 if none; 0 for tiles not visited.
 *   hist      DEVICE uint64 [ntau][4]: visited tiles, tiles with 0, 1, 2+
 *             flagged sub-blocks at taus[i] (zeroed, then written).
 *   stats     optional; counters as for lamp_attn_fwd except the flag-based
 *             ones (HIST0..2, FLAGGED, RECOMP_STEPS, SPEC_WASTE, RECOMP_LATE
 *             stay 0);
 *             stats->mask is not written.
 * shapes->pv_mode is not used (the pass computes no P.V); shapes->qk_accum
 * must be LAMP_QK_EXACT (LAMP_ERR_UNSUPPORTED otherwise).
 * Asynchronous on shapes->stream; errors as lamp_attn_fwd.
 */
int lamp_attn_tau_sweep(const void* q, const void* k, const lamp_shapes* shapes,
                        int mask_kind, float delta, const float* taus, int ntau,
                        uint32_t* records, uint64_t* hist, lamp_stats* stats);

/* Static, human-readable text for a lamp_status value. */
const char* lamp_strerror(int status);

/* Library version string, e.g. "lamp-attn 0.2 sm_103a". */
const char* lamp_version(void);

/* The 8-bit exponential the kernels use, as a table (host memory, 256
 * bytes): out[c] = E4M3 code of fl8(exp(x)) for the E4M3 code c of x (round
 * to nearest even, saturating; 0 for the NaN codes).  Abstract of the paper:
 * exponentials evaluated in 8-bit formats.  For diagnostics and tests. */
void lamp_exp8_table(uint8_t out[256]);

/*
 * lamp_selftest: device checks of the tensor-core building blocks used by
 * lamp_attn_fwd (no counterpart in the paper), run on caller data with the
 * same shared-memory layouts and instruction sequences:
 *   which 0: out[128 x 64]    = A . B^T, A [128 x d], B [64 x d] E4M3 codes (uint8)
 *   which 1: out[128 x 64]    = A . B^T, A [128 x d], B [64 x d] BF16
 *   which 2: out[128 x d]      = P . V, P [128 x 64], V [64 x d] FP16 (V MN-major)
 *   which 3: out[i] = the 8-bit logit the exact re-derivation produces for
 *            the dot product a[i] * 2^-18 (a: int64[d]) and the scale b[0]
 *            (b: double[1]): E4M3 rounding of the float64 product, as a
 *            float; d = count, 1..65536.
 *   which 4: out[i] = fl8(exp(x)) as the fused kernel computes it, for the
 *            E4M3 code a[i] of x <= 0 (a: uint8[d]; b: any non-NULL device
 *            pointer, unused); d = count, 1..65536.
 *   which 5: out[i] = x8 = fl8(S8 - m) as the fused kernel's P8 path
 *            computes it (f16 difference, then E4M3 rounding), for the E4M3
 *            codes a[i] of S8 and b[i] of m (a, b: uint8[d]); d = count,
 *            1..65536.
 *   which 6: as 5, through the fp32 difference the detector uses.
 * a, b: DEVICE, row-major as listed; out: DEVICE float32, row-major.
 * Returns LAMP_OK or an error code after synchronising `stream`.
 */
int lamp_selftest(int which, const void* a, const void* b, float* out, int d,
                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LAMP_ATTN_H */

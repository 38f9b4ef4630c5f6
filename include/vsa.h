/*
 * vsa.h - C ABI of libvsa.so: VSA coarse-to-fine video sparse attention on
 * one GB300 (sm_103a), forward and backward.
 *
 * The operation ("VSA: Faster Video Diffusion with Trainable Sparse
 * Attention", §2 Methods and App. B "Pseudocode of VSA"):
 *   1. tile   : a (T,H,W) video latent is cut into (4,4,4) cubes; each cube's
 *               64 tokens form one tile (§2 "VSA design").
 *   2. pool   : Q_c, K_c, V_c = per-cube means of Q, K, V (§2 "Coarse stage").
 *   3. coarse : A_c = softmax(Q_c K_c^T * scale), O_c = A_c V_c; each query
 *               cube keeps its top-K key cubes (default K = 32), turned into an
 *               index list in the same kernel (paper notes, 损失函数/训练策略:
 *               softmax, top-K and mask-to-index fused).  The dynamic-compute
 *               variant keeps a variable count per query cube ("Improving Video
 *               Sparse Attention with Fine-grained Router and Sparse Rebasing",
 *               abstract): the smallest top-ranked set with coarse mass >= mass,
 *               clamped to [kmin, kmax].
 *   4. fine   : token-level softmax(Q K^T * scale) V over the 64x64 tiles of the
 *               selected key cubes only (§2 "Fine stage"; App. B masked fine
 *               attention).
 *   5. combine: O = repeat(O_c over its cube) (.) G_c + O_f (.) G_f, then untile
 *               (paper notes 关键设计 3 gating; App. B).
 * Backward returns dQ, dK, dV, dG_c, dG_f; the selection is held fixed.
 *
 * Conventions for every entry point:
 *  - Tensors are contiguous [batch, heads, N, head_dim] with N = T*H*W, either
 *    in raster order (token (t,h,w) at row (t*H + h)*W + w) or in cube order
 *    (row c*64 + o, c = ((t/4)*(H/4) + h/4)*(W/4) + w/4,
 *    o = (t%4)*16 + (h%4)*4 + w%4), as cfg->layout says.  Q, K, V, G_c, G_f,
 *    dO and O are bf16; the pooled/coarse tensors and log-sum-exps are fp32;
 *    the saved fine output O_f is fp16 (cube order).  The gradients dQ, dK,
 *    dV, dG_c, dG_f are fp32 or bf16 as cfg->grad_dtype says (bf16: the fp32
 *    result rounded to nearest even once, at the store; everything before it
 *    is the same).  The pooled and coarse gradients stay fp32.
 *  - The tensor-core operands Q, K, V are staged as fp16 copies in cube order
 *    ("staged" below): bf16 -> fp16 is exact for magnitudes in
 *    [6.1e-5, 65504], and the fp16 significand keeps the rounding of the
 *    softmax probabilities 8x smaller than bf16 would.  Q, K or V values whose
 *    magnitude exceeds 65504 (or that are not finite) are reported as
 *    VSA_ERR_DEVICE_CHECK, not computed.
 *  - The backward's operand dO_f = dO (.) G_f is staged in fp16 times a power
 *    of two per (batch, head) slice (the "gradient scale"), chosen so that the
 *    slice's largest |dO (.) G_f| lies in [4, 8); the fine backward divides its
 *    results by it (exact).  Upstream gradients of any magnitude down to the
 *    fp32 normal range (1e-5 .. 1e-8 is common in bf16 training without loss
 *    scaling) thus keep fp16's full precision; only non-finite values are
 *    reported (VSA_ERR_DEVICE_CHECK).
 *  - All pointers named without a "host" prefix are device pointers owned by
 *    the caller, 16-byte aligned.  The library never allocates, frees or
 *    synchronises (except vsa_check_device_status).  Scratch comes from the
 *    caller's `ws` buffer of vsa_workspace_bytes() bytes; data the backward
 *    pass needs comes from the caller's `saved` buffer of vsa_saved_bytes().
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.  vsa_forward and vsa_backward also fork
 *    independent kernels to a second stream the library creates once per
 *    device, and join back to `stream` with two events of their own per call
 *    (this works inside stream capture; concurrent calls from several host
 *    threads are serialised while they enqueue).
 *  - Arguments are checked on the host before anything is launched; an error
 *    return leaves every output untouched.  VSA_ERR_CUDA reports a launch
 *    failure.  Faults found on the device (a bounded wait that expired, an
 *    index out of range) are recorded in a status word inside `ws` and read
 *    back by vsa_check_device_status().
 *  - Gradients are written (not accumulated).
 */
#ifndef VSA_H_
#define VSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VSA_OK = 0,
  VSA_ERR_INVALID_ARG = 1,  /* null pointer, bad count, K out of range */
  VSA_ERR_SHAPE = 2,        /* T, H or W not a multiple of 4, or too large */
  VSA_ERR_UNSUPPORTED = 3,  /* head_dim not 64 or 128 */
  VSA_ERR_ALIGNMENT = 4,    /* a pointer is not 16-byte aligned */
  VSA_ERR_CUDA = 5,         /* a CUDA call or launch failed */
  VSA_ERR_TIMEOUT = 6,      /* a device-side bounded wait expired */
  VSA_ERR_DEVICE_CHECK = 7  /* a device-side range check failed (index list, fp16 range) */
} vsa_status_t;

enum { VSA_SELECT_TOPK = 0, VSA_SELECT_MASS = 1 };
enum { VSA_LAYOUT_RASTER = 0, VSA_LAYOUT_CUBE = 1 };
enum { VSA_GRAD_FP32 = 0, VSA_GRAD_BF16 = 1 };

/* Largest supported sizes. */
#define VSA_MAX_CUBES 8192   /* cubes per (batch, head) */
#define VSA_MAX_LIST 256     /* index-list capacity per query cube */
#define VSA_NOALLOC_SCRATCH_BYTES (8u << 20)  /* fixed scratch of vsa_fine_fwd_noalloc */

typedef struct {
  int32_t batch, heads;     /* B, number of heads */
  int32_t T, H, W;          /* latent size, each a positive multiple of 4 */
  int32_t head_dim;         /* D: 64 or 128 */
  int32_t select_mode;      /* VSA_SELECT_TOPK or VSA_SELECT_MASS */
  int32_t topk;             /* TOPK: cubes kept per query cube, 1..min(Nc, VSA_MAX_LIST) */
  float mass;               /* MASS: coarse-probability threshold in (0, 1] */
  int32_t kmin, kmax;       /* MASS: count clamp, 1 <= kmin <= kmax <= VSA_MAX_LIST */
  float scale;              /* softmax scale for both stages; <= 0 means 1/sqrt(D) */
  int32_t layout;           /* VSA_LAYOUT_RASTER or VSA_LAYOUT_CUBE (caller tensors) */
  int32_t grad_dtype;       /* VSA_GRAD_FP32 or VSA_GRAD_BF16: dq, dk, dv, dgc, dgf */
} vsa_config_t;

/* Byte offsets of the pieces of the `saved` buffer written by vsa_forward.
 * Each piece starts on a 256-byte boundary.  The offsets are the same for
 * every use; the pieces only training needs come last (qc .. lse_f, then
 * q16, k16, v16, then o_f), so a smaller `total` (vsa_saved_bytes_for with
 * with_backward = 0) simply leaves off what lies at or beyond it. */
typedef struct {
  size_t q16, k16, v16;          /* fp16 [B,heads,N,D] cube order: staged Q, K, V */
  size_t qc, kc, vc, oc;         /* fp32 [B,heads,Nc,D]: pooled Q/K/V, coarse output */
  size_t lse_c;                  /* fp32 [B,heads,Nc]: coarse log-sum-exp (natural log) */
  size_t idx;                    /* int32 [B,heads,Nc,list_cap]: ascending key-cube ids, -1 padded */
  size_t cnt;                    /* int32 [B,heads,Nc]: entries used per list */
  size_t o_f;                    /* fp16 [B,heads,N,D] cube order: fine output */
  size_t lse_f;                  /* fp32 [B,heads,N] cube order: fine log-sum-exp */
  size_t total;                  /* bytes of the buffer for this use */
  int32_t list_cap;              /* topk (TOPK) or kmax (MASS) */
} vsa_saved_layout_t;

/* Checks a configuration.  VSA_OK or the reason it is rejected. */
vsa_status_t vsa_validate(const vsa_config_t* cfg);

/* Short English text for a status code (static storage). */
const char* vsa_status_string(vsa_status_t s);

/* Bytes of the caller-owned `saved` buffer; fills *layout if not NULL.
 * Returns 0 for an invalid configuration.  This is the training size (every
 * piece), which every entry point that takes `saved` accepts. */
size_t vsa_saved_bytes(const vsa_config_t* cfg, vsa_saved_layout_t* layout);

/* The same for one use: with_backward != 0 gives vsa_saved_bytes(); 0 gives the
 * smaller buffer an inference vsa_forward (with_backward = 0) needs: without
 * o_f, and without the staged q16, k16, v16 unless it stages them (raster
 * layout, head_dim 128).  The offsets are those of vsa_saved_bytes();
 * vsa_backward and vsa_forward_fp8 need the training size. */
size_t vsa_saved_bytes_for(const vsa_config_t* cfg, int with_backward,
                           vsa_saved_layout_t* layout);

/* Bytes of the caller-owned scratch buffer `ws` for the forward pass
 * (with_backward = 0) or for forward and backward (with_backward = 1).
 * Returns 0 for an invalid configuration. */
size_t vsa_workspace_bytes(const vsa_config_t* cfg, int with_backward);

/* Zeroes the device status word at the start of `ws` (asynchronously).  Call
 * once after allocating `ws`. */
vsa_status_t vsa_reset_device_status(void* ws, void* stream);

/* Synchronises `stream` and returns VSA_ERR_TIMEOUT / VSA_ERR_DEVICE_CHECK if
 * a kernel recorded a device-side failure in `ws` since the last reset. */
vsa_status_t vsa_check_device_status(void* ws, void* stream);

/* Diagnostic (no counterpart in the method): runs one CTA that waits, with
 * the same bounded mbarrier wait every pipelined kernel of this library uses,
 * on a barrier nothing ever arrives at.  After `limit_us` microseconds
 * (1..10,000,000) the wait gives up, records a time-out in the status word of
 * `ws` and the kernel returns, leaving the context usable; the next
 * vsa_check_device_status() then returns VSA_ERR_TIMEOUT.  ws: as for every
 * other entry point (only its status word is touched).  Returns
 * VSA_ERR_INVALID_ARG for a NULL ws or a limit outside the range. */
vsa_status_t vsa_probe_wait_timeout(void* ws, uint32_t limit_us, void* stream);

/* Tile / untile (App. B: tiling and untiling rearrange tokens between
 * sequence and cube order).  inverse = 0: raster -> cube order; 1: cube ->
 * raster.  in, out: bf16 [B,heads,N,D], distinct buffers.  cfg->layout is
 * ignored. */
vsa_status_t vsa_permute(const vsa_config_t* cfg, const void* in, void* out, int inverse,
                         void* stream);

/* Staging of one tensor-core operand: x (bf16, cfg->layout order) ->
 * x16 (fp16, cube order; may be NULL) and its cube means pooled (fp32
 * [B,heads,Nc,D]; may be NULL, not both).  ws receives the range flag. */
vsa_status_t vsa_stage(const vsa_config_t* cfg, const void* x, void* x16, float* pooled,
                       void* ws, void* stream);

/* Coarse stage (§2 "Coarse stage"): per-cube means, dense attention on the
 * pooled sequence, selection and index lists, in one pass.
 * q, k, v : bf16 [B,heads,N,D] in cfg->layout order; or all three NULL, when
 *           qc, kc, vc already hold the cube means (e.g. from vsa_stage) and
 *           are read instead of written (one NULL among three non-NULL is
 *           VSA_ERR_INVALID_ARG).
 * qc, kc, vc, oc : fp32 [B,heads,Nc,D] outputs (pooled inputs, O_c).
 * lse_c   : fp32 [B,heads,Nc] output, natural-log log-sum-exp of the logits.
 * idx     : int32 [B,heads,Nc,list_cap] output, ascending key-cube ids, -1 padded.
 * cnt     : int32 [B,heads,Nc] output. */
vsa_status_t vsa_coarse_select(const vsa_config_t* cfg, const void* q, const void* k,
                               const void* v, float* qc, float* kc, float* vc, float* oc,
                               float* lse_c, int32_t* idx, int32_t* cnt, void* ws,
                               void* stream);

/* Fine stage and combine (§2 "Fine stage"; App. B): block-sparse attention
 * over the listed key cubes, fused with O = repeat(O_c) G_c + O_f G_f.
 * q16, k16, v16 : staged fp16 CUBE order (vsa_stage).  idx, cnt: lists as written by vsa_coarse_select
 * (any ascending lists with entries in [0, Nc) work, e.g. injected ones).
 * gc, gf  : bf16 gates in cfg->layout order.  oc: fp32 [B,heads,Nc,D].
 * o       : bf16 output in cfg->layout order.
 * o_f     : fp16 CUBE order fine output (rounded from fp32; it feeds only the
 *           combine backward), or NULL (not needed for inference).
 * lse_f   : fp32 [B,heads,N] CUBE order, or NULL. */
vsa_status_t vsa_fine_fwd(const vsa_config_t* cfg, const void* q16, const void* k16,
                          const void* v16, const int32_t* idx, const int32_t* cnt, const void* gc,
                          const void* gf, const float* oc, void* o, void* o_f, float* lse_f,
                          void* ws, void* stream);

/* Fine stage and combine reading the caller's bf16 tensors in place (no staged
 * copies; App. B: tiling "can be moved outside individual attention layers" --
 * here it happens inside the tile copies): in raster layout each 64-token tile
 * is one 5-D copy of a (4,4,4) cube of the [B*heads, T, H, W, D] view, landing
 * in the in-cube token order.  Operands, P and the MMAs are bf16 (fp32
 * accumulation), for inference: no O_f.
 * q, k, v, gc, gf: bf16 [B,heads,N,D] in cfg->layout order; idx, cnt, oc, o,
 * lse_f (may be NULL), ws: as for vsa_fine_fwd.  Q, K, V need no fp16 range. */
vsa_status_t vsa_fine_fwd_bf16(const vsa_config_t* cfg, const void* q, const void* k,
                               const void* v, const int32_t* idx, const int32_t* cnt,
                               const void* gc, const void* gf, const float* oc, void* o,
                               float* lse_f, void* ws, void* stream);

/* vsa_fine_fwd for callers that cannot provide a scratch buffer.  The pages
 * have no counterpart: this is a calling convention, not a step of the method.
 * A caller with no device allocator of its own (for example a plugin run by a
 * host engine that owns all device memory and hands the plugin only its
 * inputs and outputs) cannot supply the `ws` buffer of vsa_fine_fwd; this
 * entry point takes no `ws` and allocates nothing.  Its scratch (status word,
 * schedule counter, query-pair work items and union lists) lives in a fixed array of
 * VSA_NOALLOC_SCRATCH_BYTES inside the library, held on every GPU that loads
 * the library until the process exits.
 *  - Arguments and results are those of vsa_fine_fwd, without `ws`.
 *  - status: optional device pointer to a uint32 (4-byte aligned, NULL to
 *    skip) that receives this call's device status bits (1: a bounded wait
 *    expired, 2: a bad index list entry, 4: a value outside the fp16 range).
 *  - Returns VSA_ERR_SHAPE when the configuration needs more scratch than
 *    VSA_NOALLOC_SCRATCH_BYTES (B*heads*ceil(Nc/2) query pairs, each with 20
 *    bytes + 8*list_cap bytes): checked after vsa_validate() has accepted the
 *    configuration (an invalid one returns vsa_validate's code), before the
 *    pointer checks and before any launch.
 *  - The query pairs are handed out in their natural order (slice by slice,
 *    neighbouring cubes together), not in the largest-first order vsa_fine_fwd
 *    uses for layers whose K and V fit in L2 (that order needs more scratch);
 *    results are bitwise the same, only the load balance differs.
 *  - The first call on each device (with that device current) looks up the
 *    array's device address; make that first call before any stream capture.
 *  - Every call shares the one array: calls that overlap on the GPU (other
 *    streams, other threads) race and must be serialised by the caller. */
vsa_status_t vsa_fine_fwd_noalloc(const vsa_config_t* cfg, const void* q16, const void* k16,
                                  const void* v16, const int32_t* idx, const int32_t* cnt,
                                  const void* gc, const void* gf, const float* oc, void* o,
                                  void* o_f, float* lse_f, uint32_t* status, void* stream);

/* ---------------------------------------------------------------------------
 * e4m3 (fp8) variant of the fine stage, head_dim 128, inference only.
 *
 * The pages give the fine stage no precision ("VSA: Faster Video Diffusion
 * with Trainable Sparse Attention", §2 "Fine stage"; the successor "Improving
 * Video Sparse Attention with Fine-grained Router and Sparse Rebasing",
 * abstract, halves VSA's attention compute): this variant runs the same
 * block-sparse attention and combine with Q, K, V and P in e4m3 and fp32
 * accumulation, reading half the bytes per tile.  Its accuracy is that of e4m3
 * (3 significand bits): results are not bit- or tolerance-equal to the fp16
 * path's; the index lists, which the fp32 coarse stage decides, are identical.
 * D = 64 returns VSA_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------ */

/* Staging: bf16 q, k, v (cfg->layout order) -> e4m3 copies, each (batch, head)
 * slice multiplied by a power of two 2^e that puts its largest |x| in
 * [128, 256) (e4m3's range ends at 448).
 * q8, k8  : [B*heads*N, 128] bytes, CUBE order (row c*64 + o of each slice).
 * v8t     : [B*heads*Nc, 128, 64] bytes: each cube's V transposed (row d holds
 *           the cube's 64 values of channel d).
 * scales  : fp32 [B,heads,3] output, 2^-e of Q, K, V (the factors that undo
 *           the scaling).
 * qc,kc,vc: fp32 [B,heads,Nc,D] cube means (as vsa_coarse_select writes them),
 *           each may be NULL.
 * Non-finite inputs are reported as VSA_ERR_DEVICE_CHECK; ws also holds the
 * slice maxima. */
vsa_status_t vsa_stage_fp8(const vsa_config_t* cfg, const void* q, const void* k,
                           const void* v, void* q8, void* k8, void* v8t, float* scales,
                           float* qc, float* kc, float* vc, void* ws, void* stream);

/* Fine stage and combine on the e4m3 copies (as vsa_fine_fwd, without O_f):
 * idx, cnt, gc, gf, oc, o, ws as for vsa_fine_fwd; lse_f: fp32 [B,heads,N]
 * CUBE order, or NULL. */
vsa_status_t vsa_fine_fwd_fp8(const vsa_config_t* cfg, const void* q8, const void* k8,
                              const void* v8t, const float* scales, const int32_t* idx,
                              const int32_t* cnt, const void* gc, const void* gf, const float* oc,
                              void* o, float* lse_f, void* ws, void* stream);

/* Whole forward with the e4m3 fine stage (inference): e4m3 staging with the
 * cube means, the fp32 coarse stage (identical lists), the e4m3 fine stage and
 * combine.  saved: vsa_saved_bytes() bytes; the e4m3 copies go to the q16,
 * k16, v16 offsets of its layout, their factors to the o_f offset, the coarse
 * results and lse_f where vsa_forward puts them.  The result cannot feed
 * vsa_backward. */
vsa_status_t vsa_forward_fp8(const vsa_config_t* cfg, const void* q, const void* k,
                             const void* v, const void* gc, const void* gf, void* o, void* saved,
                             void* ws, void* stream);

/* Backward of the combine: the gradient of O = repeat(O_c) G_c + O_f G_f
 * (paper notes 关键设计 3, the gating formula; App. B "Pseudocode of VSA": the
 * coarse output is repeated across its cube; the abstract: the whole operator
 * is one differentiable kernel trained end to end).
 * d_o, gc, gf: bf16 in cfg->layout order; o_f: fp16 CUBE order; oc: fp32.
 * dgc, dgf   : outputs in cfg->layout order (dO (.) repeat(O_c), dO (.) O_f),
 *              of cfg->grad_dtype.
 * dof16      : fp16 CUBE order output, dO (.) G_f times gscale[slice].
 * doc        : fp32 [B,heads,Nc,D] output, per-cube sum of dO (.) G_c.
 * delta      : fp32 [B,heads,N] CUBE order output, rowsum(dof16 (.) o_f)
 *              (so it carries the same factor).
 * gscale     : fp32 [B,heads] output, the power-of-two gradient scale of each
 *              slice (see the conventions above); pass it to vsa_fine_bwd.
 * ws receives the range flag (non-finite dO (.) G_f) and holds the slice
 * maxima. */
vsa_status_t vsa_combine_bwd(const vsa_config_t* cfg, const void* d_o, const void* gc,
                             const void* gf, const void* o_f, const float* oc, void* dgc,
                             void* dgf, void* dof16, float* doc, float* delta, float* gscale,
                             void* ws, void* stream);

/* Backward of the coarse attention on the pooled sequence, selection held
 * fixed (§2 "Coarse stage": dense attention over the cube means; abstract:
 * trained end to end; the top-K choice is piecewise constant and passes no
 * gradient).  Outputs dqc, dkc, dvc: fp32 [B,heads,Nc,D] (gradients w.r.t. the
 * pooled means). */
vsa_status_t vsa_coarse_bwd(const vsa_config_t* cfg, const float* qc, const float* kc,
                            const float* vc, const float* oc, const float* lse_c,
                            const float* doc, float* dqc, float* dkc, float* dvc, void* ws,
                            void* stream);

/* Backward of the fine stage plus the pooling (§2 "Fine stage" and App. B:
 * the masked fine attention over the selected 64x64 blocks, differentiated with
 * the selection held fixed; §2 "Coarse stage": each token's share of its cube
 * mean is 1/64): writes
 *   dq = dQ_fine / gscale + repeat(dqc)/64, dk = dK_fine / gscale + repeat(dkc)/64,
 *   dv = dV_fine / gscale + repeat(dvc)/64
 * in cfg->layout order, of cfg->grad_dtype.  q16, k16, v16, dof16: staged fp16 CUBE
 * order; lse_f, delta: fp32 CUBE order; gscale: fp32 [B,heads], the factor
 * dof16 and delta carry (vsa_combine_bwd's output), or NULL for 1;
 * dqc/dkc/dvc may be NULL (no pooled contribution). */
vsa_status_t vsa_fine_bwd(const vsa_config_t* cfg, const void* q16, const void* k16,
                          const void* v16, const int32_t* idx, const int32_t* cnt,
                          const float* lse_f, const void* dof16, const float* delta,
                          const float* gscale, const float* dqc, const float* dkc,
                          const float* dvc, void* dq, void* dk, void* dv, void* ws,
                          void* stream);

/* Whole forward (§2 Methods, the coarse stage feeding the fine stage; App. B
 * "Pseudocode of VSA"; paper notes 关键设计 1-3): tile, coarse stage, fine
 * stage + combine, untile.
 * q, k, v, gc, gf: bf16 in cfg->layout order; o: bf16 output, same order.
 * saved: vsa_saved_bytes() bytes, or vsa_saved_bytes_for(cfg, 0, ...) bytes for
 *   with_backward == 0.
 * with_backward != 0: stages fp16 copies of Q, K, V with the cube means, and
 *   fills everything vsa_backward needs (O_f included).
 * with_backward == 0 (inference): no O_f.  In cube layout, or at head_dim 64,
 *   computes only the cube means, the coarse results and lse_f into `saved` and
 *   runs the fine stage on q, k, v in place (vsa_fine_fwd_bf16): no staged
 *   copies, no fp16 range limit.  Raster tensors of head_dim 128 are staged as
 *   for training (a raster cube of 128 channels reads slower in place than its
 *   staged copy).  Either way the result cannot feed vsa_backward. */
vsa_status_t vsa_forward(const vsa_config_t* cfg, const void* q, const void* k, const void* v,
                         const void* gc, const void* gf, void* o, void* saved,
                         int with_backward, void* ws, void* stream);

/* Whole backward (abstract: VSA is a single differentiable kernel trained end
 * to end; the gradients of every step of vsa_forward with the selection held
 * fixed): combine backward, coarse backward, fine backward + unpooling, from
 * the upstream gradient d_o (bf16, cfg->layout order).
 * gc, gf: the forward's gates; saved: as filled by vsa_forward with
 * with_backward = 1 (it holds the staged Q, K, V).  Outputs dq, dk, dv, dgc,
 * dgf of cfg->grad_dtype in cfg->layout order. */
vsa_status_t vsa_backward(const vsa_config_t* cfg, const void* gc, const void* gf,
                          const void* saved, const void* d_o, void* dq, void* dk, void* dv,
                          void* dgc, void* dgf, void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VSA_H_ */

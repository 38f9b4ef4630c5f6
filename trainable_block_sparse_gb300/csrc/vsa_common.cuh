// Shared definitions for the VSA kernels: problem geometry, the cube <-> raster
// index maps, the internal launch interface between the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/vsa.h"

namespace vsa {

constexpr int kTile = 64;  // tokens per (4,4,4) cube

// Geometry of one call, derived from vsa_config_t on the host.
struct Geom {
  int B, heads, T, H, W, D;
  int BH;        // batch * heads
  int N;         // tokens per (batch, head)
  int Nc;        // cubes per (batch, head)
  int ct, ch, cw;  // cubes along T, H, W
  int cap;       // index-list capacity per query cube
  int raster;    // 1: caller tensors in raster order, 0: cube order
  int grad_bf16; // 1: dQ, dK, dV, dG_c, dG_f are written as bf16, 0: fp32
  float scale;   // softmax scale (both stages)
};

// Checks a configuration and derives its geometry (api.cu): VSA_OK, or the
// reason the configuration is rejected (then *g is not written).
vsa_status_t make_geom(const vsa_config_t* cfg, Geom* g);

// Raster row of token o (0..63) of cube c: cube (4,4,4) with in-cube order
// o = (t%4)*16 + (h%4)*4 + w%4, cubes ordered (t/4, h/4, w/4) row-major.
__host__ __device__ __forceinline__ int raster_row(const Geom& g, int c, int o) {
  const int cw_ = c % g.cw;
  const int tmp = c / g.cw;
  const int ch_ = tmp % g.ch;
  const int ct_ = tmp / g.ch;
  const int t = ct_ * 4 + (o >> 4);
  const int h = ch_ * 4 + ((o >> 2) & 3);
  const int w = cw_ * 4 + (o & 3);
  return (t * g.H + h) * g.W + w;
}

// Row (within one (batch, head) slice) where a caller-layout tensor holds
// token o of cube c.
__host__ __device__ __forceinline__ int caller_row(const Geom& g, int c, int o) {
  return g.raster ? raster_row(g, c, o) : c * kTile + o;
}

// Union-list entry of a query-cube pair: key cube id in the low 16 bits, bit
// 16 set when the first query cube selected it, bit 17 for the second.
constexpr uint32_t kSelA = 1u << 16;
constexpr uint32_t kSelB = 1u << 17;

// A unit of block-sparse work: two query cubes (or two key cubes) of one
// (batch, head) and the union of their lists.
struct PairItem {
  int bh;
  int a;       // first cube
  int b;       // second cube, or -1
  int count;   // entries in the union list
  int off;     // offset of the union list in its list array
};

// Pieces of the workspace, carved by the host (api.cu).
// Schedule counters of the persistent fine kernels (Workspace::counter):
// each launch takes item positions from its own counter, zeroed just before.
enum { kCounterFwd = 0, kCounterBwdQ = 1, kCounterBwdK = 2 };

struct Workspace {
  uint32_t* status;       // device status word
  int* counter;           // scratch counters (16)
  PairItem* qpairs;       // query-cube pairs
  uint32_t* qlist;        // [n_qpairs][2*cap] union lists
  int n_qpairs;
  float* clogit;          // fp32 [BH, Nc, Nc] coarse logits (forward)
  // coarse GEMM operands: Q_c and K_c as tf32 hi/lo pairs (x = hi + lo, for
  // the logits), the rest rounded to tf32 alone; the "t" arrays are
  // [BH, D, ldc], A_c / dL / P^T / dL^T [BH, Nc, ldc] with ldc = Nc rounded up
  // to 4, the others [BH, Nc, D]
  float *qh, *ql, *kh, *kl;        // Q_c, K_c
  float* vth;                      // V_c^T
  float* ach;                      // A_c (fwd), dL (bwd)
  float *vh, *doh;                 // V_c, dO_c (bwd)
  float *kth, *qth, *doth;         // K_c^T, Q_c^T, dO_c^T (bwd)
  float *pth, *dlth;               // P^T, dL^T (bwd)
  // backward: per-slice scale of dO (.) G_f (see launch_combine_bwd)
  uint32_t* gamax;        // [3*BH] slice maxima as float bits: |dO (.) G_f| (the
                          // first BH), or |Q|, |K|, |V| for the e4m3 staging
  float* gscale;          // [BH] power-of-two factor applied to dO_f and delta
  void* dof;              // fp16 cube order, dO (.) G_f times gscale
  float* delta;           // fp32 [BH, N]
  float* doc;             // fp32 [BH, Nc, D]
  float* dqc; float* dkc; float* dvc;
  float* cdelta;          // fp32 [BH, Nc]      rowsum(dO_c (.) O_c)
  uint32_t* tmask;        // [BH, Nc, ceil(Nc/32)] selection bit matrix
  int* toff;              // [BH, Nc + 1] offsets of transposed lists
  int* tlist;             // [BH, Nc * cap] transposed lists (query cubes per key cube)
  PairItem* kpairs;       // key-cube pairs
  uint32_t* klist;        // [BH, Nc * cap] union lists of key-cube pairs
  int n_kpairs;
  // schedule orders of the pair items (null: item order); order scratch
  int* qorder;
  int* korder;
  int* order_tmp;         // histogram / bucket cursors of the order
};

// ------------------------------------------------------------------ launches
// Each returns cudaSuccess or the launch error.
cudaError_t launch_permute(const Geom& g, const __nv_bfloat16* in, __nv_bfloat16* out,
                           int inverse, cudaStream_t s);
// bf16 caller tensor (raster when in_raster, else cube order) -> fp16 cube-order
// staged copy (nullable) and fp32 cube means (nullable); values outside the
// fp16 range set kDevRange in *status.
cudaError_t launch_stage(const Geom& g, const __nv_bfloat16* in, int in_raster, __half* out16,
                         float* pooled, uint32_t* status, cudaStream_t s);
cudaError_t launch_coarse_select(const Geom& g, int mode, int topk, float mass, int kmin,
                                 int kmax, const float* qc, const float* kc, const float* vc,
                                 float* oc, float* lse_c, int* idx, int* cnt, const Workspace& ws,
                                 cudaStream_t s);
// The same in two phases: logits, softmax statistics, selection and A_c
// (needs only Q_c, K_c), then O_c = A_c V_c.
cudaError_t launch_coarse_logits_select(const Geom& g, int mode, int topk, float mass, int kmin,
                                        int kmax, const float* qc, const float* kc, float* lse_c,
                                        int* idx, int* cnt, const Workspace& ws, cudaStream_t s);
cudaError_t launch_coarse_out(const Geom& g, const float* vc, float* oc, const Workspace& ws,
                              cudaStream_t s);
cudaError_t launch_build_qpairs(const Geom& g, const int* idx, const int* cnt,
                                const Workspace& ws, cudaStream_t s);
cudaError_t launch_fine_fwd(const Geom& g, const __half* q, const __half* k, const __half* v,
                            const __nv_bfloat16* gc, const __nv_bfloat16* gf, const float* oc,
                            __nv_bfloat16* o, __half* o_f, float* lse_f, const Workspace& ws,
                            cudaStream_t s);
// Combine backward.  dO_f = dO (.) G_f and delta are written scaled by a power
// of two per (batch, head) slice, gscale[bh] (chosen from the slice's largest
// |dO (.) G_f|, found first by a max-reduction into amax[bh], so that this
// largest value lands in [4, 8)): fp16 then keeps full precision for the
// magnitudes that matter, whatever the size of the upstream gradient.  The
// fine backward is linear in dO_f and divides its results by gscale.
cudaError_t launch_combine_bwd(const Geom& g, const __nv_bfloat16* d_o,
                               const __nv_bfloat16* gc, const __nv_bfloat16* gf,
                               const __half* o_f, const float* oc, void* dgc, void* dgf,
                               __half* dof, float* doc, float* delta, uint32_t* amax,
                               float* gscale, uint32_t* status, cudaStream_t s);
cudaError_t launch_coarse_bwd(const Geom& g, const float* qc, const float* kc, const float* vc,
                              const float* oc, const float* lse_c, const float* doc,
                              float* dqc, float* dkc, float* dvc, const Workspace& ws,
                              cudaStream_t s);
// The same in two parts: the tf32 operands of Q_c, K_c, V_c (no dependence on
// dO), then the rest.
cudaError_t launch_coarse_bwd_operands(const Geom& g, const float* qc, const float* kc,
                                       const float* vc, const Workspace& ws, cudaStream_t s);
cudaError_t launch_coarse_bwd_products(const Geom& g, const float* oc, const float* lse_c,
                                       const float* doc, float* dqc, float* dkc, float* dvc,
                                       const Workspace& ws, cudaStream_t s);
cudaError_t launch_build_kpairs(const Geom& g, const int* idx, const int* cnt,
                                const Workspace& ws, cudaStream_t s);
// Schedule order of n pair items: sorted by step count, largest first.  The
// persistent kernels' CTAs take schedule positions from a shared counter as
// they free up (item_seq.cuh), so this is the longest-processing-time rule:
// every CTA's total work ends within about one small item of the others.
cudaError_t launch_item_order(const PairItem* items, int n, int* order, int* tmp,
                              cudaStream_t s);
// Grid of the persistent fine kernels for n items: min(n, SMs).
int persistent_grid(int n);
// Whether the fine kernels run their items in the cost-sorted order: only when
// the fp16 K and V of all slices fit in twice the L2 (256 MB).  Otherwise the
// plain item order wins: the 152 items in flight are neighbouring cubes of one
// slice, which select the same K/V tiles, and those stay in L2.
inline bool use_cost_order(const Geom& g) {
  const double kv_bytes = 2.0 * 2.0 * g.BH * static_cast<double>(g.N) * g.D;
  return kv_bytes <= 256.0 * 1024 * 1024;
}
// gscale: [BH] factor dof and delta were scaled by (null: 1); the fine
// gradients are divided by it before the pooled ones are added.
cudaError_t launch_fine_bwd(const Geom& g, const __half* q, const __half* k, const __half* v,
                            const float* lse_f, const __half* dof, const float* delta,
                            const float* gscale, const float* dqc, const float* dkc,
                            const float* dvc, void* dq, void* dk, void* dv,
                            const Workspace& ws, cudaStream_t s);

// ------------------------------------------------ tensor-core fp32 GEMM
// D[b] = A[b] B[b]^T, A [M x K], B [N x K], both K-major, each passed as a
// tf32 pair hi + lo (fp32 arrays of tf32 values; hi = round(x), lo = round(x -
// hi)), accumulated in fp32 from three tf32 products (tgemm.cu); with every lo
// null, one plain tf32 product from the hi parts.  The attention-backward
// mode computes a second product E = A2 B2^T of the same tile into a second
// accumulator.
enum TgemmMode {
  kTgScale = 0,   // v = alpha * D
  kTgAttnBwd = 1  // p = exp2(alpha * D - beta * v1[m]),  v = p * (E - v2[m])
};
struct TgemmOperand {
  const float* hi;
  const float* lo;
  int ld;                 // elements between rows (multiple of 4)
  long long stride;       // elements between batches
};
struct TgemmArgs {
  int batch, M, N, K;
  int mode;
  float alpha, beta;
  const float* v1; const float* v2; long long vec_stride;  // per-row or per-column vectors
  // outputs, each optional: fp32 v [M][N]; v as a tf32 pair [M][N] (a null
  // lo writes the hi part alone); the tf32 hi parts of v and p transposed,
  // [N][M] (kTgAttnBwd)
  float* out; int out_ld; long long out_stride;
  float *out_hi, *out_lo; int split_ld; long long split_stride;
  float *vt_hi, *pt_hi; int t_ld; long long t_stride;
};
cudaError_t launch_tgemm(const TgemmArgs& a, const TgemmOperand& A, const TgemmOperand& B,
                         uint32_t* status, cudaStream_t s);
cudaError_t launch_tgemm_dual(const TgemmArgs& a, const TgemmOperand& A, const TgemmOperand& B,
                              const TgemmOperand& A2, const TgemmOperand& B2, uint32_t* status,
                              cudaStream_t s);
// tf32-pair splits, up to 8 per launch: fp32 [batch][rows][cols] (row stride
// ld_src) -> hi, lo in the same orientation or transposed ([batch][cols][rows]),
// row stride ld_dst; a null lo writes the hi parts alone.
struct SplitSpec {
  const float* src; int ld_src; long long stride_src; int rows, cols;
  float* hi; float* lo; int ld_dst; long long stride_dst; bool transpose;
};
cudaError_t launch_split_tf32(const SplitSpec* specs, int n, int batch, cudaStream_t s);
// Rank-3 tiled tensor map over fp32 [batch][rows][ld] with a box of
// (box_cols, box_rows, 1), 128-byte swizzle (api.cu).
bool encode_tiled_3d_f32(void* map, const float* base, uint64_t batch, uint64_t rows,
                         uint64_t cols, uint64_t ld, uint64_t batch_stride, uint32_t box_cols,
                         uint32_t box_rows);

// Driver entry point for tensor-map encoding, resolved once (api.cu).
bool encode_tiled_2d(void* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_cols);
// bf16 tensors read in place by the fine forward, 128-byte swizzle, boxes of
// 64 columns: 2-D over [rows, cols] (64-row boxes: a cube in cube order), or
// 5-D over a raster [BH, T, H, W, D] (boxes of 64 x 4 x 4 x 4 x 1: one (4,4,4)
// cube, its rows landing in the in-cube order (t%4)*16 + (h%4)*4 + w%4).
bool encode_tiled_2d_bf16(void* map, const void* base, uint64_t rows, uint64_t cols);
bool encode_raster_cubes_bf16(void* map, const void* base, const Geom& g);
// The same over bytes (e4m3 data), with a 64- or 128-byte swizzle.
bool encode_tiled_2d_u8(void* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, uint32_t box_cols, int swizzle_bytes);

// Head_dim 64 forms of the two above (fine_fwd64.cu: two CTAs per SM).
cudaError_t launch_fine_fwd64(const Geom& g, const __half* q, const __half* k, const __half* v,
                              const __nv_bfloat16* gc, const __nv_bfloat16* gf, const float* oc,
                              __nv_bfloat16* o, __half* o_f, float* lse_f, const Workspace& ws,
                              cudaStream_t s);
cudaError_t launch_fine_fwd64_bf16(const Geom& g, const __nv_bfloat16* q,
                                   const __nv_bfloat16* k, const __nv_bfloat16* v,
                                   const __nv_bfloat16* gc, const __nv_bfloat16* gf,
                                   const float* oc, __nv_bfloat16* o, float* lse_f,
                                   const Workspace& ws, cudaStream_t s);

// The fine forward + combine reading the caller's bf16 q, k, v (cfg layout)
// in place: no staged copies (fine_fwd.cu; inference: no O_f).
cudaError_t launch_fine_fwd_bf16(const Geom& g, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                 const __nv_bfloat16* v, const __nv_bfloat16* gc,
                                 const __nv_bfloat16* gf, const float* oc, __nv_bfloat16* o,
                                 float* lse_f, const Workspace& ws, cudaStream_t s);

// ------------------------------------------------ e4m3 variant of the fine forward
// Staging (stage_fp8.cu, head_dim 128): bf16 q, k, v (caller layout) -> e4m3
// copies Q8, K8 ([BH*N, 128] bytes, cube order) and V8T ([BH*Nc, 128, 64]
// bytes, each cube transposed), scales [BH][3] (1/s of Q, K, V: the power of
// two each slice was multiplied by), and optionally the fp32 cube means.
// amax: [3*BH] scratch.
cudaError_t launch_stage_fp8(const Geom& g, const __nv_bfloat16* q, const __nv_bfloat16* k,
                             const __nv_bfloat16* v, uint8_t* q8, uint8_t* k8, uint8_t* v8t,
                             float* scales, float* pq, float* pk, float* pv, uint32_t* amax,
                             uint32_t* status, cudaStream_t s);
// The fine forward + combine on those copies (fine_fwd.cu; inference: no O_f).
cudaError_t launch_fine_fwd_fp8(const Geom& g, const uint8_t* q8, const uint8_t* k8,
                                const uint8_t* v8t, const float* scales,
                                const __nv_bfloat16* gc, const __nv_bfloat16* gf, const float* oc,
                                __nv_bfloat16* o, float* lse_f, const Workspace& ws,
                                cudaStream_t s);

}  // namespace vsa

// Host side of the C ABI declared in include/vsa.h: argument checks, carving
// of the caller's `saved` and `ws` buffers, and the launch sequences of the
// forward and backward passes.  Nothing here allocates device memory.
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/vsa.h"
#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

vsa_status_t make_geom(const vsa_config_t* cfg, Geom* g) {
  if (!cfg) return VSA_ERR_INVALID_ARG;
  if (cfg->batch < 1 || cfg->heads < 1) return VSA_ERR_INVALID_ARG;
  if (cfg->T < 4 || cfg->H < 4 || cfg->W < 4 || cfg->T % 4 || cfg->H % 4 || cfg->W % 4)
    return VSA_ERR_SHAPE;
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return VSA_ERR_UNSUPPORTED;
  if (cfg->layout != VSA_LAYOUT_RASTER && cfg->layout != VSA_LAYOUT_CUBE)
    return VSA_ERR_INVALID_ARG;
  if (cfg->grad_dtype != VSA_GRAD_FP32 && cfg->grad_dtype != VSA_GRAD_BF16)
    return VSA_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(cfg->batch) * cfg->heads;
  const long long n = static_cast<long long>(cfg->T) * cfg->H * cfg->W;
  const long long nc = n / kTile;
  if (bh > 65535) return VSA_ERR_SHAPE;
  if (nc > VSA_MAX_CUBES || bh * n > 0x7fffffffLL) return VSA_ERR_SHAPE;
  int cap;
  if (cfg->select_mode == VSA_SELECT_TOPK) {
    if (cfg->topk < 1 || cfg->topk > nc || cfg->topk > VSA_MAX_LIST) return VSA_ERR_INVALID_ARG;
    cap = cfg->topk;
  } else if (cfg->select_mode == VSA_SELECT_MASS) {
    if (!(cfg->mass > 0.f && cfg->mass <= 1.f)) return VSA_ERR_INVALID_ARG;
    if (cfg->kmin < 1 || cfg->kmin > cfg->kmax || cfg->kmax > VSA_MAX_LIST)
      return VSA_ERR_INVALID_ARG;
    cap = cfg->kmax;
  } else {
    return VSA_ERR_INVALID_ARG;
  }
  if (bh * nc * cap > 0x7fffffffLL) return VSA_ERR_SHAPE;
  float scale = cfg->scale;
  if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(cfg->head_dim));
  if (!std::isfinite(scale)) return VSA_ERR_INVALID_ARG;
  g->B = cfg->batch;
  g->heads = cfg->heads;
  g->T = cfg->T;
  g->H = cfg->H;
  g->W = cfg->W;
  g->D = cfg->head_dim;
  g->BH = static_cast<int>(bh);
  g->N = static_cast<int>(n);
  g->Nc = static_cast<int>(nc);
  g->ct = cfg->T / 4;
  g->ch = cfg->H / 4;
  g->cw = cfg->W / 4;
  g->cap = cap;
  g->raster = cfg->layout == VSA_LAYOUT_RASTER;
  g->grad_bf16 = cfg->grad_dtype == VSA_GRAD_BF16;
  g->scale = scale;
  return VSA_OK;
}

namespace {

size_t half_tensor(const Geom& g) { return static_cast<size_t>(g.BH) * g.N * g.D * 2; }
size_t pooled_bytes(const Geom& g) { return static_cast<size_t>(g.BH) * g.Nc * g.D * 4; }

// Whether an inference forward (with_backward = 0) stages fp16 copies of Q, K,
// V: only raster tensors of head_dim 128 (vsa_forward explains why); it reads
// the others in place.
bool inference_stages(const Geom& g) { return g.raster && g.D == 128; }

// One layout for every use, ordered so that what an inference forward does
// not write comes last: the coarse results and lse_f, then the staged fp16
// copies (an inference forward writes them only when it stages), then O_f
// (training only).  with_backward = 0 gives the total of an inference
// forward; 1 the total of every piece (the training forward, the backward,
// the e4m3 forward).
void saved_layout(const Geom& g, int with_backward, vsa_saved_layout_t* L) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  L->qc = take(pooled_bytes(g));
  L->kc = take(pooled_bytes(g));
  L->vc = take(pooled_bytes(g));
  L->oc = take(pooled_bytes(g));
  L->lse_c = take(static_cast<size_t>(g.BH) * g.Nc * 4);
  L->idx = take(static_cast<size_t>(g.BH) * g.Nc * g.cap * 4);
  L->cnt = take(static_cast<size_t>(g.BH) * g.Nc * 4);
  L->lse_f = take(static_cast<size_t>(g.BH) * g.N * 4);
  const size_t end_in_place = off;
  L->q16 = take(half_tensor(g));
  L->k16 = take(half_tensor(g));
  L->v16 = take(half_tensor(g));
  const size_t end_staged = off;
  L->o_f = take(half_tensor(g));
  L->total = with_backward ? off : (inference_stages(g) ? end_staged : end_in_place);
  L->list_cap = g.cap;
}

// Carves `ws`; returns the bytes needed.  With base == nullptr only sizes.
size_t carve_ws(const Geom& g, int with_backward, void* base, Workspace* w) {
  size_t off = 0;
  char* b = static_cast<char*>(base);
  auto take = [&](size_t bytes) -> void* {
    void* p = b ? b + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  Workspace ws{};
  const int npairs = g.BH * ((g.Nc + 1) / 2);
  ws.status = static_cast<uint32_t*>(take(4));
  ws.counter = static_cast<int*>(take(64));
  ws.n_qpairs = npairs;
  ws.qpairs = static_cast<PairItem*>(take(sizeof(PairItem) * npairs));
  ws.qlist = static_cast<uint32_t*>(take(sizeof(uint32_t) * npairs * 2 * g.cap));
  ws.qorder = static_cast<int*>(take(sizeof(int) * npairs));
  ws.order_tmp = static_cast<int*>(take(sizeof(int) * (npairs + 512)));
  ws.gamax = static_cast<uint32_t*>(take(sizeof(uint32_t) * 3 * g.BH));
  // coarse logits [BH, Nc, ldc] and the coarse GEMM operands: tf32 pairs of
  // Q_c and K_c for the logits, everything else rounded to tf32 alone
  const size_t ldc = static_cast<size_t>((g.Nc + 3) & ~3);
  ws.clogit = static_cast<float*>(take(static_cast<size_t>(g.BH) * g.Nc * ldc * 4));
  const size_t pc_bytes = static_cast<size_t>(g.BH) * g.Nc * ldc * 4;  // [BH, Nc, ldc]
  const size_t dc_bytes = static_cast<size_t>(g.BH) * g.D * ldc * 4;   // [BH, D, ldc]
  auto f32 = [&](size_t bytes) { return static_cast<float*>(take(bytes)); };
  ws.qh = f32(pooled_bytes(g));
  ws.ql = f32(pooled_bytes(g));
  ws.kh = f32(pooled_bytes(g));
  ws.kl = f32(pooled_bytes(g));
  ws.vth = f32(dc_bytes);
  ws.ach = f32(pc_bytes);
  if (with_backward) {
    const size_t words = (g.Nc + 31) / 32;
    ws.gscale = static_cast<float*>(take(sizeof(float) * g.BH));
    ws.dof = take(half_tensor(g));
    ws.delta = static_cast<float*>(take(static_cast<size_t>(g.BH) * g.N * 4));
    ws.doc = static_cast<float*>(take(pooled_bytes(g)));
    ws.dqc = static_cast<float*>(take(pooled_bytes(g)));
    ws.dkc = static_cast<float*>(take(pooled_bytes(g)));
    ws.dvc = static_cast<float*>(take(pooled_bytes(g)));
    ws.vh = f32(pooled_bytes(g));
    ws.doh = f32(pooled_bytes(g));
    ws.kth = f32(dc_bytes);
    ws.qth = f32(dc_bytes);
    ws.doth = f32(dc_bytes);
    ws.pth = f32(pc_bytes);
    ws.dlth = f32(pc_bytes);
    ws.cdelta = static_cast<float*>(take(static_cast<size_t>(g.BH) * g.Nc * 4));
    ws.tmask = static_cast<uint32_t*>(take(static_cast<size_t>(g.BH) * g.Nc * words * 4));
    ws.toff = static_cast<int*>(take(static_cast<size_t>(g.BH) * (g.Nc + 1) * 4));
    ws.tlist = static_cast<int*>(take(static_cast<size_t>(g.BH) * g.Nc * g.cap * 4));
    ws.n_kpairs = npairs;
    ws.kpairs = static_cast<PairItem*>(take(sizeof(PairItem) * npairs));
    ws.korder = static_cast<int*>(take(sizeof(int) * npairs));
    ws.klist = static_cast<uint32_t*>(take(static_cast<size_t>(g.BH) * g.Nc * g.cap * 4));
  }
  if (w) *w = ws;
  return off;
}

vsa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? VSA_OK : VSA_ERR_CUDA; }

namespace {

// A second stream per device for the backward's list building, which needs
// only the saved selection and so runs beside the combine and coarse
// backward kernels (latency-bound small kernels next to bandwidth-bound
// ones).  Created on first use; each call forks to it and joins back with
// events of its own, under a lock so that two host threads never interleave
// their fork / join on it.
constexpr int kMaxSideDevices = 64;
std::mutex g_side_mutex;
cudaStream_t g_side_stream[kMaxSideDevices] = {};

cudaError_t side_stream(cudaStream_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxSideDevices) return cudaErrorInvalidDevice;
  if (!g_side_stream[dev]) {
    e = cudaStreamCreateWithFlags(&g_side_stream[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *out = g_side_stream[dev];
  return cudaSuccess;
}

// Events of one fork and up to two joins, destroyed when the call returns (the
// waits already enqueued keep their effect).
struct ForkJoin {
  cudaEvent_t fork = nullptr, join = nullptr, join2 = nullptr;
  ~ForkJoin() {
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    if (join2) cudaEventDestroy(join2);
  }
  cudaError_t create() {
    cudaError_t e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
    return e != cudaSuccess ? e : cudaEventCreateWithFlags(&join2, cudaEventDisableTiming);
  }
};

}  // namespace

template <typename... Ptrs>
bool all_aligned(Ptrs... ps) {
  return (aligned16(ps) && ...);
}

template <typename... Ptrs>
bool all_set(Ptrs... ps) {
  return ((ps != nullptr) && ...);
}

using bf16 = __nv_bfloat16;
using f16 = __half;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

// 2-D fp16 tensor map with 128-byte swizzle (the staged operands).
// The driver's tensor-map encoder, looked up once per process.
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q{};
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

bool encode_tiled_2d(void* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_cols) {
  if (!encoder()) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_2d_bf16(void* map, const void* base, uint64_t rows, uint64_t cols) {
  if (!encoder()) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_raster_cubes_bf16(void* map, const void* base, const Geom& g) {
  if (!encoder()) return false;
  const uint64_t D = static_cast<uint64_t>(g.D);
  const cuuint64_t dims[5] = {D, static_cast<cuuint64_t>(g.W), static_cast<cuuint64_t>(g.H),
                              static_cast<cuuint64_t>(g.T), static_cast<cuuint64_t>(g.BH)};
  const cuuint64_t strides[4] = {D * 2, D * 2 * g.W, D * 2 * g.W * g.H,
                                 D * 2 * g.W * g.H * g.T};
  const cuuint32_t box[5] = {64, 4, 4, 4, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return g_encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_2d_u8(void* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, uint32_t box_cols, int swizzle_bytes) {
  if (!encoder()) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return g_encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_3d_f32(void* map, const float* base, uint64_t batch, uint64_t rows,
                         uint64_t cols, uint64_t ld, uint64_t batch_stride, uint32_t box_cols,
                         uint32_t box_rows) {
  if (!encoder()) return false;
  const cuuint64_t dims[3] = {cols, rows, batch};
  const cuuint64_t strides[2] = {ld * 4, batch_stride * 4};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encoder()(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                   const_cast<float*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace vsa

using namespace vsa;

extern "C" {

vsa_status_t vsa_validate(const vsa_config_t* cfg) {
  Geom g;
  return make_geom(cfg, &g);
}

const char* vsa_status_string(vsa_status_t s) {
  switch (s) {
    case VSA_OK: return "ok";
    case VSA_ERR_INVALID_ARG: return "invalid argument";
    case VSA_ERR_SHAPE: return "unsupported shape (T, H, W must be positive multiples of 4; size limits)";
    case VSA_ERR_UNSUPPORTED: return "unsupported head_dim (64 or 128)";
    case VSA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case VSA_ERR_CUDA: return "CUDA error";
    case VSA_ERR_TIMEOUT: return "device-side wait timed out";
    case VSA_ERR_DEVICE_CHECK:
      return "device-side range check failed (bad index list, or a value outside the fp16 range)";
  }
  return "unknown status";
}

size_t vsa_saved_bytes(const vsa_config_t* cfg, vsa_saved_layout_t* layout) {
  return vsa_saved_bytes_for(cfg, 1, layout);
}

size_t vsa_saved_bytes_for(const vsa_config_t* cfg, int with_backward,
                           vsa_saved_layout_t* layout) {
  Geom g;
  if (make_geom(cfg, &g) != VSA_OK) return 0;
  vsa_saved_layout_t L;
  saved_layout(g, with_backward != 0, &L);
  if (layout) *layout = L;
  return L.total;
}

size_t vsa_workspace_bytes(const vsa_config_t* cfg, int with_backward) {
  Geom g;
  if (make_geom(cfg, &g) != VSA_OK) return 0;
  return carve_ws(g, with_backward, nullptr, nullptr);
}

vsa_status_t vsa_reset_device_status(void* ws, void* stream) {
  if (!ws) return VSA_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, 4, static_cast<cudaStream_t>(stream)));
}

vsa_status_t vsa_check_device_status(void* ws, void* stream) {
  if (!ws) return VSA_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, ws, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return VSA_ERR_CUDA;
  if (word & kDevTimeout) return VSA_ERR_TIMEOUT;
  if (word & (kDevBadIndex | kDevRange)) return VSA_ERR_DEVICE_CHECK;
  return VSA_OK;
}

vsa_status_t vsa_permute(const vsa_config_t* cfg, const void* in, void* out, int inverse,
                         void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(in, out) || in == out || (inverse != 0 && inverse != 1))
    return VSA_ERR_INVALID_ARG;
  if (!all_aligned(in, out)) return VSA_ERR_ALIGNMENT;
  return cuda_status(launch_permute(g, static_cast<const bf16*>(in), static_cast<bf16*>(out),
                                    inverse, static_cast<cudaStream_t>(stream)));
}

vsa_status_t vsa_stage(const vsa_config_t* cfg, const void* x, void* x16, float* pooled,
                       void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(x, ws) || (!x16 && !pooled)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(x, ws) || !aligned16(x16) || !aligned16(pooled)) return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 0, ws, &w);
  return cuda_status(launch_stage(g, static_cast<const bf16*>(x), g.raster, static_cast<f16*>(x16),
                                  pooled, w.status, static_cast<cudaStream_t>(stream)));
}

vsa_status_t vsa_coarse_select(const vsa_config_t* cfg, const void* q, const void* k,
                               const void* v, float* qc, float* kc, float* vc, float* oc,
                               float* lse_c, int32_t* idx, int32_t* cnt, void* ws,
                               void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  const bool pooled = !q && !k && !v;  // qc, kc, vc are inputs
  if ((!pooled && !all_set(q, k, v)) || !all_set(qc, kc, vc, oc, lse_c, idx, cnt, ws))
    return VSA_ERR_INVALID_ARG;
  if (!all_aligned(q, k, v, qc, kc, vc, oc, lse_c, idx, cnt, ws)) return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 0, ws, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!pooled &&
      (launch_stage(g, static_cast<const bf16*>(q), g.raster, nullptr, qc, w.status, s) ||
       launch_stage(g, static_cast<const bf16*>(k), g.raster, nullptr, kc, w.status, s) ||
       launch_stage(g, static_cast<const bf16*>(v), g.raster, nullptr, vc, w.status, s)))
    return VSA_ERR_CUDA;
  return cuda_status(launch_coarse_select(g, cfg->select_mode, cfg->topk, cfg->mass, cfg->kmin,
                                          cfg->kmax, qc, kc, vc, oc, lse_c, idx, cnt, w, s));
}

vsa_status_t vsa_fine_fwd(const vsa_config_t* cfg, const void* q16, const void* k16,
                          const void* v16, const int32_t* idx, const int32_t* cnt, const void* gc,
                          const void* gf, const float* oc, void* o, void* o_f, float* lse_f,
                          void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(q16, k16, v16, idx, cnt, gc, gf, oc, o, ws)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(q16, k16, v16, idx, cnt, gc, gf, oc, o, ws) || !aligned16(o_f) ||
      !aligned16(lse_f))
    return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 0, ws, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_build_qpairs(g, idx, cnt, w, s) != cudaSuccess) return VSA_ERR_CUDA;
  return cuda_status(launch_fine_fwd(g, static_cast<const f16*>(q16), static_cast<const f16*>(k16),
                                     static_cast<const f16*>(v16), static_cast<const bf16*>(gc),
                                     static_cast<const bf16*>(gf), oc, static_cast<bf16*>(o),
                                     static_cast<f16*>(o_f), lse_f, w, s));
}

vsa_status_t vsa_fine_fwd_bf16(const vsa_config_t* cfg, const void* q, const void* k,
                               const void* v, const int32_t* idx, const int32_t* cnt,
                               const void* gc, const void* gf, const float* oc, void* o,
                               float* lse_f, void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(q, k, v, idx, cnt, gc, gf, oc, o, ws)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(q, k, v, idx, cnt, gc, gf, oc, o, ws) || !aligned16(lse_f))
    return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 0, ws, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_build_qpairs(g, idx, cnt, w, s) != cudaSuccess) return VSA_ERR_CUDA;
  return cuda_status(launch_fine_fwd_bf16(g, static_cast<const bf16*>(q),
                                          static_cast<const bf16*>(k),
                                          static_cast<const bf16*>(v),
                                          static_cast<const bf16*>(gc),
                                          static_cast<const bf16*>(gf), oc, static_cast<bf16*>(o),
                                          lse_f, w, s));
}

vsa_status_t vsa_combine_bwd(const vsa_config_t* cfg, const void* d_o, const void* gc,
                             const void* gf, const void* o_f, const float* oc, void* dgc,
                             void* dgf, void* dof16, float* doc, float* delta, float* gscale,
                             void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(d_o, gc, gf, o_f, oc, dgc, dgf, dof16, doc, delta, gscale, ws))
    return VSA_ERR_INVALID_ARG;
  if (!all_aligned(d_o, gc, gf, o_f, oc, dgc, dgf, dof16, doc, delta, gscale, ws))
    return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 0, ws, &w);
  return cuda_status(launch_combine_bwd(
      g, static_cast<const bf16*>(d_o), static_cast<const bf16*>(gc),
      static_cast<const bf16*>(gf), static_cast<const f16*>(o_f), oc, dgc, dgf,
      static_cast<f16*>(dof16), doc, delta, w.gamax, gscale,
      w.status, static_cast<cudaStream_t>(stream)));
}

vsa_status_t vsa_coarse_bwd(const vsa_config_t* cfg, const float* qc, const float* kc,
                            const float* vc, const float* oc, const float* lse_c,
                            const float* doc, float* dqc, float* dkc, float* dvc, void* ws,
                            void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(qc, kc, vc, oc, lse_c, doc, dqc, dkc, dvc, ws)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(qc, kc, vc, oc, lse_c, doc, dqc, dkc, dvc, ws)) return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 1, ws, &w);
  return cuda_status(launch_coarse_bwd(g, qc, kc, vc, oc, lse_c, doc, dqc, dkc, dvc, w,
                                       static_cast<cudaStream_t>(stream)));
}

vsa_status_t vsa_fine_bwd(const vsa_config_t* cfg, const void* q16, const void* k16,
                          const void* v16, const int32_t* idx, const int32_t* cnt,
                          const float* lse_f, const void* dof16, const float* delta,
                          const float* gscale, const float* dqc, const float* dkc,
                          const float* dvc, void* dq, void* dk, void* dv, void* ws,
                          void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(q16, k16, v16, idx, cnt, lse_f, dof16, delta, dq, dk, dv, ws))
    return VSA_ERR_INVALID_ARG;
  if (!all_aligned(q16, k16, v16, idx, cnt, lse_f, dof16, delta, dq, dk, dv, ws) ||
      !aligned16(dqc) || !aligned16(dkc) || !aligned16(dvc) ||
      (reinterpret_cast<uintptr_t>(gscale) & 3u))
    return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 1, ws, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_build_qpairs(g, idx, cnt, w, s) != cudaSuccess) return VSA_ERR_CUDA;
  if (launch_build_kpairs(g, idx, cnt, w, s) != cudaSuccess) return VSA_ERR_CUDA;
  return cuda_status(launch_fine_bwd(g, static_cast<const f16*>(q16), static_cast<const f16*>(k16),
                                     static_cast<const f16*>(v16), lse_f,
                                     static_cast<const f16*>(dof16), delta, gscale, dqc, dkc, dvc,
                                     dq, dk, dv, w, s));
}

vsa_status_t vsa_forward(const vsa_config_t* cfg, const void* q, const void* k, const void* v,
                         const void* gc, const void* gf, void* o, void* saved,
                         int with_backward, void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(q, k, v, gc, gf, o, saved, ws)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(q, k, v, gc, gf, o, saved, ws)) return VSA_ERR_ALIGNMENT;
  vsa_saved_layout_t L;
  saved_layout(g, with_backward != 0, &L);
  char* sv = static_cast<char*>(saved);
  Workspace w;
  carve_ws(g, 0, ws, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // V is staged on the side stream while Q and K are staged and the logits,
  // selection and lists are computed on `s` (V is needed first by O_c).
  std::lock_guard<std::mutex> lock(g_side_mutex);
  cudaStream_t side = nullptr;
  ForkJoin fj;
  if (side_stream(&side) != cudaSuccess || fj.create() != cudaSuccess ||
      cudaEventRecord(fj.fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(side, fj.fork, 0) != cudaSuccess)
    return VSA_ERR_CUDA;
  float* qc = reinterpret_cast<float*>(sv + L.qc);
  float* kc = reinterpret_cast<float*>(sv + L.kc);
  float* vc = reinterpret_cast<float*>(sv + L.vc);
  float* oc = reinterpret_cast<float*>(sv + L.oc);
  float* lse_c = reinterpret_cast<float*>(sv + L.lse_c);
  int* idx = reinterpret_cast<int*>(sv + L.idx);
  int* cnt = reinterpret_cast<int*>(sv + L.cnt);
  // Inference reads q, k, v in place unless they are raster tensors of head_dim
  // 128: there a cube's 64-channel box is 16 runs spread over a 4 x 4 patch of
  // image rows, and the fine stage measured 23-31% slower than on the staged
  // cube-order copy (which is one contiguous block per cube); at head_dim 64
  // (whole 512-byte runs) and in cube layout it runs at the staged speed.
  const bool in_place = !with_backward && !inference_stages(g);
  f16* q16 = in_place ? nullptr : reinterpret_cast<f16*>(sv + L.q16);
  f16* k16 = in_place ? nullptr : reinterpret_cast<f16*>(sv + L.k16);
  f16* v16 = in_place ? nullptr : reinterpret_cast<f16*>(sv + L.v16);
  if (launch_stage(g, static_cast<const bf16*>(v), g.raster, v16, vc, w.status, side) ||
      cudaEventRecord(fj.join, side) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (launch_stage(g, static_cast<const bf16*>(q), g.raster, q16, qc, w.status, s) ||
      launch_stage(g, static_cast<const bf16*>(k), g.raster, k16, kc, w.status, s))
    return VSA_ERR_CUDA;
  if (launch_coarse_logits_select(g, cfg->select_mode, cfg->topk, cfg->mass, cfg->kmin,
                                  cfg->kmax, qc, kc, lse_c, idx, cnt, w, s) != cudaSuccess ||
      launch_build_qpairs(g, idx, cnt, w, s) != cudaSuccess ||
      cudaStreamWaitEvent(s, fj.join, 0) != cudaSuccess ||
      launch_coarse_out(g, vc, oc, w, s) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (in_place)
    return cuda_status(launch_fine_fwd_bf16(
        g, static_cast<const bf16*>(q), static_cast<const bf16*>(k), static_cast<const bf16*>(v),
        static_cast<const bf16*>(gc), static_cast<const bf16*>(gf), oc, static_cast<bf16*>(o),
        reinterpret_cast<float*>(sv + L.lse_f), w, s));
  return cuda_status(launch_fine_fwd(g, q16, k16, v16, static_cast<const bf16*>(gc),
                                     static_cast<const bf16*>(gf), oc, static_cast<bf16*>(o),
                                     with_backward ? reinterpret_cast<f16*>(sv + L.o_f) : nullptr,
                                     reinterpret_cast<float*>(sv + L.lse_f), w, s));
}

vsa_status_t vsa_backward(const vsa_config_t* cfg, const void* gc, const void* gf,
                          const void* saved, const void* d_o, void* dq, void* dk, void* dv,
                          void* dgc, void* dgf, void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (!all_set(gc, gf, saved, d_o, dq, dk, dv, dgc, dgf, ws)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(gc, gf, saved, d_o, dq, dk, dv, dgc, dgf, ws)) return VSA_ERR_ALIGNMENT;
  vsa_saved_layout_t L;
  saved_layout(g, 1, &L);
  const char* sv = static_cast<const char*>(saved);
  Workspace w;
  carve_ws(g, 1, ws, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const f16* q16 = reinterpret_cast<const f16*>(sv + L.q16);
  const f16* k16 = reinterpret_cast<const f16*>(sv + L.k16);
  const f16* v16 = reinterpret_cast<const f16*>(sv + L.v16);
  const f16* of = reinterpret_cast<const f16*>(sv + L.o_f);
  const float* oc = reinterpret_cast<const float*>(sv + L.oc);
  const int* idx = reinterpret_cast<const int*>(sv + L.idx);
  const int* cnt = reinterpret_cast<const int*>(sv + L.cnt);
  // The coarse backward's tf32 operands of Q_c, K_c, V_c, then the pair lists
  // and the transposed lists (ws regions of their own; none needs dO) on the
  // side stream, after everything already on `s`; `s` waits for the operands
  // before the coarse backward's products and for the lists before the fine
  // backward.
  std::lock_guard<std::mutex> lock(g_side_mutex);
  cudaStream_t side = nullptr;
  ForkJoin fj;
  if (side_stream(&side) != cudaSuccess || fj.create() != cudaSuccess ||
      cudaEventRecord(fj.fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(side, fj.fork, 0) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (launch_coarse_bwd_operands(g, reinterpret_cast<const float*>(sv + L.qc),
                                 reinterpret_cast<const float*>(sv + L.kc),
                                 reinterpret_cast<const float*>(sv + L.vc), w,
                                 side) != cudaSuccess ||
      cudaEventRecord(fj.join, side) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (launch_build_qpairs(g, idx, cnt, w, side) != cudaSuccess) return VSA_ERR_CUDA;
  if (launch_build_kpairs(g, idx, cnt, w, side) != cudaSuccess) return VSA_ERR_CUDA;
  if (cudaEventRecord(fj.join2, side) != cudaSuccess) return VSA_ERR_CUDA;
  if (launch_combine_bwd(g, static_cast<const bf16*>(d_o), static_cast<const bf16*>(gc),
                         static_cast<const bf16*>(gf), of, oc, dgc, dgf,
                         static_cast<f16*>(w.dof), w.doc, w.delta, w.gamax, w.gscale, w.status,
                         s) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (cudaStreamWaitEvent(s, fj.join, 0) != cudaSuccess) return VSA_ERR_CUDA;
  if (launch_coarse_bwd_products(g, oc, reinterpret_cast<const float*>(sv + L.lse_c), w.doc,
                                 w.dqc, w.dkc, w.dvc, w, s) != cudaSuccess ||
      cudaStreamWaitEvent(s, fj.join2, 0) != cudaSuccess)
    return VSA_ERR_CUDA;
  return cuda_status(launch_fine_bwd(g, q16, k16, v16, reinterpret_cast<const float*>(sv + L.lse_f),
                                     static_cast<const f16*>(w.dof), w.delta, w.gscale, w.dqc,
                                     w.dkc, w.dvc, dq, dk, dv, w, s));
}

vsa_status_t vsa_stage_fp8(const vsa_config_t* cfg, const void* q, const void* k,
                           const void* v, void* q8, void* k8, void* v8t, float* scales,
                           float* qc, float* kc, float* vc, void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (g.D != 128) return VSA_ERR_UNSUPPORTED;
  if (!all_set(q, k, v, q8, k8, v8t, scales, ws)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(q, k, v, q8, k8, v8t, scales, ws) || !aligned16(qc) || !aligned16(kc) ||
      !aligned16(vc))
    return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 0, ws, &w);
  return cuda_status(launch_stage_fp8(g, static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                                      static_cast<const bf16*>(v), static_cast<uint8_t*>(q8),
                                      static_cast<uint8_t*>(k8), static_cast<uint8_t*>(v8t),
                                      scales, qc, kc, vc, w.gamax, w.status,
                                      static_cast<cudaStream_t>(stream)));
}

vsa_status_t vsa_fine_fwd_fp8(const vsa_config_t* cfg, const void* q8, const void* k8,
                              const void* v8t, const float* scales, const int32_t* idx,
                              const int32_t* cnt, const void* gc, const void* gf, const float* oc,
                              void* o, float* lse_f, void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (g.D != 128) return VSA_ERR_UNSUPPORTED;
  if (!all_set(q8, k8, v8t, scales, idx, cnt, gc, gf, oc, o, ws)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(q8, k8, v8t, scales, idx, cnt, gc, gf, oc, o, ws) || !aligned16(lse_f))
    return VSA_ERR_ALIGNMENT;
  Workspace w;
  carve_ws(g, 0, ws, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_build_qpairs(g, idx, cnt, w, s) != cudaSuccess) return VSA_ERR_CUDA;
  return cuda_status(launch_fine_fwd_fp8(g, static_cast<const uint8_t*>(q8),
                                         static_cast<const uint8_t*>(k8),
                                         static_cast<const uint8_t*>(v8t), scales,
                                         static_cast<const bf16*>(gc), static_cast<const bf16*>(gf),
                                         oc, static_cast<bf16*>(o), lse_f, w, s));
}

vsa_status_t vsa_forward_fp8(const vsa_config_t* cfg, const void* q, const void* k,
                             const void* v, const void* gc, const void* gf, void* o, void* saved,
                             void* ws, void* stream) {
  Geom g;
  vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  if (g.D != 128) return VSA_ERR_UNSUPPORTED;
  if (!all_set(q, k, v, gc, gf, o, saved, ws)) return VSA_ERR_INVALID_ARG;
  if (!all_aligned(q, k, v, gc, gf, o, saved, ws)) return VSA_ERR_ALIGNMENT;
  vsa_saved_layout_t L;
  saved_layout(g, 1, &L);
  char* sv = static_cast<char*>(saved);
  Workspace w;
  carve_ws(g, 0, ws, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* q8 = reinterpret_cast<uint8_t*>(sv + L.q16);
  uint8_t* k8 = reinterpret_cast<uint8_t*>(sv + L.k16);
  uint8_t* v8t = reinterpret_cast<uint8_t*>(sv + L.v16);
  float* scales = reinterpret_cast<float*>(sv + L.o_f);
  float* qc = reinterpret_cast<float*>(sv + L.qc);
  float* kc = reinterpret_cast<float*>(sv + L.kc);
  float* vc = reinterpret_cast<float*>(sv + L.vc);
  float* oc = reinterpret_cast<float*>(sv + L.oc);
  int* idx = reinterpret_cast<int*>(sv + L.idx);
  int* cnt = reinterpret_cast<int*>(sv + L.cnt);
  if (launch_stage_fp8(g, static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                       static_cast<const bf16*>(v), q8, k8, v8t, scales, qc, kc, vc, w.gamax,
                       w.status, s) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (launch_coarse_select(g, cfg->select_mode, cfg->topk, cfg->mass, cfg->kmin, cfg->kmax, qc,
                           kc, vc, oc, reinterpret_cast<float*>(sv + L.lse_c), idx, cnt, w,
                           s) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (launch_build_qpairs(g, idx, cnt, w, s) != cudaSuccess) return VSA_ERR_CUDA;
  return cuda_status(launch_fine_fwd_fp8(g, q8, k8, v8t, scales, static_cast<const bf16*>(gc),
                                         static_cast<const bf16*>(gf), oc, static_cast<bf16*>(o),
                                         reinterpret_cast<float*>(sv + L.lse_f), w, s));
}

}  // extern "C"

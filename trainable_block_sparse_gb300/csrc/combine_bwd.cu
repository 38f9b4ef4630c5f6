// Backward of the gated combine O = repeat(O_c) (.) G_c + O_f (.) G_f (paper
// notes 关键设计 3; "VSA: Faster Video Diffusion with Trainable Sparse
// Attention", App. B: the coarse output is repeated across its block):
//   dG_c = dO (.) repeat(O_c)          dG_f = dO (.) O_f
//   dO_f = dO (.) G_f (fp16, the tensor-core operand of the fine backward)
//   dO_c[cube] = sum over the cube of dO (.) G_c
//   delta[row] = sum_d dO_f (.) O_f    (the softmax-backward row term of the fine stage)
// HBM-bound: one CTA per (batch, head, cube) reads dO, G_c, G_f (bf16, caller
// layout) and O_f (fp16, cube order) once and writes each output once (dG_c
// and dG_f as fp32, or rounded once to bf16 when the caller asks for bf16
// gradients).
//
// dO_f is the fp16 tensor-core operand of the fine backward.  Upstream
// gradients of bf16 training are often far below fp16's normal range (1e-5 to
// 1e-8 without loss scaling), where fp16 loses significand bits or flushes to
// zero.  So dO_f and delta are written times a power of two s per (batch, head)
// slice, chosen so that the slice's largest |dO (.) G_f| lands in [4, 8): a
// max-reduction over the slice (amax_kernel) runs first.  Everything the fine
// backward computes from dO_f is linear in it, and a power of two scales
// exactly, so the fine backward divides its results by s and nothing else
// changes.  A per-slice (not per-row) factor is what the key-side gradients
// need: dK and dV sum over query rows, which must share one factor.
#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 256;
constexpr int kAmaxCtasPerSm = 4;

// Largest |dO (.) G_f| of each slice, as the bits of a non-negative float
// (which order like the floats), max-reduced into amax[bh] (zeroed before).
// NaNs are skipped here (fmaxf); the combine kernel flags every non-finite
// product itself.
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint4* __restrict__ d_o,
                                                        const uint4* __restrict__ gf,
                                                        size_t vec_per_slice, uint32_t* amax) {
  const int bh = blockIdx.y;
  const size_t base = static_cast<size_t>(bh) * vec_per_slice;
  float m = 0.f;
  for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < vec_per_slice;
       i += static_cast<size_t>(gridDim.x) * kThreads) {
    const uint4 ud = d_o[base + i], uf = gf[base + i];
    const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&ud);
    const __nv_bfloat162* pf = reinterpret_cast<const __nv_bfloat162*>(&uf);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 dd = __bfloat1622float2(pd[e]);
      const float2 ff = __bfloat1622float2(pf[e]);
      m = fmaxf(m, fmaxf(fabsf(dd.x * ff.x), fabsf(dd.y * ff.y)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ float wmax[kThreads / 32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, wmax[w]);
    atomicMax(amax + bh, __float_as_uint(m));
  }
}

// The power of two s that brings a slice maximum `bits` (a non-negative float)
// into [4, 8): s = 2^(3 - x) for a maximum in [2^(x-1), 2^x), clamped so that s
// and 1/s are normal floats.  A zero or non-finite maximum gives s = 1.
__device__ __forceinline__ float grad_scale_of(uint32_t bits) {
  const int E = static_cast<int>((bits >> 23) & 0xFFu);
  if (bits == 0u || E == 0xFF) return 1.f;
  const int e = E == 0 ? 126 : min(126, max(-126, 3 - (E - 126)));
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// Eight fp32 values rounded to bf16 (nearest even), packed in order.
__device__ __forceinline__ uint4 pack_bf16x8(const float (&v)[8]) {
  uint4 u;
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) p[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
  return u;
}

template <int D>
__global__ void __launch_bounds__(kThreads) combine_bwd_kernel(
    Geom g, const uint4* __restrict__ d_o, const uint4* __restrict__ gc,
    const uint4* __restrict__ gf, const uint4* __restrict__ o_f, const float* __restrict__ oc,
    void* __restrict__ dgc, void* __restrict__ dgf, uint4* __restrict__ dof,
    float* __restrict__ doc, float* __restrict__ delta, const uint32_t* __restrict__ amax,
    float* __restrict__ gscale, uint32_t* status) {
  constexpr int VPR = D / 8;              // 8-element vectors per row
  constexpr int GROUPS = kThreads / VPR;  // rows processed side by side
  __shared__ float red[GROUPS][D];
  const int c = blockIdx.x, bh = blockIdx.y;
  const int col = threadIdx.x % VPR, grp = threadIdx.x / VPR;
  const size_t slice = static_cast<size_t>(bh) * g.N;
  const float gs = grad_scale_of(amax[bh]);  // the same in every CTA of the slice
  if (c == 0 && threadIdx.x == 0) gscale[bh] = gs;
  const float* ocr = oc + (static_cast<size_t>(bh) * g.Nc + c) * D + col * 8;
  float ocv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ocv[i] = ocr[i];
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  bool bad = false;
  for (int o = grp; o < kTile; o += GROUPS) {
    const size_t crow = slice + caller_row(g, c, o);
    const size_t frow = slice + static_cast<size_t>(c) * kTile + o;
    const uint4 ud = d_o[crow * VPR + col], uc = gc[crow * VPR + col], uf = gf[crow * VPR + col];
    const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&ud);
    const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&uc);
    const __nv_bfloat162* pf = reinterpret_cast<const __nv_bfloat162*>(&uf);
    const uint4 uo = o_f[frow * VPR + col];  // fp16 O_f, 8 values
    const __half2* po = reinterpret_cast<const __half2*>(&uo);
    float ofv[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(po[e]);
      ofv[2 * e] = f.x;
      ofv[2 * e + 1] = f.y;
    }
    float vdgc[8], vdgf[8];
    uint4 udof;
    __half2* pof = reinterpret_cast<__half2*>(&udof);
    float dsum = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 dd = __bfloat1622float2(pd[e]);
      const float2 cc = __bfloat1622float2(pc[e]);
      const float2 ff = __bfloat1622float2(pf[e]);
      vdgc[2 * e] = dd.x * ocv[2 * e];
      vdgc[2 * e + 1] = dd.y * ocv[2 * e + 1];
      vdgf[2 * e] = dd.x * ofv[2 * e];
      vdgf[2 * e + 1] = dd.y * ofv[2 * e + 1];
      acc[2 * e] += dd.x * cc.x;
      acc[2 * e + 1] += dd.y * cc.y;
      // exact: a product of two bf16 values times a power of two
      const float2 raw = make_float2(dd.x * ff.x * gs, dd.y * ff.y * gs);
      bad |= !(fabsf(raw.x) <= 65504.f) || !(fabsf(raw.y) <= 65504.f);
      pof[e] = __floats2half2_rn(raw.x, raw.y);
      const float2 r = __half22float2(pof[e]);  // delta uses the rounded dO_f the MMAs see
      dsum = fmaf(r.x, ofv[2 * e], fmaf(r.y, ofv[2 * e + 1], dsum));
    }
    const size_t o8 = crow * D + col * 8;  // first of this thread's 8 elements
    if (g.grad_bf16) {
      reinterpret_cast<uint4*>(dgc)[o8 / 8] = pack_bf16x8(vdgc);
      reinterpret_cast<uint4*>(dgf)[o8 / 8] = pack_bf16x8(vdgf);
    } else {
      float4* dc = reinterpret_cast<float4*>(static_cast<float*>(dgc) + o8);
      float4* df = reinterpret_cast<float4*>(static_cast<float*>(dgf) + o8);
      dc[0] = make_float4(vdgc[0], vdgc[1], vdgc[2], vdgc[3]);
      dc[1] = make_float4(vdgc[4], vdgc[5], vdgc[6], vdgc[7]);
      df[0] = make_float4(vdgf[0], vdgf[1], vdgf[2], vdgf[3]);
      df[1] = make_float4(vdgf[4], vdgf[5], vdgf[6], vdgf[7]);
    }
    dof[frow * VPR + col] = udof;
    // row sum over the VPR consecutive lanes that share this row
#pragma unroll
    for (int off = VPR / 2; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    if (col == 0) delta[frow] = dsum;
  }
  if (bad) flag_error(status, kDevRange);
#pragma unroll
  for (int i = 0; i < 8; ++i) red[grp][col * 8 + i] = acc[i];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += kThreads) {
    float s = 0.f;
#pragma unroll 8
    for (int r = 0; r < GROUPS; ++r) s += red[r][d];
    doc[(static_cast<size_t>(bh) * g.Nc + c) * D + d] = s;
  }
}

}  // namespace

cudaError_t launch_combine_bwd(const Geom& g, const __nv_bfloat16* d_o,
                               const __nv_bfloat16* gc, const __nv_bfloat16* gf,
                               const __half* o_f, const float* oc, void* dgc, void* dgf,
                               __half* dof, float* doc, float* delta, uint32_t* amax,
                               float* gscale, uint32_t* status, cudaStream_t s) {
  auto u4 = [](const void* p) { return reinterpret_cast<const uint4*>(p); };
  // slice maxima first: a few CTAs per SM in total, strided over each slice
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t) * g.BH, s);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const size_t vec = static_cast<size_t>(g.N) * g.D / 8;  // uint4 vectors per slice
  const size_t per_slice_max = (vec + kThreads - 1) / kThreads;
  const size_t want = (static_cast<size_t>(sms) * kAmaxCtasPerSm + g.BH - 1) / g.BH;
  const dim3 agrid(static_cast<unsigned>(want < per_slice_max ? want : per_slice_max), g.BH);
  amax_kernel<<<agrid, kThreads, 0, s>>>(u4(d_o), u4(gf), vec, amax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dim3 grid(g.Nc, g.BH);
  if (g.D == 64)
    combine_bwd_kernel<64><<<grid, kThreads, 0, s>>>(g, u4(d_o), u4(gc), u4(gf), u4(o_f), oc, dgc, dgf,
                                                     reinterpret_cast<uint4*>(dof), doc, delta,
                                                     amax, gscale, status);
  else
    combine_bwd_kernel<128><<<grid, kThreads, 0, s>>>(g, u4(d_o), u4(gc), u4(gf), u4(o_f), oc, dgc,
                                                      dgf, reinterpret_cast<uint4*>(dof), doc,
                                                      delta, amax, gscale, status);
  return cudaGetLastError();
}

}  // namespace vsa

// Backward of the gated combine O = repeat(O_c) (.) G_c + O_f (.) G_f (paper
// notes 关键设计 3; "VSA: Faster Video Diffusion with Trainable Sparse
// Attention", App. B: the coarse output is repeated across its block):
//   dG_c = dO (.) repeat(O_c)          dG_f = dO (.) O_f
//   dO_f = dO (.) G_f (fp16, the tensor-core operand of the fine backward)
//   dO_c[cube] = sum over the cube of dO (.) G_c
//   delta[row] = sum_d dO_f (.) O_f    (the softmax-backward row term of the fine stage)
// HBM-bound: one CTA per (batch, head, cube) reads dO, G_c, G_f (bf16, caller
// layout) and O_f (fp16, cube order) once and writes each output once.
#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 256;

template <int D>
__global__ void __launch_bounds__(kThreads) combine_bwd_kernel(
    Geom g, const uint4* __restrict__ d_o, const uint4* __restrict__ gc,
    const uint4* __restrict__ gf, const uint4* __restrict__ o_f, const float* __restrict__ oc,
    float* __restrict__ dgc, float* __restrict__ dgf, uint4* __restrict__ dof,
    float* __restrict__ doc, float* __restrict__ delta, uint32_t* status) {
  constexpr int VPR = D / 8;              // 8-element vectors per row
  constexpr int GROUPS = kThreads / VPR;  // rows processed side by side
  __shared__ float red[GROUPS][D];
  const int c = blockIdx.x, bh = blockIdx.y;
  const int col = threadIdx.x % VPR, grp = threadIdx.x / VPR;
  const size_t slice = static_cast<size_t>(bh) * g.N;
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
      const float2 raw = make_float2(dd.x * ff.x, dd.y * ff.y);
      bad |= !(fabsf(raw.x) <= 65504.f) || !(fabsf(raw.y) <= 65504.f);
      pof[e] = __floats2half2_rn(raw.x, raw.y);
      const float2 r = __half22float2(pof[e]);  // delta uses the rounded dO_f the MMAs see
      dsum = fmaf(r.x, ofv[2 * e], fmaf(r.y, ofv[2 * e + 1], dsum));
    }
    float4* dc = reinterpret_cast<float4*>(dgc + crow * D + col * 8);
    float4* df = reinterpret_cast<float4*>(dgf + crow * D + col * 8);
    dc[0] = make_float4(vdgc[0], vdgc[1], vdgc[2], vdgc[3]);
    dc[1] = make_float4(vdgc[4], vdgc[5], vdgc[6], vdgc[7]);
    df[0] = make_float4(vdgf[0], vdgf[1], vdgf[2], vdgf[3]);
    df[1] = make_float4(vdgf[4], vdgf[5], vdgf[6], vdgf[7]);
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
                               const __half* o_f, const float* oc, float* dgc, float* dgf,
                               __half* dof, float* doc, float* delta, uint32_t* status,
                               cudaStream_t s) {
  dim3 grid(g.Nc, g.BH);
  auto u4 = [](const void* p) { return reinterpret_cast<const uint4*>(p); };
  if (g.D == 64)
    combine_bwd_kernel<64><<<grid, kThreads, 0, s>>>(g, u4(d_o), u4(gc), u4(gf), u4(o_f), oc, dgc, dgf,
                                                     reinterpret_cast<uint4*>(dof), doc, delta, status);
  else
    combine_bwd_kernel<128><<<grid, kThreads, 0, s>>>(g, u4(d_o), u4(gc), u4(gf), u4(o_f), oc, dgc,
                                                      dgf, reinterpret_cast<uint4*>(dof), doc,
                                                      delta, status);
  return cudaGetLastError();
}

}  // namespace vsa

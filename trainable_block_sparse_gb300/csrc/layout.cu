// Tile / untile and cube mean-pooling ("VSA: Faster Video Diffusion with
// Trainable Sparse Attention", App. B: tiling rearranges tokens between
// sequence and cube order; §2 "Coarse stage": Q_c, K_c, V_c are cube means),
// and the staging of the tensor-core operands as fp16 cube-order copies.
//
// Both kernels are HBM-bound copies: one CTA moves one (batch, head,
// cube) block of 64 rows x D bf16 with 16-byte vector loads and stores.  In
// raster order a cube's rows come in runs of 4 consecutive tokens (512 B or
// 1 KB contiguous for D = 64 or 128); in cube order the block is one
// contiguous 8 or 16 KB span.
#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 256;

template <int D>
__global__ void __launch_bounds__(kThreads) permute_kernel(Geom g, const uint4* __restrict__ in,
                                                           uint4* __restrict__ out, int inverse) {
  constexpr int VPR = D / 8;  // 16-byte vectors per row
  const int c = blockIdx.x, bh = blockIdx.y;
  const size_t slice = static_cast<size_t>(bh) * g.N * VPR;
  for (int v = threadIdx.x; v < kTile * VPR; v += kThreads) {
    const int o = v / VPR, col = v % VPR;
    const size_t cube_pos = slice + static_cast<size_t>(c * kTile + o) * VPR + col;
    const size_t rast_pos = slice + static_cast<size_t>(raster_row(g, c, o)) * VPR + col;
    if (inverse)
      out[rast_pos] = in[cube_pos];
    else
      out[cube_pos] = in[rast_pos];
  }
}

// Cube means of one (batch, head, cube) block, and optionally its fp16
// cube-order staged copy (the tensor-core operand format).  bf16 -> fp16 is
// exact for |x| < 65504 (subnormal below 6.1e-5, absolute error < 3e-8);
// larger or non-finite values set kDevRange in the status word.
template <int D>
__global__ void __launch_bounds__(kThreads) stage_kernel(Geom g, const uint4* __restrict__ in,
                                                         int in_raster, uint4* __restrict__ out16,
                                                         float* __restrict__ pooled,
                                                         uint32_t* status) {
  constexpr int VPR = D / 8;
  constexpr int GROUPS = kThreads / VPR;  // row groups
  __shared__ float red[GROUPS][D];
  const int c = blockIdx.x, bh = blockIdx.y;
  const int col = threadIdx.x % VPR, grp = threadIdx.x / VPR;
  const size_t slice = static_cast<size_t>(bh) * g.N * VPR;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  bool bad = false;
  for (int o = grp; o < kTile; o += GROUPS) {
    const int row = in_raster ? raster_row(g, c, o) : c * kTile + o;
    const uint4 u = in[slice + static_cast<size_t>(row) * VPR + col];
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
    uint4 h;
    __half2* ph = reinterpret_cast<__half2*>(&h);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p[i]);
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
      bad |= !(fabsf(f.x) <= 65504.f) || !(fabsf(f.y) <= 65504.f);
      ph[i] = __floats2half2_rn(f.x, f.y);
    }
    if (out16) out16[slice + static_cast<size_t>(c * kTile + o) * VPR + col] = h;
  }
  if (bad && out16) flag_error(status, kDevRange);
#pragma unroll
  for (int i = 0; i < 8; ++i) red[grp][col * 8 + i] = acc[i];
  __syncthreads();
  if (pooled) {
    for (int d = threadIdx.x; d < D; d += kThreads) {
      float s = 0.f;
#pragma unroll 8
      for (int r = 0; r < GROUPS; ++r) s += red[r][d];
      pooled[(static_cast<size_t>(bh) * g.Nc + c) * D + d] = s * (1.0f / kTile);
    }
  }
}

}  // namespace

cudaError_t launch_permute(const Geom& g, const __nv_bfloat16* in, __nv_bfloat16* out,
                           int inverse, cudaStream_t s) {
  dim3 grid(g.Nc, g.BH);
  if (g.D == 64)
    permute_kernel<64><<<grid, kThreads, 0, s>>>(g, reinterpret_cast<const uint4*>(in),
                                                 reinterpret_cast<uint4*>(out), inverse);
  else
    permute_kernel<128><<<grid, kThreads, 0, s>>>(g, reinterpret_cast<const uint4*>(in),
                                                  reinterpret_cast<uint4*>(out), inverse);
  return cudaGetLastError();
}

cudaError_t launch_stage(const Geom& g, const __nv_bfloat16* in, int in_raster, __half* out16,
                         float* pooled, uint32_t* status, cudaStream_t s) {
  dim3 grid(g.Nc, g.BH);
  const uint4* src = reinterpret_cast<const uint4*>(in);
  uint4* dst = reinterpret_cast<uint4*>(out16);
  if (g.D == 64)
    stage_kernel<64><<<grid, kThreads, 0, s>>>(g, src, in_raster, dst, pooled, status);
  else
    stage_kernel<128><<<grid, kThreads, 0, s>>>(g, src, in_raster, dst, pooled, status);
  return cudaGetLastError();
}

}  // namespace vsa

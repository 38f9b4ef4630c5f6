// Staging of the fine-stage operands as e4m3 (fp8) for the fp8 variant of the
// fine forward: the same cube-order tiles as the fp16 staging ("VSA: Faster
// Video Diffusion with Trainable Sparse Attention", App. B: tiling), half the
// bytes.  The pages fix no precision; this variant trades accuracy for the
// bytes each product reads (a fine-forward step at head_dim 128 reads 32 KB of
// K and V instead of 64 KB).
//
// Each (batch, head) slice of Q, K and V gets its own power-of-two factor
// s = 2^e, chosen so that the slice's largest |x| times s lies in [128, 256)
// (e4m3 holds magnitudes up to 448 and keeps 3 significand bits down to 2^-6):
// x8 = e4m3(x * s), and 1/s is written to scales[bh][tensor] for the
// consumer (a power of two, so scaling adds no rounding).  Two passes:
// slice_amax_kernel (max |x| of each slice, read once), then quantize_kernel
// (read again, write the e4m3 copy and, optionally, the fp32 cube means the
// coarse stage needs).
//
// Layouts (D = 128 only):
//   Q8, K8 : [B*heads*N, 128] bytes, cube order (row c*64 + o of a slice), so a
//            64-row tile is one TMA box of 128-byte rows (K-major operands).
//   V8T    : [B*heads*Nc, 128, 64] bytes: each cube's V transposed, row d holds
//            the cube's 64 keys of channel d, so the P V product reads V as a
//            K-major operand (K = keys) through 64-byte rows.
#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 256;
constexpr int kAmaxCtasPerSm = 4;

// max |x| of every slice of up to three bf16 tensors (blockIdx.z picks one),
// as the bits of a non-negative float, max-reduced into amax[z * BH + bh].
__global__ void __launch_bounds__(kThreads) slice_amax_kernel(const uint4* __restrict__ x0,
                                                              const uint4* __restrict__ x1,
                                                              const uint4* __restrict__ x2,
                                                              size_t vec_per_slice, int bh_total,
                                                              uint32_t* amax) {
  const uint4* x = blockIdx.z == 0 ? x0 : (blockIdx.z == 1 ? x1 : x2);
  const int bh = blockIdx.y;
  const size_t base = static_cast<size_t>(bh) * vec_per_slice;
  float m = 0.f;
  for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < vec_per_slice;
       i += static_cast<size_t>(gridDim.x) * kThreads) {
    const uint4 u = x[base + i];
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(p[e]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ float wmax[kThreads / 32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, wmax[w]);
    atomicMax(amax + static_cast<size_t>(blockIdx.z) * bh_total + bh, __float_as_uint(m));
  }
}

// The power of two s with (slice maximum) * s in [128, 256); a zero or
// non-finite maximum gives s = 1 (non-finite values are flagged when quantized).
__device__ __forceinline__ float fp8_scale_of(uint32_t bits) {
  const int E = static_cast<int>((bits >> 23) & 0xFFu);
  if (bits == 0u || E == 0xFF) return 1.f;
  // maximum in [2^(x-1), 2^x) with x = E - 126 (normal) -> s = 2^(8 - x)
  const int e = E == 0 ? 126 : min(126, max(-126, 8 - (E - 126)));
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// One (batch, head, cube) block of one tensor (blockIdx.z: 0 Q, 1 K, 2 V):
// 64 rows x 128 bf16 -> e4m3 (Q, K row-major, V transposed) and the fp32 cube
// mean.
__global__ void __launch_bounds__(kThreads) quantize_kernel(
    Geom g, const uint4* __restrict__ q, const uint4* __restrict__ k,
    const uint4* __restrict__ v, int in_raster, uint2* __restrict__ q8, uint2* __restrict__ k8,
    uint4* __restrict__ v8t, const uint32_t* __restrict__ amax, float* __restrict__ scales,
    float* pq, float* pk, float* pv, uint32_t* status) {
  constexpr int D = 128, VPR = D / 8, GROUPS = kThreads / VPR;  // 16 groups of 16 threads
  __shared__ float red[GROUPS][D];
  __shared__ float vt[kTile][D + 1];  // V block (fp32, scaled) for the transposed write
  const int c = blockIdx.x, bh = blockIdx.y, z = blockIdx.z;
  const uint4* x = z == 0 ? q : (z == 1 ? k : v);
  float* pooled = z == 0 ? pq : (z == 1 ? pk : pv);
  const float s = fp8_scale_of(amax[static_cast<size_t>(z) * g.BH + bh]);
  if (c == 0 && threadIdx.x == 0) scales[bh * 3 + z] = 1.f / s;
  const int col = threadIdx.x % VPR, grp = threadIdx.x / VPR;
  const size_t slice = static_cast<size_t>(bh) * g.N;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  bool bad = false;
  for (int o = grp; o < kTile; o += GROUPS) {
    const int row = in_raster ? raster_row(g, c, o) : c * kTile + o;
    const uint4 u = x[(slice + row) * VPR + col];
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(p[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      acc[i] += f[i];
      bad |= !isfinite(f[i]);
    }
    if (z < 2) {
      uint2 w;
      w.x = pack_e4m3x4(f[0] * s, f[1] * s, f[2] * s, f[3] * s);
      w.y = pack_e4m3x4(f[4] * s, f[5] * s, f[6] * s, f[7] * s);
      (z == 0 ? q8 : k8)[(slice + static_cast<size_t>(c) * kTile + o) * VPR + col] = w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) vt[o][col * 8 + i] = f[i] * s;
    }
  }
  if (bad) flag_error(status, kDevRange);
#pragma unroll
  for (int i = 0; i < 8; ++i) red[grp][col * 8 + i] = acc[i];
  __syncthreads();
  if (z == 2) {
    // row d of the transposed block: 64 keys = 64 bytes; thread -> (d, 32-key half)
    const int d = threadIdx.x >> 1, h = threadIdx.x & 1;
    uint4* dst = v8t + ((static_cast<size_t>(bh) * g.Nc + c) * D + d) * 4 + 2 * h;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int k0 = 32 * h + 16 * u;
      uint4 w;
      w.x = pack_e4m3x4(vt[k0][d], vt[k0 + 1][d], vt[k0 + 2][d], vt[k0 + 3][d]);
      w.y = pack_e4m3x4(vt[k0 + 4][d], vt[k0 + 5][d], vt[k0 + 6][d], vt[k0 + 7][d]);
      w.z = pack_e4m3x4(vt[k0 + 8][d], vt[k0 + 9][d], vt[k0 + 10][d], vt[k0 + 11][d]);
      w.w = pack_e4m3x4(vt[k0 + 12][d], vt[k0 + 13][d], vt[k0 + 14][d], vt[k0 + 15][d]);
      dst[u] = w;
    }
  }
  if (pooled) {
    for (int d = threadIdx.x; d < D; d += kThreads) {
      float t = 0.f;
#pragma unroll 8
      for (int r = 0; r < GROUPS; ++r) t += red[r][d];
      pooled[(static_cast<size_t>(bh) * g.Nc + c) * D + d] = t * (1.0f / kTile);
    }
  }
}

}  // namespace

cudaError_t launch_stage_fp8(const Geom& g, const __nv_bfloat16* q, const __nv_bfloat16* k,
                             const __nv_bfloat16* v, uint8_t* q8, uint8_t* k8, uint8_t* v8t,
                             float* scales, float* pq, float* pk, float* pv, uint32_t* amax,
                             uint32_t* status, cudaStream_t s) {
  if (g.D != 128) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t) * 3 * g.BH, s);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  auto u4 = [](const void* p) { return reinterpret_cast<const uint4*>(p); };
  const size_t vec = static_cast<size_t>(g.N) * g.D / 8;
  const size_t per_slice_max = (vec + kThreads - 1) / kThreads;
  const size_t want = (static_cast<size_t>(sms) * kAmaxCtasPerSm + 3 * g.BH - 1) / (3 * g.BH);
  const dim3 agrid(static_cast<unsigned>(want < per_slice_max ? want : per_slice_max), g.BH, 3);
  slice_amax_kernel<<<agrid, kThreads, 0, s>>>(u4(q), u4(k), u4(v), vec, g.BH, amax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const dim3 grid(g.Nc, g.BH, 3);
  quantize_kernel<<<grid, kThreads, 0, s>>>(g, u4(q), u4(k), u4(v), g.raster,
                                            reinterpret_cast<uint2*>(q8),
                                            reinterpret_cast<uint2*>(k8),
                                            reinterpret_cast<uint4*>(v8t), amax, scales, pq, pk,
                                            pv, status);
  return cudaGetLastError();
}

}  // namespace vsa

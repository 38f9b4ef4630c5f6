// Coarse stage of VSA ("VSA: Faster Video Diffusion with Trainable Sparse
// Attention", §2 "Coarse stage"; paper notes 关键设计 1): dense attention on
// the pooled (64x shorter) sequence, the row-wise selection of key cubes and
// the mask-to-index conversion, in one kernel; and its backward.
//
// The contraction runs in fp32 on the CUDA cores, not on the tensor cores:
// the selection is an integer decision taken on these logits, and rounding
// the pooled vectors to bf16 or tf32 moves a logit by ~1e-3, the size of the
// smallest gap the selection has to resolve.  In fp32 the error is ~1e-6.
//
// One CTA owns R query cubes of one (batch, head) and streams all key/value
// cubes through shared memory in tiles of 64.
#include <cfloat>

#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kKT = 64;  // key cubes per tile

// Rows [r0, r0+R) of a [rows, D] fp32 matrix into smem [R][D] (zero past `rows`).
template <int D, int R>
__device__ void load_rows(float* dst, const float* src, int r0, int rows) {
  for (int i = threadIdx.x; i < R * D / 4; i += kThreads) {
    const int r = i / (D / 4), c4 = i % (D / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 + r < rows) v = reinterpret_cast<const float4*>(src + static_cast<size_t>(r0 + r) * D)[c4];
    reinterpret_cast<float4*>(dst + r * D)[c4] = v;
  }
}

// Tile of 64 rows starting at j0, stored transposed: dst[d * (kKT+1) + j].
template <int D>
__device__ void load_tile_t(float* dst, const float* src, int j0, int rows) {
  for (int i = threadIdx.x; i < kKT * D / 4; i += kThreads) {
    const int j = i % kKT, c4 = i / kKT;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j0 + j < rows) v = reinterpret_cast<const float4*>(src + static_cast<size_t>(j0 + j) * D)[c4];
    dst[(4 * c4 + 0) * (kKT + 1) + j] = v.x;
    dst[(4 * c4 + 1) * (kKT + 1) + j] = v.y;
    dst[(4 * c4 + 2) * (kKT + 1) + j] = v.z;
    dst[(4 * c4 + 3) * (kKT + 1) + j] = v.w;
  }
}

// Tile of 64 rows starting at j0, row-major dst[j * D + d].
template <int D>
__device__ void load_tile(float* dst, const float* src, int j0, int rows) {
  for (int i = threadIdx.x; i < kKT * D / 4; i += kThreads) {
    const int j = i / (D / 4), c4 = i % (D / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j0 + j < rows) v = reinterpret_cast<const float4*>(src + static_cast<size_t>(j0 + j) * D)[c4];
    reinterpret_cast<float4*>(dst + j * D)[c4] = v;
  }
}

// out[r * ld + j] = mul * dot(A[r, :], Bt[:, j]) for r < R, j < 64.
// Thread (j = tid % 64, g = tid / 64) computes rows g, g+4, ...
template <int D, int R>
__device__ void dots_tile(const float* A, const float* Bt, float* out, int ld, float mul) {
  constexpr int RPT = R / 4;
  const int j = threadIdx.x % kKT, g = threadIdx.x / kKT;
  float acc[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (int d = 0; d < D; d += 4) {
    const float b0 = Bt[(d + 0) * (kKT + 1) + j], b1 = Bt[(d + 1) * (kKT + 1) + j];
    const float b2 = Bt[(d + 2) * (kKT + 1) + j], b3 = Bt[(d + 3) * (kKT + 1) + j];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float4 a = *reinterpret_cast<const float4*>(A + (g + 4 * i) * D + d);
      acc[i] = fmaf(a.x, b0, fmaf(a.y, b1, fmaf(a.z, b2, fmaf(a.w, b3, acc[i]))));
    }
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) out[(g + 4 * i) * ld + j] = acc[i] * mul;
}

// acc[i] += sum_j P[(row_i) * 64 + j] * V[j * D + d], thread (d = tid % D,
// rows tid / D + i * (256 / D)).
template <int D, int R>
__device__ __forceinline__ void accum_tile(float (&acc)[R * D / kThreads], const float* P,
                                           const float* V) {
  constexpr int STEP = kThreads / D;
  constexpr int RPT = R * D / kThreads;
  const int d = threadIdx.x % D, r0 = threadIdx.x / D;
#pragma unroll 8
  for (int j = 0; j < kKT; ++j) {
    const float v = V[j * D + d];
#pragma unroll
    for (int i = 0; i < RPT; ++i) acc[i] = fmaf(P[(r0 + i * STEP) * kKT + j], v, acc[i]);
  }
}

__device__ __forceinline__ void argmax_pair(float& v, int& j) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
    const int j2 = __shfl_xor_sync(0xffffffffu, j, off);
    if (v2 > v || (v2 == v && j2 < j)) {
      v = v2;
      j = j2;
    }
  }
}

struct SelectArgs {
  int mode, topk, kmin, kmax;
  float mass;
};

// Forward: logits, softmax statistics, O_c, selection, ascending index lists.
template <int D, int R>
__global__ void __launch_bounds__(kThreads) coarse_select_kernel(Geom g, SelectArgs sa,
                                                                 const float* __restrict__ qc,
                                                                 const float* __restrict__ kc,
                                                                 const float* __restrict__ vc,
                                                                 float* __restrict__ oc,
                                                                 float* __restrict__ lse_c,
                                                                 int* __restrict__ idx,
                                                                 int* __restrict__ cnt) {
  extern __shared__ __align__(16) float sm[];
  const int Nc = g.Nc, bh = blockIdx.y, r0 = blockIdx.x * R;
  float* Qs = sm;                       // [R][D]
  float* Ts = Qs + R * D;               // key tile (transposed) or value tile
  float* Ps = Ts + D * (kKT + 1);       // [R][64]
  float* rowm = Ps + R * kKT;           // [R]
  float* rowinv = rowm + R;             // [R]
  int* sel = reinterpret_cast<int*>(rowinv + R);  // [R][cap]
  float* Ls = reinterpret_cast<float*>(sel + R * g.cap);  // [R][Nc]
  const size_t base = static_cast<size_t>(bh) * Nc;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  load_rows<D, R>(Qs, qc + base * D, r0, Nc);
  // ---- logits
  for (int j0 = 0; j0 < Nc; j0 += kKT) {
    __syncthreads();
    load_tile_t<D>(Ts, kc + base * D, j0, Nc);
    __syncthreads();
    dots_tile<D, R>(Qs, Ts, Ps, kKT, g.scale);
    __syncthreads();
    for (int i = threadIdx.x; i < R * kKT; i += kThreads) {
      const int r = i / kKT, j = i % kKT;
      if (j0 + j < Nc) Ls[r * Nc + j0 + j] = Ps[i];
    }
  }
  __syncthreads();
  // ---- softmax statistics per row (one warp per row)
  for (int r = warp; r < R; r += kWarps) {
    float m = -FLT_MAX;
    for (int j = lane; j < Nc; j += 32) m = fmaxf(m, Ls[r * Nc + j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float s = 0.f;
    for (int j = lane; j < Nc; j += 32) s += expf(Ls[r * Nc + j] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
      rowm[r] = m;
      rowinv[r] = 1.f / s;
      if (r0 + r < Nc) lse_c[base + r0 + r] = m + logf(s);
    }
  }
  // ---- O_c = A_c V_c
  constexpr int RPT = R * D / kThreads;
  float acc[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < Nc; j0 += kKT) {
    __syncthreads();
    load_tile<D>(Ts, vc + base * D, j0, Nc);
    for (int i = threadIdx.x; i < R * kKT; i += kThreads) {
      const int r = i / kKT, j = i % kKT;
      Ps[i] = (j0 + j < Nc) ? expf(Ls[r * Nc + j0 + j] - rowm[r]) * rowinv[r] : 0.f;
    }
    __syncthreads();
    accum_tile<D, R>(acc, Ps, Ts);
  }
  {
    constexpr int STEP = kThreads / D;
    const int d = threadIdx.x % D, rr = threadIdx.x / D;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = rr + i * STEP;
      if (r0 + r < Nc) oc[(base + r0 + r) * D + d] = acc[i];
    }
  }
  __syncthreads();
  // ---- selection: repeated warp argmax over the row (ties -> lower id)
  const int kmax_eff = min(sa.kmax, Nc);
  const int kmin_eff = min(sa.kmin, kmax_eff);
  for (int r = warp; r < R; r += kWarps) {
    if (r0 + r >= Nc) continue;
    float* L = Ls + r * Nc;
    int* S = sel + r * g.cap;
    int n = 0;
    if (sa.mode == 0) {
      for (; n < sa.topk; ++n) {
        float v = -INFINITY;
        int j = 0x7fffffff;
        for (int t = lane; t < Nc; t += 32)
          if (L[t] > v) { v = L[t]; j = t; }
        argmax_pair(v, j);
        if (lane == 0) { S[n] = j; L[j] = -INFINITY; }
        __syncwarp();
      }
    } else {
      float cum = 0.f;
      int n_raw = 0;
      while (true) {
        float v = -INFINITY;
        int j = 0x7fffffff;
        for (int t = lane; t < Nc; t += 32)
          if (L[t] > v) { v = L[t]; j = t; }
        argmax_pair(v, j);
        if (lane == 0) { S[n] = j; L[j] = -INFINITY; }
        __syncwarp();
        cum += expf(v - rowm[r]) * rowinv[r];
        ++n;
        if (n_raw == 0 && cum >= sa.mass) n_raw = n;
        if ((n >= kmin_eff && n_raw > 0) || n >= kmax_eff) break;
      }
    }
    __syncwarp();
    // ascending order: the rank of each selected id among the selected ones
    int* out = idx + (base + r0 + r) * g.cap;
    for (int e = lane; e < n; e += 32) {
      const int me = S[e];
      int pos = 0;
      for (int f = 0; f < n; ++f) pos += (S[f] < me);
      out[pos] = me;
    }
    for (int e = n + lane; e < g.cap; e += 32) out[e] = -1;
    if (lane == 0) cnt[base + r0 + r] = n;
  }
}

// Backward, row pass: P = exp(L - lse), dA = dO_c V_c^T, dL = P (dA - rowsum(dO_c O_c)),
// written to global; dQ_c = scale * dL K_c.
template <int D, int R>
__global__ void __launch_bounds__(kThreads) coarse_bwd_rows_kernel(
    Geom g, const float* __restrict__ qc, const float* __restrict__ kc,
    const float* __restrict__ vc, const float* __restrict__ oc, const float* __restrict__ lse_c,
    const float* __restrict__ doc, float* __restrict__ prob, float* __restrict__ dlog,
    float* __restrict__ dqc) {
  extern __shared__ __align__(16) float sm[];
  const int Nc = g.Nc, bh = blockIdx.y, r0 = blockIdx.x * R;
  float* Qs = sm;                   // [R][D]
  float* Gs = Qs + R * D;           // dO_c rows [R][D]
  float* Ts = Gs + R * D;           // tile buffer, max(D*(65), 64*D)
  float* Ls = Ts + D * (kKT + 1);   // [R][64] logits -> P
  float* As = Ls + R * kKT;         // [R][64] dA -> dL
  float* rl = As + R * kKT;         // [R] lse
  float* rd = rl + R;               // [R] delta
  const size_t base = static_cast<size_t>(bh) * Nc;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  load_rows<D, R>(Qs, qc + base * D, r0, Nc);
  load_rows<D, R>(Gs, doc + base * D, r0, Nc);
  __syncthreads();
  for (int r = warp; r < R; r += kWarps) {
    float s = 0.f;
    if (r0 + r < Nc) {
      const float* o = oc + (base + r0 + r) * D;
      for (int d = lane; d < D; d += 32) s += Gs[r * D + d] * o[d];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
      rd[r] = s;
      rl[r] = (r0 + r < Nc) ? lse_c[base + r0 + r] : 0.f;
    }
  }
  constexpr int RPT = R * D / kThreads;
  float acc[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < Nc; j0 += kKT) {
    __syncthreads();
    load_tile_t<D>(Ts, kc + base * D, j0, Nc);
    __syncthreads();
    dots_tile<D, R>(Qs, Ts, Ls, kKT, g.scale);
    __syncthreads();
    load_tile_t<D>(Ts, vc + base * D, j0, Nc);
    __syncthreads();
    dots_tile<D, R>(Gs, Ts, As, kKT, 1.f);
    __syncthreads();
    for (int i = threadIdx.x; i < R * kKT; i += kThreads) {
      const int r = i / kKT, j = i % kKT;
      const bool ok = (r0 + r < Nc) && (j0 + j < Nc);
      const float p = ok ? expf(Ls[i] - rl[r]) : 0.f;
      const float dl = p * (As[i] - rd[r]);
      Ls[i] = p;
      As[i] = dl;
      if (ok) {
        prob[(base + r0 + r) * Nc + j0 + j] = p;
        dlog[(base + r0 + r) * Nc + j0 + j] = dl;
      }
    }
    __syncthreads();
    load_tile<D>(Ts, kc + base * D, j0, Nc);
    __syncthreads();
    accum_tile<D, R>(acc, As, Ts);
  }
  constexpr int STEP = kThreads / D;
  const int d = threadIdx.x % D, rr = threadIdx.x / D;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rr + i * STEP;
    if (r0 + r < Nc) dqc[(base + r0 + r) * D + d] = acc[i] * g.scale;
  }
}

// Backward, column pass: dK_c[j] = scale * sum_i dL[i,j] Q_c[i];
// dV_c[j] = sum_i P[i,j] dO_c[i], for R key cubes j per CTA.
template <int D, int R>
__global__ void __launch_bounds__(kThreads) coarse_bwd_cols_kernel(
    Geom g, const float* __restrict__ qc, const float* __restrict__ doc,
    const float* __restrict__ prob, const float* __restrict__ dlog, float* __restrict__ dkc,
    float* __restrict__ dvc) {
  extern __shared__ __align__(16) float sm[];
  const int Nc = g.Nc, bh = blockIdx.y, j0 = blockIdx.x * R;
  float* Qs = sm;               // [64][D] query-cube tile
  float* Gs = Qs + kKT * D;     // [64][D] dO_c tile
  float* Pt = Gs + kKT * D;     // [R][64]  P^T block
  float* Dt = Pt + R * kKT;     // [R][64]  dL^T block
  const size_t base = static_cast<size_t>(bh) * Nc;
  constexpr int RPT = R * D / kThreads;
  float ak[RPT], av[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) ak[i] = av[i] = 0.f;
  for (int i0 = 0; i0 < Nc; i0 += kKT) {
    __syncthreads();
    load_tile<D>(Qs, qc + base * D, i0, Nc);
    load_tile<D>(Gs, doc + base * D, i0, Nc);
    for (int t = threadIdx.x; t < R * kKT; t += kThreads) {
      const int i = t / R, r = t % R;  // consecutive threads read consecutive columns
      const bool ok = (i0 + i < Nc) && (j0 + r < Nc);
      const size_t off = (base + i0 + i) * Nc + j0 + r;
      Pt[r * kKT + i] = ok ? prob[off] : 0.f;
      Dt[r * kKT + i] = ok ? dlog[off] : 0.f;
    }
    __syncthreads();
    accum_tile<D, R>(ak, Dt, Qs);
    accum_tile<D, R>(av, Pt, Gs);
  }
  constexpr int STEP = kThreads / D;
  const int d = threadIdx.x % D, rr = threadIdx.x / D;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rr + i * STEP;
    if (j0 + r < Nc) {
      dkc[(base + j0 + r) * D + d] = ak[i] * g.scale;
      dvc[(base + j0 + r) * D + d] = av[i];
    }
  }
}

template <int D, int R>
size_t select_smem(const Geom& g) {
  return sizeof(float) * (R * D + D * (kKT + 1) + R * kKT + 2 * R) +
         sizeof(int) * R * g.cap + sizeof(float) * static_cast<size_t>(R) * g.Nc;
}

template <int D, int R>
cudaError_t run_select(const Geom& g, SelectArgs sa, const float* qc, const float* kc,
                       const float* vc, float* oc, float* lse_c, int* idx, int* cnt,
                       cudaStream_t s) {
  const size_t smem = select_smem<D, R>(g);
  auto kern = coarse_select_kernel<D, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((g.Nc + R - 1) / R, g.BH);
  kern<<<grid, kThreads, smem, s>>>(g, sa, qc, kc, vc, oc, lse_c, idx, cnt);
  return cudaGetLastError();
}

template <int D>
cudaError_t select_dispatch(const Geom& g, SelectArgs sa, const float* qc, const float* kc,
                            const float* vc, float* oc, float* lse_c, int* idx, int* cnt,
                            cudaStream_t s) {
  constexpr size_t kBudget = 200 * 1024;
  if (select_smem<D, 16>(g) <= kBudget)
    return run_select<D, 16>(g, sa, qc, kc, vc, oc, lse_c, idx, cnt, s);
  if (select_smem<D, 8>(g) <= kBudget)
    return run_select<D, 8>(g, sa, qc, kc, vc, oc, lse_c, idx, cnt, s);
  return run_select<D, 4>(g, sa, qc, kc, vc, oc, lse_c, idx, cnt, s);
}

template <int D>
cudaError_t coarse_bwd_impl(const Geom& g, const float* qc, const float* kc, const float* vc,
                            const float* oc, const float* lse_c, const float* doc, float* dqc,
                            float* dkc, float* dvc, const Workspace& ws, cudaStream_t s) {
  constexpr int R = 16;
  {
    const size_t smem = sizeof(float) * (2 * R * D + D * (kKT + 1) + 2 * R * kKT + 2 * R);
    auto kern = coarse_bwd_rows_kernel<D, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<dim3((g.Nc + R - 1) / R, g.BH), kThreads, smem, s>>>(g, qc, kc, vc, oc, lse_c, doc,
                                                                 ws.cprob, ws.cgrad, dqc);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const size_t smem = sizeof(float) * (2 * kKT * D + 2 * R * kKT);
    auto kern = coarse_bwd_cols_kernel<D, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<dim3((g.Nc + R - 1) / R, g.BH), kThreads, smem, s>>>(g, qc, doc, ws.cprob, ws.cgrad,
                                                                 dkc, dvc);
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_coarse_select(const Geom& g, int mode, int topk, float mass, int kmin,
                                 int kmax, const float* qc, const float* kc, const float* vc,
                                 float* oc, float* lse_c, int* idx, int* cnt, cudaStream_t s) {
  SelectArgs sa{mode, topk, kmin, kmax, mass};
  if (g.D == 64) return select_dispatch<64>(g, sa, qc, kc, vc, oc, lse_c, idx, cnt, s);
  return select_dispatch<128>(g, sa, qc, kc, vc, oc, lse_c, idx, cnt, s);
}

cudaError_t launch_coarse_bwd(const Geom& g, const float* qc, const float* kc, const float* vc,
                              const float* oc, const float* lse_c, const float* doc,
                              float* dqc, float* dkc, float* dvc, const Workspace& ws,
                              cudaStream_t s) {
  if (g.D == 64) return coarse_bwd_impl<64>(g, qc, kc, vc, oc, lse_c, doc, dqc, dkc, dvc, ws, s);
  return coarse_bwd_impl<128>(g, qc, kc, vc, oc, lse_c, doc, dqc, dkc, dvc, ws, s);
}

}  // namespace vsa

// Coarse stage of VSA ("VSA: Faster Video Diffusion with Trainable Sparse
// Attention", §2 "Coarse stage"; paper notes 关键设计 1 and 损失函数/训练策略):
// dense attention on the pooled (64x shorter) sequence, the row-wise selection
// of key cubes and the mask-to-index conversion; and its backward.
//
// All contractions are fp32 on the CUDA cores, not on the tensor cores: the
// selection is an integer decision taken on these logits, and rounding the
// pooled vectors to bf16 or tf32 moves a logit by ~1e-3, the size of the
// smallest gap the selection has to resolve.  In fp32 the error is ~1e-6.
//
// Structure (per (batch, head) slice, Nc cubes):
//   forward : L = scale Q_c K_c^T            (batched fp32 GEMM)
//             softmax statistics, A_c, top-K / mass selection, index lists
//                                            (one fused kernel, warp per row)
//             O_c = A_c V_c                  (batched fp32 GEMM)
//   backward: A_c = exp(scale Q_c K_c^T - lse)            (GEMM, fused exp)
//             dL  = A_c (.) (dO_c V_c^T - rowsum(dO_c O_c)) (GEMM, fused)
//             dQ_c = scale dL K_c, dK_c = scale dL^T Q_c, dV_c = A_c^T dO_c
// The GEMM is register-tiled: a CTA computes a 128 x 64 tile with 256
// threads, 8 x 4 outputs per thread, operands staged k-major in shared memory
// (double-buffered through registers), so each 16-wide k step costs 3
// vector shared loads per 32 FMAs.
#include <cfloat>

#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kBM = 128, kBN = 64, kBK = 16;
constexpr int kGemmThreads = 256;

enum Epi { kEpiStore = 0, kEpiExpLse = 1, kEpiDLogit = 2 };

struct GemmArgs {
  int M, N, K;
  const float* A; long long lda, strideA;  // element strides; batch stride
  const float* B; long long ldb, strideB;
  float* C; long long ldc, strideC;
  float alpha;
  // epilogue operands (per batch, row-major M x N like C; row vectors of M)
  const float* rowvec; long long strideRow;  // lse (kEpiExpLse) or delta (kEpiDLogit)
  const float* P; long long ldp, strideP;    // probabilities (kEpiDLogit)
};

// C[b] = alpha * op(A[b]) op(B[b]) with op(A) M x K, op(B) K x N.
// TA: A is stored K x M (so op(A) = A^T); otherwise M x K.  TB: B is stored
// N x K; otherwise K x N.  All row-major.
template <bool TA, bool TB, int EPI>
__global__ void __launch_bounds__(kGemmThreads) sgemm_kernel(GemmArgs g) {
  __shared__ __align__(16) float As[2][kBK][kBM + 4];
  __shared__ __align__(16) float Bs[2][kBK][kBN + 4];
  const int b = blockIdx.z;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const float* A = g.A + b * g.strideA;
  const float* B = g.B + b * g.strideB;
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;  // 16 x 16 threads; outputs rows ty*8.., cols tx*4..

  // per-thread load slots: A tile 128 x 16 = 2048 values = 8 per thread,
  // B tile 16 x 64 = 1024 values = 4 per thread
  float ra[8], rb[4];
  auto load_a = [&](int k0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = tid + i * kGemmThreads;  // 0..2047
      int m, k;
      if (TA) { k = e / kBM; m = e % kBM; }  // contiguous along m
      else    { m = e / kBK; k = e % kBK; }  // contiguous along k
      const int gm = m0 + m, gk = k0 + k;
      float v = 0.f;
      if (gm < g.M && gk < g.K) v = TA ? A[gk * g.lda + gm] : A[gm * g.lda + gk];
      ra[i] = v;
    }
  };
  auto store_a = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = tid + i * kGemmThreads;
      int m, k;
      if (TA) { k = e / kBM; m = e % kBM; }
      else    { m = e / kBK; k = e % kBK; }
      As[buf][k][m] = ra[i];
    }
  };
  auto load_b = [&](int k0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + i * kGemmThreads;  // 0..1023
      int n, k;
      if (TB) { n = e / kBK; k = e % kBK; }  // contiguous along k
      else    { k = e / kBN; n = e % kBN; }  // contiguous along n
      const int gn = n0 + n, gk = k0 + k;
      float v = 0.f;
      if (gn < g.N && gk < g.K) v = TB ? B[gn * g.ldb + gk] : B[gk * g.ldb + gn];
      rb[i] = v;
    }
  };
  auto store_b = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + i * kGemmThreads;
      int n, k;
      if (TB) { n = e / kBK; k = e % kBK; }
      else    { k = e / kBN; n = e % kBN; }
      Bs[buf][k][n] = rb[i];
    }
  };

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  const int nk = (g.K + kBK - 1) / kBK;
  load_a(0);
  load_b(0);
  store_a(0);
  store_b(0);
  __syncthreads();
  for (int t = 0; t < nk; ++t) {
    const int cur = t & 1;
    if (t + 1 < nk) {
      load_a((t + 1) * kBK);
      load_b((t + 1) * kBK);
    }
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 8 + 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[cur][k][tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bw[j], acc[i][j]);
    }
    if (t + 1 < nk) {
      store_a(cur ^ 1);
      store_b(cur ^ 1);
    }
    __syncthreads();
  }

  float* C = g.C + b * g.strideC;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + ty * 8 + i;
    if (gm >= g.M) continue;
    float rv = 0.f;
    if (EPI != kEpiStore) rv = g.rowvec[b * g.strideRow + gm];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= g.N) continue;
      float v = g.alpha * acc[i][j];
      if (EPI == kEpiExpLse) v = expf(v - rv);
      if (EPI == kEpiDLogit) v = g.P[b * g.strideP + gm * g.ldp + gn] * (v - rv);
      C[gm * g.ldc + gn] = v;
    }
  }
}

template <bool TA, bool TB, int EPI>
cudaError_t sgemm(const GemmArgs& a, int batch, cudaStream_t s) {
  dim3 grid((a.N + kBN - 1) / kBN, (a.M + kBM - 1) / kBM, batch);
  sgemm_kernel<TA, TB, EPI><<<grid, kGemmThreads, 0, s>>>(a);
  return cudaGetLastError();
}

constexpr int kSelThreads = 256;

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

// One warp per query cube: softmax statistics of its logits row, the row of
// A_c written in place of the logits, the selection by repeated warp argmax
// (ties go to the lower cube id), and the ascending index list.
__global__ void __launch_bounds__(kSelThreads) select_kernel(Geom g, SelectArgs sa, int rows_per_cta,
                                                             float* __restrict__ logits,
                                                             float* __restrict__ lse_c,
                                                             int* __restrict__ idx,
                                                             int* __restrict__ cnt) {
  extern __shared__ float sel_smem[];
  const int Nc = g.Nc, bh = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row = blockIdx.x * rows_per_cta + warp;
  if (warp >= rows_per_cta || row >= Nc) return;
  float* Lsm = sel_smem + static_cast<size_t>(warp) * (Nc + g.cap);
  int* S = reinterpret_cast<int*>(Lsm + Nc);
  float* Lg = logits + (static_cast<size_t>(bh) * Nc + row) * Nc;
  float m = -FLT_MAX;
  for (int j = lane; j < Nc; j += 32) {
    const float v = Lg[j];
    Lsm[j] = v;
    m = fmaxf(m, v);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float z = 0.f;
  for (int j = lane; j < Nc; j += 32) z += expf(Lsm[j] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  const float inv = 1.f / z;
  for (int j = lane; j < Nc; j += 32) Lg[j] = expf(Lsm[j] - m) * inv;  // A_c row
  if (lane == 0) lse_c[static_cast<size_t>(bh) * Nc + row] = m + logf(z);
  __syncwarp();

  const int kmax_eff = min(sa.kmax, Nc);
  const int kmin_eff = min(sa.kmin, kmax_eff);
  const int want = sa.mode == 0 ? sa.topk : kmax_eff;
  int n = 0, n_raw = 0;
  float cum = 0.f;
  while (n < want) {
    float v = -INFINITY;
    int j = 0x7fffffff;
    for (int t = lane; t < Nc; t += 32)
      if (Lsm[t] > v) {
        v = Lsm[t];
        j = t;
      }
    argmax_pair(v, j);
    if (j >= Nc) break;  // no finite entry left (non-finite logits)
    if (lane == 0) {
      S[n] = j;
      Lsm[j] = -INFINITY;
    }
    __syncwarp();
    ++n;
    if (sa.mode != 0) {
      cum += expf(v - m) * inv;
      if (n_raw == 0 && cum >= sa.mass) n_raw = n;
      if (n >= kmin_eff && n_raw > 0) break;
    }
  }
  __syncwarp();
  int* out = idx + (static_cast<size_t>(bh) * Nc + row) * g.cap;
  for (int e = lane; e < n; e += 32) {
    const int me = S[e];
    int pos = 0;
    for (int f = 0; f < n; ++f) pos += (S[f] < me);
    out[pos] = me;
  }
  for (int e = n + lane; e < g.cap; e += 32) out[e] = -1;
  if (lane == 0) cnt[static_cast<size_t>(bh) * Nc + row] = n;
}

// delta_c[row] = sum_d dO_c[row, d] * O_c[row, d], one warp per row.
__global__ void rowdot_kernel(int rows, int D, const float* __restrict__ a,
                              const float* __restrict__ b, float* __restrict__ out) {
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  float s = 0.f;
  for (int d = lane; d < D; d += 32) s += a[static_cast<size_t>(row) * D + d] * b[static_cast<size_t>(row) * D + d];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) out[row] = s;
}

GemmArgs gemm_args(const Geom& g, int M, int N, int K, const float* A, long long lda, long long sA,
                   const float* B, long long ldb, long long sB, float* C, long long ldc,
                   long long sC, float alpha) {
  GemmArgs a{};
  a.M = M; a.N = N; a.K = K;
  a.A = A; a.lda = lda; a.strideA = sA;
  a.B = B; a.ldb = ldb; a.strideB = sB;
  a.C = C; a.ldc = ldc; a.strideC = sC;
  a.alpha = alpha;
  (void)g;
  return a;
}

}  // namespace

cudaError_t launch_coarse_select(const Geom& g, int mode, int topk, float mass, int kmin,
                                 int kmax, const float* qc, const float* kc, const float* vc,
                                 float* logits, float* oc, float* lse_c, int* idx, int* cnt,
                                 cudaStream_t s) {
  const long long Nc = g.Nc, D = g.D, NN = Nc * Nc, ND = Nc * D;
  cudaError_t e;
  // L = scale * Q_c K_c^T
  GemmArgs a = gemm_args(g, g.Nc, g.Nc, g.D, qc, D, ND, kc, D, ND, logits, Nc, NN, g.scale);
  if ((e = sgemm<false, true, kEpiStore>(a, g.BH, s)) != cudaSuccess) return e;
  // softmax, selection and index lists; A_c replaces the logits
  const size_t per_row = sizeof(float) * (static_cast<size_t>(g.Nc) + g.cap);
  int rows = static_cast<int>((160 * 1024) / per_row);
  rows = rows < 1 ? 1 : (rows > 8 ? 8 : rows);
  const size_t smem = per_row * rows;
  if ((e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem))) != cudaSuccess)
    return e;
  SelectArgs sa{mode, topk, kmin, kmax, mass};
  select_kernel<<<dim3((g.Nc + rows - 1) / rows, g.BH), kSelThreads, smem, s>>>(
      g, sa, rows, logits, lse_c, idx, cnt);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // O_c = A_c V_c
  a = gemm_args(g, g.Nc, g.D, g.Nc, logits, Nc, NN, vc, D, ND, oc, D, ND, 1.f);
  return sgemm<false, false, kEpiStore>(a, g.BH, s);
}

cudaError_t launch_coarse_bwd(const Geom& g, const float* qc, const float* kc, const float* vc,
                              const float* oc, const float* lse_c, const float* doc,
                              float* dqc, float* dkc, float* dvc, const Workspace& ws,
                              cudaStream_t s) {
  const long long Nc = g.Nc, D = g.D, NN = Nc * Nc, ND = Nc * D;
  cudaError_t e;
  const int rows = g.BH * g.Nc;
  rowdot_kernel<<<(rows + 7) / 8, 256, 0, s>>>(rows, g.D, doc, oc, ws.cdelta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // A_c = exp(scale Q_c K_c^T - lse_c)
  GemmArgs a = gemm_args(g, g.Nc, g.Nc, g.D, qc, D, ND, kc, D, ND, ws.cprob, Nc, NN, g.scale);
  a.rowvec = lse_c;
  a.strideRow = Nc;
  if ((e = sgemm<false, true, kEpiExpLse>(a, g.BH, s)) != cudaSuccess) return e;
  // dL = A_c (.) (dO_c V_c^T - delta_c)
  a = gemm_args(g, g.Nc, g.Nc, g.D, doc, D, ND, vc, D, ND, ws.cgrad, Nc, NN, 1.f);
  a.rowvec = ws.cdelta;
  a.strideRow = Nc;
  a.P = ws.cprob;
  a.ldp = Nc;
  a.strideP = NN;
  if ((e = sgemm<false, true, kEpiDLogit>(a, g.BH, s)) != cudaSuccess) return e;
  // dQ_c = scale dL K_c
  a = gemm_args(g, g.Nc, g.D, g.Nc, ws.cgrad, Nc, NN, kc, D, ND, dqc, D, ND, g.scale);
  if ((e = sgemm<false, false, kEpiStore>(a, g.BH, s)) != cudaSuccess) return e;
  // dK_c = scale dL^T Q_c
  a = gemm_args(g, g.Nc, g.D, g.Nc, ws.cgrad, Nc, NN, qc, D, ND, dkc, D, ND, g.scale);
  if ((e = sgemm<true, false, kEpiStore>(a, g.BH, s)) != cudaSuccess) return e;
  // dV_c = A_c^T dO_c
  a = gemm_args(g, g.Nc, g.D, g.Nc, ws.cprob, Nc, NN, doc, D, ND, dvc, D, ND, 1.f);
  return sgemm<true, false, kEpiStore>(a, g.BH, s);
}

}  // namespace vsa

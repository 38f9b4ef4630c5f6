// Coarse stage of VSA ("VSA: Faster Video Diffusion with Trainable Sparse
// Attention", §2 "Coarse stage"; paper notes 关键设计 1 and 损失函数/训练策略):
// dense attention on the pooled (64x shorter) sequence, the row-wise selection
// of key cubes and the mask-to-index conversion; and its backward.
//
// The selection is an integer decision taken on the logits, so their
// contraction keeps fp32 accuracy: it runs on the tensor cores as
// error-compensated tf32 products (each operand split into a tf32 pair
// hi + lo, three products per step; tgemm.cu), about 1e-6 relative, where a
// single bf16 or tf32 product would move a logit by ~1e-3, the size of the
// smallest gap the selection has to resolve.  The other products decide
// nothing and run as plain tf32 (operands rounded to tf32, relative error
// 2^-11 per element): O_c, which reaches O through a gate and a bf16
// rounding, and the backward, whose gradients reach dq, dk, dv divided by 64.
//
// Structure (per (batch, head) slice, Nc cubes; "pair" = tf32 hi/lo pair):
//   forward : L = scale Q_c K_c^T                   (pair GEMM -> L, fp32)
//             softmax statistics, A_c, top-K / mass selection, index lists
//                                                   (one kernel, warp per row;
//                                                    A_c rounded to tf32)
//             O_c = A_c V_c                         (plain tf32 GEMM)
//   backward: P  = exp(scale Q_c K_c^T - lse),
//             dL = P (.) (dO_c V_c^T - rowsum(dO_c O_c))
//                 (dual GEMM, query-major tiles -> dL, dL^T and P^T rounded
//                  to tf32; P is never stored in fp32)
//             dQ_c = scale dL K_c, dK_c = scale dL^T Q_c, dV_c = P^T dO_c
#include <cfloat>

#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

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

// exp(v - m) of the softmax sums and A_c, as 2^((v - m) log2 e) on the
// hardware exponential (about 2 ulp; A_c is then rounded to tf32, 2^-11).
// Both selection kernels use it, in the same summation order, so their A_c
// and lse_c agree bit for bit.  (The mass rule's running sum keeps expf.)
__device__ __forceinline__ float softmax_term(float v, float m) {
  return ex2_approx((v - m) * 1.4426950408889634f);
}

struct SelectArgs {
  int mode, topk, kmin, kmax;
  float mass;
};

// One warp per query cube: softmax statistics of its logits row (row stride
// ldc), its row of A_c rounded to tf32 (ach; row stride ldc), the selection by repeated
// warp argmax (ties go to the lower cube id), and the ascending index list.
__global__ void __launch_bounds__(kSelThreads) select_kernel(Geom g, SelectArgs sa, int rows_per_cta,
                                                             const float* __restrict__ logits,
                                                             float* __restrict__ ach, int ldc,
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
  const size_t arow = (static_cast<size_t>(bh) * Nc + row) * ldc;  // logits and A_c rows
  const float* Lg = logits + arow;
  float m = -FLT_MAX;
  for (int j = lane; j < Nc; j += 32) {
    const float v = Lg[j];
    Lsm[j] = v;
    m = fmaxf(m, v);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float z = 0.f;
  for (int j = lane; j < Nc; j += 32) z += softmax_term(Lsm[j], m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  const float inv = 1.f / z;
  for (int j = lane; j < Nc; j += 32) {  // A_c row
    ach[arow + j] = round_tf32(softmax_term(Lsm[j], m) * inv);
  }
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

// The same computation with the row in registers (lane l holds columns
// l, l + 32, ...; kPer * 32 >= Nc) and the selection by threshold instead of
// repeated argmax: the K-th largest logit is found by bisection on its
// order-preserving 32-bit key (count of keys >= mid, one warp reduction per
// halving, early exit when exactly K keys lie above), then the chosen columns
// are written in ascending order by ballots over the register rows, equal
// keys at the threshold going to the lower cube ids.  The mass rule ranks the
// kmax largest candidates and sums their probabilities in descending order,
// as the argmax loop did, so lists, A_c and lse_c are bit-identical to
// select_kernel's.
__device__ __forceinline__ uint32_t order_key(float v) {
  // v > -inf and not NaN -> a key >= 1 that orders like v; others -> 0
  const uint32_t u = v == 0.f ? 0u : __float_as_uint(v);  // -0 and +0 compare equal
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return v > -INFINITY ? k : 0u;
}

// Per-warp shared scratch of the mass rule (kmax <= 64): candidate columns in
// ascending order, their keys, their descending ranks, the columns by rank.
// Then the row's threshold candidates (below).
constexpr int kCand = 256;  // candidates held by a warp, kCand / 32 per lane
struct MassScratch {
  int ci[64];
  uint32_t ck[64];
  int rk[64];
  int cr[64];
  uint32_t cand_key[kCand];
  int cand_col[kCand];
};

// Selection of one row held in registers by one warp (lane l holds columns
// l, l + 32, ...; v[i] = -inf past Nc): the top-K by bisection on the order
// key, or the mass rule over the kmax candidates; writes the ascending list
// (-1 padded to the capacity) and the count.  Lrow: the row's logits (global
// or shared memory) for the mass rule's probabilities, m and inv its softmax
// maximum and 1 / sum.
template <int kPer>
__device__ __forceinline__ void select_row(const Geom& g, const SelectArgs& sa,
                                           const float (&v)[kPer], float m, float inv,
                                           const float* Lrow, int* out, int* cnt_out,
                                           MassScratch& ms) {
  constexpr uint32_t kFull = 0xffffffffu;
  const int Nc = g.Nc;
  const int lane = threadIdx.x % 32;
  uint32_t key[kPer];
  uint32_t kmin_l = 0xffffffffu, kmax_l = 0u, k2_l = 0u;  // k2_l: the lane's second largest
  int nvalid = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    key[i] = order_key(v[i]);  // 0 past the row (v = -inf there)
    if (key[i]) {
      kmin_l = min(kmin_l, key[i]);
      k2_l = max(k2_l, min(kmax_l, key[i]));
      kmax_l = max(kmax_l, key[i]);
      ++nvalid;
    }
  }
  nvalid = __reduce_add_sync(kFull, nvalid);
  const int kmax_eff = min(sa.kmax, Nc);
  const int kmin_eff = min(sa.kmin, kmax_eff);
  const int want = sa.mode == 0 ? sa.topk : kmax_eff;
  const int K = min(want, nvalid);
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t t = 1u;  // the K-th largest key (or a key with exactly K keys at or above it)
  // Candidates: when the start lo below already leaves at most kCand keys at
  // or above it, those keys (every key the threshold search and the
  // selection can touch, since both only look at keys >= lo) are compacted
  // into shared memory in ascending column order, and the search and the
  // selection run over kCand / 32 slots a lane instead of the kPer-wide row.
  // The threshold and the chosen set are the same either way.  (Rows of
  // more than 36 x 32 cubes skip it: their registers are taken.)
  constexpr int kSlots = kCand / 32;
  constexpr bool kUseCand = kPer <= 36;
  bool cand = false;
  int ncand = 0;
  uint32_t ck[kSlots];
  if (K > 0) {
    uint32_t lo = __reduce_min_sync(kFull, kmin_l), hi = __reduce_max_sync(kFull, kmax_l);
    // When every lane holds r = ceil(K / 32) <= 2 valid keys, the smallest of
    // the lanes' r-th largest keys has at least 32 r >= K keys at or above
    // it: a tighter start.
    bool tight = false;
    if (K <= 32 && nvalid >= 32 && __all_sync(kFull, kmax_l != 0u)) {
      lo = max(lo, __reduce_min_sync(kFull, kmax_l));
      tight = true;
    } else if (K <= 64 && nvalid >= 64 && __all_sync(kFull, k2_l != 0u)) {
      lo = max(lo, __reduce_min_sync(kFull, k2_l));
      tight = true;
    }
    if (kUseCand && tight) {
      int c = 0;
#pragma unroll
      for (int i = 0; i < kPer; ++i) c += key[i] >= lo;
      ncand = __reduce_add_sync(kFull, c);
      cand = ncand <= kCand;
    }
    if (cand) {
      int base = 0;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const bool in = key[i] >= lo;
        const uint32_t b = __ballot_sync(kFull, in);
        if (in) {
          const int p = base + __popc(b & lt_mask);
          ms.cand_key[p] = key[i];
          ms.cand_col[p] = 32 * i + lane;
        }
        base += __popc(b);
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < kSlots; ++j) {
        const int p = 32 * j + lane;
        ck[j] = p < ncand ? ms.cand_key[p] : 0u;  // 0: below every valid key
      }
    }
    // invariant: count(key >= lo) >= K; the answer lies in [lo, hi]
    while (lo < hi) {
      const uint32_t mid = lo + (hi - lo + 1) / 2;
      int c = 0;
      if (cand) {
#pragma unroll
        for (int j = 0; j < kSlots; ++j) c += ck[j] >= mid;
      } else {
#pragma unroll
        for (int i = 0; i < kPer; ++i) c += key[i] >= mid;
      }
      c = __reduce_add_sync(kFull, c);
      if (c == K) { lo = mid; break; }
      if (c > K) lo = mid;
      else hi = mid - 1;
    }
    t = lo;
  }
  int n_gt = 0;
  if (cand) {
#pragma unroll
    for (int j = 0; j < kSlots; ++j) n_gt += ck[j] > t;
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) n_gt += key[i] > t;
  }
  n_gt = __reduce_add_sync(kFull, n_gt);
  const int need_eq = K - n_gt;  // keys equal to t to take, lowest columns first
  // the K chosen columns in ascending order
  int* dst = sa.mode == 0 ? out : ms.ci;
  int nout = 0, eq_seen = 0;
  if (cand) {
    // candidate p holds the p-th smallest candidate column
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      if (32 * j >= ncand) break;
      const uint32_t kk = ck[j];
      const bool eq = kk == t;
      const uint32_t beq = __ballot_sync(kFull, eq);
      const bool sel = kk > t || (eq && eq_seen + __popc(beq & lt_mask) < need_eq);
      eq_seen += __popc(beq);
      const uint32_t bsel = __ballot_sync(kFull, sel);
      if (sel) {
        const int pos = nout + __popc(bsel & lt_mask);
        dst[pos] = ms.cand_col[32 * j + lane];
        if (sa.mode != 0) ms.ck[pos] = kk;
      }
      nout += __popc(bsel);
    }
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const bool eq = K > 0 && key[i] == t;
      const uint32_t beq = __ballot_sync(kFull, eq);
      const bool sel =
          K > 0 && (key[i] > t || (eq && eq_seen + __popc(beq & lt_mask) < need_eq));
      eq_seen += __popc(beq);
      const uint32_t bsel = __ballot_sync(kFull, sel);
      if (sel) {
        const int pos = nout + __popc(bsel & lt_mask);
        dst[pos] = 32 * i + lane;
        if (sa.mode != 0) ms.ck[pos] = key[i];
      }
      nout += __popc(bsel);
    }
  }
  int n = K;
  if (sa.mode != 0) {
    // mass rule over the K (<= 64) candidates: descending rank (larger key
    // first, the lower column on ties), then the probabilities summed in
    // rank order by one lane, as the argmax loop summed them
    __syncwarp();
    for (int c = lane; c < K; c += 32) {
      const uint32_t kc = ms.ck[c];
      int r = 0;
      for (int d = 0; d < K; ++d) {
        const uint32_t kd = ms.ck[d];
        r += kd > kc || (kd == kc && d < c);
      }
      ms.rk[c] = r;
      ms.cr[r] = ms.ci[c];
    }
    __syncwarp();
    int nn = 0;
    if (lane == 0) {
      float cum = 0.f;
      int n_raw = 0;
      for (int r = 0; r < K; ++r) {
        cum += expf(Lrow[ms.cr[r]] - m) * inv;
        nn = r + 1;
        if (n_raw == 0 && cum >= sa.mass) n_raw = nn;
        if (nn >= kmin_eff && n_raw > 0) break;
      }
    }
    n = __shfl_sync(kFull, nn, 0);
    // the n highest-ranked candidates, in ascending column order
    int nsel = 0;
    for (int c0 = 0; c0 < K; c0 += 32) {
      const int c = c0 + lane;
      const bool sel = c < K && ms.rk[c] < n;
      const uint32_t bsel = __ballot_sync(kFull, sel);
      if (sel) out[nsel + __popc(bsel & lt_mask)] = ms.ci[c];
      nsel += __popc(bsel);
    }
  }
  for (int e2 = n + lane; e2 < g.cap; e2 += 32) out[e2] = -1;
  if (lane == 0) *cnt_out = n;
}

template <int kPer>
__global__ void __launch_bounds__(kSelThreads) select_reg_kernel(Geom g, SelectArgs sa,
                                                                 const float* __restrict__ logits,
                                                                 float* __restrict__ ach, int ldc,
                                                                 float* __restrict__ lse_c,
                                                                 int* __restrict__ idx,
                                                                 int* __restrict__ cnt) {
  constexpr int kWarps = kSelThreads / 32;
  __shared__ MassScratch s_mass[kWarps];
  constexpr uint32_t kFull = 0xffffffffu;
  const int Nc = g.Nc, bh = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row = blockIdx.x * kWarps + warp;
  if (row >= Nc) return;
  const size_t arow = (static_cast<size_t>(bh) * Nc + row) * ldc;
  const float* Lg = logits + arow;
  float v[kPer];  // -inf past the row: no term in the max, exp gives 0, order key 0
  float m = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = 32 * i + lane;
    v[i] = j < Nc ? Lg[j] : -INFINITY;
    m = fmaxf(m, v[i]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  float e[kPer];
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    e[i] = softmax_term(v[i], m);
    z += e[i];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(kFull, z, off);
  const float inv = 1.f / z;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {  // A_c row
    const int j = 32 * i + lane;
    if (j < Nc) {
      ach[arow + j] = round_tf32(e[i] * inv);
    }
  }
  if (lane == 0) lse_c[static_cast<size_t>(bh) * Nc + row] = m + logf(z);
  const size_t lrow = static_cast<size_t>(bh) * Nc + row;
  select_row<kPer>(g, sa, v, m, inv, Lg, idx + lrow * g.cap, cnt + lrow, s_mass[warp]);
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

int ldc_of(const Geom& g) { return (g.Nc + 3) & ~3; }

TgemmOperand pair(const float* hi, const float* lo, int ld, long long stride) {
  return TgemmOperand{hi, lo, ld, stride};
}

TgemmArgs gemm(const Geom& g, int M, int N, int K, float alpha) {
  TgemmArgs a{};
  a.batch = g.BH;
  a.M = M;
  a.N = N;
  a.K = K;
  a.mode = kTgScale;
  a.alpha = alpha;
  return a;
}

}  // namespace

cudaError_t launch_coarse_logits_select(const Geom& g, int mode, int topk, float mass, int kmin,
                                        int kmax, const float* qc, const float* kc, float* lse_c,
                                        int* idx, int* cnt, const Workspace& ws, cudaStream_t s) {
  const int Nc = g.Nc, D = g.D, ldc = ldc_of(g);
  const long long ND = static_cast<long long>(Nc) * D, NC = static_cast<long long>(Nc) * ldc;
  cudaError_t e;
  // operand pairs Q_c, K_c ([Nc, D]) as tf32 hi + lo
  {
    const SplitSpec sp[2] = {{qc, D, ND, Nc, D, ws.qh, ws.ql, D, ND, false},
                             {kc, D, ND, Nc, D, ws.kh, ws.kl, D, ND, false}};
    if ((e = launch_split_tf32(sp, 2, g.BH, s))) return e;
  }
  // L = scale Q_c K_c^T
  TgemmArgs a = gemm(g, Nc, Nc, D, g.scale);
  a.out = ws.clogit;
  a.out_ld = ldc;
  a.out_stride = NC;
  if ((e = launch_tgemm(a, pair(ws.qh, ws.ql, D, ND), pair(ws.kh, ws.kl, D, ND), ws.status, s)))
    return e;
  // softmax, selection and index lists; A_c rounded to tf32
  const size_t per_row = sizeof(float) * (static_cast<size_t>(Nc) + g.cap);
  int rows = static_cast<int>((160 * 1024) / per_row);
  rows = rows < 1 ? 1 : (rows > 8 ? 8 : rows);
  const size_t smem = per_row * rows;
  if ((e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem))) != cudaSuccess)
    return e;
  SelectArgs sa{mode, topk, kmin, kmax, mass};
  // rows in registers when they fit (and the mass rule's candidates in 64 slots)
  const dim3 rgrid((Nc + kSelThreads / 32 - 1) / (kSelThreads / 32), g.BH);
  const bool reg_ok = mode == 0 || (kmax < Nc ? kmax : Nc) <= 64;
  if (reg_ok && Nc <= 8 * 32) {
    select_reg_kernel<8><<<rgrid, kSelThreads, 0, s>>>(g, sa, ws.clogit, ws.ach, ldc, lse_c, idx, cnt);
  } else if (reg_ok && Nc <= 16 * 32) {
    select_reg_kernel<16><<<rgrid, kSelThreads, 0, s>>>(g, sa, ws.clogit, ws.ach, ldc, lse_c, idx, cnt);
  } else if (reg_ok && Nc <= 36 * 32) {
    select_reg_kernel<36><<<rgrid, kSelThreads, 0, s>>>(g, sa, ws.clogit, ws.ach, ldc, lse_c, idx, cnt);
  } else if (reg_ok && Nc <= 64 * 32) {
    select_reg_kernel<64><<<rgrid, kSelThreads, 0, s>>>(g, sa, ws.clogit, ws.ach, ldc, lse_c, idx, cnt);
  } else {
    select_kernel<<<dim3((Nc + rows - 1) / rows, g.BH), kSelThreads, smem, s>>>(
        g, sa, rows, ws.clogit, ws.ach, ldc, lse_c, idx, cnt);
  }
  return cudaGetLastError();
}

cudaError_t launch_coarse_out(const Geom& g, const float* vc, float* oc, const Workspace& ws,
                              cudaStream_t s) {
  const int Nc = g.Nc, D = g.D, ldc = ldc_of(g);
  const long long ND = static_cast<long long>(Nc) * D, NC = static_cast<long long>(Nc) * ldc;
  const long long DC = static_cast<long long>(D) * ldc;
  cudaError_t e;
  // V_c^T ([D, Nc]) rounded to tf32
  {
    const SplitSpec sp[1] = {{vc, D, ND, Nc, D, ws.vth, nullptr, ldc, DC, true}};
    if ((e = launch_split_tf32(sp, 1, g.BH, s))) return e;
  }
  // O_c = A_c V_c, plain tf32
  TgemmArgs a = gemm(g, Nc, D, Nc, 1.f);
  a.out = oc;
  a.out_ld = D;
  a.out_stride = ND;
  return launch_tgemm(a, TgemmOperand{ws.ach, nullptr, ldc, NC},
                      TgemmOperand{ws.vth, nullptr, ldc, DC}, ws.status, s);
}

cudaError_t launch_coarse_select(const Geom& g, int mode, int topk, float mass, int kmin,
                                 int kmax, const float* qc, const float* kc, const float* vc,
                                 float* oc, float* lse_c, int* idx, int* cnt, const Workspace& ws,
                                 cudaStream_t s) {
  const cudaError_t e =
      launch_coarse_logits_select(g, mode, topk, mass, kmin, kmax, qc, kc, lse_c, idx, cnt, ws, s);
  return e != cudaSuccess ? e : launch_coarse_out(g, vc, oc, ws, s);
}

// The backward's products run as plain tf32 (operands rounded to tf32, one
// product per k-step): unlike the forward's logits they decide no selection,
// and their gradients reach dq, dk, dv divided by 64.  Operands in both
// orientations where a product contracts over cubes; no lo parts.  Those of
// Q_c, K_c, V_c need only the forward's results, so they can be made while
// the combine backward computes dO_c.
cudaError_t launch_coarse_bwd_operands(const Geom& g, const float* qc, const float* kc,
                                       const float* vc, const Workspace& ws, cudaStream_t s) {
  const int Nc = g.Nc, D = g.D, ldc = ldc_of(g);
  const long long ND = static_cast<long long>(Nc) * D, DC = static_cast<long long>(D) * ldc;
  const SplitSpec sp[5] = {{qc, D, ND, Nc, D, ws.qh, nullptr, D, ND, false},
                           {kc, D, ND, Nc, D, ws.kh, nullptr, D, ND, false},
                           {vc, D, ND, Nc, D, ws.vh, nullptr, D, ND, false},
                           {qc, D, ND, Nc, D, ws.qth, nullptr, ldc, DC, true},
                           {kc, D, ND, Nc, D, ws.kth, nullptr, ldc, DC, true}};
  return launch_split_tf32(sp, 5, g.BH, s);
}

cudaError_t launch_coarse_bwd_products(const Geom& g, const float* oc, const float* lse_c,
                                       const float* doc, float* dqc, float* dkc, float* dvc,
                                       const Workspace& ws, cudaStream_t s) {
  const int Nc = g.Nc, D = g.D, ldc = ldc_of(g);
  const long long ND = static_cast<long long>(Nc) * D, NC = static_cast<long long>(Nc) * ldc;
  const long long DC = static_cast<long long>(D) * ldc;
  cudaError_t e;
  const int rows = g.BH * Nc;
  rowdot_kernel<<<(rows + 7) / 8, 256, 0, s>>>(rows, D, doc, oc, ws.cdelta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    const SplitSpec sp[2] = {{doc, D, ND, Nc, D, ws.doh, nullptr, D, ND, false},
                             {doc, D, ND, Nc, D, ws.doth, nullptr, ldc, DC, true}};
    if ((e = launch_split_tf32(sp, 2, g.BH, s))) return e;
  }
  auto hi = [](const float* h, int ld, long long stride) {
    return TgemmOperand{h, nullptr, ld, stride};
  };
  // query-major tiles: P = exp(scale Q_c K_c^T - lse) and dL = P (.) (dO_c V_c^T - delta)
  // in registers from two accumulators; dL leaves rounded to tf32, and so do
  // its transpose dL^T and P^T (through transposed shared-memory blocks)
  constexpr float kLog2e = 1.4426950408889634f;
  TgemmArgs a = gemm(g, Nc, Nc, D, g.scale * kLog2e);
  a.mode = kTgAttnBwd;
  a.beta = kLog2e;
  a.v1 = lse_c;
  a.v2 = ws.cdelta;
  a.vec_stride = Nc;
  a.out_hi = ws.ach;
  a.split_ld = ldc;
  a.split_stride = NC;
  a.vt_hi = ws.dlth;
  a.pt_hi = ws.pth;
  a.t_ld = ldc;
  a.t_stride = NC;
  if ((e = launch_tgemm_dual(a, hi(ws.qh, D, ND), hi(ws.kh, D, ND), hi(ws.doh, D, ND),
                             hi(ws.vh, D, ND), ws.status, s)))
    return e;
  // dQ_c = scale dL K_c
  a = gemm(g, Nc, D, Nc, g.scale);
  a.out = dqc;
  a.out_ld = D;
  a.out_stride = ND;
  if ((e = launch_tgemm(a, hi(ws.ach, ldc, NC), hi(ws.kth, ldc, DC), ws.status, s))) return e;
  // dK_c = scale dL^T Q_c
  a.out = dkc;
  if ((e = launch_tgemm(a, hi(ws.dlth, ldc, NC), hi(ws.qth, ldc, DC), ws.status, s))) return e;
  // dV_c = P^T dO_c
  a.alpha = 1.f;
  a.out = dvc;
  return launch_tgemm(a, hi(ws.pth, ldc, NC), hi(ws.doth, ldc, DC), ws.status, s);
}

cudaError_t launch_coarse_bwd(const Geom& g, const float* qc, const float* kc, const float* vc,
                              const float* oc, const float* lse_c, const float* doc,
                              float* dqc, float* dkc, float* dvc, const Workspace& ws,
                              cudaStream_t s) {
  const cudaError_t e = launch_coarse_bwd_operands(g, qc, kc, vc, ws, s);
  return e != cudaSuccess ? e
                          : launch_coarse_bwd_products(g, oc, lse_c, doc, dqc, dkc, dvc, ws, s);
}

}  // namespace vsa

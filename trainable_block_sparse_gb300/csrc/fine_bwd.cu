// Fine stage of VSA, backward (the method trains end to end: "VSA: Faster
// Video Diffusion with Trainable Sparse Attention", abstract; gradients of the
// masked fine attention of App. B with the selection held fixed):
//   P  = exp(S * scale - lse)           (recomputed from the saved log-sum-exp)
//   dP = dO_f V^T,  dS = P (.) (dP - delta),  delta = rowsum(dO_f (.) O_f)
//   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO_f
// over the selected 64x64 blocks only.  The pooled (coarse) gradients enter
// as dQ += repeat(dQ_c)/64 etc. in the epilogue, which also un-permutes.
//
// One tcgen05 kernel template runs two deterministic, atomic-free passes:
//  * kKeyMajor = false (dQ pass): work item = two query cubes (M = 128 query
//    rows), walking the union of their index lists.  Per step of two key
//    cubes: S = Q K^T and dP = dO V^T into TMEM, the softmax warps turn them
//    into dS (fp16, back into TMEM), then dQ += dS K.
//  * kKeyMajor = true (dK/dV pass): work item = two key cubes (M = 128 key
//    rows), walking the union of their transposed lists (query cubes that
//    selected them).  Per step of two query cubes: S^T = K Q^T and
//    dP^T = V dO^T, the softmax warps write P^T and dS^T into TMEM (the
//    per-column lse and delta come through shared memory), then
//    dV += P^T dO and dK += dS^T Q.
// TMEM: S at column 0, dP at 128, accumulators at 256 and 384 (512 columns).
// Operands are the fp16 staged copies of Q, K, V and dO_f; P and dS are fp16.
//
// Overlap with one S and one dP buffer: the softmax warps work in two phases
// per step, each with its own signal to the UMMA warp.
//   phase 1: S -> P in registers (and P^T into TMEM in the key-major pass);
//            from here the S columns are free again;
//   phase 2: dP -> dS into TMEM.
// The UMMA warp issues, per step t:  [dV(t)]  S(t+1)  dQ(t)|dK(t)  dP(t+1),
// each waiting only for the phase it reads, so the next step's S product runs
// while the softmax warps compute dS, and dP(t+1) while they compute P(t+1).
// (In-order execution of one CTA's UMMAs keeps S(t+1) from overwriting the P^T
// that dV(t) reads, and dP(t+1) from overwriting the dS that dQ/dK(t) read.)
// Warps 0-7: softmax and epilogue; warp w reads TMEM lane quarter w%4 (32
// rows) and the 64 columns of step tile w/4, so each thread owns half a row.
// Warp 8: TMA producer.  Warp 9: UMMA issue.
// Bounded waits and the abort path are as in the forward kernel.
#include "umma_pipe.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreadsBwd = 320;  // 10 warps
constexpr int kSoftmaxWarpsBwd = 8;
constexpr int kWarpLoad = 8, kWarpIssue = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColA1 = 256, kColA2 = 384;

template <int D>
struct BwdSmem {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 128;       // 128 rows x 128 bytes
  static constexpr int kXBytes = kChunks * kChunkBytes;  // one 128-row operand
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kTileBytes = 64 * D * 2;
  static constexpr int kColBytes = 4 * 64 * 4;        // lse, delta of two query cubes
  static constexpr int kBytes = 2 * kXBytes + kStages * (2 * kXBytes + kColBytes) + 1024;
};

struct BwdBars {
  uint64_t x_full, x_empty;
  uint64_t y_full[4], y_empty[4];
  uint64_t s_full, dp_full, p_done, ds_done;
  uint64_t acc_full, acc_free, final_mma;
  uint32_t tmem_base;
  int abort;
};

struct BwdParams {
  Geom g;
  const PairItem* items;
  const uint32_t* lists;
  int n_items;
  const float* lse;     // [BH, N] cube order, natural log
  const float* delta;   // [BH, N] cube order
  const float* pooled1; // dQ_c (dQ pass) or dV_c (key-major pass), may be null
  const float* pooled2; // dK_c (key-major pass), may be null
  float* out1;          // dQ (dQ pass) or dV (key-major pass), caller layout fp32
  float* out2;          // dK (key-major pass)
  uint32_t* status;
};

__device__ __forceinline__ void warp_arrive_bwd(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Writes columns [c0, c0 + D/2) of one fp32 row from a TMEM accumulator
// (times `mul`) plus pooled[cube]/64 into a caller-layout tensor.
template <int D>
__device__ __forceinline__ void store_half_row(uint32_t tacc, int c0, float mul,
                                               const float* pooled, size_t pooled_row, float* out,
                                               size_t out_row, bool have_acc) {
#pragma unroll 1
  for (int cc = c0; cc < c0 + D / 2; cc += 32) {
    uint32_t v[32];
    if (have_acc) {
      tmem_ld32(tacc + cc, v);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;
    }
    float4* dst = reinterpret_cast<float4*>(out + out_row * D + cc);
    const float4* pp =
        pooled ? reinterpret_cast<const float4*>(pooled + pooled_row * D + cc) : nullptr;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 r = make_float4(__uint_as_float(v[4 * i]) * mul, __uint_as_float(v[4 * i + 1]) * mul,
                             __uint_as_float(v[4 * i + 2]) * mul,
                             __uint_as_float(v[4 * i + 3]) * mul);
      if (pp) {
        const float4 a = pp[i];
        r.x += a.x * (1.f / kTile);
        r.y += a.y * (1.f / kTile);
        r.z += a.z * (1.f / kTile);
        r.w += a.w * (1.f / kTile);
      }
      dst[i] = r;
    }
  }
}

template <int D, bool kKeyMajor>
__global__ void __launch_bounds__(kThreadsBwd, 1)
    fine_bwd_kernel(const __grid_constant__ CUtensorMap tx1, const __grid_constant__ CUtensorMap tx2,
                    const __grid_constant__ CUtensorMap ty1, const __grid_constant__ CUtensorMap ty2,
                    BwdParams P) {
  using L = BwdSmem<D>;
  constexpr int kS = L::kStages;
  constexpr int kKSteps = D / 16;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sX1 = smem;
  uint8_t* sX2 = sX1 + L::kXBytes;
  uint8_t* sY = sX2 + L::kXBytes;  // stage s: Y1 at s*2*kXBytes, Y2 right after
  // key-major pass, per stage: lse[128] then delta[128] of the step's query cubes
  float* sCol = reinterpret_cast<float*>(sY + kS * 2 * L::kXBytes);
  __shared__ BwdBars sb;
  int* abort_flag = &sb.abort;
  const Geom& g = P.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&sb.x_full, 1);
    mbar_init(&sb.x_empty, 1);
    for (int i = 0; i < kS; ++i) {
      mbar_init(&sb.y_full[i], 1);
      mbar_init(&sb.y_empty[i], 1);
    }
    mbar_init(&sb.s_full, 1);
    mbar_init(&sb.dp_full, 1);
    mbar_init(&sb.p_done, kSoftmaxWarpsBwd);   // one arrival per softmax warp
    mbar_init(&sb.ds_done, kSoftmaxWarpsBwd);
    mbar_init(&sb.acc_full, 1);
    mbar_init(&sb.acc_free, kSoftmaxWarpsBwd);
    mbar_init(&sb.final_mma, 1);
    sb.abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpIssue) {
    tmem_alloc(&sb.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = sb.tmem_base;

  if (warp == kWarpLoad) {
    // ===================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tx1);
      tma_prefetch_desc(&tx2);
      tma_prefetch_desc(&ty1);
      tma_prefetch_desc(&ty2);
      uint32_t step = 0;
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < P.n_items && ok && !is_aborted(abort_flag);
           item += gridDim.x) {
        const PairItem pi = P.items[item];
        if (pi.count == 0) continue;
        const uint32_t* list = P.lists + pi.off;
        if (it > 0 && !wait1(&sb.x_empty, (it - 1) & 1, abort_flag, P.status)) break;
        mbar_arrive_expect_tx(&sb.x_full, 2 * L::kXBytes);
        const int ra = pi.bh * g.N + pi.a * kTile;
        const int rb = pi.bh * g.N + (pi.b >= 0 ? pi.b : pi.a) * kTile;
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          tma_load_2d(sX1 + c * L::kChunkBytes, &tx1, c * 64, ra, &sb.x_full);
          tma_load_2d(sX1 + c * L::kChunkBytes + 8192, &tx1, c * 64, rb, &sb.x_full);
          tma_load_2d(sX2 + c * L::kChunkBytes, &tx2, c * 64, ra, &sb.x_full);
          tma_load_2d(sX2 + c * L::kChunkBytes + 8192, &tx2, c * 64, rb, &sb.x_full);
        }
        ++it;
        const int nsteps = (pi.count + 1) / 2;
        for (int s = 0; s < nsteps; ++s) {
          const uint32_t slot = step % kS, ph = (step / kS) & 1;
          const bool two = 2 * s + 1 < pi.count;
          const int t0 = static_cast<int>(list[2 * s] & 0xFFFFu);
          const int t1 = two ? static_cast<int>(list[2 * s + 1] & 0xFFFFu) : t0;
          if (step >= static_cast<uint32_t>(kS) &&
              !wait1(&sb.y_empty[slot], ph ^ 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          uint8_t* y1 = sY + slot * 2 * L::kXBytes;
          uint8_t* y2 = y1 + L::kXBytes;
          const int r0 = pi.bh * g.N + t0 * kTile, r1 = pi.bh * g.N + t1 * kTile;
          mbar_arrive_expect_tx(&sb.y_full[slot], 2 * (two ? 2 : 1) * L::kTileBytes +
                                                      (kKeyMajor ? L::kColBytes : 0));
          if (kKeyMajor) {
            float* col = sCol + slot * 256;
            bulk_load(col, P.lse + r0, 256, &sb.y_full[slot]);
            bulk_load(col + 64, P.lse + r1, 256, &sb.y_full[slot]);
            bulk_load(col + 128, P.delta + r0, 256, &sb.y_full[slot]);
            bulk_load(col + 192, P.delta + r1, 256, &sb.y_full[slot]);
          }
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_2d(y1 + c * L::kChunkBytes, &ty1, c * 64, r0, &sb.y_full[slot]);
            tma_load_2d(y2 + c * L::kChunkBytes, &ty2, c * 64, r0, &sb.y_full[slot]);
            if (two) {
              tma_load_2d(y1 + c * L::kChunkBytes + 8192, &ty1, c * 64, r1, &sb.y_full[slot]);
              tma_load_2d(y2 + c * L::kChunkBytes + 8192, &ty2, c * 64, r1, &sb.y_full[slot]);
            }
          }
          ++step;
        }
      }
      const uint32_t first = step > static_cast<uint32_t>(kS) ? step - kS : 0;
      for (uint32_t t = first; t < step; ++t) mbar_wait(&sb.y_full[t % kS], (t / kS) & 1, kWaitNs);
      if (it > 0) mbar_wait(&sb.x_full, (it - 1) & 1, kWaitNs);
    }
  } else if (warp == kWarpIssue) {
    // ===================================================== UMMA issuer
    const uint32_t id_s128 = idesc_f16(128, 128, 0, 0);
    const uint32_t id_s64 = idesc_f16(128, 64, 0, 0);
    const uint32_t id_acc = idesc_f16(128, D, 0, 1);
    const uint64_t x1d0 = sdesc_sw128(smem_u32(sX1), 16, 1024);
    const uint64_t x2d0 = sdesc_sw128(smem_u32(sX2), 16, 1024);
    const uint64_t yk0 = sdesc_sw128(smem_u32(sY), 16, 1024);                 // K-major view
    const uint64_t ym0 = sdesc_sw128(smem_u32(sY), L::kChunkBytes, 1024);     // MN-major view
    uint64_t x1d[kKSteps], x2d[kKSteps];
#pragma unroll
    for (int k = 0; k < kKSteps; ++k) {
      const uint32_t o = ((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4;
      x1d[k] = x1d0 + o;
      x2d[k] = x2d0 + o;
    }
    // K-major descriptors of operand `which` (0: Y1, 1: Y2) of stage `slot`
    auto ydesc = [&](uint32_t slot, int which, uint64_t (&yd)[kKSteps]) {
      const uint32_t off = (slot * 2 * L::kXBytes + which * L::kXBytes) >> 4;
#pragma unroll
      for (int k = 0; k < kKSteps; ++k)
        yd[k] = yk0 + off + (((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4);
    };
    auto ymn = [&](uint32_t slot, int which) -> uint64_t {
      return ym0 + ((slot * 2 * L::kXBytes + which * L::kXBytes) >> 4);
    };
    uint32_t step = 0;  // global index of the current item's first step
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < P.n_items && ok && !is_aborted(abort_flag);
         item += gridDim.x) {
      const PairItem pi = P.items[item];
      if (pi.count == 0) continue;
      const int nsteps = (pi.count + 1) / 2;
      if (!waitw(&sb.x_full, it & 1, abort_flag, P.status)) break;
      // S(0) and dP(0) of this item
      {
        const uint32_t slot = step % kS;
        const uint32_t ids = pi.count > 1 ? id_s128 : id_s64;
        if (!waitw(&sb.y_full[slot], (step / kS) & 1, abort_flag, P.status)) break;
        tc_fence_after();
        uint64_t yd[kKSteps];
        ydesc(slot, 0, yd);
        issue_ss_chain<kKSteps>(tb + kColS, x1d, yd, ids);   // S   (or S^T)
        commit_elect(&sb.s_full);
        ydesc(slot, 1, yd);
        issue_ss_chain<kKSteps>(tb + kColDP, x2d, yd, ids);  // dP  (or dP^T)
        commit_elect(&sb.dp_full);
        if (nsteps == 1) commit_elect(&sb.x_empty);
      }
      for (int s = 0; s < nsteps; ++s) {
        const uint32_t t = step + s;
        const uint32_t slot = t % kS;
        const bool two = 2 * s + 1 < pi.count;
        const bool more = s + 1 < nsteps;
        const uint32_t nslot = (t + 1) % kS;
        const uint32_t nids = (2 * s + 3 < pi.count) ? id_s128 : id_s64;
        if (kKeyMajor) {
          // dV += P^T dO   (P^T in the S columns, dO = Y2 of this stage)
          if (!waitw(&sb.p_done, t & 1, abort_flag, P.status)) { ok = false; break; }
          if (s == 0 && it > 0 && !waitw(&sb.acc_free, (it - 1) & 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_ts_rows(tb + kColA1, tb + kColS, ymn(slot, 1), two, id_acc, s > 0, 64);
        }
        if (more) {
          // S(t+1): the softmax warps are done reading S(t)
          if (!kKeyMajor && !waitw(&sb.p_done, t & 1, abort_flag, P.status)) { ok = false; break; }
          if (!waitw(&sb.y_full[nslot], ((t + 1) / kS) & 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint64_t yd[kKSteps];
          ydesc(nslot, 0, yd);
          issue_ss_chain<kKSteps>(tb + kColS, x1d, yd, nids);
          commit_elect(&sb.s_full);
        }
        if (!waitw(&sb.ds_done, t & 1, abort_flag, P.status)) { ok = false; break; }
        if (!kKeyMajor && s == 0 && it > 0 &&
            !waitw(&sb.acc_free, (it - 1) & 1, abort_flag, P.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (!kKeyMajor) {
          // dQ += dS K   (dS in the dP columns, K = Y1 as an MN-major operand)
          issue_ts_rows(tb + kColA1, tb + kColDP, ymn(slot, 0), two, id_acc, s > 0, 64);
        } else {
          // dK += dS^T Q   (Q = Y1)
          issue_ts_rows(tb + kColA2, tb + kColDP, ymn(slot, 0), two, id_acc, s > 0, 64);
        }
        commit_elect(&sb.y_empty[slot]);
        if (more) {
          uint64_t yd[kKSteps];
          ydesc(nslot, 1, yd);
          issue_ss_chain<kKSteps>(tb + kColDP, x2d, yd, nids);
          commit_elect(&sb.dp_full);
          if (s + 2 == nsteps) commit_elect(&sb.x_empty);  // last read of X1/X2 issued
        }
      }
      if (!ok) break;
      commit_elect(&sb.acc_full);
      step += nsteps;
      ++it;
    }
    commit_elect(&sb.final_mma);
    mbar_wait(&sb.final_mma, 0, kWaitNs);
  } else if (warp < kSoftmaxWarpsBwd) {
    // ===================================================== softmax-backward + epilogue
    const int quarter = warp & 3;
    const int hc = warp >> 2;                 // step tile = column half of S and dP
    const int row = quarter * 32 + lane;
    const int half = row >> 6;
    const uint32_t mybit = half ? kSelB : kSelA;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr float kLog2e = 1.4426950408889634f;
    const float c = g.scale * kLog2e;
    const uint32_t ts = tb + lane_addr + kColS + 64 * hc;
    const uint32_t tdp = tb + lane_addr + kColDP + 64 * hc;
    uint32_t step = 0;
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < P.n_items && ok && !is_aborted(abort_flag);
         item += gridDim.x) {
      const PairItem pi = P.items[item];
      const int cube = half ? pi.b : pi.a;
      const bool row_live = half == 0 || pi.b >= 0;
      if (pi.count == 0) {
        // no fine contribution: only the pooled gradient reaches these rows
        if (row_live) {
          const size_t orow = static_cast<size_t>(pi.bh) * g.N + caller_row(g, cube, row & 63);
          const size_t prow = static_cast<size_t>(pi.bh) * g.Nc + cube;
          store_half_row<D>(0, hc * (D / 2), 0.f, P.pooled1, prow, P.out1, orow, false);
          if (kKeyMajor)
            store_half_row<D>(0, hc * (D / 2), 0.f, P.pooled2, prow, P.out2, orow, false);
        }
        continue;
      }
      const uint32_t* list = P.lists + pi.off;
      float row_lse = 0.f, row_delta = 0.f;
      if (!kKeyMajor && row_live) {
        const size_t frow = static_cast<size_t>(pi.bh) * g.N + cube * kTile + (row & 63);
        row_lse = P.lse[frow] * kLog2e;
        row_delta = P.delta[frow];
      }
      const int nsteps = (pi.count + 1) / 2;
      for (int s = 0; s < nsteps; ++s, ++step) {
        const bool two = 2 * s + 1 < pi.count;
        const bool have = hc == 0 || two;   // this step has a tile for this column half
        const bool valid = have && (list[2 * s + hc] & mybit) != 0;
        const uint32_t slot = step % kS;
        if (!waitw(&sb.s_full, step & 1, abort_flag, P.status)) { ok = false; break; }
        // the column data arrived with the stage's tiles (already complete: the
        // MMAs that produced S waited for it); waiting makes it visible here
        if (kKeyMajor && !waitw(&sb.y_full[slot], (step / kS) & 1, abort_flag, P.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* col_lse = sCol + slot * 256 + 64 * hc;
        const float* col_delta = col_lse + 128;
        // ---- phase 1: P from S
        float p[64];
        if (valid) {
          uint32_t sv[64];
          tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
          tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float lse2 = kKeyMajor ? col_lse[j] * kLog2e : row_lse;
            p[j] = ex2_approx(fmaf(__uint_as_float(sv[j]), c, -lse2));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) p[j] = 0.f;
        }
        if (kKeyMajor && have) {
          // P^T of this tile: 64 values pack into 32 columns at the tile's start
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_f16x2(p[2 * i], p[2 * i + 1]);
          tmem_st32(ts, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        warp_arrive_bwd(&sb.p_done);
        // ---- phase 2: dS = P (.) (dP - delta)
        if (!waitw(&sb.dp_full, step & 1, abort_flag, P.status)) { ok = false; break; }
        tc_fence_after();
        if (have) {
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t dk[16];
            if (valid) {
              uint32_t dv[32];
              tmem_ld32(tdp + 32 * ch, dv);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float d[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int j = 32 * ch + 2 * i + u;
                  const float dl = kKeyMajor ? col_delta[j] : row_delta;
                  d[u] = p[j] * (__uint_as_float(dv[2 * i + u]) - dl);
                }
                dk[i] = pack_f16x2(d[0], d[1]);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) dk[i] = 0u;
            }
            // chunk ch (32 values) packs into 16 columns at 16*ch: already-read columns
            tmem_st16(tdp + 16 * ch, dk);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        warp_arrive_bwd(&sb.ds_done);
      }
      if (!ok) break;
      // ---------------------------------------------- epilogue
      if (!waitw(&sb.acc_full, it & 1, abort_flag, P.status)) break;
      tc_fence_after();
      if (row_live) {
        const size_t orow = static_cast<size_t>(pi.bh) * g.N + caller_row(g, cube, row & 63);
        const size_t prow = static_cast<size_t>(pi.bh) * g.Nc + cube;
        const uint32_t ta = tb + lane_addr;
        if (!kKeyMajor) {
          store_half_row<D>(ta + kColA1, hc * (D / 2), g.scale, P.pooled1, prow, P.out1, orow, true);
        } else {
          store_half_row<D>(ta + kColA1, hc * (D / 2), 1.f, P.pooled1, prow, P.out1, orow, true);
          store_half_row<D>(ta + kColA2, hc * (D / 2), g.scale, P.pooled2, prow, P.out2, orow, true);
        }
      }
      tc_fence_before();
      warp_arrive_bwd(&sb.acc_free);
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpIssue) tmem_dealloc(tb, kTmemCols);
}

template <int D, bool kKeyMajor>
cudaError_t run_bwd(const Geom& g, const void* x1, const void* x2, const void* y1, const void* y2,
                    BwdParams p, cudaStream_t s) {
  alignas(64) CUtensorMap m1, m2, m3, m4;
  const uint64_t rows = static_cast<uint64_t>(g.BH) * g.N;
  if (!encode_tiled_2d(&m1, x1, rows, D, 64, 64) || !encode_tiled_2d(&m2, x2, rows, D, 64, 64) ||
      !encode_tiled_2d(&m3, y1, rows, D, 64, 64) || !encode_tiled_2d(&m4, y2, rows, D, 64, 64))
    return cudaErrorInvalidValue;
  const int smem = BwdSmem<D>::kBytes;
  auto kern = fine_bwd_kernel<D, kKeyMajor>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = p.n_items < sms ? p.n_items : sms;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreadsBwd, smem, s>>>(m1, m2, m3, m4, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_impl(const Geom& g, const __half* q, const __half* k, const __half* v,
                     const float* lse_f, const __half* dof,
                     const float* delta, const float* dqc, const float* dkc, const float* dvc,
                     float* dq, float* dk, float* dv, const Workspace& ws, cudaStream_t s) {
  BwdParams pq{g, ws.qpairs, ws.qlist, ws.n_qpairs, lse_f, delta, dqc, nullptr, dq, nullptr,
               ws.status};
  cudaError_t e = run_bwd<D, false>(g, q, dof, k, v, pq, s);
  if (e != cudaSuccess) return e;
  BwdParams pk{g, ws.kpairs, ws.klist, ws.n_kpairs, lse_f, delta, dvc, dkc, dv, dk, ws.status};
  return run_bwd<D, true>(g, k, v, q, dof, pk, s);
}

}  // namespace

cudaError_t launch_fine_bwd(const Geom& g, const __half* q, const __half* k, const __half* v,
                            const float* lse_f, const __half* dof, const float* delta,
                            const float* dqc, const float* dkc, const float* dvc, float* dq,
                            float* dk, float* dv, const Workspace& ws, cudaStream_t s) {
  if (g.D == 64) return bwd_impl<64>(g, q, k, v, lse_f, dof, delta, dqc, dkc, dvc, dq, dk, dv, ws, s);
  return bwd_impl<128>(g, q, k, v, lse_f, dof, delta, dqc, dkc, dvc, dq, dk, dv, ws, s);
}

}  // namespace vsa
